"""bench.py's host-side bookkeeping (CPU only): the launch count it claims for
each schedule, and the workload shape both arms report."""
import types

import pytest

import bench
import workloads as wl


def _count(name, schedule, attn_kernels=2):
    cfg = wl.CONFIGS[name]
    w = types.SimpleNamespace(cfg=cfg, L=cfg.L, schedule=schedule, attn_kernels=attn_kernels,
                              restore=object() if cfg.label_reset else None)
    return bench.HybridWorkload.launches_per_step(w)


@pytest.mark.parametrize("name,schedule,want", [
    # thresholds + per layer: main kernel, a lookup launch of its own (128 groups), merge
    ("qwen25_14b_step_b16_64k", "fused", 1 + 48 * 3),
    # 8 and 64 groups: the lookup rides in the merge launch
    ("llama3_8b_step_b1_128k", "fused", 1 + 32 * 2),
    ("llama3_8b_layer_b8_32k", "fused", 1 + 2),
    ("llama3_8b_layer_b8_32k", "serial", 1 + 3),  # lookup, main kernel, merge
    # + the label restore copy and one fill a layer
    ("llama3_8b_layer_b8_32k_miss_fill", "pipelined", 1 + 2 + 1 + 1),
    ("llama3_8b_layer_b8_32k_miss_fill", "overlap", 1 + 3 + 1 + 1),
])
def test_launches_per_step(name, schedule, want):
    assert _count(name, schedule) == want


def test_one_cta_attention_has_no_merge_launch():
    # a single main-kernel CTA leaves nothing to merge: a large lookup then
    # follows the main kernel alone, a small one still rides in a merge launch
    assert _count("qwen25_14b_step_b16_64k", "fused", attn_kernels=1) == 1 + 48 * 2
    assert _count("llama3_8b_step_b1_128k", "fused", attn_kernels=1) == 1 + 32 * 2


def test_shape_config_names_every_workload():
    names = list(wl.CONFIGS) + list(wl.PAGED_CONFIGS) + list(wl.FILL_CONFIGS) + \
        list(wl.TOPK_CONFIGS)
    for n in names:
        c = bench.shape_config(n)
        assert c["workload"] == n and c["batch"] > 0 and c["head_dim"] == 128
