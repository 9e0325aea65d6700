"""clo_hybrid_decode_attn on the GPU vs the fp64 oracle.

Small cases run the whole oracle (several tiles per head, ragged tails,
GQA 1/4/5/8, no / some / all persistent heads, token-addressed and compact
Cache Buffers, several CTA counts).  The full-size workloads run the kernel in
the configuration the benchmark uses and check every (batch, KV head) group
against the oracle's dense attention over the group's rows.
"""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
import workloads as wl
from gpu_util import LSE_ATOL, assert_close, dev, parallel_map, rel_l2, scale_for

pytestmark = pytest.mark.gpu


def run_gpu(q, cbK, cbV, idx, pK, pV, pid, num_ctas=0, want_lse=True):
    """All inputs are device tensors; returns (out fp16 host, lse host, err flag)."""
    B, Hq, d = q.shape
    Hkv = cbK.shape[1] if cbK is not None else pid.numel()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=q.device) if want_lse else None
    ws = torch.empty(clo.clo_hybrid_workspace_size(B, Hq, Hkv, d, num_ctas), dtype=torch.uint8,
                     device=q.device)
    err = torch.zeros(1, dtype=torch.int32, device=q.device)
    clo.clo_hybrid_decode_attn(q, cbK, cbV, idx, pK, pV, pid, out, ws, lse=lse, err_flag=err,
                               num_ctas=num_ctas)
    torch.cuda.synchronize()
    return (out.cpu().numpy().astype(np.float64),
            None if lse is None else lse.cpu().numpy().astype(np.float64), int(err.item()))


def small_case(seed, B, Hq, Hkv, T, k, Np, C=None, dup=False):
    rng = np.random.Generator(np.random.PCG64(seed))
    C = T if C is None else C
    f16 = lambda *s: rng.standard_normal(s).astype(np.float16)
    q = f16(B, Hq, 128)
    cbK, cbV = f16(B, Hkv, C, 128), f16(B, Hkv, C, 128)
    if dup:
        idx = rng.integers(0, C, size=(B, Hkv, k)).astype(np.int32)
    else:
        idx = np.stack([np.stack([rng.permutation(C)[:k] for _ in range(Hkv)])
                        for _ in range(B)]).astype(np.int32)
    pK, pV = f16(B, Np, max(T, 1), 128), f16(B, Np, max(T, 1), 128)
    pid = rng.permutation(Hkv)[:Np].astype(np.int32)
    return q, cbK, cbV, idx, pK, pV, pid


def to_dev(*arrs):
    return [None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev()) for a in arrs]


def check_small(case, num_ctas=0, what=""):
    q, cbK, cbV, idx, pK, pV, pid = case
    ref, ref_lse = oracle.get().hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale_for())
    got, lse, err = run_gpu(*to_dev(q, cbK, cbV, idx, pK, pV, pid), num_ctas=num_ctas)
    assert err == 0
    assert_close(got, ref, what)
    assert np.max(np.abs(lse - ref_lse)) < LSE_ATOL
    return got


SMALL = [
    # name, seed, B, Hq, Hkv, T, k, Np, C
    ("tiny_shape", 1, 1, 32, 8, 1024, 102, 2, None),
    ("ragged_b3", 2, 3, 32, 8, 1000, 37, 1, None),
    ("gqa5", 3, 2, 40, 8, 517, 49, 1, None),
    ("mha", 4, 2, 8, 8, 300, 33, 3, None),
    ("gqa8", 5, 2, 64, 8, 200, 20, 2, None),
    ("no_persistent", 6, 2, 32, 8, 500, 16, 0, None),
    ("all_persistent", 7, 2, 32, 8, 33, 3, 8, None),
    ("k1_t1", 8, 2, 32, 8, 1, 1, 2, None),
    ("compact", 9, 2, 32, 8, 2000, 200, 2, 200),
    ("one_kv_head", 10, 3, 4, 1, 77, 9, 0, None),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("num_ctas", [0, 1, 3])
def test_small_vs_oracle(case, num_ctas):
    name, seed, B, Hq, Hkv, T, k, Np, C = case
    check_small(small_case(seed, B, Hq, Hkv, T, k, Np, C), num_ctas, name)


def test_duplicate_indices_allowed():
    check_small(small_case(11, 2, 32, 8, 400, 60, 2, dup=True), 0, "dup")


def test_split_count_independence():
    """The same problem cut into 1, 2, 5, 13 or all-SM CTA ranges agrees to
    well under the oracle tolerance (fixed split points, fixed merge order)."""
    case = to_dev(*small_case(12, 2, 32, 8, 3000, 300, 2))
    outs = [run_gpu(*case, num_ctas=c)[0] for c in (1, 2, 5, 13, 0)]
    for o in outs[1:]:
        assert rel_l2(o, outs[0]) < 1e-3
    again = run_gpu(*case, num_ctas=0)[0]
    assert np.array_equal(again, outs[-1]), "same launch must be bit-reproducible"


@pytest.mark.parametrize("num_ctas", [7, 37, 100])
def test_ranges_cross_segments_in_both_parts(num_ctas):
    """Segment boundaries crossed in both parts (8 batch rows; 2 persistent heads
    of 128 tiles and 6 Cache Buffer heads of 21 tiles each), so some CTAs flush
    three to five segments: every partial lands in the slot the merge reads."""
    check_small(small_case(13, 8, 32, 8, 2048, 330, 2), num_ctas, "weighted cut")


def test_index_order_does_not_matter():
    """The Cache Buffer indices of each head in random, ascending and reversed
    order name the same token set: the outputs agree within the bound of the
    split-count test.  Only the order of the tiles differs, and with it the
    running maximum at each tile, which sets how each softmax weight rounds
    to fp16 for the P.V product (2^-11 relative a weight)."""
    q, cbK, cbV, idx, pK, pV, pid = small_case(14, 3, 32, 8, 2500, 700, 2)
    outs = []
    for order in (idx, np.sort(idx, axis=-1), np.sort(idx, axis=-1)[..., ::-1]):
        outs.append(run_gpu(*to_dev(q, cbK, cbV, np.ascontiguousarray(order), pK, pV, pid))[0])
    for o in outs[1:]:
        assert rel_l2(o, outs[0]) < 1e-3
        assert np.max(np.abs(o - outs[0])) < 2e-3


def test_tiny_config_from_generator():
    cfg = wl.CONFIGS["tiny"]
    q, _ = wl.queries_and_labels(cfg, 0, "cpu")
    cbK, cbV, idx = wl.cache_buffer(cfg, 0, "cpu")
    pK, pV = wl.persistent_cache(cfg, 0, "cpu")
    pid = wl.persist_ids(cfg, 0)
    check_small((q.numpy(), cbK.numpy(), cbV.numpy(), idx.numpy(), pK.numpy(), pV.numpy(), pid))


def test_bad_index_zeroes_group_and_flags():
    q, cbK, cbV, idx, pK, pV, pid = small_case(13, 2, 32, 8, 300, 40, 2)
    g_bad = [g for g in range(8) if g not in pid.tolist()][0]
    ref, _ = oracle.get().hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale_for())
    idx_bad = idx.copy()
    idx_bad[1, g_bad, 7] = 300          # == C: out of range
    idx_bad[1, g_bad, 9] = -5
    got, lse, err = run_gpu(*to_dev(q, cbK, cbV, idx_bad, pK, pV, pid))
    assert err & clo.FLAG_BAD_INDEX
    assert clo.check_error_flag(err) == clo.CLO_ERR_BAD_INDEX
    sl = slice(4 * g_bad, 4 * g_bad + 4)
    assert np.all(got[1, sl] == 0) and np.all(np.isneginf(lse[1, sl]))
    mask = np.ones(got.shape[:2], dtype=bool)
    mask[1, sl] = False
    assert_close(got[mask], ref[mask], "other groups")


def test_bad_persist_ids_zero_everything():
    q, cbK, cbV, idx, pK, pV, _ = small_case(14, 2, 32, 8, 100, 10, 2)
    for bad in ([3, 3], [1, 8], [-1, 2]):
        got, lse, err = run_gpu(*to_dev(q, cbK, cbV, idx, pK, pV, np.array(bad, dtype=np.int32)))
        assert err & clo.FLAG_BAD_PERSIST
        assert np.all(got == 0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------- full size, every group

def full_size_check(name, layers=(0,), groups=None):
    """The workload at full size, in the launch configuration the benchmark
    uses; every (batch row, KV head) group (or the `groups` subset) of each
    layer compared with the oracle's dense attention over the group's rows,
    gathered on the GPU and copied to the host.  Returns the groups checked."""
    cfg = wl.CONFIGS[name]
    scale = scale_for()
    orc = oracle.get()
    checked = 0
    for layer in layers:
        q, _ = wl.queries_and_labels(cfg, layer, dev())
        cbK, cbV, idx = wl.cache_buffer(cfg, layer, dev())
        pK, pV = wl.persistent_cache(cfg, layer, dev())
        pid_np = wl.persist_ids(cfg, layer)
        pid = torch.from_numpy(pid_np).to(dev())
        got, lse, err = run_gpu(q, cbK, cbV, idx, pK, pV, pid)
        assert err == 0
        qh = q.cpu().numpy()
        G = cfg.G
        todo = groups(cfg, pid_np) if groups is not None else \
            [(b, g) for b in range(cfg.B) for g in range(cfg.Hkv)]
        rows = {}
        for (b, g) in todo:
            if g in pid_np.tolist():
                j = pid_np.tolist().index(g)
                rows[(b, g)] = (pK[b, j].cpu().numpy(), pV[b, j].cpu().numpy())
            else:
                sel = idx[b, g].long()
                rows[(b, g)] = (cbK[b, g][sel].cpu().numpy(), cbV[b, g][sel].cpu().numpy())
        refs = parallel_map(
            lambda bg: orc.attention_dense(qh[bg[0], bg[1] * G:(bg[1] + 1) * G], *rows[bg], scale),
            todo)
        for (b, g), (ref, ref_lse) in zip(todo, refs):
            assert_close(got[b, g * G:(g + 1) * G], ref, f"{name} layer {layer} b{b} g{g}")
            assert np.max(np.abs(lse[b, g * G:(g + 1) * G] - ref_lse)) < LSE_ATOL
        checked += len(todo)
        del q, cbK, cbV, idx, pK, pV, rows
        torch.cuda.empty_cache()
    print(f"{name}: {checked} groups checked against the oracle over layers {list(layers)}")
    return checked


@pytest.mark.parametrize("name,layers", [("llama3_8b_layer_b8_32k", (0, 1)),
                                         ("llama3_8b_step_b1_128k", (0, 1)),
                                         ("llama3_8b_step_b4_128k", (0,)),
                                         ("qwen25_14b_step_b16_64k", (0,))])
def test_full_size_every_group(name, layers):
    cfg = wl.CONFIGS[name]
    assert full_size_check(name, layers) == len(layers) * cfg.B * cfg.Hkv
