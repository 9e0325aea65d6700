"""bench.py end to end on small cases of every workload kind: the JSON line
carries the contract's keys and sane values."""
import contextlib
import dataclasses
import io
import json

import pytest

import bench

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("args", [
    ["--workload", "tiny"],
    ["--workload", "tiny", "--lookup-schedule", "stream"],
    ["--workload", "tiny", "--lookup-schedule", "serial"],
    ["--workload", "tiny", "--lookup-schedule", "pipelined"],
    ["--workload", "paged_llama2_7b_b256", "--batch", "8"],
    ["--workload", "fill_hbm_llama3_8b_b8_32k", "--batch", "1"],
    ["--workload", "fill_c2c_llama3_8b_b8_32k", "--batch", "1"],
    ["--workload", "topk_llama3_8b_b8_32k", "--batch", "1"],
    ["--workload", "qwen25_14b_step_b16_64k", "--batch", "1"],
    ["--workload", "llama3_8b_layer_b8_32k_miss", "--batch", "2"],
    ["--workload", "llama3_8b_layer_b8_32k_miss", "--batch", "2", "--lookup-schedule", "serial"],
    ["--workload", "llama3_8b_layer_b8_32k_miss_fill", "--batch", "1"],
    ["--workload", "llama3_8b_layer_b8_32k_miss_fill", "--batch", "1", "--lookup-schedule",
     "overlap"],
    ["--workload", "llama3_8b_layer_b8_32k_miss_fill", "--batch", "1", "--lookup-schedule",
     "stream"],
    ["--workload", "llama3_8b_layer_b8_32k_miss_fill", "--batch", "1", "--lookup-schedule",
     "pipelined"],
], ids=lambda a: "_".join(x.lstrip("-") for x in a[1::2] if x not in ("--batch",)))
def test_bench_line(args):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(args + ["--steps", "3", "--warmup", "3", "--max-rounds", "1",
                           "--no-cpu-baseline"])
    d = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "roofline", "e2e",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["gpu_launches"] > 0
    r = d["roofline"]
    assert r["bound"] in ("hbm", "c2c") and r["achieved"] > 0 and r["peak"] > 0
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0
    if "lookup" in d:
        assert d["lookup"]["looked_up_heads"] > 0 and d["tokens_per_s"] > 0
    if "_miss" in d["config"]["workload"]:
        # the misses recur every step (labels restored) and their bytes are counted
        assert d["config"]["misses_per_step"] > 0 and d["config"]["miss_bytes_per_step"] > 0
        assert 0.0 < d["lookup"]["hit_rate"] < 1.0


def test_overlapped_fill_schedule_orders_the_fill_before_its_attention():
    """The miss-path fill on the second stream (the next layer's fill beside
    the current layer's attention, "overlap"; or lookup and fill there,
    "stream"), or carried beside the attention in one layer call
    ("pipelined"), must leave every layer's attention output bit-identical to
    the serial schedule's with the same CTA counts: an attention that ran
    before its fill would read the old rows (the full KV copy holds other
    values than the Cache Buffer)."""
    import torch
    import workloads as wl

    cfg = dataclasses.replace(wl.CONFIGS["llama3_8b_layer_b8_32k_miss_fill"], B=1)
    dev = torch.device("cuda:0")
    outs = {}
    for sched in ("serial", "overlap", "stream", "pipelined"):
        W = bench.HybridWorkload(cfg, dev, 0, replicas=3, schedule=sched, side_ctas=32)
        assert W.misses_per_step > 0
        for i in range(2 * W.n_inst):  # every buffer set filled at least once
            W.launch(i)
        torch.cuda.synchronize()
        for it in W.inst:
            it["out"].fill_(float("nan"))
        for i in range(2 * W.n_inst, 3 * W.n_inst):
            W.launch(i)
        torch.cuda.synchronize()
        assert int(W.err.item()) == 0
        outs[sched] = [it["out"].clone() for it in W.inst]
        del W
        torch.cuda.empty_cache()
    for sched in ("overlap", "stream", "pipelined"):
        for a, b in zip(outs["serial"], outs[sched]):
            assert not torch.isnan(a).any()
            assert torch.equal(a, b), sched


def test_overlapped_fill_schedule_across_layers():
    """The same check on a three-layer step with a ring of five buffer sets
    and the fill from a full KV copy in HBM: the attention of layer l+1 must
    wait for the fill issued beside layer l, for every l, and for the next
    step's layer 0 (with "pipelined" the lookups run two layers ahead, so the
    step's last two calls look up the next step's first two layers)."""
    import torch
    import workloads as wl

    cfg = wl.small_hybrid("three_layers_miss_fill", B=3, L=3, Hq=32, Hkv=8, T=2048, Np=2,
                          qmode="cos", c_lo=0.725, c_hi=0.925, smode="one", label_reset=True,
                          miss_fill="device", ring=5, seed=4242)
    dev = torch.device("cuda:0")
    outs = {}
    for sched in ("serial", "overlap", "pipelined"):
        W = bench.HybridWorkload(cfg, dev, 0, schedule=sched, side_ctas=24)
        assert W.n_inst == 5 and W.misses_per_step > 0
        for i in range(4 * W.n_inst):
            W.launch(i)
        torch.cuda.synchronize()
        for it in W.inst:
            it["out"].fill_(float("nan"))
        for i in range(4 * W.n_inst, 6 * W.n_inst):
            W.launch(i)
        torch.cuda.synchronize()
        assert int(W.err.item()) == 0
        outs[sched] = [it["out"].clone() for it in W.inst]
        del W
        torch.cuda.empty_cache()
    for sched in ("overlap", "pipelined"):
        for a, b in zip(outs["serial"], outs[sched]):
            assert not torch.isnan(a).any()
            assert torch.equal(a, b), sched
