"""clo_lookup_update on the GPU vs the fp64 oracle: flags, label updates and
the miss list bit-exact (except groups whose similarity is within 1e-4 of tau,
which are counted), similarities within fp32 rounding."""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
import workloads as wl
from gpu_util import NEAR_TAU, assert_lookup_matches, dev

pytestmark = pytest.mark.gpu


def run_gpu(q, lab, w, tau32, pm):
    B, Hq, _ = q.shape
    Hkv = tau32.size
    d = dev()
    qd, labd = torch.from_numpy(q).to(d), torch.from_numpy(lab).to(d)
    flag = torch.full((B * Hkv,), 255, dtype=torch.uint8, device=d)
    sim = torch.empty(B * Hkv, dtype=torch.float32, device=d)
    ml = torch.full((max(B * Hkv, 1),), -7, dtype=torch.int32, device=d)
    mc = torch.full((1,), -7, dtype=torch.int32, device=d)
    clo.clo_lookup_update(qd, labd, torch.from_numpy(w).to(d), torch.from_numpy(tau32).to(d),
                          None if pm is None else torch.from_numpy(pm).to(d), flag, sim, ml, mc)
    torch.cuda.synchronize()
    n = int(mc.item())
    return dict(flag=flag.cpu().numpy().reshape(B, Hkv), sim=sim.cpu().numpy().reshape(B, Hkv),
                labels=labd.cpu().numpy(), miss_list=ml.cpu().numpy()[:n], miss_count=n)


def compare(q, lab, w, tau32, pm):
    """Runs both sides; returns the number of near-tau groups."""
    ref = oracle.get().lookup_update(q, lab, w.astype(np.float64), tau32.astype(np.float64), pm)
    got = run_gpu(q, lab, w, tau32, pm)
    return assert_lookup_matches(ref, got, tau32, pm, q.shape[1] // tau32.size)


def cfg_inputs(cfg, layer=0):
    """The workload's lookup inputs; tau is the library's (clo_thresholds_host),
    which both sides then take, and it must match the oracle's Eqs. 7-9."""
    q, lab = wl.queries_and_labels(cfg, layer, "cpu")
    s = wl.importance(cfg, layer)
    tau = clo.clo_thresholds_host(s, cfg.Hkv, cfg.G, wl.ETA, wl.N_EXP)
    ref = oracle.get().thresholds(s.astype(np.float64), cfg.Hkv, cfg.G, wl.ETA, wl.N_EXP)
    assert np.max(np.abs(tau.astype(np.float64) - ref)) < 1e-6
    return q.numpy(), lab.numpy(), s, tau, wl.persist_mask(cfg, layer)


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_layer_b8_32k", "llama3_8b_layer_b8_32k_miss",
                                  "llama3_8b_step_b4_128k",
                                  "qwen25_14b_step_b16_64k"])
def test_lookup_configs(name):
    cfg = wl.CONFIGS[name]
    for layer in range(min(cfg.L, 4)):
        near = compare(*cfg_inputs(cfg, layer))
        print(f"{name} layer {layer}: {near} near-tau groups")


def test_lookup_many_groups_half_miss():
    """512 groups spread over the 8-CTA cluster, tau set so about half miss:
    exercises the cross-CTA ordered miss list."""
    rng = np.random.Generator(np.random.PCG64(5))
    B, Hq, Hkv = 64, 32, 8
    lab = rng.standard_normal((B, Hq, 128)).astype(np.float16)
    q = (0.5 * lab + rng.standard_normal((B, Hq, 128))).astype(np.float16)
    w = rng.uniform(0, 1, Hq).astype(np.float32)
    tau = np.full(Hkv, 0.447, dtype=np.float32)
    pm = np.zeros(Hkv, dtype=np.uint8)
    pm[3] = 1
    compare(q, lab, w, tau, pm)


@pytest.mark.parametrize("B", [4, 5, 16, 17])
def test_lookup_cta_width_boundary(B):
    """32 groups run on 4-warp CTAs, 40 and more on 16-warp CTAs (one group a
    warp per pass); both sides of the switch, with about half of them missing."""
    rng = np.random.Generator(np.random.PCG64(50 + B))
    Hq, Hkv = 32, 8
    lab = rng.standard_normal((B, Hq, 128)).astype(np.float16)
    q = (0.5 * lab + rng.standard_normal((B, Hq, 128))).astype(np.float16)
    w = rng.uniform(0, 1, Hq).astype(np.float32)
    tau = np.full(Hkv, 0.447, dtype=np.float32)
    pm = np.zeros(Hkv, dtype=np.uint8)
    pm[5] = 1
    compare(q, lab, w, tau, pm)


def test_lookup_mha_and_gqa8():
    rng = np.random.Generator(np.random.PCG64(6))
    for (B, Hq, Hkv) in [(5, 32, 32), (3, 64, 8), (257, 8, 8)]:
        lab = rng.standard_normal((B, Hq, 128)).astype(np.float16)
        q = (0.8 * lab + 0.6 * rng.standard_normal((B, Hq, 128))).astype(np.float16)
        w = rng.uniform(0, 1, Hq).astype(np.float32)
        tau = rng.uniform(0.6, 0.9, Hkv).astype(np.float32)
        compare(q, lab, w, tau, None)


def test_lookup_degenerate_cases():
    """Zero query (cosine 0), all-zero weights (plain mean), an exact tie
    sim == tau (a hit), and a second call that sees the replaced labels."""
    B, Hq, Hkv = 2, 8, 2
    v = np.zeros((B, Hq, 128), dtype=np.float16)
    v[:, :, :64] = 0.5  # norm exactly 4: cosine of v with itself is exactly 1
    q = v.copy()
    q[1, 4:8] = -v[1, 4:8]          # (1, 1): cosine -1 -> miss
    q[0, 5] = 0                      # (0, 1): one zero query -> cosine 0 in the mean
    w = np.zeros(Hq, dtype=np.float32)
    tau = np.array([1.0, 0.5], dtype=np.float32)
    compare(q, v, w, tau, None)
    got = run_gpu(q, v, w, tau, None)
    assert got["flag"][0, 0] == 0            # tie: sim == tau == 1 is a hit
    assert got["flag"][0, 1] == 0 and abs(got["sim"][0, 1] - 0.75) < 1e-6
    assert got["flag"][1, 1] == 1 and got["miss_list"].tolist() == [3]
    # Next step with the same queries: the replaced labels now match exactly.
    again = run_gpu(q, got["labels"], w, tau, None)
    assert again["flag"][1, 1] == 0 and again["miss_count"] == 0


def test_lookup_empty_batch():
    d = dev()
    mc = torch.full((1,), 99, dtype=torch.int32, device=d)
    z = torch.empty((0, 32, 128), dtype=torch.float16, device=d)
    clo.clo_lookup_update(z, z.clone(), torch.ones(32, device=d), torch.zeros(8, device=d), None,
                          torch.empty(0, dtype=torch.uint8, device=d),
                          torch.empty(0, device=d), torch.empty(0, dtype=torch.int32, device=d),
                          mc)
    torch.cuda.synchronize()
    assert mc.item() == 0


def test_lookup_maximum_groups():
    """The largest lookup a call takes: 8192 batch rows x 8 KV heads = 65536
    groups (one past it is refused on the host), about a third of them
    missing, so each of the cluster's 8 CTAs writes thousands of misses at
    offsets read from the others."""
    rng = np.random.Generator(np.random.PCG64(65536))
    B, Hq, Hkv = 8192, 32, 8
    lab = rng.standard_normal((B, Hq, 128)).astype(np.float16)
    q = (0.8 * lab.astype(np.float32) + 0.6 * rng.standard_normal((B, Hq, 128))).astype(np.float16)
    w = rng.uniform(0, 1, Hq).astype(np.float32)
    tau = np.array([0.79, 0.8, -1.0, 0.81, 0.8, 0.79, 0.5, 0.8], dtype=np.float32)
    pm = np.zeros(Hkv, dtype=np.uint8)
    pm[2] = 1
    ref = oracle.get().lookup_update(q, lab, w.astype(np.float64), tau.astype(np.float64), pm)
    assert B * Hkv // 5 < ref["miss_count"] < B * Hkv // 2
    near = compare(q, lab, w, tau, pm)
    print(f"65536 groups: {ref['miss_count']} misses, {near} near tau")
