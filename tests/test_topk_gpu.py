"""clo_topk_retrieve on the GPU vs the fp64 oracle.  The selection is an
integer decision taken on fp32 scores on the GPU and fp64 scores in the
oracle, so the two sets must agree except for keys whose fp64 score lies
within the fp32 error bound of the k-th largest; those are checked for
validity instead (right count, ascending, distinct, all on the right side of
the cut within the bound)."""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _gen(seed, B, Hq, Hkv, T, d=128):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, d), generator=g).to(torch.float16)
    K = torch.randn((B, Hkv, T, d), generator=g).to(torch.float16)
    return q, K


def run_gpu(q, K, k):
    d = dev()
    B, Hkv, T = K.shape[0], K.shape[1], K.shape[2]
    idx = torch.full((B, Hkv, k), -1, dtype=torch.int32, device=d)
    ws = torch.empty(max(clo.clo_topk_workspace_size(B, Hkv, T), 16), dtype=torch.uint8, device=d)
    clo.clo_topk_retrieve(q.to(d), K.to(d), k, idx, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy()


def check_head(got, ref, qs64, K64, k):
    """got/ref: index lists of one head; qs64: the group's summed query (fp64)."""
    assert len(got) == k and list(got) == sorted(set(got)), "not k distinct ascending tokens"
    if set(got) == set(ref):
        return 0
    sc = K64 @ qs64
    mag = np.abs(K64) @ np.abs(qs64)
    tol = 4e-6 * mag + 1e-6        # fp32 dot of 128 terms + the fp32 query sum
    cut = np.sort(sc)[::-1][k - 1]
    for t in set(got) ^ set(ref):
        assert abs(sc[t] - cut) <= tol[t], f"token {t} differs outside the fp32 band"
    return len(set(got) ^ set(ref))


def compare(q, K, k):
    got = run_gpu(q, K, k)
    ref = oracle.get().topk_retrieve(q.numpy(), K.numpy(), k)
    B, Hq = q.shape[:2]
    Hkv = K.shape[1]
    G = Hq // Hkv
    q64, K64 = q.numpy().astype(np.float64), K.numpy().astype(np.float64)
    swaps = 0
    for b in range(B):
        for g in range(Hkv):
            swaps += check_head(got[b, g], ref[b, g], q64[b, g * G:(g + 1) * G].sum(0), K64[b, g], k)
    return swaps


@pytest.mark.parametrize("B,Hq,Hkv,T,k", [
    (2, 32, 8, 1000, 100),    # GQA 4, ragged T
    (3, 40, 8, 777, 77),      # GQA 5
    (1, 8, 8, 5000, 500),     # MHA
    (2, 16, 4, 300, 1),       # argmax
    (1, 16, 4, 130, 130),     # everything
    (2, 32, 8, 90, 9),        # less than one CTA step of keys
    (1, 8, 2, 60000, 6000),   # more keys than the select kernel keeps in shared memory
    (1, 4, 1, 8193, 820),     # one key past a one-CTA slice: a cluster of 2
    (2, 8, 1, 100000, 1000),  # a cluster of 8, slices of 12500 keys
    (1, 4, 1, 300000, 30000), # a cluster of 8 near the largest slice (37500 keys)
    (1, 4, 1, 385024, 38502), # the largest context a call takes: 8 slices of 48128 keys
])
def test_topk_vs_oracle(B, Hq, Hkv, T, k):
    q, K = _gen(B * 1000 + T, B, Hq, Hkv, T)
    assert compare(q, K, k) <= B * Hkv  # at most a boundary swap per head, each checked


def test_topk_ties_take_lower_tokens():
    q, K = _gen(5, 1, 8, 2, 400)
    K[0, 1, 100:300] = K[0, 1, 50]          # 200 identical keys in head 1
    K[0, 1, 50] = K[0, 1, 50]
    q[0, 4:8] = K[0, 1, 50].to(torch.float32).mul(0.5).to(torch.float16)   # and make them the best
    got = run_gpu(q, K, 40)
    tied = [50] + list(range(100, 300))
    assert got[0, 1].tolist() == tied[:40]


def test_topk_deterministic():
    q, K = _gen(7, 2, 32, 8, 3000)
    a, b = run_gpu(q, K, 300), run_gpu(q, K, 300)
    assert np.array_equal(a, b)


def test_topk_full_size_every_head():
    """The bench's top-k workload (batch 8, 8 KV heads, 32K keys, k = 3276):
    all 64 heads checked against the oracle."""
    d = dev()
    B, Hq, Hkv, T, k = 8, 32, 8, 32768, 3276
    g = torch.Generator(device=d).manual_seed(11)
    q = torch.randn((B, Hq, 128), generator=g, device=d).to(torch.float16)
    K = torch.randn((B, Hkv, T, 128), generator=g, device=d).to(torch.float16)
    idx = torch.empty((B, Hkv, k), dtype=torch.int32, device=d)
    ws = torch.empty(clo.clo_topk_workspace_size(B, Hkv, T), dtype=torch.uint8, device=d)
    clo.clo_topk_retrieve(q, K, k, idx, ws)
    torch.cuda.synchronize()
    got = idx.cpu().numpy()
    G = Hq // Hkv
    orc = oracle.get()
    qn, Kn = q.cpu().numpy(), K.cpu().numpy()

    def one(bh):
        b, h = bh
        qh, Kh = qn[b:b + 1, h * G:(h + 1) * G], Kn[b:b + 1, h:h + 1]
        ref = orc.topk_retrieve(qh, Kh, k)[0, 0]
        return check_head(got[b, h], ref, qh.astype(np.float64)[0].sum(0),
                          Kh.astype(np.float64)[0, 0], k)

    # One head at a time: the oracle's top-k sorts through a file-level
    # comparator context, so it must not run on several threads at once.
    swaps = [one((b, h)) for b in range(B) for h in range(Hkv)]
    assert sum(swaps) <= B * Hkv
    print(f"top-k full size: 64 heads, {sum(swaps)} boundary swaps")


def test_retrieval_fill_attention_chain():
    """CLO's miss path with retrieval, on one stream with no host round trip:
    the lookup flags the missed heads; top-k retrieval ranks every key of
    every head against the queries (CLO Eq. 6); the fill copies the missed
    heads' new top-k rows from the full KV copy in pinned host memory into
    the token-addressed Cache Buffer; the attention reads them through the
    same indices.  The retrieval is checked against the oracle's as above,
    and the oracle then runs the lookup, fill and attention on the indices the
    GPU chose, which the GPU results must match (the fill bit for bit)."""
    import workloads as wl
    from gpu_util import assert_close, scale_for

    cfg = wl.small_hybrid("retrieval_chain", B=2, Hq=32, Hkv=8, T=1200, Np=2, qmode="cos",
                          c_lo=0.5, c_hi=0.95, seed=5500)
    orc = oracle.get()
    d = dev()
    q, lab = wl.queries_and_labels(cfg, 0, "cpu")
    srcK, srcV = wl.full_kv(cfg, 0, "cpu")
    cbK, cbV, _ = wl.cache_buffer(cfg, 0, "cpu")  # old rows, partly overwritten by the fill
    pK, pV = wl.persistent_cache(cfg, 0, "cpu")
    pid = wl.persist_ids(cfg, 0)
    pm = wl.persist_mask(cfg, 0)
    s = np.ones(cfg.Hq, dtype=np.float32)  # tau = eta: groups with cosine below 0.8 miss
    tau = clo.clo_thresholds_host(s, cfg.Hkv, cfg.G, 0.8, 3.0)

    qd, labd = q.to(d), lab.to(d)
    n = cfg.B * cfg.Hkv
    flag = torch.empty(n, dtype=torch.uint8, device=d)
    sim = torch.empty(n, dtype=torch.float32, device=d)
    ml = torch.empty(n, dtype=torch.int32, device=d)
    mc = torch.empty(1, dtype=torch.int32, device=d)
    idx = torch.empty((cfg.B, cfg.Hkv, cfg.k), dtype=torch.int32, device=d)
    tws = torch.empty(clo.clo_topk_workspace_size(cfg.B, cfg.Hkv, cfg.T), dtype=torch.uint8,
                      device=d)
    gK, gV = cbK.to(d), cbV.to(d)
    out = torch.empty_like(qd)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv), dtype=torch.uint8,
                     device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    hK, hV = srcK.pin_memory(), srcV.pin_memory()
    clo.clo_lookup_update(qd, labd, torch.from_numpy(s).to(d), torch.from_numpy(tau).to(d),
                          torch.from_numpy(pm).to(d), flag, sim, ml, mc)
    clo.clo_topk_retrieve(qd, srcK.to(d), cfg.k, idx, tws)
    clo.clo_fill_cache_buffer(hK, hV, idx, None, gK, gV, ml, mc, err_flag=err)
    clo.clo_hybrid_decode_attn(qd, gK, gV, idx, pK.to(d), pV.to(d), torch.from_numpy(pid).to(d),
                               out, ws, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # The retrieval against the oracle's (boundary swaps inside the fp32 band only).
    got_idx = idx.cpu().numpy()
    ref_idx = orc.topk_retrieve(q.numpy(), srcK.numpy(), cfg.k)
    q64, K64 = q.numpy().astype(np.float64), srcK.numpy().astype(np.float64)
    for b in range(cfg.B):
        for g in range(cfg.Hkv):
            check_head(got_idx[b, g], ref_idx[b, g], q64[b, g * cfg.G:(g + 1) * cfg.G].sum(0),
                       K64[b, g], cfg.k)
    # The oracle chain on the GPU's indices.
    lk = orc.lookup_update(q.numpy(), lab.numpy(), s.astype(np.float64), tau.astype(np.float64),
                           pm)
    assert not (np.abs(lk["sim"] - tau.astype(np.float64)[None, :]) < 1e-4).any()
    assert int(mc.item()) == lk["miss_count"] > 0
    rK, rV, rc = orc.fill_cache_buffer(srcK.numpy(), srcV.numpy(), got_idx, None, cbK.numpy(),
                                       cbV.numpy(), lk["miss_list"])
    assert rc == 0
    assert np.array_equal(gK.cpu().numpy().view(np.uint16), rK)
    assert np.array_equal(gV.cpu().numpy().view(np.uint16), rV)
    ref, _ = orc.hybrid_attn(q.numpy(), rK, rV, got_idx, pK.numpy(), pV.numpy(), pid, scale_for())
    assert_close(out.cpu().numpy(), ref, "retrieval + fill + attention")
