"""Seeded random-shape sweeps of both attention entry points against the fp64
oracle (GPU).

Each case draws its own batch, head counts (GQA 1 to 8), context, top-k size,
number of persistent heads, Cache Buffer addressing, CTA count and, for the
paged layout, per-request lengths (empty requests included), so the tile
ranges, segment flushes, partial merges and ragged tails meet shapes the
hand-picked cases do not.  The shapes are drawn by a fixed generator: a
failure names its case and reproduces.
"""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
from gpu_util import LSE_ATOL, assert_close, dev, scale_for

pytestmark = pytest.mark.gpu

N_CASES = 16


def _hybrid_shape(i):
    r = np.random.Generator(np.random.PCG64(1000 + i))
    Hkv = int(r.choice([1, 2, 4, 8]))
    G = int(r.integers(1, 9))
    B = int(r.integers(1, 5))
    T = int(r.integers(1, 2500))
    k = int(r.integers(1, T + 1))
    Np = int(r.integers(0, Hkv + 1))
    compact = bool(r.integers(0, 2))
    C = k if compact else T
    num_ctas = int(r.choice([0, 0, 1, 2, 5, 17, 64]))
    return B, Hkv * G, Hkv, T, k, Np, C, num_ctas


@pytest.mark.parametrize("i", range(N_CASES))
def test_hybrid_random_shape(i):
    B, Hq, Hkv, T, k, Np, C, num_ctas = _hybrid_shape(i)
    r = np.random.Generator(np.random.PCG64(2000 + i))
    f16 = lambda *s: r.standard_normal(s).astype(np.float16)
    q = f16(B, Hq, 128)
    cbK, cbV = f16(B, Hkv, C, 128), f16(B, Hkv, C, 128)
    idx = np.stack([np.stack([r.permutation(C)[:k] for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    pK, pV = f16(B, Np, T, 128), f16(B, Np, T, 128)
    pid = r.permutation(Hkv)[:Np].astype(np.int32)
    ref, ref_lse = oracle.get().hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale_for())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=dev())
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev())
    ws = torch.empty(clo.clo_hybrid_workspace_size(B, Hq, Hkv, 128, num_ctas), dtype=torch.uint8,
                     device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    has_cb = Np < Hkv
    clo.clo_hybrid_decode_attn(t(q), t(cbK) if has_cb else None, t(cbV) if has_cb else None,
                               t(idx) if has_cb else None, t(pK) if Np else None,
                               t(pV) if Np else None, t(pid) if Np else None, out, ws, lse=lse,
                               err_flag=err, num_ctas=num_ctas)
    torch.cuda.synchronize()
    case = f"B{B} Hq{Hq} Hkv{Hkv} T{T} k{k} Np{Np} C{C} ctas{num_ctas}"
    assert int(err.item()) == 0, case
    assert_close(out.cpu().numpy().astype(np.float64), ref, case)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) < LSE_ATOL, case


def _paged_case(i):
    r = np.random.Generator(np.random.PCG64(3000 + i))
    Hkv = int(r.choice([1, 2, 8, 32]))
    G = int(r.choice([1, 1, 4, 5, 8])) if Hkv <= 8 else 1
    B = int(r.integers(1, 40))
    max_ctx = int(r.integers(1, 1200))
    ctx = r.integers(0, max_ctx + 1, size=B).astype(np.int32)
    ctx[r.random(B) < 0.1] = 0  # idle slots
    mb = -(-max_ctx // 16)
    nb = B * mb + int(r.integers(0, 8))
    bt = np.stack([r.permutation(nb)[:mb] for _ in range(B)]).astype(np.int32)
    num_ctas = int(r.choice([0, 0, 1, 3, 19, 100]))
    return B, Hkv * G, Hkv, nb, bt, ctx, num_ctas, r


@pytest.mark.parametrize("i", range(N_CASES))
def test_paged_random_shape(i):
    B, Hq, Hkv, nb, bt, ctx, num_ctas, r = _paged_case(i)
    f16 = lambda *s: r.standard_normal(s).astype(np.float16)
    q = f16(B, Hq, 128)
    kc, vc = f16(nb, Hkv, 16, 128), f16(nb, Hkv, 16, 128)
    ref, ref_lse = oracle.get().paged_attn(q, kc, vc, bt, ctx, scale_for())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=dev())
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev())
    ws = torch.empty(clo.clo_paged_workspace_size(B, Hq, Hkv, 128, num_ctas), dtype=torch.uint8,
                     device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    clo.clo_paged_decode_attn(t(q), t(kc), t(vc), t(bt), t(ctx), out, ws, lse=lse, err_flag=err,
                              num_ctas=num_ctas)
    torch.cuda.synchronize()
    case = f"B{B} Hq{Hq} Hkv{Hkv} blocks{nb} max_ctx{int(ctx.max())} ctas{num_ctas}"
    assert int(err.item()) == 0, case
    got = out.cpu().numpy().astype(np.float64)
    assert_close(got, ref, case)
    lse_h = lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.max(np.abs(lse_h[fin] - ref_lse[fin]), initial=0) < LSE_ATOL, case
    assert np.array_equal(np.isneginf(lse_h), ~fin), case
    assert np.all(got[ctx == 0] == 0), case


def test_hybrid_at_the_head_limits():
    """The largest query group (G = 8) over the most KV heads a call takes (64),
    with persistent and Cache Buffer heads, against the oracle."""
    r = np.random.Generator(np.random.PCG64(4001))
    B, Hkv, G, T, k, Np = 2, 64, 8, 90, 23, 13
    Hq = Hkv * G
    f16 = lambda *s: r.standard_normal(s).astype(np.float16)
    q = f16(B, Hq, 128)
    cbK, cbV = f16(B, Hkv, T, 128), f16(B, Hkv, T, 128)
    idx = np.stack([np.stack([r.permutation(T)[:k] for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    pK, pV = f16(B, Np, T, 128), f16(B, Np, T, 128)
    pid = r.permutation(Hkv)[:Np].astype(np.int32)
    ref, ref_lse = oracle.get().hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale_for())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=dev())
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev())
    ws = torch.empty(clo.clo_hybrid_workspace_size(B, Hq, Hkv), dtype=torch.uint8, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    clo.clo_hybrid_decode_attn(t(q), t(cbK), t(cbV), t(idx), t(pK), t(pV), t(pid), out, ws,
                               lse=lse, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.cpu().numpy().astype(np.float64), ref, "64 KV heads, G = 8")
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) < LSE_ATOL


def test_paged_at_the_request_limit():
    """The most requests a paged call takes (4096) at G = 8, short contexts with
    idle slots, against the oracle."""
    r = np.random.Generator(np.random.PCG64(4002))
    B, Hkv, G = 4096, 1, 8
    Hq = Hkv * G
    ctx = r.integers(0, 41, size=B).astype(np.int32)
    mb = 3
    nb = B * mb
    bt = r.permutation(nb).reshape(B, mb).astype(np.int32)
    f16 = lambda *s: r.standard_normal(s).astype(np.float16)
    q = f16(B, Hq, 128)
    kc, vc = f16(nb, Hkv, 16, 128), f16(nb, Hkv, 16, 128)
    ref, ref_lse = oracle.get().paged_attn(q, kc, vc, bt, ctx, scale_for())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=dev())
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev())
    ws = torch.empty(clo.clo_paged_workspace_size(B, Hq, Hkv), dtype=torch.uint8, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    clo.clo_paged_decode_attn(t(q), t(kc), t(vc), t(bt), t(ctx), out, ws, lse=lse, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert_close(got, ref, "4096 requests, G = 8")
    lse_h = lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.max(np.abs(lse_h[fin] - ref_lse[fin]), initial=0) < LSE_ATOL
    assert np.array_equal(np.isneginf(lse_h), ~fin)
    assert np.all(got[ctx == 0] == 0)


@pytest.mark.parametrize("gain", [8.0, 40.0])
def test_peaked_softmax(gain):
    """Queries scaled so the scores spread over tens to hundreds of nats: one
    or a few tokens carry the softmax, the running maximum moves late in the
    stream, and the split partials differ in scale by far more than fp32's
    range (their merge must rescale, not add)."""
    r = np.random.Generator(np.random.PCG64(5000 + int(gain)))
    B, Hkv, G, T, k, Np = 2, 8, 4, 3000, 300, 2
    Hq = Hkv * G
    q = (r.standard_normal((B, Hq, 128)) * gain).astype(np.float16)
    f16 = lambda *s: r.standard_normal(s).astype(np.float16)
    cbK, cbV = f16(B, Hkv, T, 128), f16(B, Hkv, T, 128)
    idx = np.stack([np.stack([r.permutation(T)[:k] for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    pK, pV = f16(B, Np, T, 128), f16(B, Np, T, 128)
    pid = r.permutation(Hkv)[:Np].astype(np.int32)
    ref, ref_lse = oracle.get().hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale_for())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    for num_ctas in (0, 7):
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=dev())
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev())
        ws = torch.empty(clo.clo_hybrid_workspace_size(B, Hq, Hkv, 128, num_ctas),
                         dtype=torch.uint8, device=dev())
        clo.clo_hybrid_decode_attn(t(q), t(cbK), t(cbV), t(idx), t(pK), t(pV), t(pid), out, ws,
                                   lse=lse, num_ctas=num_ctas)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy().astype(np.float64), ref, f"gain {gain}, {num_ctas} CTAs")
        # lse grows with the gain; hold it to the same relative precision
        err = np.abs(lse.cpu().numpy() - ref_lse)
        assert np.all(err < LSE_ATOL * np.maximum(1.0, np.abs(ref_lse))), f"gain {gain}"


@pytest.mark.parametrize("i", range(N_CASES))
def test_fused_lookup_random_shape(i):
    """clo_hybrid_decode_attn_lookup on a random shape: the attention against
    the oracle's, and the carried lookup (about half the KV heads at s = 1, so
    tau = eta and some groups miss) against oracle_lookup_update bit for bit."""
    from gpu_util import assert_lookup_matches

    B, Hq, Hkv, T, k, Np, C, num_ctas = _hybrid_shape(500 + i)
    G = Hq // Hkv
    r = np.random.Generator(np.random.PCG64(3000 + i))
    f16 = lambda *s: r.standard_normal(s).astype(np.float16)
    q = f16(B, Hq, 128)
    cbK, cbV = f16(B, Hkv, C, 128), f16(B, Hkv, C, 128)
    idx = np.stack([np.stack([r.permutation(C)[:k] for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    pK, pV = f16(B, Np, T, 128), f16(B, Np, T, 128)
    pid = r.permutation(Hkv)[:Np].astype(np.int32)
    # The next layer's lookup inputs.
    lab = r.standard_normal((B, Hq, 128))
    qn = (0.8 * lab + 0.6 * r.standard_normal((B, Hq, 128))).astype(np.float16)
    lab = lab.astype(np.float16)
    s = r.uniform(0, 1, Hq).astype(np.float32)
    for g in range(Hkv):
        if r.integers(0, 2):
            s[g * G:(g + 1) * G] = 1.0
    tau = clo.clo_thresholds_host(s, Hkv, G)
    pm = np.zeros(Hkv, dtype=np.uint8)
    pm[r.permutation(Hkv)[:int(r.integers(0, Hkv + 1))]] = 1
    ref, ref_lse = oracle.get().hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale_for())
    ref_lk = oracle.get().lookup_update(qn, lab, s.astype(np.float64), tau.astype(np.float64), pm)

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    d = dev()
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=d)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=d)
    ws = torch.empty(clo.clo_hybrid_workspace_size(B, Hq, Hkv, 128, num_ctas), dtype=torch.uint8,
                     device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    labd = t(lab)
    n = B * Hkv
    flag = torch.full((n,), 9, dtype=torch.uint8, device=d)
    sim = torch.full((n,), -9.0, device=d)
    miss = torch.full((n,), -9, dtype=torch.int32, device=d)
    cnt = torch.full((1,), -9, dtype=torch.int32, device=d)
    has_cb = Np < Hkv
    clo.clo_hybrid_decode_attn_lookup(
        t(q), t(cbK) if has_cb else None, t(cbV) if has_cb else None, t(idx) if has_cb else None,
        t(pK) if Np else None, t(pV) if Np else None, t(pid) if Np else None, out, ws,
        t(qn), labd, t(s), t(tau), t(pm), flag, sim, miss, cnt, lse=lse, err_flag=err,
        num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    what = f"case {i}: B{B} Hq{Hq} Hkv{Hkv} T{T} k{k} Np{Np} C{C} ctas{num_ctas}"
    assert_close(out.cpu().numpy(), ref, what)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) < LSE_ATOL
    m = int(cnt.item())
    got = dict(flag=flag.cpu().numpy(), sim=sim.cpu().numpy(), labels=labd.cpu().numpy(),
               miss_list=miss.cpu().numpy()[:max(m, 0)], miss_count=m)
    assert_lookup_matches(ref_lk, got, tau, pm, G)


@pytest.mark.parametrize("i", range(N_CASES))
def test_layer_call_random_shape(i):
    """clo_hybrid_decode_layer on a random shape: the attention against the
    oracle's, the next layer's fill (a random miss list, rows from pinned host
    memory or HBM, token or compact addressing) bit for bit, and the carried
    lookup (about half the KV heads at s = 1) against oracle_lookup_update."""
    from gpu_util import assert_lookup_matches

    B, Hq, Hkv, T, k, Np, C, num_ctas = _hybrid_shape(700 + i)
    G = Hq // Hkv
    r = np.random.Generator(np.random.PCG64(4000 + i))
    f16 = lambda *s: r.standard_normal(s).astype(np.float16)
    q = f16(B, Hq, 128)
    cbK, cbV = f16(B, Hkv, C, 128), f16(B, Hkv, C, 128)
    idx = np.stack([np.stack([r.permutation(C)[:k] for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    pK, pV = f16(B, Np, T, 128), f16(B, Np, T, 128)
    pid = r.permutation(Hkv)[:Np].astype(np.int32)
    # The fill: the next layer's full KV copy, its new top-k tokens and their rows.
    Tf = int(r.integers(1, 2000))
    kf = int(r.integers(1, Tf + 1))
    compact = bool(r.integers(0, 2))
    Cf = kf if compact else Tf
    srcK, srcV = f16(B, Hkv, Tf, 128), f16(B, Hkv, Tf, 128)
    tok = np.stack([np.stack([r.permutation(Tf)[:kf] for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    slot = np.stack([np.stack([r.permutation(kf) for _ in range(Hkv)])
                     for _ in range(B)]).astype(np.int32) if compact else None
    fK0, fV0 = f16(B, Hkv, Cf, 128), f16(B, Hkv, Cf, 128)
    fmiss = sorted(r.permutation(B * Hkv)[:int(r.integers(0, B * Hkv + 1))].tolist())
    host_src = bool(r.integers(0, 2))
    fill_ctas = int(r.choice([0, 0, 1, 7, 40]))
    # The lookup of the layer after.
    lab = r.standard_normal((B, Hq, 128))
    qn = (0.8 * lab + 0.6 * r.standard_normal((B, Hq, 128))).astype(np.float16)
    lab = lab.astype(np.float16)
    s = r.uniform(0, 1, Hq).astype(np.float32)
    for g in range(Hkv):
        if r.integers(0, 2):
            s[g * G:(g + 1) * G] = 1.0
    tau = clo.clo_thresholds_host(s, Hkv, G)
    pm = np.zeros(Hkv, dtype=np.uint8)
    pm[r.permutation(Hkv)[:int(r.integers(0, Hkv + 1))]] = 1
    orc = oracle.get()
    ref, ref_lse = orc.hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale_for())
    rK, rV, rc = orc.fill_cache_buffer(srcK, srcV, tok, slot, fK0, fV0, fmiss)
    assert rc == 0
    ref_lk = orc.lookup_update(qn, lab, s.astype(np.float64), tau.astype(np.float64), pm)

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    h = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    d = dev()
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=d)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=d)
    ws = torch.empty(clo.clo_hybrid_workspace_size(B, Hq, Hkv, 128, num_ctas), dtype=torch.uint8,
                     device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    fK, fV = t(fK0), t(fV0)
    fml = torch.full((B * Hkv,), -3, dtype=torch.int32)
    fml[:len(fmiss)] = torch.tensor(fmiss, dtype=torch.int32)
    fill = ((h(srcK), h(srcV)) if host_src else (t(srcK), t(srcV))) + \
        (t(tok), None if slot is None else t(slot), fK, fV, fml.to(d),
         torch.tensor([len(fmiss)], dtype=torch.int32, device=d))
    labd = t(lab)
    n = B * Hkv
    flag = torch.full((n,), 9, dtype=torch.uint8, device=d)
    sim = torch.full((n,), -9.0, device=d)
    miss = torch.full((n,), -9, dtype=torch.int32, device=d)
    cnt = torch.full((1,), -9, dtype=torch.int32, device=d)
    has_cb = Np < Hkv
    clo.clo_hybrid_decode_layer(
        t(q), t(cbK) if has_cb else None, t(cbV) if has_cb else None, t(idx) if has_cb else None,
        t(pK) if Np else None, t(pV) if Np else None, t(pid) if Np else None, out, ws,
        fill=fill, lookup=(t(qn), labd, t(s), t(tau), t(pm), flag, sim, miss, cnt), lse=lse,
        err_flag=err, num_ctas=num_ctas, fill_ctas=fill_ctas)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    what = (f"case {i}: B{B} Hq{Hq} Hkv{Hkv} T{T} k{k} Np{Np} C{C} ctas{num_ctas}; fill T{Tf} "
            f"k{kf} C{Cf} {len(fmiss)} heads {'host' if host_src else 'hbm'} ctas{fill_ctas}")
    assert_close(out.cpu().numpy(), ref, what)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) < LSE_ATOL, what
    assert np.array_equal(fK.cpu().numpy().view(np.uint16), rK), what
    assert np.array_equal(fV.cpu().numpy().view(np.uint16), rV), what
    m = int(cnt.item())
    got = dict(flag=flag.cpu().numpy(), sim=sim.cpu().numpy(), labels=labd.cpu().numpy(),
               miss_list=miss.cpu().numpy()[:max(m, 0)], miss_count=m)
    assert_lookup_matches(ref_lk, got, tau, pm, G)
