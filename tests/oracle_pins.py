"""Pins for the fp64 oracle: each check ties it to something other than itself.

Every ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
on a mismatch.  They are run on the real oracle by test_oracle_pins.py and on
copies with planted mistakes by test_oracle_mutants.py (which expects at
least one pin to fail for every planted mistake).

The anchors used:
  * values printed on the CLO page (golden files under tests/golden/),
  * library routines (numpy's binary16 decoding, scipy's cosine distance,
    numpy's weighted average, torch's scaled_dot_product_attention and
    logsumexp in float64),
  * closed forms and invariants (norm invariance of the cosine, Eq. 6;
    equal-similarity collapse of Eq. 10; constant-V and single-token
    attention; permutation invariance of the attended set).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
from scipy.spatial.distance import cosine as scipy_cosine_distance

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _f16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


def _sdpa64(q16, K16, V16, scale):
    """torch SDPA in float64: q [G][d], K/V [n][d] -> out [G][d]."""
    q = torch.from_numpy(q16.astype(np.float64))[None, :, None, :]
    K = torch.from_numpy(K16.astype(np.float64))[None, None].expand(1, q.shape[1], -1, -1)
    V = torch.from_numpy(V16.astype(np.float64))[None, None].expand(1, q.shape[1], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=scale)
    return o[0, :, 0, :].numpy()


def _lse64(q16, K16, scale):
    s = torch.from_numpy(q16.astype(np.float64)) @ torch.from_numpy(K16.astype(np.float64)).T
    return torch.logsumexp(s * scale, dim=1).numpy()


# ---------------------------------------------------------------- fp16 decode

def pin_half_decode(orc):
    """Decoder equals numpy's binary16 -> float64 for every bit pattern."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = orc.half_to_double(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "NaN patterns differ"
    assert np.array_equal(got[~nan], ref[~nan]), "binary16 decode differs from numpy"


# ---------------------------------------------------------------- Eqs. 7-9

def pin_threshold_limits(orc):
    """The page's printed ends of the chain: s=1 -> tau=eta, s=0 -> tau=-1."""
    for eta, n, s, tau in _read_golden("threshold_limits.txt"):
        got = orc.thresholds([s], 1, 1, eta, n)[0]
        assert abs(got - tau) <= 1e-12, (eta, n, s, got, tau)
    # s = 1 gives tau = eta for any eta (the derivation in the same check).
    for eta in (0.3, 0.5, 0.8, 0.95):
        got = orc.thresholds([1.0], 1, 1, eta, 3.0)[0]
        assert abs(got - eta) <= 1e-12, (eta, got)


def pin_threshold_monotone_range(orc):
    """Important heads get stricter thresholds: tau non-decreasing in s and
    within [-1, eta]."""
    s = np.linspace(0.0, 1.0, 201)
    tau = orc.thresholds(s, s.size, 1, 0.8, 3.0)
    assert np.all(np.diff(tau) >= -1e-15), "tau not monotone in s"
    assert tau.min() >= -1.0 - 1e-15 and tau.max() <= 0.8 + 1e-12


def pin_threshold_angle_affine(orc):
    """With n = 1 the chain interpolates in angle space: arccos(tau) is an
    affine function of s through (0, pi) and (1, arccos eta)."""
    eta = 0.8
    s = np.array([0.0, 0.1, 0.25, 0.5, 0.8, 1.0])
    ang = np.arccos(np.clip(orc.thresholds(s, s.size, 1, eta, 1.0), -1, 1))
    a, b = np.polyfit(s, ang, 1)
    assert np.max(np.abs(a * s + b - ang)) < 1e-7, "arccos(tau) not affine in s"
    assert abs(b - math.pi) < 1e-7 and abs(a + b - math.acos(eta)) < 1e-7


def pin_threshold_exponent(orc):
    """lambda = s^n (Eq. 8): the chain at exponent n equals the n = 1 chain
    evaluated at s^n."""
    s = np.array([0.05, 0.3, 0.5, 0.7, 0.9, 0.99])
    for n in (2.0, 3.0, 5.0):
        a = orc.thresholds(s, s.size, 1, 0.8, n)
        b = orc.thresholds(s ** n, s.size, 1, 0.8, 1.0)
        assert np.max(np.abs(a - b)) < 1e-12, n


def pin_threshold_group_mean(orc):
    """Group score = mean of the group's query-head scores: a group of equal
    scores gives the single-head threshold, and the order inside a group
    does not matter."""
    s = np.array([0.2, 0.7, 0.4, 0.9])
    one = orc.thresholds([0.55], 1, 1, 0.8, 3.0)[0]
    got = orc.thresholds(s, 1, 4, 0.8, 3.0)[0]
    assert abs(got - one) < 1e-12
    eq = orc.thresholds([0.6] * 4, 1, 4, 0.8, 3.0)[0]
    assert abs(eq - orc.thresholds([0.6], 1, 1, 0.8, 3.0)[0]) < 1e-12


# ---------------------------------------------------------------- lookup / Eq. 10

def _lookup_case(seed=7, B=3, Hq=16, Hkv=4, d=128):
    rng = _rng(seed)
    lab = _f16(rng, (B, Hq, d))
    q = (0.8 * lab.astype(np.float32) + 0.6 * rng.standard_normal((B, Hq, d))).astype(np.float16)
    w = rng.uniform(0.0, 1.0, Hq)
    return q, lab, w


def pin_lookup_cosine_scipy(orc):
    """Per-query-head cosine equals scipy's (1 - cosine distance)."""
    q, lab, w = _lookup_case()
    r = orc.lookup_update(q, lab, w, np.full(4, -2.0))
    B, Hq, _ = q.shape
    for b in range(B):
        for h in range(Hq):
            ref = 1.0 - scipy_cosine_distance(q[b, h].astype(np.float64),
                                              lab[b, h].astype(np.float64))
            assert abs(r["cos"][b, h] - ref) < 1e-12, (b, h)


def pin_lookup_eq10_weighted_mean(orc):
    """Eq. 10: the KV head's similarity is numpy's importance-weighted average
    of the cosines of its G query heads (query head h -> KV head h // G)."""
    q, lab, w = _lookup_case(seed=11)
    r = orc.lookup_update(q, lab, w, np.full(4, -2.0))
    B, Hq, _ = q.shape
    G = Hq // 4
    for b in range(B):
        for g in range(4):
            c = [1.0 - scipy_cosine_distance(q[b, h].astype(np.float64),
                                             lab[b, h].astype(np.float64))
                 for h in range(g * G, (g + 1) * G)]
            ref = np.average(c, weights=w[g * G:(g + 1) * G])
            assert abs(r["sim"][b, g] - ref) < 1e-12, (b, g)


def pin_lookup_eq10_equal_sims(orc):
    """Eq. 10 rule 2 (page check 3): equal similarities collapse to that value
    for any weights (golden weight sets)."""
    rng = _rng(3)
    for row in _read_golden("eq10_equal_sims.txt"):
        G = int(row[0])
        w = np.array(row[1:1 + G])
        lab1 = _f16(rng, (128,))
        q1 = (0.7 * lab1.astype(np.float32) + 0.7 * rng.standard_normal(128)).astype(np.float16)
        lab = np.broadcast_to(lab1, (1, G, 128)).copy()
        q = np.broadcast_to(q1, (1, G, 128)).copy()
        r = orc.lookup_update(q, lab, w, np.array([-2.0]))
        c = 1.0 - scipy_cosine_distance(q1.astype(np.float64), lab1.astype(np.float64))
        assert abs(r["sim"][0, 0] - c) < 1e-12, (row, r["sim"][0, 0], c)


def pin_lookup_norm_invariance(orc):
    """Eq. 6: ranking and similarity do not depend on ||q|| -- scaling q by 2
    and the labels by 4 (exact in binary16 for these magnitudes) leaves sims
    and flags unchanged."""
    q, lab, w = _lookup_case(seed=5)
    tau = np.array([0.5, 0.75, 0.8, 0.85])
    r1 = orc.lookup_update(q, lab, w, tau)
    r2 = orc.lookup_update((q.astype(np.float32) * 2).astype(np.float16),
                           (lab.astype(np.float32) * 4).astype(np.float16), w, tau)
    assert np.max(np.abs(r1["sim"] - r2["sim"])) < 1e-12
    assert np.array_equal(r1["flag"], r2["flag"])


def pin_lookup_self_hit(orc):
    """q equal to its label has cosine 1: every head hits for tau <= 1 and no
    label changes."""
    _, lab, w = _lookup_case(seed=9)
    tau = np.array([0.999999, 0.8, 0.0, -1.0])
    r = orc.lookup_update(lab, lab, w, tau)
    assert np.all(r["flag"] == 0) and r["miss_count"] == 0
    assert np.array_equal(r["labels"], lab.view(np.uint16))


def pin_lookup_tau_minus_one(orc):
    """s = 0 gives tau = -1, which the page calls always a hit (check 2)."""
    q, lab, w = _lookup_case(seed=13)
    q = (-lab.astype(np.float32) + 0.01 * _rng(1).standard_normal(lab.shape)).astype(np.float16)
    tau = np.full(4, orc.thresholds([0.0], 1, 1, 0.8, 3.0)[0])
    r = orc.lookup_update(q, lab, w, tau)
    assert np.all(r["flag"] == 0), r["sim"]


def pin_lookup_exact_tie_hits(orc):
    """sim == tau is a hit ("cos >= tau_i hits", section 2).  Vectors of 0.5 in
    64 slots have norm exactly 4, so the cosine of q with itself is exactly 1."""
    v = np.zeros((1, 4, 128), dtype=np.float16)
    v[:, :, :64] = 0.5
    r = orc.lookup_update(v, v, np.ones(4), np.array([1.0]))
    assert r["sim"][0, 0] == 1.0 and r["flag"][0, 0] == 0


def pin_lookup_miss_replaces_group(orc):
    """A miss replaces all G labels of the KV head with the current queries, a
    hit leaves them, a persistent head is flagged 2 and left alone; the miss
    list is the ascending b*Hkv+g of the misses.  Group pattern chosen so a
    wrong query-head -> KV-head mapping changes the flags."""
    rng = _rng(21)
    B, Hkv, G, d = 2, 4, 4, 128
    lab = _f16(rng, (B, Hkv * G, d))
    q = lab.copy()
    # (b, g) pattern of misses: q opposite to the label.
    miss = {(0, 1), (0, 3), (1, 0), (1, 2)}
    for (b, g) in miss:
        q[b, g * G:(g + 1) * G] = -lab[b, g * G:(g + 1) * G]
    persist = np.array([0, 0, 1, 0], dtype=np.uint8)  # KV head 2 persistent
    w = rng.uniform(0.1, 1.0, Hkv * G)
    r = orc.lookup_update(q, lab, w, np.full(Hkv, 0.5), persist)
    exp_list = []
    for b in range(B):
        for g in range(Hkv):
            sl = slice(g * G, (g + 1) * G)
            if persist[g]:
                assert r["flag"][b, g] == 2
                assert np.array_equal(r["labels"][b, sl], lab.view(np.uint16)[b, sl])
            elif (b, g) in miss:
                assert r["flag"][b, g] == 1
                assert np.array_equal(r["labels"][b, sl], q.view(np.uint16)[b, sl])
                exp_list.append(b * Hkv + g)
            else:
                assert r["flag"][b, g] == 0
                assert np.array_equal(r["labels"][b, sl], lab.view(np.uint16)[b, sl])
    assert r["miss_list"].tolist() == exp_list and r["miss_count"] == len(exp_list)


def pin_lookup_degenerate(orc):
    """A zero query has cosine 0; all-zero weights fall back to the plain mean."""
    rng = _rng(17)
    lab = _f16(rng, (1, 4, 128))
    q = lab.copy()
    q[0, 0] = 0
    r = orc.lookup_update(q, lab, np.zeros(4), np.array([-2.0]))
    assert r["cos"][0, 0] == 0.0
    assert abs(r["sim"][0, 0] - np.mean(r["cos"][0])) < 1e-15
    assert abs(r["sim"][0, 0] - 0.75) < 1e-12


# ---------------------------------------------------------------- attention

def pin_attention_sdpa(orc):
    """Dense attention equals torch's float64 scaled_dot_product_attention, and
    lse equals torch's logsumexp of the scaled scores."""
    rng = _rng(31)
    for (G, n) in ((4, 37), (5, 1), (1, 200), (8, 64)):
        q, K, V = _f16(rng, (G, 128)), _f16(rng, (n, 128)), _f16(rng, (n, 128))
        scale = 1.0 / math.sqrt(128)
        out, lse = orc.attention_dense(q, K, V, scale)
        assert np.max(np.abs(out - _sdpa64(q, K, V, scale))) < 1e-12, (G, n)
        assert np.max(np.abs(lse - _lse64(q, K, scale))) < 1e-12, (G, n)


def pin_attention_closed_forms(orc):
    """Constant V rows give that row; one token gives its V row and lse equal to
    its scaled score; zero scale gives the plain mean of V."""
    rng = _rng(33)
    q, K = _f16(rng, (4, 128)), _f16(rng, (50, 128))
    row = _f16(rng, (128,))
    V = np.broadcast_to(row, (50, 128)).copy()
    out, _ = orc.attention_dense(q, K, V, 0.09)
    assert np.max(np.abs(out - row.astype(np.float64))) < 1e-12
    V1 = _f16(rng, (1, 128))
    out, lse = orc.attention_dense(q, K[:1], V1, 0.09)
    assert np.max(np.abs(out - V1.astype(np.float64))) == 0.0
    s0 = q.astype(np.float64) @ K[0].astype(np.float64) * 0.09
    assert np.max(np.abs(lse - s0)) < 1e-12
    V = _f16(rng, (50, 128))
    out, lse = orc.attention_dense(q, K, V, 0.0)
    assert np.max(np.abs(out - V.astype(np.float64).mean(0))) < 1e-12
    assert np.max(np.abs(lse - math.log(50))) < 1e-12


def _hybrid_case(seed, B=2, Hkv=4, G=4, C=40, k=9, Np=2, T=23, pid=(3, 1)):
    rng = _rng(seed)
    q = _f16(rng, (B, Hkv * G, 128))
    cbK, cbV = _f16(rng, (B, Hkv, C, 128)), _f16(rng, (B, Hkv, C, 128))
    pK, pV = _f16(rng, (B, Np, T, 128)), _f16(rng, (B, Np, T, 128))
    idx = np.stack([np.stack([rng.permutation(C)[:k] for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    return q, cbK, cbV, idx, pK, pV, np.array(pid[:Np], dtype=np.int32)


def pin_hybrid_gather_vs_sdpa(orc):
    """Each KV head attends to its indexed Cache Buffer rows, or to all rows of
    the Persistent Cache slot that lists it (unsorted persist_ids): checked
    against SDPA on rows gathered here with numpy indexing."""
    q, cbK, cbV, idx, pK, pV, pid = _hybrid_case(41)
    B, Hq, _ = q.shape
    Hkv, G = cbK.shape[1], Hq // cbK.shape[1]
    scale = 1.0 / math.sqrt(128)
    out, lse = orc.hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale)
    for b in range(B):
        for g in range(Hkv):
            if g in pid.tolist():
                j = pid.tolist().index(g)
                K, V = pK[b, j], pV[b, j]
            else:
                K, V = cbK[b, g][idx[b, g]], cbV[b, g][idx[b, g]]
            qs = q[b, g * G:(g + 1) * G]
            assert np.max(np.abs(out[b, g * G:(g + 1) * G] - _sdpa64(qs, K, V, scale))) < 1e-12
            assert np.max(np.abs(lse[b, g * G:(g + 1) * G] - _lse64(qs, K, scale))) < 1e-12


def pin_hybrid_reductions(orc):
    """Special cases: idx = all rows with no persistent heads is dense attention
    over the Cache Buffer; all heads persistent is dense attention over the
    Persistent Cache; a permutation of idx changes nothing; k = 1 gives the
    selected V row."""
    scale = 1.0 / math.sqrt(128)
    q, cbK, cbV, idx, pK, pV, _ = _hybrid_case(43, C=30, k=30, Np=0)
    idx_all = np.broadcast_to(np.arange(30, dtype=np.int32), idx.shape).copy()
    none = np.zeros(0, dtype=np.int32)
    pK0, pV0 = pK[:, :0], pV[:, :0]
    out, _ = orc.hybrid_attn(q, cbK, cbV, idx_all, pK0, pV0, none, scale)
    for b in range(2):
        for g in range(4):
            ref = _sdpa64(q[b, 4 * g:4 * g + 4], cbK[b, g], cbV[b, g], scale)
            assert np.max(np.abs(out[b, 4 * g:4 * g + 4] - ref)) < 1e-12
    perm = idx_all[..., ::-1].copy()
    out2, _ = orc.hybrid_attn(q, cbK, cbV, perm, pK0, pV0, none, scale)
    assert np.max(np.abs(out - out2)) < 1e-12
    q, cbK, cbV, idx, pK, pV, _ = _hybrid_case(44, Np=4, pid=(2, 0, 3, 1))
    pid = np.array([2, 0, 3, 1], dtype=np.int32)
    out, _ = orc.hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale)
    for b in range(2):
        for j, g in enumerate(pid):
            ref = _sdpa64(q[b, 4 * g:4 * g + 4], pK[b, j], pV[b, j], scale)
            assert np.max(np.abs(out[b, 4 * g:4 * g + 4] - ref)) < 1e-12
    q, cbK, cbV, idx, pK, pV, pid = _hybrid_case(45, k=1)
    out, _ = orc.hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, scale)
    for b in range(2):
        for g in (0, 2):  # not persistent in this case
            row = cbV[b, g, idx[b, g, 0]].astype(np.float64)
            assert np.max(np.abs(out[b, 4 * g:4 * g + 4] - row)) == 0.0


def pin_hybrid_bad_index(orc):
    """An index outside the Cache Buffer is reported, not read."""
    q, cbK, cbV, idx, pK, pV, pid = _hybrid_case(47)
    idx[1, 0, 3] = cbK.shape[2]
    try:
        orc.hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, 0.1)
    except ValueError as e:
        assert "rc=4" in str(e)
    else:
        raise AssertionError("out-of-range index accepted")


def _paged_case(seed, B=3, Hkv=2, G=2, bs=16, mb=5, lens=(33, 80, 1)):
    rng = _rng(seed)
    nb = B * mb + 3
    q = _f16(rng, (B, Hkv * G, 128))
    kc, vc = _f16(rng, (nb, Hkv, bs, 128)), _f16(rng, (nb, Hkv, bs, 128))
    bt = rng.permutation(nb)[:B * mb].reshape(B, mb).astype(np.int32)
    return q, kc, vc, bt, np.array(lens[:B], dtype=np.int32)


def pin_paged_vs_sdpa(orc):
    """Token t of request r is row t % 16 of block block_table[r][t // 16]:
    checked against SDPA on K/V reassembled here block by block."""
    q, kc, vc, bt, cl = _paged_case(51)
    scale = 1.0 / math.sqrt(128)
    out, lse = orc.paged_attn(q, kc, vc, bt, cl, scale)
    B, Hq, _ = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    for r in range(B):
        for h in range(Hkv):
            K = np.concatenate([kc[bt[r, j], h] for j in range(bt.shape[1])])[:cl[r]]
            V = np.concatenate([vc[bt[r, j], h] for j in range(bt.shape[1])])[:cl[r]]
            qs = q[r, h * G:(h + 1) * G]
            assert np.max(np.abs(out[r, h * G:(h + 1) * G] - _sdpa64(qs, K, V, scale))) < 1e-12
            assert np.max(np.abs(lse[r, h * G:(h + 1) * G] - _lse64(qs, K, scale))) < 1e-12


def pin_paged_identity_and_empty(orc):
    """An identity block table over a contiguous pool is contiguous attention;
    a request with no tokens gives zeros and lse = -inf."""
    rng = _rng(53)
    n = 40
    q = _f16(rng, (2, 1, 128))
    K, V = _f16(rng, (n, 128)), _f16(rng, (n, 128))
    kc = np.zeros((3, 1, 16, 128), dtype=np.float16)
    vc = np.zeros_like(kc)
    kc.reshape(48, 128)[:n] = K
    vc.reshape(48, 128)[:n] = V
    bt = np.array([[0, 1, 2], [0, 1, 2]], dtype=np.int32)
    out, lse = orc.paged_attn(q, kc, vc, bt, np.array([n, 0], dtype=np.int32), 0.1)
    assert np.max(np.abs(out[0] - _sdpa64(q[0], K, V, 0.1))) < 1e-12
    assert np.all(out[1] == 0.0) and np.all(np.isneginf(lse[1]))


# -- miss-path fill (CLO page, section 3, Fig. 7: new KV rows go straight to
#    their final position; section 2: only missed heads are transferred) ------

def _h(vals):
    return np.asarray(vals, dtype=np.float16)


def pin_fill_worked_example(orc):
    """A case small enough to write the answer out by hand."""
    # Full KV of B=1 batch row, 2 KV heads, T=3 tokens, d=2: K row (g, t) is
    # [10g + t, -(10g + t)], V row is [100 + 10g + t, 0.5].
    srcK = _h([[[[0, -0], [1, -1], [2, -2]], [[10, -10], [11, -11], [12, -12]]]])
    srcV = _h([[[[100, .5], [101, .5], [102, .5]], [[110, .5], [111, .5], [112, .5]]]])
    tok = np.array([[[2, 0], [1, 2]]], dtype=np.int32)
    zero = np.zeros((1, 2, 3, 2), dtype=np.float16)
    # Token-addressed (slot = token), only head 1 on the miss list.
    K, V, rc = orc.fill_cache_buffer(srcK, srcV, tok, None, zero, zero, [1])
    assert rc == 0
    wantK = _h([[[[0, 0], [0, 0], [0, 0]], [[0, 0], [11, -11], [12, -12]]]])
    wantV = _h([[[[0, 0], [0, 0], [0, 0]], [[0, 0], [111, .5], [112, .5]]]])
    assert np.array_equal(K.view(np.float16), wantK), K.view(np.float16)
    assert np.array_equal(V.view(np.float16), wantV), V.view(np.float16)
    # Compact (slot = position in the set), both heads missed, C = 2.
    zero2 = np.zeros((1, 2, 2, 2), dtype=np.float16)
    slot = np.array([[[0, 1], [0, 1]]], dtype=np.int32)
    K, V, rc = orc.fill_cache_buffer(srcK, srcV, tok, slot, zero2, zero2, [0, 1])
    assert rc == 0
    wantK = _h([[[[2, -2], [0, -0]], [[11, -11], [12, -12]]]])
    wantV = _h([[[[102, .5], [100, .5]], [[111, .5], [112, .5]]]])
    assert np.array_equal(K.view(np.float16), wantK), K.view(np.float16)
    assert np.array_equal(V.view(np.float16), wantV), V.view(np.float16)


def _fill_case(seed, B=2, Hkv=3, T=29, k=7, d=16, compact=False):
    rng = _rng(seed)
    srcK, srcV = _f16(rng, (B, Hkv, T, d)), _f16(rng, (B, Hkv, T, d))
    tok = np.stack([rng.choice(T, k, replace=False) for _ in range(B * Hkv)])
    tok = tok.reshape(B, Hkv, k).astype(np.int32)
    if compact:
        C = k
        slot = np.stack([rng.permutation(k) for _ in range(B * Hkv)]).reshape(B, Hkv, k)
        slot = slot.astype(np.int32)
    else:
        C, slot = T, None
    cbK, cbV = _f16(rng, (B, Hkv, C, d)), _f16(rng, (B, Hkv, C, d))
    return srcK, srcV, tok, slot, cbK, cbV


def pin_fill_then_attention_vs_sdpa(orc):
    """After every head is filled, the hybrid attention over the Cache Buffer
    (rows named by the slots) equals torch SDPA over the selected rows of the
    full KV copy: the rows landed where the attention reads them."""
    for compact in (False, True):
        B, Hkv, G, d = 2, 3, 2, 16
        srcK, srcV, tok, slot, cbK, cbV = _fill_case(11 + compact, B=B, Hkv=Hkv, d=d,
                                                     compact=compact)
        K, V, rc = orc.fill_cache_buffer(srcK, srcV, tok, slot, cbK, cbV,
                                         np.arange(B * Hkv))
        assert rc == 0
        q = _f16(_rng(5), (B, Hkv * G, d))
        idx = tok if slot is None else slot
        empty = np.zeros((B, 0, 1, d), dtype=np.float16)
        out, _ = orc.hybrid_attn(q, K, V, idx, empty, empty, [], 1.0 / math.sqrt(d))
        for b in range(B):
            for g in range(Hkv):
                ref = _sdpa64(q[b, g * G:(g + 1) * G], srcK[b, g, tok[b, g]],
                              srcV[b, g, tok[b, g]], 1.0 / math.sqrt(d))
                assert np.allclose(out[b, g * G:(g + 1) * G], ref, atol=1e-12, rtol=0), (b, g)


def pin_fill_leaves_the_rest(orc):
    """Heads not on the miss list, and rows not selected, keep their bytes."""
    srcK, srcV, tok, slot, cbK, cbV = _fill_case(21)
    B, Hkv, T = tok.shape[0], tok.shape[1], srcK.shape[2]
    miss = [0 * Hkv + 2, 1 * Hkv + 0]
    K, V, rc = orc.fill_cache_buffer(srcK, srcV, tok, slot, cbK, cbV, miss)
    assert rc == 0
    cbK16, cbV16 = cbK.view(np.uint16), cbV.view(np.uint16)
    sK, sV = srcK.view(np.uint16), srcV.view(np.uint16)
    for b in range(B):
        for g in range(Hkv):
            chosen = set(tok[b, g].tolist()) if (b * Hkv + g) in miss else set()
            for t in range(T):
                wantK = sK[b, g, t] if t in chosen else cbK16[b, g, t]
                wantV = sV[b, g, t] if t in chosen else cbV16[b, g, t]
                assert np.array_equal(K[b, g, t], wantK), (b, g, t)
                assert np.array_equal(V[b, g, t], wantV), (b, g, t)


def pin_fill_bad_entries_skipped(orc):
    """Out-of-range list entries, tokens and slots are skipped and reported;
    every valid row is still written."""
    srcK, srcV, tok, slot, cbK, cbV = _fill_case(31, compact=True)
    B, Hkv, k = tok.shape
    tok = tok.copy()
    slot = slot.copy()
    tok[0, 1, 3] = srcK.shape[2]      # token past the end
    slot[1, 2, 0] = -1                # slot before the start
    good = [0 * Hkv + 1, 1 * Hkv + 2]
    K, V, rc = orc.fill_cache_buffer(srcK, srcV, tok, slot, cbK, cbV, good + [B * Hkv, -3])
    assert rc == 4
    Kg, Vg, rcg = orc.fill_cache_buffer(srcK, srcV, tok, slot, cbK, cbV, good)
    assert rcg == 4 and np.array_equal(K, Kg) and np.array_equal(V, Vg)
    # The skipped rows kept their old contents; the others hold the new rows.
    for (b, g) in ((0, 1), (1, 2)):
        for j in range(k):
            bad = (b, g, j) in ((0, 1, 3), (1, 2, 0))
            r = slot[b, g, j]
            if bad:
                continue
            assert np.array_equal(K[b, g, r], srcK.view(np.uint16)[b, g, tok[b, g, j]])
    assert np.array_equal(K[0, 1, slot[0, 1, 3]], cbK.view(np.uint16)[0, 1, slot[0, 1, 3]])


def pin_fill_list_order(orc):
    """The order of the miss list does not matter (the heads are disjoint)."""
    srcK, srcV, tok, slot, cbK, cbV = _fill_case(41, compact=True)
    n = tok.shape[0] * tok.shape[1]
    a = orc.fill_cache_buffer(srcK, srcV, tok, slot, cbK, cbV, np.arange(n))
    b = orc.fill_cache_buffer(srcK, srcV, tok, slot, cbK, cbV, np.arange(n)[::-1])
    assert a[2] == b[2] == 0
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# -- offline persistent-head plan (CLO page, section 3.3, Eqs. 11-13) ---------

_PLAN_TAU = [[0.8, 0.5, -1.0, 0.7], [0.6, 0.6, 0.2, -0.5]]
_PLAN_SHAT = [[0.75, 0.9, 0.2, 0.5], [0.4, 0.45, 0.9, 0.1]]


def pin_plan_worked_example(orc):
    """Eqs. 11-13 on numbers worked out by hand.  D = tau - (s^ - 0.1):
    layer 0: 0.15, -0.3, -1.1, 0.3 (hard: heads 3, 0); layer 1: 0.3, 0.25,
    -0.6, -0.5 (hard: heads 0, 1).  mem_head = 10 MB over 10 GB/s: one head
    per ms of compute."""
    want_D = [[0.15, -0.3, -1.1, 0.3], [0.3, 0.25, -0.6, -0.5]]
    for t_comp, n_p, n_persist, ids in (
            (0.5e-3, 0, [2, 2], [[3, 0, -1, -1], [0, 1, -1, -1]]),
            (1.5e-3, 1, [1, 1], [[3, -1, -1, -1], [0, -1, -1, -1]]),
            (2.5e-3, 2, [0, 0], [[-1] * 4, [-1] * 4]),
            (40e-3, 40, [0, 0], [[-1] * 4, [-1] * 4])):
        r = orc.plan_persistent(_PLAN_TAU, _PLAN_SHAT, 0.1, t_comp, 10e9, 10e6)
        assert np.allclose(r["D"], want_D, atol=1e-12, rtol=0), r["D"]
        assert r["n_p"] == n_p, (t_comp, r["n_p"])
        assert r["n_persist"].tolist() == n_persist, (t_comp, r["n_persist"])
        assert r["persist_ids"].tolist() == ids, (t_comp, r["persist_ids"])


def pin_plan_zero_difficulty_is_not_hard(orc):
    """D = 0 exactly (0.5 - (0.75 - 0.25)) is not hard: Eq. 11 needs D > 0."""
    r = orc.plan_persistent([[0.5, 0.5]], [[0.75, 0.5]], 0.25, 0.0, 1e9, 1e6)
    assert r["D"].tolist() == [[0.0, 0.25]]
    assert r["n_p"] == 0 and r["n_persist"].tolist() == [1]
    assert r["persist_ids"].tolist() == [[1, -1]]


def pin_plan_tie_goes_to_lower_head(orc):
    """Heads 1 and 2 are equally hard (D = 0.2) and harder than head 0
    (D = 0.1); with one head to keep, head 1 is kept, with two, heads 1, 2."""
    tau, sh = [[0.5, 0.6, 0.6]], [[0.4, 0.4, 0.4]]   # D = tau - s^ (eps = 0)
    r = orc.plan_persistent(tau, sh, 0.0, 2.5e-3, 1e9, 1e6)    # N_p = 2 of 3 hard
    assert r["n_p"] == 2 and r["n_persist"].tolist() == [1]
    assert r["persist_ids"].tolist() == [[1, -1, -1]]
    r = orc.plan_persistent(tau, sh, 0.0, 1.5e-3, 1e9, 1e6)    # N_p = 1
    assert r["persist_ids"].tolist() == [[1, 2, -1]]


def pin_plan_invariants(orc):
    """Random plans: N_p is dimensionless (scaling time and head bytes
    together leaves it alone), Eq. 13 is never negative, more bandwidth never
    keeps more heads resident, the resident heads are the hardest ones, and
    ties go to the lower head index."""
    rng = _rng(61)
    L, Hkv = 6, 8
    tau = rng.uniform(-1, 0.8, (L, Hkv))
    sh = rng.uniform(0.2, 1.0, (L, Hkv))
    tau[2, 5] = tau[2, 1]
    sh[2, 5] = sh[2, 1]          # equal difficulty in layer 2
    last = None
    for bw in (0.0, 1e9, 3e9, 6e9, 2e10):
        r = orc.plan_persistent(tau, sh, 0.05, 2e-3, bw, 2e6)
        r2 = orc.plan_persistent(tau, sh, 0.05, 4e-3, bw, 4e6)
        assert r2["n_p"] == r["n_p"]
        hard = (r["D"] > 0).sum(axis=1)
        assert np.array_equal(r["n_persist"], np.maximum(hard - r["n_p"], 0))
        assert (r["n_persist"] >= 0).all()
        if last is not None:
            assert (r["n_persist"] <= last).all()
        last = r["n_persist"]
        for l in range(L):
            kept = [i for i in r["persist_ids"][l] if i >= 0]
            assert len(kept) == r["n_persist"][l] and len(set(kept)) == len(kept)
            rest = [i for i in range(Hkv) if r["D"][l, i] > 0 and i not in kept]
            if kept and rest:
                assert min(r["D"][l, kept]) >= max(r["D"][l, rest])
            assert list(r["D"][l, kept]) == sorted(r["D"][l, kept], reverse=True)
            if l == 2 and 5 in kept:   # the tie: head 1 goes first
                assert 1 in kept and kept.index(1) < kept.index(5)


# -- top-k retrieval (CLO page, section 2, Eq. 6; the decode flow's top-k
#    retrieval stage), exact ranking by the group's summed qk-score ----------

def pin_topk_worked_example(orc):
    """Two query heads [1, 0] and [0, 1] share one KV head, so the score of a
    key is its coordinate sum: 2, 1, 3, -2, 2 for the five keys below."""
    q = _h([[[1, 0], [0, 1]]])
    K = _h([[[[1, 1], [2, -1], [0, 3], [-1, -1], [1, 1]]]])
    for k, want in ((5, [0, 1, 2, 3, 4]), (3, [0, 2, 4]), (2, [0, 2]), (1, [2]), (0, [])):
        got = orc.topk_retrieve(q, K, k)
        assert got.shape == (1, 1, k) and got[0, 0].tolist() == want, (k, got)


def pin_topk_is_the_best_set(orc):
    """On random inputs (several KV heads, GQA 4) the selected set beats every
    unselected key, in float64 scores computed here with torch, and other
    groups' queries do not matter."""
    rng = _rng(71)
    B, Hkv, G, T, d, k = 2, 3, 4, 97, 32, 13
    q = _f16(rng, (B, Hkv * G, d))
    K = _f16(rng, (B, Hkv, T, d))
    idx = orc.topk_retrieve(q, K, k)
    for b in range(B):
        for g in range(Hkv):
            qs = torch.from_numpy(q[b, g * G:(g + 1) * G].astype(np.float64)).sum(0)
            sc = (torch.from_numpy(K[b, g].astype(np.float64)) @ qs).numpy()
            sel = idx[b, g].tolist()
            assert sel == sorted(set(sel)) and len(sel) == k
            rest = np.setdiff1d(np.arange(T), sel)
            assert sc[sel].min() > sc[rest].max(), (b, g)
    q2 = q.copy()
    q2[:, :G] = _f16(rng, (B, G, d), scale=50.0)   # only group 0's queries change
    idx2 = orc.topk_retrieve(q2, K, k)
    assert np.array_equal(idx2[:, 1:], idx[:, 1:])


def pin_topk_norm_invariance(orc):
    """Eq. 6: scaling every query of the group by the same positive factor
    (powers of two, exact in binary16) leaves the selection unchanged."""
    rng = _rng(72)
    q = _f16(rng, (1, 8, 64))
    K = _f16(rng, (1, 2, 150, 64))
    base = orc.topk_retrieve(q, K, 15)
    for f in (0.25, 4.0):
        assert np.array_equal(orc.topk_retrieve((q.astype(np.float32) * f).astype(np.float16), K, 15),
                              base)


def pin_topk_ties_to_lower_token(orc):
    """Identical keys tie; the cut takes the lower token indices."""
    q = _h([[[1, 2]]])
    K = _h([[[[1, 1]] * 6 + [[5, 5]] * 2]])
    assert orc.topk_retrieve(q, K, 4)[0, 0].tolist() == [0, 1, 6, 7]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def run_all(orc):
    """Runs every pin; returns the names of the pins that failed."""
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError) as e:  # noqa: PERF203
            failed.append(f"{pin.__name__}: {e!s:.200}")
    return failed
