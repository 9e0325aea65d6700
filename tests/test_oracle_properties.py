"""Property checks of the fp64 oracle over drawn shapes (CPU only).

The fixed-seed pins tie the oracle's attention to torch's float64
scaled_dot_product_attention on a few hand-picked shapes; here hypothesis
draws the shapes (GQA group, KV heads, persistent heads and their order,
Cache Buffer size and k, context lengths, block tables with idle requests)
and the same comparison must hold for every draw.
"""
import math

import numpy as np
import pytest

import oracle
from oracle_pins import _lse64, _sdpa64

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")

SCALE = 1.0 / math.sqrt(128)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@hyp.settings(max_examples=60, deadline=None)
@hyp.given(data=st.data())
def test_hybrid_matches_gathered_sdpa(orc, data):
    Hkv = data.draw(st.integers(1, 6), label="Hkv")
    G = data.draw(st.integers(1, 8), label="G")
    B = data.draw(st.integers(1, 3), label="B")
    C = data.draw(st.integers(1, 50), label="C")
    k = data.draw(st.integers(1, C), label="k")
    Np = data.draw(st.integers(0, Hkv), label="Np")
    T = data.draw(st.integers(1, 40), label="T")
    seed = data.draw(st.integers(0, 2 ** 31), label="seed")
    rng = np.random.Generator(np.random.PCG64(seed))
    f16 = lambda *s: rng.standard_normal(s).astype(np.float16)
    q = f16(B, Hkv * G, 128)
    cbK, cbV = f16(B, Hkv, C, 128), f16(B, Hkv, C, 128)
    pK, pV = f16(B, Np, T, 128), f16(B, Np, T, 128)
    idx = np.stack([np.stack([rng.permutation(C)[:k] for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    pid = rng.permutation(Hkv)[:Np].astype(np.int32)
    out, lse = orc.hybrid_attn(q, cbK, cbV, idx, pK, pV, pid, SCALE)
    for b in range(B):
        for g in range(Hkv):
            if g in pid.tolist():
                j = pid.tolist().index(g)
                K, V = pK[b, j], pV[b, j]
            else:
                K, V = cbK[b, g][idx[b, g]], cbV[b, g][idx[b, g]]
            qs = q[b, g * G:(g + 1) * G]
            assert np.max(np.abs(out[b, g * G:(g + 1) * G] - _sdpa64(qs, K, V, SCALE))) < 1e-12
            assert np.max(np.abs(lse[b, g * G:(g + 1) * G] - _lse64(qs, K, SCALE))) < 1e-12


@hyp.settings(max_examples=60, deadline=None)
@hyp.given(data=st.data())
def test_paged_matches_reassembled_sdpa(orc, data):
    Hkv = data.draw(st.integers(1, 4), label="Hkv")
    G = data.draw(st.integers(1, 8), label="G")
    B = data.draw(st.integers(1, 5), label="B")
    mb = data.draw(st.integers(1, 4), label="blocks per request")
    lens = data.draw(st.lists(st.integers(0, 16 * mb), min_size=B, max_size=B), label="ctx")
    spare = data.draw(st.integers(0, 5), label="spare blocks")
    seed = data.draw(st.integers(0, 2 ** 31), label="seed")
    rng = np.random.Generator(np.random.PCG64(seed))
    f16 = lambda *s: rng.standard_normal(s).astype(np.float16)
    nb = B * mb + spare
    q = f16(B, Hkv * G, 128)
    kc, vc = f16(nb, Hkv, 16, 128), f16(nb, Hkv, 16, 128)
    bt = rng.permutation(nb)[:B * mb].reshape(B, mb).astype(np.int32)
    cl = np.array(lens, dtype=np.int32)
    out, lse = orc.paged_attn(q, kc, vc, bt, cl, SCALE)
    for r in range(B):
        for h in range(Hkv):
            sl = slice(h * G, (h + 1) * G)
            if cl[r] == 0:
                assert np.all(out[r, sl] == 0.0) and np.all(np.isneginf(lse[r, sl]))
                continue
            K = np.concatenate([kc[bt[r, j], h] for j in range(mb)])[:cl[r]]
            V = np.concatenate([vc[bt[r, j], h] for j in range(mb)])[:cl[r]]
            assert np.max(np.abs(out[r, sl] - _sdpa64(q[r, sl], K, V, SCALE))) < 1e-12
            assert np.max(np.abs(lse[r, sl] - _lse64(q[r, sl], K, SCALE))) < 1e-12
