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
