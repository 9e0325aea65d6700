"""clo_paged_decode_attn on the GPU vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
import workloads as wl
from gpu_util import LSE_ATOL, assert_close, dev, parallel_map, scale_for

pytestmark = pytest.mark.gpu


def run_gpu(q, kc, vc, bt, cl, num_ctas=0):
    B, Hq, d = q.shape
    Hkv = kc.shape[1]
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=q.device)
    ws = torch.empty(clo.clo_paged_workspace_size(B, Hq, Hkv, d, num_ctas), dtype=torch.uint8,
                     device=q.device)
    err = torch.zeros(1, dtype=torch.int32, device=q.device)
    clo.clo_paged_decode_attn(q, kc, vc, bt, cl, out, ws, lse=lse, err_flag=err, num_ctas=num_ctas)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), int(err.item())


def check(pc, num_ctas=0, mutate=None):
    q, kc, vc, bt, cl = wl.paged_inputs(pc, "cpu")
    if mutate is not None:
        mutate(bt, cl)
    ref, ref_lse = oracle.get().paged_attn(q.numpy(), kc.numpy(), vc.numpy(), bt.numpy(),
                                           cl.numpy(), scale_for())
    got, lse, err = run_gpu(*[t.to(dev()) for t in (q, kc, vc, bt, cl)], num_ctas=num_ctas)
    assert err == 0
    assert_close(got, ref, pc.name)
    fin = np.isfinite(ref_lse)
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0) < LSE_ATOL
    assert np.array_equal(np.isneginf(lse), ~fin)


@pytest.mark.parametrize("num_ctas", [0, 1, 4])
@pytest.mark.parametrize("shape", [(6, 8, 8, 1, 300), (5, 32, 8, 1, 700), (9, 40, 8, 16, 64),
                                   (3, 32, 32, 100, 2500)])
def test_small_vs_oracle(shape, num_ctas):
    B, Hq, Hkv, lo, hi = shape
    check(wl.small_paged(B=B, Hq=Hq, Hkv=Hkv, ctx_lo=lo, ctx_hi=hi, seed=B * 7 + Hq), num_ctas)


def test_empty_and_full_requests():
    def mut(bt, cl):
        cl[0] = 0                       # idle slot
        cl[2] = bt.shape[1] * 16        # exactly full
        cl[3] = 1                       # single token
    check(wl.small_paged(B=6, Hq=32, Hkv=8, ctx_lo=1, ctx_hi=200, seed=77), 0, mut)


def test_all_requests_empty():
    pc = wl.small_paged(B=3, Hq=8, Hkv=8, ctx_lo=1, ctx_hi=40, seed=78)
    q, kc, vc, bt, cl = [t.to(dev()) for t in wl.paged_inputs(pc, "cpu")]
    cl.zero_()
    got, lse, err = run_gpu(q, kc, vc, bt, cl)
    assert err == 0 and np.all(got == 0) and np.all(np.isneginf(lse))


def test_bad_block_and_length_flagged():
    pc = wl.small_paged(B=4, Hq=8, Hkv=8, ctx_lo=50, ctx_hi=100, seed=79)
    q, kc, vc, bt, cl = wl.paged_inputs(pc, "cpu")
    ref, _ = oracle.get().paged_attn(q.numpy(), kc.numpy(), vc.numpy(), bt.numpy(), cl.numpy(),
                                     scale_for())
    bt2, cl2 = bt.clone(), cl.clone()
    bt2[1, 1] = kc.shape[0]      # block id out of range (request 1 uses >= 4 blocks)
    cl2[2] = -3                  # negative length
    got, lse, err = run_gpu(*[t.to(dev()) for t in (q, kc, vc, bt2, cl2)])
    assert err & clo.FLAG_BAD_INDEX and err & clo.FLAG_BAD_CTX
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    assert_close(got[[0, 3]], ref[[0, 3]], "untouched requests")


def test_full_size_many_pairs():
    """The B256 workload at full size: every head of twelve requests (the
    shortest, the longest, the first and last, and eight drawn at random),
    384 (request, head) pairs against the oracle."""
    pc = wl.PAGED_CONFIGS["paged_llama2_7b_b256"]
    q, kc, vc, bt, cl = wl.paged_inputs(pc, dev())
    got, lse, err = run_gpu(q, kc, vc, bt, cl)
    assert err == 0
    orc = oracle.get()
    cln, btn, qn = cl.cpu().numpy(), bt.cpu().numpy(), q.cpu().numpy()
    rng = np.random.Generator(np.random.PCG64(pc.seed))
    rs = [int(np.argmin(cln)), int(np.argmax(cln)), 0, pc.B - 1]
    rs += [int(x) for x in rng.choice([r for r in range(pc.B) if r not in rs], 8, replace=False)]
    pairs = [(r, h) for r in rs for h in range(pc.Hkv)]
    rows = {}
    for r in rs:
        nb = -(-int(cln[r]) // 16)
        blocks = torch.from_numpy(btn[r, :nb].astype(np.int64)).to(dev())
        Kr = kc[blocks].permute(1, 0, 2, 3).reshape(pc.Hkv, -1, 128)[:, : cln[r]].cpu().numpy()
        Vr = vc[blocks].permute(1, 0, 2, 3).reshape(pc.Hkv, -1, 128)[:, : cln[r]].cpu().numpy()
        rows[r] = (Kr, Vr)
    G = pc.G
    refs = parallel_map(lambda rh: orc.attention_dense(
        qn[rh[0], rh[1] * G:(rh[1] + 1) * G], np.ascontiguousarray(rows[rh[0]][0][rh[1]]),
        np.ascontiguousarray(rows[rh[0]][1][rh[1]]), scale_for()), pairs)
    for (r, h), (ref, ref_lse) in zip(pairs, refs):
        assert_close(got[r, h * G:(h + 1) * G], ref, f"paged r{r} h{h}")
        assert np.max(np.abs(lse[r, h * G:(h + 1) * G] - ref_lse)) < LSE_ATOL
    print(f"paged B256: {len(pairs)} (request, head) pairs checked against the oracle")
