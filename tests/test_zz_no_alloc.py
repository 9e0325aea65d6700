"""The no-allocation hybrid attention entry point (GPU).

clo_hybrid_decode_attn_noalloc exists for callers that cannot allocate device
memory when they run the decode path -- engines whose own pool holds all
free device memory, deployments that freeze allocation after start-up, host
programs with no allocator of their own.  It must give the same results as the
workspace entry point; here both are called through the C ABI on the same
inputs, twice in a row for the fixed-scratch variant (the scratch keeps the
previous call's contents), and compared at the parity tolerance; and it is
held to the fp64 oracle itself with explicit CTA counts (the opts argument
passed through) and with an out-of-range index.  This file is collected last
on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
from gpu_util import LSE_ATOL, assert_close, dev, scale_for

pytestmark = pytest.mark.gpu


def _case(seed, B, Hq, Hkv, T, k, Np):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((B, Hq, 128), generator=g).half()
    cbK = torch.randn((B, Hkv, T, 128), generator=g).half()
    cbV = torch.randn((B, Hkv, T, 128), generator=g).half()
    idx = torch.stack([torch.randperm(T, generator=g)[:k] for _ in range(B * Hkv)])
    idx = idx.reshape(B, Hkv, k).to(torch.int32)
    pK = torch.randn((B, Np, T, 128), generator=g).half()
    pV = torch.randn((B, Np, T, 128), generator=g).half()
    pid = torch.randperm(Hkv, generator=g)[:Np].to(torch.int32)
    return [t.to(dev()) for t in (q, cbK, cbV, idx, pK, pV, pid)]


@pytest.mark.parametrize("shape", [(1, 32, 8, 1024, 102, 2), (3, 40, 8, 777, 61, 1),
                                   (2, 8, 8, 300, 33, 0)])
def test_noalloc_matches_workspace_entry_twice(shape):
    q, cbK, cbV, idx, pK, pV, pid = _case(99, *shape)
    B, Hq, Hkv = shape[0], shape[1], shape[2]
    ws = torch.empty(clo.clo_hybrid_workspace_size(B, Hq, Hkv), dtype=torch.uint8, device=dev())
    ref = torch.empty_like(q)
    ref_lse = torch.empty((B, Hq), dtype=torch.float32, device=dev())
    clo.clo_hybrid_decode_attn(q, cbK, cbV, idx, pK, pV, pid, ref, ws, lse=ref_lse)
    torch.cuda.synchronize()
    ref_np = ref.cpu().numpy().astype(np.float64)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev())
        err = torch.zeros(1, dtype=torch.int32, device=dev())
        clo.clo_hybrid_decode_attn_noalloc(q, cbK, cbV, idx, pK, pV, pid, out, lse=lse,
                                           err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.cpu().numpy(), ref_np, "noalloc vs workspace entry")
        assert torch.allclose(lse, ref_lse, atol=1e-4, rtol=0)


def test_noalloc_rejects_problems_beyond_its_scratch():
    cap = clo.clo_hybrid_noalloc_max_scratch()
    assert cap == 8 << 20
    B = 4096  # (2*CTAs + B*Hkv) partials of 4 heads exceed 8 MiB
    assert clo.clo_hybrid_workspace_size(B, 32, 8) > cap
    q = torch.zeros((B, 32, 128), dtype=torch.float16, device=dev())
    cb = torch.zeros((1, 8, 16, 128), dtype=torch.float16, device=dev())
    idx = torch.zeros((B, 8, 1), dtype=torch.int32, device=dev())
    with pytest.raises(clo.CloError) as e:
        clo.clo_hybrid_decode_attn_noalloc(q, cb, cb, idx, None, None, None, torch.empty_like(q))
    assert e.value.status == clo.CLO_ERR_WORKSPACE


def _oracle(q, cbK, cbV, idx, pK, pV, pid):
    return oracle.get().hybrid_attn(*(t.cpu().numpy() for t in (q, cbK, cbV, idx, pK, pV, pid)),
                                    scale_for())


@pytest.mark.parametrize("num_ctas", [1, 37])
def test_noalloc_explicit_ctas_vs_oracle(num_ctas):
    """opts->num_ctas reaches the kernel through the no-allocation entry
    point: one CTA (no partials) and 37 CTAs (ranges cut inside segments of
    both parts, partials merged from the fixed scratch), against the oracle."""
    q, cbK, cbV, idx, pK, pV, pid = _case(123, 3, 32, 8, 2000, 200, 2)
    ref, ref_lse = _oracle(q, cbK, cbV, idx, pK, pV, pid)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((3, 32), float("nan"), dtype=torch.float32, device=dev())
        err = torch.zeros(1, dtype=torch.int32, device=dev())
        clo.clo_hybrid_decode_attn_noalloc(q, cbK, cbV, idx, pK, pV, pid, out, lse=lse,
                                           err_flag=err, num_ctas=num_ctas)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.cpu().numpy(), ref, f"noalloc, {num_ctas} CTAs")
        assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) < LSE_ATOL


def test_noalloc_bad_index_vs_oracle():
    """An out-of-range Cache Buffer index: its group's outputs are zeros with
    lse = -inf and the flag is raised; every other group matches the oracle."""
    q, cbK, cbV, idx, pK, pV, pid = _case(321, 2, 32, 8, 600, 60, 2)
    ref, _ = _oracle(q, cbK, cbV, idx, pK, pV, pid)
    g_bad = [g for g in range(8) if g not in pid.cpu().tolist()][0]
    idx_bad = idx.clone()
    idx_bad[1, g_bad, 5] = 600  # == C
    out = torch.full_like(q, float("nan"))
    lse = torch.full((2, 32), float("nan"), dtype=torch.float32, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    clo.clo_hybrid_decode_attn_noalloc(q, cbK, cbV, idx_bad, pK, pV, pid, out, lse=lse,
                                       err_flag=err, num_ctas=7)
    torch.cuda.synchronize()
    assert int(err.item()) & clo.FLAG_BAD_INDEX
    got, lg = out.cpu().numpy().astype(np.float64), lse.cpu().numpy()
    sl = slice(4 * g_bad, 4 * g_bad + 4)
    assert np.all(got[1, sl] == 0) and np.all(np.isneginf(lg[1, sl]))
    mask = np.ones(got.shape[:2], dtype=bool)
    mask[1, sl] = False
    assert_close(got[mask], ref[mask], "noalloc, other groups")

