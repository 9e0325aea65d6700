"""Prepared calls and the host-buffer copy call (GPU).

A prepared call is checked once and re-issued on the same buffers; it must
give exactly what the direct call gives, also after the inputs change in
place.  clo_copy_async must move bytes between pinned host memory and the GPU
unchanged, in order.  Both are what the end-to-end timing of the benchmark
uses.
"""
import numpy as np
import pytest
import torch

import offloaded_kv_decode_gb300 as clo
import workloads as wl
from gpu_util import dev

pytestmark = pytest.mark.gpu


def test_copy_async_round_trip():
    g = torch.Generator().manual_seed(5)
    h_a = torch.randint(0, 2 ** 15, (3000,), dtype=torch.int16, generator=g).pin_memory()
    h_b = torch.randn(517, generator=g).pin_memory()
    d_a = torch.empty(3000, dtype=torch.int16, device=dev())
    d_b = torch.empty(517, device=dev())
    empty_h = torch.empty(0).pin_memory()
    empty_d = torch.empty(0, device=dev())
    clo.clo_copy_async([(d_a, h_a), (empty_d, empty_h), (d_b, h_b)])
    back_a = torch.empty_like(h_a).pin_memory()
    back_b = torch.empty_like(h_b).pin_memory()
    d_b.mul_(2.0)  # ordered on the stream between the two copy calls
    clo.clo_copy_async([(back_a, d_a), (back_b, d_b)])
    torch.cuda.synchronize()
    assert torch.equal(back_a, h_a)
    assert torch.equal(back_b, h_b * 2.0)


def test_copy_async_many_large_and_mixed():
    """More copies than one launch takes (20), one of 40 MB (many CTAs), and
    unaligned sizes (copy-engine copies) between them, in both directions."""
    g = torch.Generator().manual_seed(6)
    sizes = [16 * (i + 1) for i in range(19)] + [40 << 20]
    sizes[7] = 1001  # not a multiple of 16 bytes
    hs = [torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory() for n in sizes]
    ds = [torch.empty(n, dtype=torch.uint8, device=dev()) for n in sizes]
    clo.clo_copy_async(list(zip(ds, hs)))
    backs = [torch.empty_like(h).pin_memory() for h in hs]
    clo.clo_copy_async(list(zip(backs, ds)))
    torch.cuda.synchronize()
    for h, d, b in zip(hs, ds, backs):
        assert torch.equal(d.cpu(), h)
        assert torch.equal(b, h)


def test_copy_async_unaligned_ends():
    """Ends off the 16-byte grid: small copies go byte by byte through the
    kernel, a large one (past 64 KiB) through the copy engine; both directions."""
    g = torch.Generator().manual_seed(7)
    sizes = [1, 4, 13, 4099, 70000]
    hs = [torch.randint(0, 256, (n + 3,), dtype=torch.uint8, generator=g).pin_memory()
          for n in sizes]
    ds = [torch.zeros(n + 5, dtype=torch.uint8, device=dev()) for n in sizes]
    clo.clo_copy_async([(d[1:1 + n], h[3:3 + n]) for d, h, n in zip(ds, hs, sizes)])
    backs = [torch.zeros(n + 2, dtype=torch.uint8).pin_memory() for n in sizes]
    clo.clo_copy_async([(b[2:2 + n], d[1:1 + n]) for b, d, n in zip(backs, ds, sizes)])
    torch.cuda.synchronize()
    for h, d, b, n in zip(hs, ds, backs, sizes):
        dc = d.cpu()
        assert torch.equal(dc[1:1 + n], h[3:3 + n])
        assert dc[0] == 0 and torch.all(dc[1 + n:] == 0)  # nothing written outside the copy
        assert torch.equal(b[2:2 + n], h[3:3 + n])
        assert torch.all(b[:2] == 0)


def test_copy_lists_may_not_overlap():
    h = torch.zeros(64, dtype=torch.uint8).pin_memory()
    d = torch.zeros(128, dtype=torch.uint8, device=dev())
    with pytest.raises(clo.CloError):
        clo.clo_copy_async([(d[:64], h), (d[32:96], h)])
    # reads may overlap reads: one source into two places
    h[:] = torch.arange(64, dtype=torch.uint8)
    clo.clo_copy_async([(d[:64], h), (d[64:], h)])
    torch.cuda.synchronize()
    assert torch.equal(d[:64].cpu(), h) and torch.equal(d[64:].cpu(), h)


def test_copy_pairs_device_or_pinned():
    """Device-to-device copies are made too (a caller restoring state between
    steps); host-to-host and mismatched sizes are refused."""
    src = torch.arange(1000, dtype=torch.int32, device=dev())
    d = torch.zeros(1000, dtype=torch.int32, device=dev())
    clo.clo_copy_async([(d, src)])
    torch.cuda.synchronize()
    assert torch.equal(d, src)
    with pytest.raises(clo.CloError):
        clo.prepare_copies([(torch.empty(4).pin_memory(), torch.empty(4).pin_memory())])
    with pytest.raises(clo.CloError):
        clo.prepare_copies([(torch.empty(4, device=dev()), torch.empty(5).pin_memory())])


def _layer(cfg, layer):
    q, lab = wl.queries_and_labels(cfg, layer, dev())
    cbK, cbV, idx = wl.cache_buffer(cfg, layer, dev())
    pK, pV = wl.persistent_cache(cfg, layer, dev())
    n = cfg.B * cfg.Hkv
    return dict(q=q, labels=lab, cbK=cbK, cbV=cbV, idx=idx, pK=pK, pV=pV,
                pid=torch.from_numpy(wl.persist_ids(cfg, layer)).to(dev()),
                pmask=torch.from_numpy(wl.persist_mask(cfg, layer)).to(dev()),
                w=torch.from_numpy(wl.importance(cfg, layer)).to(dev()),
                tau=torch.full((cfg.Hkv,), 0.85, dtype=torch.float32, device=dev()),
                out=torch.empty_like(q),
                flag=torch.empty(n, dtype=torch.uint8, device=dev()),
                sim=torch.empty(n, dtype=torch.float32, device=dev()),
                miss=torch.empty(n, dtype=torch.int32, device=dev()),
                nmiss=torch.zeros(1, dtype=torch.int32, device=dev()))


def _fused_args(a, b, ws):
    return (a["q"], a["cbK"], a["cbV"], a["idx"], a["pK"], a["pV"], a["pid"], a["out"], ws,
            b["q"], b["labels"], b["w"], b["tau"], b["pmask"], b["flag"], b["sim"], b["miss"],
            b["nmiss"])


def test_prepared_fused_call_equals_direct_call():
    cfg = wl.small_hybrid(B=3, T=1500)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv), dtype=torch.uint8,
                     device=dev())
    a, b = _layer(cfg, 0), _layer(cfg, 1)
    a2, b2 = ({k: v.clone() for k, v in x.items()} for x in (a, b))
    call = clo.prepare_hybrid_decode_attn_lookup(*_fused_args(a, b, ws))
    for rep in range(2):
        if rep == 1:  # new contents in place: the prepared call reads them
            for x in (a, a2):
                x["q"].copy_(torch.flip(a2["q"], dims=[1]))
            for x in (b, b2):
                x["q"].copy_(-b2["q"])
        call()
        torch.cuda.synchronize()
        clo.clo_hybrid_decode_attn_lookup(*_fused_args(a2, b2, ws))
        torch.cuda.synchronize()
        for key in ("out",):
            assert torch.equal(a[key], a2[key]), key
        for key in ("labels", "flag", "sim", "nmiss"):
            assert torch.equal(b[key], b2[key]), key
        m = int(b["nmiss"].item())
        assert torch.equal(b["miss"][:m], b2["miss"][:m])
    assert int(b["nmiss"].item()) > 0  # the negated queries miss


def test_prepared_thresholds_and_paged_equal_direct_calls():
    s = torch.rand(64, device=dev())
    t1 = torch.empty(16, device=dev())
    t2 = torch.empty(16, device=dev())
    clo.prepare_thresholds(s, t1, 4, 0.8, 3.0)()
    clo.clo_thresholds(s, t2, 4, 0.8, 3.0)
    pc = wl.small_paged(B=5)
    q, kc, vc, bt, ctx = wl.paged_inputs(pc, dev())
    ws = torch.empty(clo.clo_paged_workspace_size(pc.B, pc.Hq, pc.Hkv), dtype=torch.uint8,
                     device=dev())
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    clo.prepare_paged_decode_attn(q, kc, vc, bt, ctx, o1, ws)()
    torch.cuda.synchronize()
    clo.clo_paged_decode_attn(q, kc, vc, bt, ctx, o2, ws)
    torch.cuda.synchronize()
    assert torch.equal(t1, t2)
    assert torch.equal(o1, o2)
