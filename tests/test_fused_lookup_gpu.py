"""clo_hybrid_decode_attn_lookup: the attention of one layer and the lookup
of the next in one launch sequence must give exactly what the two separate
calls give (and so what the oracle gives)."""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
import workloads as wl
from gpu_util import assert_close, dev, scale_for

pytestmark = pytest.mark.gpu


def _layer(cfg, layer, d):
    q, lab = wl.queries_and_labels(cfg, layer, d)
    cbK, cbV, idx = wl.cache_buffer(cfg, layer, d)
    pK, pV = wl.persistent_cache(cfg, layer, d)
    pid = torch.from_numpy(wl.persist_ids(cfg, layer)).to(d)
    return dict(q=q, lab=lab, cbK=cbK, cbV=cbV, idx=idx, pK=pK, pV=pV, pid=pid)


def _lookup_inputs(cfg, layer, d):
    s = wl.importance(cfg, layer)
    tau = oracle.get().thresholds(s.astype(np.float64), cfg.Hkv, cfg.G, wl.ETA,
                                  wl.N_EXP).astype(np.float32)
    return (torch.from_numpy(s).to(d), torch.from_numpy(tau).to(d),
            torch.from_numpy(wl.persist_mask(cfg, layer)).to(d))


def _outs(cfg, d):
    n = cfg.B * cfg.Hkv
    return dict(flag=torch.full((n,), 9, dtype=torch.uint8, device=d),
                sim=torch.full((n,), -9.0, device=d),
                miss=torch.full((n,), -9, dtype=torch.int32, device=d),
                count=torch.full((1,), -9, dtype=torch.int32, device=d))


@pytest.mark.parametrize("name,kw,num_ctas", [
    ("gqa4", dict(B=2, Hq=32, Hkv=8, T=1000, Np=2, qmode="cos", c_lo=0.5, c_hi=0.95), 0),
    ("gqa5_b3", dict(B=3, Hq=40, Hkv=8, T=700, Np=1, qmode="cos", c_lo=0.5, c_hi=0.95), 0),
    ("one_cta", dict(B=1, Hq=32, Hkv=8, T=300, Np=2, qmode="cos", c_lo=0.5, c_hi=0.95), 1),
    ("all_persistent", dict(B=2, Hq=16, Hkv=4, T=200, Np=4), 0),
])
def test_fused_equals_separate(name, kw, num_ctas):
    cfg = wl.small_hybrid(**kw)
    d = dev()
    cur = _layer(cfg, 0, d)
    nxt = _layer(cfg, 1, d)
    w, tau, pm = _lookup_inputs(cfg, 1, d)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, 128, num_ctas),
                     dtype=torch.uint8, device=d)
    has_cb = cfg.Np < cfg.Hkv
    cb = (cur["cbK"], cur["cbV"], cur["idx"]) if has_cb else (None, None, None)
    # Separate calls.
    out_a = torch.empty_like(cur["q"])
    lab_a = nxt["lab"].clone()
    ra = _outs(cfg, d)
    clo.clo_hybrid_decode_attn(cur["q"], *cb, cur["pK"], cur["pV"], cur["pid"], out_a, ws,
                               num_ctas=num_ctas)
    clo.clo_lookup_update(nxt["q"], lab_a, w, tau, pm, ra["flag"], ra["sim"], ra["miss"],
                          ra["count"])
    # One fused call.
    out_b = torch.empty_like(cur["q"])
    lab_b = nxt["lab"].clone()
    rb = _outs(cfg, d)
    clo.clo_hybrid_decode_attn_lookup(cur["q"], *cb, cur["pK"], cur["pV"], cur["pid"], out_b, ws,
                                      nxt["q"], lab_b, w, tau, pm, rb["flag"], rb["sim"],
                                      rb["miss"], rb["count"], num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b), "attention output differs"
    assert torch.equal(lab_a, lab_b), "labels differ"
    n = int(ra["count"].item())
    assert n == int(rb["count"].item()) and n >= 0
    for key in ("flag", "sim"):
        assert torch.equal(ra[key], rb[key]), key
    assert torch.equal(ra["miss"][:n], rb["miss"][:n])
    # And the attention against the oracle.
    ref, _ = oracle.get().hybrid_attn(
        cur["q"].cpu().numpy(),
        *(x.cpu().numpy() for x in (cb if has_cb else
          (torch.zeros(cfg.B, cfg.Hkv, 1, 128, dtype=torch.float16),) * 2 +
          (torch.zeros(cfg.B, cfg.Hkv, 0, dtype=torch.int32),))),
        cur["pK"].cpu().numpy(), cur["pV"].cpu().numpy(), cur["pid"].cpu().numpy(), scale_for())
    assert_close(out_b.cpu().numpy(), ref, name)


def test_fused_full_step_size():
    """The batch-1 128K step layer shape: fused equals separate."""
    cfg = wl.CONFIGS["llama3_8b_step_b1_128k"]
    d = dev()
    cur = _layer(cfg, 0, d)
    nxt = _layer(cfg, 1, d)
    w, tau, pm = _lookup_inputs(cfg, 1, d)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv), dtype=torch.uint8,
                     device=d)
    outs = []
    for fused in (False, True):
        out = torch.empty_like(cur["q"])
        lab = nxt["lab"].clone()
        r = _outs(cfg, d)
        if fused:
            clo.clo_hybrid_decode_attn_lookup(cur["q"], cur["cbK"], cur["cbV"], cur["idx"],
                                              cur["pK"], cur["pV"], cur["pid"], out, ws, nxt["q"],
                                              lab, w, tau, pm, r["flag"], r["sim"], r["miss"],
                                              r["count"])
        else:
            clo.clo_hybrid_decode_attn(cur["q"], cur["cbK"], cur["cbV"], cur["idx"], cur["pK"],
                                       cur["pV"], cur["pid"], out, ws)
            clo.clo_lookup_update(nxt["q"], lab, w, tau, pm, r["flag"], r["sim"], r["miss"],
                                  r["count"])
        torch.cuda.synchronize()
        outs.append((out, lab, r))
    (oa, la, ra), (ob, lb, rb) = outs
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    assert torch.equal(ra["flag"], rb["flag"]) and torch.equal(ra["count"], rb["count"])
