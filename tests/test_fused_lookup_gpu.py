"""clo_hybrid_decode_attn_lookup: the attention of one layer and the lookup
of the next in one launch sequence must give exactly what the two separate
calls give, and the carried lookup must match the fp64 oracle bit for bit on
inputs where it misses (label replacement and the cross-CTA ordered miss
list inside the merge launch's cluster)."""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
import workloads as wl
from gpu_util import assert_close, assert_lookup_matches, dev, scale_for

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


# ---------------------------------------------------------------- carried lookup vs the oracle

def _next_importance(cfg, mode, seed):
    """Importance scores of the next layer's query heads.  s = 1 puts a KV
    head's threshold at eta (CLO section 4, check 2: lambda = 1 gives
    tau = eta), so with query/label cosines around 0.5-0.95 a good share of
    those groups miss.  "all_one": every head; "half_one": the query heads of
    every other KV head, the rest drawn from U(0, 1) (tau near -1: hits)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s = rng.uniform(0.0, 1.0, cfg.Hq).astype(np.float32)
    if mode == "all_one":
        s[:] = 1.0
    else:
        for g in range(0, cfg.Hkv, 2):
            s[g * cfg.G:(g + 1) * cfg.G] = 1.0
    return s


def fused_lookup_vs_oracle(cfg, s_next, num_ctas=0, check_attn=True):
    """Runs clo_hybrid_decode_attn_lookup (attention of layer 0, lookup of
    layer 1) and compares its lookup outputs with oracle_lookup_update.  The
    next layer's queries and labels are drawn on the CPU (reproducible here)
    and copied over; tau comes from the library (clo_thresholds_host)."""
    d = dev()
    cur = _layer(cfg, 0, d)
    qn, labn = wl.queries_and_labels(cfg, 1, "cpu")
    tau = clo.clo_thresholds_host(s_next, cfg.Hkv, cfg.G, wl.ETA, wl.N_EXP)
    pm = wl.persist_mask(cfg, 1)
    ref = oracle.get().lookup_update(qn.numpy(), labn.numpy(), s_next.astype(np.float64),
                                     tau.astype(np.float64), pm)
    lab = labn.to(d)
    r = _outs(cfg, d)
    has_cb = cfg.Np < cfg.Hkv
    cb = (cur["cbK"], cur["cbV"], cur["idx"]) if has_cb else (None, None, None)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, 128, num_ctas),
                     dtype=torch.uint8, device=d)
    out = torch.empty_like(cur["q"])
    err = torch.zeros(1, dtype=torch.int32, device=d)
    clo.clo_hybrid_decode_attn_lookup(cur["q"], *cb, cur["pK"], cur["pV"], cur["pid"], out, ws,
                                      qn.to(d), lab, torch.from_numpy(s_next).to(d),
                                      torch.from_numpy(tau).to(d), torch.from_numpy(pm).to(d),
                                      r["flag"], r["sim"], r["miss"], r["count"], err_flag=err,
                                      num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    n = int(r["count"].item())
    got = dict(flag=r["flag"].cpu().numpy(), sim=r["sim"].cpu().numpy(),
               labels=lab.cpu().numpy(), miss_list=r["miss"].cpu().numpy()[:max(n, 0)],
               miss_count=n)
    near = assert_lookup_matches(ref, got, tau, pm, cfg.G)
    assert ref["miss_count"] > 0 and n > 0, "the case was meant to miss"
    assert n < int((pm == 0).sum()) * cfg.B, "the case was meant to hit too"
    # Persistent heads are never looked up: flag 2, labels untouched.
    fl = got["flag"].reshape(cfg.B, cfg.Hkv)
    assert np.all(fl[:, pm != 0] == 2)
    if check_attn and cfg.T <= 4096:
        q = cur["q"].cpu().numpy()
        cbn = [x.cpu().numpy() for x in cb] if has_cb else \
            [np.zeros((cfg.B, cfg.Hkv, 1, 128), np.float16)] * 2 + \
            [np.zeros((cfg.B, cfg.Hkv, 0), np.int32)]
        ref_o, _ = oracle.get().hybrid_attn(q, *cbn, cur["pK"].cpu().numpy(),
                                            cur["pV"].cpu().numpy(), cur["pid"].cpu().numpy(),
                                            scale_for())
        assert_close(out.cpu().numpy(), ref_o, "attention beside the carried lookup")
    return ref, got, near


MISS_CASES = [
    # name, small_hybrid overrides, importance mode, CTAs of the main kernel
    ("gqa4_b2", dict(B=2, Hq=32, Hkv=8, T=1000, Np=2), "all_one", 0),
    ("gqa5_b3", dict(B=3, Hq=40, Hkv=8, T=700, Np=1), "half_one", 0),
    ("one_cta", dict(B=1, Hq=32, Hkv=8, T=300, Np=2), "half_one", 1),
    ("b20_wide", dict(B=20, Hq=32, Hkv=8, T=200, Np=2), "all_one", 0),
    ("b64_gqa8", dict(B=64, Hq=64, Hkv=8, T=64, Np=1), "half_one", 37),
    ("mha_b5", dict(B=5, Hq=16, Hkv=16, T=300, Np=3), "all_one", 0),
    # 96 groups: the lookup runs in a launch of its own beside the main kernel,
    # and with one attention CTA no merge launch follows it.
    ("b12_beside_one_cta", dict(B=12, Hq=32, Hkv=8, T=300, Np=2), "half_one", 1),
]


@pytest.mark.parametrize("name,kw,mode,num_ctas", MISS_CASES, ids=[c[0] for c in MISS_CASES])
def test_fused_lookup_misses_vs_oracle(name, kw, mode, num_ctas):
    cfg = wl.small_hybrid(name, qmode="cos", c_lo=0.5, c_hi=0.95, seed=4400 + len(name), **kw)
    s_next = _next_importance(cfg, mode, 77 + len(name))
    ref, got, near = fused_lookup_vs_oracle(cfg, s_next, num_ctas)
    ngroups = cfg.B * cfg.Hkv
    ranks = {int(x) * 8 // ngroups for x in got["miss_list"]}
    if ngroups >= 16:
        assert len(ranks) >= 2, "misses should come from several CTAs of the lookup cluster"
    print(f"{name}: {got['miss_count']} misses of {ngroups} groups over cluster ranks "
          f"{sorted(ranks)}; {near} near tau")


def test_fused_lookup_misses_full_step_shape():
    """The batch-1, 128K-context Llama3-8B layer shape with every next-layer
    head at tau = eta: its six looked-up groups split into hits and misses."""
    cfg = wl.CONFIGS["llama3_8b_step_b1_128k"]
    s_next = _next_importance(cfg, "all_one", 5)
    ref, got, near = fused_lookup_vs_oracle(cfg, s_next, 0, check_attn=False)
    print(f"B1 128K: {got['miss_count']} misses; {near} near tau")



def test_fused_lookup_maximum_groups_vs_oracle():
    """The carried lookup at its largest size, 65536 groups (8192 batch rows x
    8 KV heads), beside an attention over the same batch (32-token contexts):
    the merge launch then has 65536 blocks ahead of the lookup's cluster."""
    cfg = wl.small_hybrid("max_groups", B=8192, Hq=32, Hkv=8, T=32, Np=2, qmode="cos",
                          c_lo=0.5, c_hi=0.95, seed=9090)
    s_next = _next_importance(cfg, "half_one", 11)
    ref, got, near = fused_lookup_vs_oracle(cfg, s_next, 0)
    print(f"65536 groups carried: {got['miss_count']} misses, {near} near tau")
