"""clo_hybrid_decode_layer: one call runs the attention of layer l, the fill
of layer l+1 beside it and the lookup of layer l+2 in its merge launch
("CLO: CPU-Light KVCache Offloading", section 3 Fig. 9).  Each of the three
must match the fp64 oracle as its own call does, and a chain of such calls
must give exactly what the same calls made one after another give: an
attention that read its Cache Buffer before the fill beside the previous
layer's attention had landed would differ."""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
import workloads as wl
from gpu_util import assert_close, assert_lookup_matches, dev, scale_for

pytestmark = pytest.mark.gpu


def _tau(s, cfg):
    return clo.clo_thresholds_host(s, cfg.Hkv, cfg.G, wl.ETA, wl.N_EXP)


def _importance_one_every_other(cfg, seed):
    """s = 1 (tau = eta) on the query heads of every other KV head, U(0, 1)
    elsewhere (tau near -1): with cosines in [0.5, 0.95] some groups miss."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s = rng.uniform(0.0, 1.0, cfg.Hq).astype(np.float32)
    for g in range(0, cfg.Hkv, 2):
        s[g * cfg.G:(g + 1) * cfg.G] = 1.0
    return s


def _lookup_bufs(cfg, d):
    n = cfg.B * cfg.Hkv
    return dict(flag=torch.full((n,), 9, dtype=torch.uint8, device=d),
                sim=torch.full((n,), -9.0, device=d),
                miss=torch.full((n,), -9, dtype=torch.int32, device=d),
                count=torch.full((1,), -9, dtype=torch.int32, device=d))


CASES = [
    # name, small_hybrid overrides, fill source in host memory, num_ctas, fill_ctas
    ("gqa4_token_host", dict(B=2, Hq=32, Hkv=8, T=1000, Np=2), True, 0, 0),
    ("gqa4_compact_hbm", dict(B=2, Hq=32, Hkv=8, T=777, Np=2, addressing="compact"), False, 0, 0),
    ("gqa5_b3_ctas", dict(B=3, Hq=40, Hkv=8, T=700, Np=1), True, 37, 5),
    ("mha_b5_one_fill_cta", dict(B=5, Hq=16, Hkv=16, T=300, Np=3), False, 0, 1),
    ("b20_wide", dict(B=20, Hq=32, Hkv=8, T=200, Np=2), True, 0, 0),
]


@pytest.mark.parametrize("name,kw,host_src,num_ctas,fill_ctas", CASES,
                         ids=[c[0] for c in CASES])
def test_layer_vs_oracle(name, kw, host_src, num_ctas, fill_ctas):
    cfg = wl.small_hybrid(name, qmode="cos", c_lo=0.5, c_hi=0.95, seed=5100 + len(name), **kw)
    orc = oracle.get()
    d = dev()
    # Layer 0: the attention.
    q0, _ = wl.queries_and_labels(cfg, 0, "cpu")
    cbK0, cbV0, idx0 = wl.cache_buffer(cfg, 0, "cpu")
    pK0, pV0 = wl.persistent_cache(cfg, 0, "cpu")
    pid0 = wl.persist_ids(cfg, 0)
    # Layer 1: the fill, from the oracle lookup's miss list of that layer.
    q1, lab1 = wl.queries_and_labels(cfg, 1, "cpu")
    s1 = _importance_one_every_other(cfg, 11)
    tau1 = _tau(s1, cfg)
    pm1 = wl.persist_mask(cfg, 1)
    lk1 = orc.lookup_update(q1.numpy(), lab1.numpy(), s1.astype(np.float64),
                            tau1.astype(np.float64), pm1)
    miss1 = [int(x) for x in lk1["miss_list"]]
    assert miss1, "the case was meant to miss"
    srcK, srcV = wl.full_kv(cfg, 1, "cpu")
    tok, slot = wl.fill_selection(cfg, 1, "cpu")
    cbK1, cbV1, _ = wl.cache_buffer(cfg, 1, "cpu")
    use_slot = None if cfg.addressing == "token" else slot
    # Layer 2: the lookup.
    q2, lab2 = wl.queries_and_labels(cfg, 2, "cpu")
    s2 = _importance_one_every_other(cfg, 12)
    tau2 = _tau(s2, cfg)
    pm2 = wl.persist_mask(cfg, 2)

    # The library: one call.
    out = torch.empty_like(q0, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, 128, num_ctas),
                     dtype=torch.uint8, device=d)
    sK, sV = (srcK.pin_memory(), srcV.pin_memory()) if host_src else (srcK.to(d), srcV.to(d))
    gK1, gV1 = cbK1.to(d), cbV1.to(d)
    ml1 = torch.full((cfg.B * cfg.Hkv,), -5, dtype=torch.int32)
    ml1[:len(miss1)] = torch.tensor(miss1, dtype=torch.int32)
    mc1 = torch.tensor([len(miss1)], dtype=torch.int32)
    fill = (sK, sV, tok.to(d), None if use_slot is None else use_slot.to(d), gK1, gV1,
            ml1.to(d), mc1.to(d))
    glab2 = lab2.to(d)
    r2 = _lookup_bufs(cfg, d)
    lookup = (q2.to(d), glab2, torch.from_numpy(s2).to(d), torch.from_numpy(tau2).to(d),
              torch.from_numpy(pm2).to(d), r2["flag"], r2["sim"], r2["miss"], r2["count"])
    clo.clo_hybrid_decode_layer(q0.to(d), cbK0.to(d), cbV0.to(d), idx0.to(d), pK0.to(d),
                                pV0.to(d), torch.from_numpy(pid0).to(d), out, ws, fill=fill,
                                lookup=lookup, err_flag=err, num_ctas=num_ctas,
                                fill_ctas=fill_ctas)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # The attention of layer 0.
    ref0, _ = orc.hybrid_attn(q0.numpy(), cbK0.numpy(), cbV0.numpy(), idx0.numpy(), pK0.numpy(),
                              pV0.numpy(), pid0, scale_for())
    assert_close(out.cpu().numpy(), ref0, f"{name}: attention")
    # The fill of layer 1, bit for bit.
    rK, rV, rc = orc.fill_cache_buffer(srcK.numpy(), srcV.numpy(), tok.numpy(),
                                       None if use_slot is None else use_slot.numpy(),
                                       cbK1.numpy(), cbV1.numpy(), miss1)
    assert rc == 0
    assert np.array_equal(gK1.cpu().numpy().view(np.uint16), rK), "filled K rows differ"
    assert np.array_equal(gV1.cpu().numpy().view(np.uint16), rV), "filled V rows differ"
    # The lookup of layer 2.
    ref2 = orc.lookup_update(q2.numpy(), lab2.numpy(), s2.astype(np.float64),
                             tau2.astype(np.float64), pm2)
    n = int(r2["count"].item())
    got = dict(flag=r2["flag"].cpu().numpy(), sim=r2["sim"].cpu().numpy(),
               labels=glab2.cpu().numpy(), miss_list=r2["miss"].cpu().numpy()[:max(n, 0)],
               miss_count=n)
    near = assert_lookup_matches(ref2, got, tau2, pm2, cfg.G)
    assert n > 0, "the carried lookup was meant to miss"
    print(f"{name}: filled {len(miss1)} heads, looked up {n} misses, {near} near tau")


def _chain_layers(cfg, L, d, host_src):
    """L layers of distinct buffers on the device (sources of the fill in
    pinned host memory or HBM), with importance s = 1 on every other KV head."""
    layers = []
    for l in range(L):
        q, lab = wl.queries_and_labels(cfg, l, "cpu")
        cbK, cbV, idx = wl.cache_buffer(cfg, l, "cpu")
        pK, pV = wl.persistent_cache(cfg, l, "cpu")
        srcK, srcV = wl.full_kv(cfg, l, "cpu")
        s = _importance_one_every_other(cfg, 300 + l)
        layers.append(dict(
            q=q.to(d), lab0=lab.to(d), cbK0=cbK.to(d), cbV0=cbV.to(d), idx=idx.to(d),
            pK=pK.to(d), pV=pV.to(d), pid=torch.from_numpy(wl.persist_ids(cfg, l)).to(d),
            srcK=srcK.pin_memory() if host_src else srcK.to(d),
            srcV=srcV.pin_memory() if host_src else srcV.to(d),
            w=torch.from_numpy(s).to(d), tau=torch.from_numpy(_tau(s, cfg)).to(d),
            pm=torch.from_numpy(wl.persist_mask(cfg, l)).to(d)))
    return layers


def _fresh(cfg, layers, d):
    """Per-layer state a run writes: labels, Cache Buffer, lookup outputs, output."""
    st = []
    for x in layers:
        st.append(dict(lab=x["lab0"].clone(), cbK=x["cbK0"].clone(), cbV=x["cbV0"].clone(),
                       out=torch.full_like(x["q"], float("nan")), **_lookup_bufs(cfg, d)))
    return st


def _lookup_tuple(x, s):
    return (x["q"], s["lab"], x["w"], x["tau"], x["pm"], s["flag"], s["sim"], s["miss"],
            s["count"])


def _fill_tuple(x, s):
    # Token-addressed: the fill writes each missed head's rows idx[b][g] (the
    # tokens themselves), which that layer's attention then reads.
    return (x["srcK"], x["srcV"], x["idx"], None, s["cbK"], s["cbV"], s["miss"], s["count"])


@pytest.mark.parametrize("host_src,full_wave", [(True, False), (False, False), (True, True)],
                         ids=["host_src", "hbm_src", "host_src_full_wave"])
def test_layer_chain_equals_serial(host_src, full_wave):
    """Five layers.  Serial: per layer lookup, fill, attention, one after
    another.  Pipelined: lookups of layers 0 and 1 and the fill of layer 0
    first, then one clo_hybrid_decode_layer call per layer (attention l, fill
    l+1 beside it, lookup l+2 in its merge launch).  Every output, label,
    lookup result and Cache Buffer must be bit-identical; the attentions use
    the same grid in both.  With full_wave the attention takes every CTA slot,
    so the fill's CTAs find room only as attention CTAs finish (nothing the
    attention does waits for the fill, so the call still completes)."""
    cfg = wl.small_hybrid("chain", B=4, Hq=32, Hkv=8, T=4096, Np=2, qmode="cos", c_lo=0.5,
                          c_hi=0.95, seed=5300)
    d = dev()
    L = 5
    layers = _chain_layers(cfg, L, d, host_src)
    sms = torch.cuda.get_device_properties(d).multi_processor_count
    fill_ctas = 64 if full_wave else 48
    main_ctas = 3 * sms if full_wave else 3 * sms - fill_ctas
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, 128, main_ctas),
                     dtype=torch.uint8, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)

    def attn_args(x, s):
        return (x["q"], s["cbK"], s["cbV"], x["idx"], x["pK"], x["pV"], x["pid"], s["out"], ws)

    serial = _fresh(cfg, layers, d)
    for x, s in zip(layers, serial):
        clo.clo_lookup_update(*_lookup_tuple(x, s))
        clo.clo_fill_cache_buffer(*_fill_tuple(x, s), err_flag=err, num_ctas=fill_ctas)
        clo.clo_hybrid_decode_attn(*attn_args(x, s), err_flag=err, num_ctas=main_ctas)
    pipe = _fresh(cfg, layers, d)
    clo.clo_lookup_update(*_lookup_tuple(layers[0], pipe[0]))
    clo.clo_lookup_update(*_lookup_tuple(layers[1], pipe[1]))
    clo.clo_fill_cache_buffer(*_fill_tuple(layers[0], pipe[0]), err_flag=err,
                              num_ctas=fill_ctas)
    for l in range(L):
        fill = _fill_tuple(layers[l + 1], pipe[l + 1]) if l + 1 < L else None
        look = _lookup_tuple(layers[l + 2], pipe[l + 2]) if l + 2 < L else None
        clo.clo_hybrid_decode_layer(*attn_args(layers[l], pipe[l]), fill=fill, lookup=look,
                                    err_flag=err, num_ctas=main_ctas, fill_ctas=fill_ctas)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    misses = 0
    for l, (a, b) in enumerate(zip(serial, pipe)):
        n = int(a["count"].item())
        misses += n
        assert n == int(b["count"].item()), f"layer {l}: miss count"
        assert torch.equal(a["miss"][:n], b["miss"][:n]), f"layer {l}: miss list"
        for key in ("flag", "sim", "lab", "cbK", "cbV", "out"):
            assert torch.equal(a[key], b[key]), f"layer {l}: {key} differs"
    assert misses > 0
    # And the chain against the oracle on its last layer: lookup, fill, attention.
    orc = oracle.get()
    x = layers[L - 1]
    q, lab = wl.queries_and_labels(cfg, L - 1, "cpu")
    lk = orc.lookup_update(q.numpy(), lab.numpy(), x["w"].cpu().numpy().astype(np.float64),
                           x["tau"].cpu().numpy().astype(np.float64), x["pm"].cpu().numpy())
    srcK, srcV = wl.full_kv(cfg, L - 1, "cpu")
    cbK, cbV, idx = wl.cache_buffer(cfg, L - 1, "cpu")
    rK, rV, rc = orc.fill_cache_buffer(srcK.numpy(), srcV.numpy(), idx.numpy(), None,
                                       cbK.numpy(), cbV.numpy(), lk["miss_list"])
    pK, pV = wl.persistent_cache(cfg, L - 1, "cpu")
    ref, _ = orc.hybrid_attn(q.numpy(), rK, rV, idx.numpy(), pK.numpy(), pV.numpy(),
                             wl.persist_ids(cfg, L - 1), scale_for())
    assert rc == 0
    assert_close(pipe[L - 1]["out"].cpu().numpy(), ref, "last layer of the chain")
    print(f"chain: {misses} misses over {L} layers")


def test_layer_rejects_overlapping_buffers():
    cfg = wl.small_hybrid(B=1, Hq=32, Hkv=8, T=300, Np=2)
    d = dev()
    x = _chain_layers(cfg, 2, d, False)
    st = _fresh(cfg, x, d)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv), dtype=torch.uint8,
                     device=d)
    args = (x[0]["q"], st[0]["cbK"], st[0]["cbV"], x[0]["idx"], x[0]["pK"], x[0]["pV"],
            x[0]["pid"], st[0]["out"], ws)
    # The fill writing the Cache Buffer this attention reads.
    with pytest.raises(clo.CloError) as e:
        clo.clo_hybrid_decode_layer(*args, fill=_fill_tuple(x[0], st[0]))
    assert e.value.status == clo.CLO_ERR_INVALID_ARG
    # The fill reading the miss list the carried lookup writes.
    with pytest.raises(clo.CloError) as e:
        clo.clo_hybrid_decode_layer(*args, fill=_fill_tuple(x[1], st[1]),
                                    lookup=_lookup_tuple(x[1], st[1]))
    assert e.value.status == clo.CLO_ERR_INVALID_ARG
    # A lookup of another shape.
    with pytest.raises(clo.CloError):
        bad = list(_lookup_tuple(x[1], st[1]))
        bad[0] = bad[0][:, :16].contiguous()
        bad[1] = bad[1][:, :16].contiguous()
        clo.clo_hybrid_decode_layer(*args, lookup=tuple(bad))


def test_layer_fill_bad_rows_flagged_and_nothing_else_changes():
    """A token outside [0, T) in a missed head's selection: the fill flags it
    in the layer call's err_flag and skips that row; the other rows and the
    attention beside it are as the oracle has them."""
    cfg = wl.small_hybrid(B=2, Hq=16, Hkv=4, T=500, Np=1, addressing="compact")
    orc = oracle.get()
    d = dev()
    q0, _ = wl.queries_and_labels(cfg, 0, "cpu")
    cbK0, cbV0, idx0 = wl.cache_buffer(cfg, 0, "cpu")
    pK0, pV0 = wl.persistent_cache(cfg, 0, "cpu")
    pid0 = wl.persist_ids(cfg, 0)
    srcK, srcV = wl.full_kv(cfg, 1, "cpu")
    tok, slot = wl.fill_selection(cfg, 1, "cpu")
    tok = tok.clone()
    tok[1, 2, 7] = cfg.T
    cbK1, cbV1, _ = wl.cache_buffer(cfg, 1, "cpu")
    miss = [6, 1]
    gK1, gV1 = cbK1.to(d), cbV1.to(d)
    out = torch.empty_like(q0, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv), dtype=torch.uint8,
                     device=d)
    fill = (srcK.to(d), srcV.to(d), tok.to(d), slot.to(d), gK1, gV1,
            torch.tensor(miss, dtype=torch.int32, device=d),
            torch.tensor([len(miss)], dtype=torch.int32, device=d))
    clo.clo_hybrid_decode_layer(q0.to(d), cbK0.to(d), cbV0.to(d), idx0.to(d), pK0.to(d),
                                pV0.to(d), torch.from_numpy(pid0).to(d), out, ws, fill=fill,
                                err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & clo.FLAG_BAD_INDEX
    rK, rV, rc = orc.fill_cache_buffer(srcK.numpy(), srcV.numpy(), tok.numpy(), slot.numpy(),
                                       cbK1.numpy(), cbV1.numpy(), miss)
    assert rc == oracle.BAD_INDEX
    assert np.array_equal(gK1.cpu().numpy().view(np.uint16), rK)
    assert np.array_equal(gV1.cpu().numpy().view(np.uint16), rV)
    ref0, _ = orc.hybrid_attn(q0.numpy(), cbK0.numpy(), cbV0.numpy(), idx0.numpy(), pK0.numpy(),
                              pV0.numpy(), pid0, scale_for())
    assert_close(out.cpu().numpy(), ref0, "attention beside a bad fill")


def test_layer_empty_batch_and_empty_fill():
    cfg = wl.small_hybrid(B=1, Hq=32, Hkv=8, T=300, Np=2)
    d = dev()
    x = _chain_layers(cfg, 3, d, False)
    st = _fresh(cfg, x, d)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv), dtype=torch.uint8,
                     device=d)
    # A fill whose miss count is 0 moves nothing; the attention and lookup run as usual.
    st[1]["count"].zero_()
    cb1 = st[1]["cbK"].clone()
    clo.clo_hybrid_decode_layer(x[0]["q"], st[0]["cbK"], st[0]["cbV"], x[0]["idx"], x[0]["pK"],
                                x[0]["pV"], x[0]["pid"], st[0]["out"], ws,
                                fill=_fill_tuple(x[1], st[1]), lookup=_lookup_tuple(x[2], st[2]))
    ref_out = torch.empty_like(x[0]["q"])
    clo.clo_hybrid_decode_attn(x[0]["q"], st[0]["cbK"], st[0]["cbV"], x[0]["idx"], x[0]["pK"],
                               x[0]["pV"], x[0]["pid"], ref_out, ws)
    torch.cuda.synchronize()
    assert torch.equal(st[1]["cbK"], cb1)
    assert int(st[2]["count"].item()) >= 0
    # 50 tiles: both grids are capped at one tile a warp (12 CTAs).
    assert torch.equal(st[0]["out"], ref_out)
    # An empty batch: the carried lookup's miss count is written, nothing else.
    q = torch.empty((0, cfg.Hq, 128), dtype=torch.float16, device=d)
    cnt = torch.full((1,), 7, dtype=torch.int32, device=d)
    z8 = torch.empty(0, dtype=torch.uint8, device=d)
    z32 = torch.empty(0, dtype=torch.float32, device=d)
    zi = torch.empty(0, dtype=torch.int32, device=d)
    lk = (q, q.clone(), x[2]["w"], x[2]["tau"], x[2]["pm"], z8, z32, zi, cnt)
    empty_cb = torch.empty((0, cfg.Hkv, cfg.C, 128), dtype=torch.float16, device=d)
    clo.clo_hybrid_decode_layer(q, empty_cb, empty_cb.clone(),
                                torch.empty((0, cfg.Hkv, cfg.k), dtype=torch.int32, device=d),
                                None, None, None, q.clone(), ws, lookup=lk)
    torch.cuda.synchronize()
    assert int(cnt.item()) == 0


def test_layer_calls_captured_in_a_graph():
    """Three chained layer calls captured into a CUDA graph and replayed give
    exactly what the same calls give issued one by one: the fill beside each
    attention and the programmatic-launch edges survive capture."""
    cfg = wl.small_hybrid("graph_chain", B=2, Hq=32, Hkv=8, T=2048, Np=2, qmode="cos", c_lo=0.5,
                          c_hi=0.95, seed=5400)
    d = dev()
    L = 4
    layers = _chain_layers(cfg, L, d, True)
    ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv), dtype=torch.uint8,
                     device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)

    def prologue(st):
        clo.clo_lookup_update(*_lookup_tuple(layers[0], st[0]))
        clo.clo_lookup_update(*_lookup_tuple(layers[1], st[1]))
        clo.clo_fill_cache_buffer(*_fill_tuple(layers[0], st[0]), err_flag=err)

    def calls(st):
        for l in range(L - 1):
            x = layers[l]
            fill = _fill_tuple(layers[l + 1], st[l + 1])
            look = _lookup_tuple(layers[l + 2], st[l + 2]) if l + 2 < L else None
            clo.clo_hybrid_decode_layer(x["q"], st[l]["cbK"], st[l]["cbV"], x["idx"], x["pK"],
                                        x["pV"], x["pid"], st[l]["out"], ws, fill=fill,
                                        lookup=look, err_flag=err)

    eager = _fresh(cfg, layers, d)
    prologue(eager)
    calls(eager)
    torch.cuda.synchronize()
    graph = _fresh(cfg, layers, d)
    prologue(graph)
    torch.cuda.synchronize()
    # Warm the calls once on a side stream (kernel attributes are set outside capture).
    warm = _fresh(cfg, layers, d)
    prologue(warm)
    calls(warm)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            calls(graph)
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(L):
        for key in ("out", "cbK", "cbV", "lab", "flag", "sim"):
            if key == "out" and l == L - 1:
                continue  # the last layer's attention is not in the captured calls
            assert torch.equal(eager[l][key], graph[l][key]), f"layer {l}: {key}"
