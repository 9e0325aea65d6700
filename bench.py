#!/usr/bin/env python3
"""Benchmark of the CLO decode hot path on GB300: fused lookup + label update
and hybrid (Cache Buffer + Persistent Cache) decode attention, or the paged
dense decode attention, through libclo.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one decode step of the workload: the thresholds launch, then for
every layer the hybrid attention with the next layer's fused lookup + label
update carried in the same launches (--lookup-schedule picks the
alternatives); for the paged workload one paged attention call; for the
fill and top-k workloads one miss-path fill or one top-k retrieval of a
layer.  Inputs are seeded synthetic tensors (workloads/), resident in device
memory (the fill's full KV copy in pinned host memory for the host-link
variant) before timing.  Every workload cycles over physical buffer sets so
that the bytes between two reads of the same address exceed the 129 MB L2
(no L2 flush is needed).

The timed steps replay a CUDA graph of several consecutive steps (a multiple
of the buffer phases that divides K, at most 16; one graph per step when there
is none), so the kernels chain across steps inside a replay; K steps are timed
with CUDA events between a barrier + synchronize on both sides, repeated in
rounds of exactly K steps until about a second of GPU time has been covered
(so the clock sampler sees the load); the median round is reported.  A second copy of each graph with CUDA events around the main
kernel (the attention's split kernel, the fill kernel or the top-k scoring
kernel) is replayed after every timed round; those events give the kernel's
duration for the roofline line.

Multi-GPU (torchrun): every rank runs an independent replica on its own
inputs (the path has no exchange step), value = bytes of all ranks / max time.

--impl reference times the fp64 CPU oracle (oracle/, test infrastructure) on
a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = ("µs per layer-step and achieved HBM GB/s (% of GB300 peak) for lookup+attention")
DEFAULT_WORKLOAD = "qwen25_14b_step_b16_64k"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal
L2_BYTES = 129 * 2 ** 20
HALF = 2


# ---------------------------------------------------------------- byte accounting

# A lookup carried by an attention call rides in its merge launch for up to
# this many (batch row, KV head) groups, else in a launch of its own
# (clo_hybrid_decode_attn_lookup, include/clo.h).
LOOKUP_IN_MERGE_MAX_GROUPS = 64


def hybrid_attn_bytes(cfg) -> int:
    """Algorithmic bytes of one hybrid attention launch (one layer): the
    selected Cache Buffer rows and the full persistent rows (K and V), the
    indices, q in and the output."""
    rows = cfg.B * ((cfg.Hkv - cfg.Np) * cfg.k + cfg.Np * cfg.T)
    kv = rows * cfg.d * HALF * 2
    idx = cfg.B * (cfg.Hkv - cfg.Np) * cfg.k * 4
    qo = 2 * cfg.B * cfg.Hq * cfg.d * HALF
    return kv + idx + qo


def hybrid_lookup_bytes(cfg) -> int:
    """Lookup: read q and labels, write flag + sim (label writes on misses are
    data dependent and not counted)."""
    return 2 * cfg.B * cfg.Hq * cfg.d * HALF + cfg.B * cfg.Hkv * 5


def paged_bytes(pc, ctx: np.ndarray) -> int:
    kv = int(ctx.astype(np.int64).sum()) * pc.Hkv * pc.d * HALF * 2
    blocks = int(((ctx.astype(np.int64) + pc.block_size - 1) // pc.block_size).sum()) * 4
    qo = 2 * pc.B * pc.Hq * pc.d * HALF
    return kv + blocks + qo + pc.B * 4


# ---------------------------------------------------------------- workloads (GPU)

class E2ECopies:
    """The host-buffer copies of an end-to-end loop over fixed buffers: each
    step copies its inputs in; the previous step's results go out in the same
    clo_copy_async call (they are adjacent on the stream and touch disjoint
    memory), and finish() copies the last step's results out."""

    def __init__(self, clo, ins, outs):
        self.only_in = clo.prepare_copies(ins)
        self.out_in = clo.prepare_copies(list(outs) + list(ins))
        self.only_out = clo.prepare_copies(outs)
        self.pending = False

    def step_in(self):
        (self.out_in if self.pending else self.only_in)()
        self.pending = True

    def finish(self):
        if self.pending:
            self.only_out()
            self.pending = False


PIPELINED_E2E = ("public API: prepared calls and clo_copy_async to and from pinned host buffers, "
                 "issued from Python each step; a step's result copy shares one call with the next "
                 "step's input copy, the last step's results are copied out inside the timed region")


class HybridWorkload:
    kind = "hybrid"
    e2e_path = PIPELINED_E2E

    def __init__(self, cfg, dev, rank: int, replicas: int = 0, schedule: str = "fused",
                 side_ctas=None):
        import torch
        import offloaded_kv_decode_gb300 as clo

        self.clo, self.torch = clo, torch
        self.cfg = cfg
        self.schedule = schedule
        self.side = torch.cuda.Stream(dev)
        self.L = cfg.L
        per_layer = hybrid_attn_bytes(cfg)
        if cfg.L > 1:
            self.n_inst = cfg.ring if cfg.ring else cfg.L
        elif replicas > 0:
            self.n_inst = replicas
        else:  # one layer: enough replicas that a buffer is re-read only after > 1 GB
            self.n_inst = int(min(8, max(2, math.ceil(2 ** 30 / per_layer))))
        self.inst = []
        s_all = []
        n = cfg.B * cfg.Hkv
        # The queries of all buffer sets sit in one device buffer, and so do
        # their results: each set's attention output, then its lookup outputs
        # (sim, miss list, miss count, flags), padded to 256 bytes.  The host
        # moves a step's inputs in and its results out with one copy each.
        out_bytes = cfg.B * cfg.Hq * cfg.d * HALF
        res_bytes = 9 * n + 4
        row = -(-(out_bytes + res_bytes) // 256) * 256
        self.q_all = torch.empty((self.n_inst, cfg.B, cfg.Hq, cfg.d), dtype=torch.float16,
                                 device=dev)
        self.io_all = torch.zeros((self.n_inst, row), dtype=torch.uint8, device=dev)
        # With label_reset, every set's labels sit in one buffer and each step
        # starts by copying the drawn labels back over it, so the same groups
        # miss every step (a miss replaces the group's labels with q).
        self.lab_all = torch.empty((self.n_inst, cfg.B, cfg.Hq, cfg.d), dtype=torch.float16,
                                   device=dev)
        for i in range(self.n_inst):
            li = i + 1000 * rank
            res = self.io_all[i, out_bytes:out_bytes + res_bytes]
            q0, lab0 = wl.queries_and_labels(cfg, li, dev)
            q = self.q_all[i]
            q.copy_(q0)
            lab = self.lab_all[i]
            lab.copy_(lab0)
            del q0, lab0
            has_cb = cfg.Np < cfg.Hkv
            cbK, cbV, idx = wl.cache_buffer(cfg, li, dev) if has_cb else (None, None, None)
            pK, pV = wl.persistent_cache(cfg, li, dev) if cfg.Np > 0 else (None, None)
            srcK = srcV = None
            if cfg.miss_fill:
                # The full KV copy the missed heads' rows come from; the fill
                # writes each missed head's rows idx[b][g] (the token itself,
                # token-addressed), which the next attention then reads.
                srcK, srcV = wl.full_kv(cfg, li, dev)
                if cfg.miss_fill == "host":
                    srcK, srcV = srcK.cpu().pin_memory(), srcV.cpu().pin_memory()
            s_np = wl.importance(cfg, li)
            s_all.append(s_np)
            self.inst.append(dict(
                q=q, labels=lab, labels0=lab.clone(), cbK=cbK, cbV=cbV, idx=idx, pK=pK, pV=pV,
                srcK=srcK, srcV=srcV,
                pid=torch.from_numpy(wl.persist_ids(cfg, li)).to(dev),
                pmask=torch.from_numpy(wl.persist_mask(cfg, li)).to(dev),
                w=torch.from_numpy(s_np).to(dev),
                out=self.io_all[i, :out_bytes].view(torch.float16).view(cfg.B, cfg.Hq, cfg.d),
                res=res,
                sim=res[0:4 * n].view(torch.float32),
                miss=res[4 * n:8 * n].view(torch.int32),
                nmiss=res[8 * n:8 * n + 4].view(torch.int32).zero_(),
                flag=res[8 * n + 4:9 * n + 4]))
        self.s = torch.from_numpy(np.concatenate(s_all)).to(dev)
        self.tau = torch.empty(self.n_inst * cfg.Hkv, dtype=torch.float32, device=dev)
        self.ws = torch.empty(clo.clo_hybrid_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.d),
                              dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        n_tiles = cfg.B * (cfg.Np * -(-cfg.T // 16) + (cfg.Hkv - cfg.Np) * -(-cfg.k // 16))
        ctas = min(torch.cuda.get_device_properties(dev).multi_processor_count,
                   max(1, n_tiles // 8))
        self.attn_kernels = 2 if ctas >= 2 else 1
        self.phases = self.n_inst // math.gcd(self.L, self.n_inst)
        # "overlap" and "pipelined": the next layer's fill runs beside this
        # layer's attention (on a second stream, or in the same layer call).
        # The fill takes side_ctas CTAs (each fits in the room of one attention
        # CTA) and the attention grid leaves that many of its 3 x SMs slots
        # free, so both are resident at once.  (None: the measured best of
        # each schedule, else the full grids; a number applies to any schedule.)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        if side_ctas is None:  # for the layer call, the library's default share (a quarter)
            side_ctas = 64 if schedule == "overlap" else \
                (3 * sms) // 4 if (schedule == "pipelined" and cfg.miss_fill) else 0
        self.side_ctas = side_ctas
        self.main_ctas = max(1, 3 * sms - self.side_ctas) if self.side_ctas else 0
        self.fill_ctas = self.side_ctas
        self.lab0_all = self.lab_all.clone()
        self.restore = clo.prepare_copies([(self.lab_all, self.lab0_all)]) \
            if cfg.label_reset else None
        self.misses_per_step = self._count_misses()
        if cfg.miss_fill:
            # The fill moves the step's rows over the host link (or reads and
            # writes them in HBM): the roofline line covers it.
            self.kernel, self.kernel_src = "fill_kernel", "clo_fill.cu"
            if schedule == "pipelined":
                # Carried beside the attention in the layer call, the fill is
                # timed by the call's events, which bracket both kernels.
                self.kernel = "fill_beside_kernel"
                self.launch_ms_source = (
                    "CUDA events around each layer call (the attention's main kernel and the "
                    "fill beside it) in a second copy of the step graph, replayed after each "
                    "timed round; the fill starts just after the main kernel's CTAs and ends "
                    "last, so the bracket is an upper bound on its duration")

    def _count_misses(self) -> float:
        """Misses of one step's L lookups, averaged over the buffer sets (one
        lookup per set on the drawn labels; with label_reset every step sees
        those labels, otherwise later lookups of a set hit after its first)."""
        torch, clo, cfg = self.torch, self.clo, self.cfg
        clo.clo_thresholds(self.s, self.tau, cfg.G, wl.ETA, wl.N_EXP)
        n = 0
        for j, it in enumerate(self.inst):
            lab = it["labels0"].clone()
            clo.clo_lookup_update(it["q"], lab, it["w"], self.tau[j * cfg.Hkv:(j + 1) * cfg.Hkv],
                                  it["pmask"], it["flag"], it["sim"], it["miss"], it["nmiss"])
            n += int(it["nmiss"].item())
        torch.cuda.synchronize()
        return n / self.n_inst * self.L if cfg.label_reset else 0.0

    def instance(self, step: int, layer: int):
        return self.inst[(step * self.L + layer) % self.n_inst]

    def miss_bytes_per_step(self) -> int:
        """Bytes the misses of a step move: each missed group's G new labels
        and its miss-list entry; with the fill, its k K and V rows read from
        the full KV copy and written into the Cache Buffer, and the k row ids."""
        cfg = self.cfg
        per = cfg.G * cfg.d * HALF + 4
        if cfg.miss_fill:
            per += cfg.k * (2 * cfg.d * HALF * 2 + 4)
        return int(round(self.misses_per_step * per))

    def bytes_per_step(self) -> int:
        return self.L * (hybrid_attn_bytes(self.cfg) + hybrid_lookup_bytes(self.cfg)) + \
            self.n_inst * (self.cfg.Hq + self.cfg.Hkv) * 4 + self.miss_bytes_per_step()

    def attn_bytes_per_launch(self) -> int:
        """Bytes the roofline kernel moves per launch: the attention's
        algorithmic bytes, or with the miss-path fill the fill's rows (read
        over the host link; read and written, plus the row ids, from HBM),
        at the mean misses of a launch."""
        cfg = self.cfg
        if not cfg.miss_fill:
            return hybrid_attn_bytes(cfg)
        rows = self.misses_per_step / self.L * cfg.k
        if cfg.miss_fill == "host":
            return int(round(rows * 2 * cfg.d * HALF))
        return int(round(rows * (2 * 2 * cfg.d * HALF + 8)))

    def roofline_peak(self):
        """(peak, source, bound) of the roofline kernel."""
        if self.cfg.miss_fill == "host":
            return measure_h2d_gbs(self.torch), "measured in this run: pinned host-to-device " \
                "cudaMemcpyAsync of 512 MiB, best of 5", "c2c"
        p, src = peak_hbm()
        return p, src, "hbm"

    def launches_per_step(self) -> int:
        extra = (1 if self.restore is not None else 0) + (self.L if self.cfg.miss_fill else 0)
        if self.schedule in ("fused", "pipelined"):
            # The main kernel; the carried lookup, in the merge launch or, for
            # more than 64 groups, in a launch of its own (include/clo.h); the
            # merge launch where there are partials to merge.
            beside = self.cfg.B * self.cfg.Hkv > LOOKUP_IN_MERGE_MAX_GROUPS
            per_layer = 1 + (1 if beside else 0) + (1 if self.attn_kernels == 2 or not beside else 0)
            return 1 + self.L * per_layer + extra
        return 1 + self.L * (1 + self.attn_kernels) + extra

    def _fill(self, step: int, l: int, events=None):
        """The miss path of layer l's lookup: its missed heads' rows from the
        full KV copy into the Cache Buffer (read on the device from the
        lookup's miss list)."""
        it = self.instance(step, l)
        self.clo.clo_fill_cache_buffer(it["srcK"], it["srcV"], it["idx"], None, it["cbK"],
                                       it["cbV"], it["miss"], it["nmiss"], err_flag=self.err,
                                       num_ctas=self.fill_ctas, events=events)

    def _lookup(self, step: int, l: int):
        cfg = self.cfg
        it = self.instance(step, l)
        j = (step * self.L + l) % self.n_inst
        tau = self.tau[j * cfg.Hkv:(j + 1) * cfg.Hkv]
        self.clo.clo_lookup_update(it["q"], it["labels"], it["w"], tau, it["pmask"], it["flag"],
                                   it["sim"], it["miss"], it["nmiss"])

    def _attention_lookup(self, step: int, l: int, events=None):
        it = self.instance(step, l)
        nx = self.instance(step, l + 1)
        j = (step * self.L + l + 1) % self.n_inst
        tau = self.tau[j * self.cfg.Hkv:(j + 1) * self.cfg.Hkv]
        self.clo.clo_hybrid_decode_attn_lookup(
            it["q"], it["cbK"], it["cbV"], it["idx"], it["pK"], it["pV"], it["pid"], it["out"],
            self.ws, nx["q"], nx["labels"], nx["w"], tau, nx["pmask"], nx["flag"], nx["sim"],
            nx["miss"], nx["nmiss"], err_flag=self.err, events=events)

    def _layer_args(self, j: int) -> dict:
        """clo_hybrid_decode_layer keyword arguments for buffer set j: its
        attention, the fill of set j + 1 (with the miss-path fill; its miss
        list came from an earlier call's lookup) and the lookup of set j + 2."""
        cfg = self.cfg
        it = self.inst[j % self.n_inst]
        fl = self.inst[(j + 1) % self.n_inst]
        j2 = (j + 2) % self.n_inst
        nx = self.inst[j2]
        tau = self.tau[j2 * cfg.Hkv:(j2 + 1) * cfg.Hkv]
        fill = (fl["srcK"], fl["srcV"], fl["idx"], None, fl["cbK"], fl["cbV"], fl["miss"],
                fl["nmiss"]) if cfg.miss_fill else None
        return dict(q=it["q"], cbK=it["cbK"], cbV=it["cbV"], idx=it["idx"], pK=it["pK"],
                    pV=it["pV"], persist_ids=it["pid"], out=it["out"], workspace=self.ws,
                    fill=fill,
                    lookup=(nx["q"], nx["labels"], nx["w"], tau, nx["pmask"], nx["flag"],
                            nx["sim"], nx["miss"], nx["nmiss"]),
                    err_flag=self.err, num_ctas=self.main_ctas, fill_ctas=self.fill_ctas)

    def _layer(self, step: int, l: int, events=None):
        self.clo.clo_hybrid_decode_layer(**self._layer_args(step * self.L + l), events=events)

    def _attention(self, step: int, l: int, events=None):
        it = self.instance(step, l)
        self.clo.clo_hybrid_decode_attn(it["q"], it["cbK"], it["cbV"], it["idx"], it["pK"],
                                        it["pV"], it["pid"], it["out"], self.ws,
                                        err_flag=self.err, num_ctas=self.main_ctas, events=events)

    def launch(self, step: int, attn_events=None):
        """One decode step.  With the "fused" schedule (the default) every
        layer is one clo_hybrid_decode_attn_lookup call: the attention of
        layer l with the lookup of layer l+1 carried in the same launch
        sequence (the step's last call looks up the next step's layer 0, so
        each step still runs exactly L lookups and L attentions).  With the
        "stream" schedule the lookup runs one
        layer ahead on a second stream, as in CLO's decode flow: the lookup of
        layer l+1 starts when layer l starts (after attention l-1) and runs
        beside attention l, and the step's last lookup is the next step's
        layer 0 (replays of the step graph are ordered on the stream, so
        attention 0 of a step always follows its lookup).  With the "overlap"
        schedule (for the miss-path fill) each layer first looks up layer l+1
        on the main stream; the fill of layer l+1's missed heads then runs on
        the second stream beside attention l, so the host-link transfer hides
        behind this layer's attention (CLO section 3: the next layer's missed
        heads move while the current layer computes), and attention l+1 waits
        for it.  With the "pipelined" schedule every layer is one
        clo_hybrid_decode_layer call on one stream: the attention of layer l,
        the fill of layer l+1 beside it (its CTAs in slots the attention grid
        leaves free) and the lookup of layer l+2 carried after it, so each
        layer's lookup runs a layer of compute ahead of the attention before
        it, and its fill beside that attention (CLO section 3 Fig. 9); the
        step's last two calls fill and look up the next step's first layers.
        With the "serial" schedule every layer runs lookup (and fill) then
        attention on one stream."""
        clo, cfg, torch = self.clo, self.cfg, self.torch
        if self.restore is not None:
            self.restore()
        if self.schedule == "fused":
            clo.clo_thresholds(self.s, self.tau, cfg.G, wl.ETA, wl.N_EXP)
            for l in range(self.L):
                ev = None if attn_events is None else attn_events[l]
                self._attention_lookup(step, l, None if cfg.miss_fill else ev)
                if cfg.miss_fill:
                    self._fill(step, l + 1, ev)
            return
        if self.schedule == "pipelined":
            clo.clo_thresholds(self.s, self.tau, cfg.G, wl.ETA, wl.N_EXP)
            for l in range(self.L):
                self._layer(step, l, None if attn_events is None else attn_events[l])
            return
        if self.schedule == "serial":
            clo.clo_thresholds(self.s, self.tau, cfg.G, wl.ETA, wl.N_EXP)
            for l in range(self.L):
                ev = None if attn_events is None else attn_events[l]
                self._lookup(step, l)
                if cfg.miss_fill:
                    self._fill(step, l, ev)
                self._attention(step, l, None if cfg.miss_fill else ev)
            return
        main = torch.cuda.current_stream()
        side = self.side
        fork = torch.cuda.Event()
        fork.record(main)
        side.wait_event(fork)
        looked = [torch.cuda.Event() for _ in range(self.L + 1)]
        if self.schedule == "overlap":
            clo.clo_thresholds(self.s, self.tau, cfg.G, wl.ETA, wl.N_EXP)
            filled = [torch.cuda.Event() for _ in range(self.L + 1)]
            for l in range(self.L):
                ev = None if attn_events is None else attn_events[l]
                self._lookup(step, l + 1)  # layer l+1; for l = L-1 the next step's layer 0
                looked[l + 1].record(main)
                with torch.cuda.stream(side):
                    side.wait_event(looked[l + 1])
                    if cfg.miss_fill:
                        self._fill(step, l + 1, ev)
                    filled[l + 1].record(side)
                if l >= 1:
                    main.wait_event(filled[l])
                self._attention(step, l, None if cfg.miss_fill else ev)
            main.wait_stream(side)  # the next step's layer 0 was filled in this step
            return
        attn_done = [torch.cuda.Event() for _ in range(self.L)]
        with torch.cuda.stream(side):
            clo.clo_thresholds(self.s, self.tau, cfg.G, wl.ETA, wl.N_EXP)
        for l in range(self.L):
            ev = None if attn_events is None else attn_events[l]
            with torch.cuda.stream(side):
                if l >= 1:
                    side.wait_event(attn_done[l - 1])
                self._lookup(step, l + 1)  # layer l+1; for l = L-1 the next step's layer 0
                if cfg.miss_fill:
                    self._fill(step, l + 1, ev)
                looked[l + 1].record(side)
            if l >= 1:
                main.wait_event(looked[l])
            self._attention(step, l, None if cfg.miss_fill else ev)
            attn_done[l].record(main)
        main.wait_stream(side)

    # e2e: each step, one H2D copy of the step's queries (those of every
    # buffer set), the step's calls, and one D2H copy of its results (every
    # set's attention output and lookup outputs).  Every call goes through the
    # public API on buffers fixed for the run: the calls and the copy lists
    # are prepared once (checked and marshalled) and re-issued each step, and
    # the copies are made by the library (clo_copy_async) from and to pinned
    # host memory.  A step's result copy and the next step's query copy are
    # next to each other on the stream and touch disjoint memory, so they go
    # out as one call (one copy launch); e2e_finish copies the last step out.
    def e2e_setup(self):
        clo, cfg = self.clo, self.cfg
        self.h_q = self.q_all.cpu().pin_memory()
        self.h_io = self.io_all.cpu().pin_memory()
        self.e2e_h2d = self.q_all.numel() * HALF
        self.e2e_d2h = self.io_all.numel()
        ins = [(self.q_all, self.h_q)]
        if self.restore is not None:  # the labels restored in the same copy launch
            ins.append((self.lab_all, self.lab0_all))
        self.e2e_pipe = E2ECopies(clo, ins, [(self.h_io, self.io_all)])
        torch = self.torch
        self.e2e_ev = [[torch.cuda.Event() for _ in range(self.L + 1)] for _ in range(3)]
        self.e2e_tau = clo.prepare_thresholds(self.s, self.tau, cfg.G, wl.ETA, wl.N_EXP)
        self.e2e_layer = []
        self.e2e_parts = []
        for j, it in enumerate(self.inst):
            def fill_of(x):
                return (clo.prepare_fill_cache_buffer(x["srcK"], x["srcV"], x["idx"], None,
                                                      x["cbK"], x["cbV"], x["miss"], x["nmiss"],
                                                      err_flag=self.err,
                                                      num_ctas=self.fill_ctas),) \
                    if cfg.miss_fill else ()
            if self.schedule == "pipelined":
                calls = (clo.prepare_hybrid_decode_layer(**self._layer_args(j)),)
            elif self.schedule == "fused":
                # This layer's attention with the next layer's lookup.
                jn = (j + 1) % self.n_inst
                nx = self.inst[jn]
                tau = self.tau[jn * cfg.Hkv:(jn + 1) * cfg.Hkv]
                calls = (clo.prepare_hybrid_decode_attn_lookup(
                    it["q"], it["cbK"], it["cbV"], it["idx"], it["pK"], it["pV"], it["pid"],
                    it["out"], self.ws, nx["q"], nx["labels"], nx["w"], tau, nx["pmask"],
                    nx["flag"], nx["sim"], nx["miss"], nx["nmiss"], err_flag=self.err),) + \
                    fill_of(nx)
            else:
                tau = self.tau[j * cfg.Hkv:(j + 1) * cfg.Hkv]
                look = (clo.prepare_lookup_update(it["q"], it["labels"], it["w"], tau,
                                                  it["pmask"], it["flag"], it["sim"], it["miss"],
                                                  it["nmiss"]),) + fill_of(it)
                attn = (clo.prepare_hybrid_decode_attn(it["q"], it["cbK"], it["cbV"], it["idx"],
                                                       it["pK"], it["pV"], it["pid"], it["out"],
                                                       self.ws, err_flag=self.err,
                                                       num_ctas=self.main_ctas),)
                self.e2e_parts.append((look, attn))
                calls = look + attn
            self.e2e_layer.append(calls)

    def e2e_step(self, step: int):
        self.e2e_pipe.step_in()  # with label_reset this also restores the labels
        if self.schedule == "overlap":  # the same two-stream order as launch()
            torch = self.torch
            main, side = torch.cuda.current_stream(), self.side
            looked, filled, _ = self.e2e_ev
            self.e2e_tau()
            for l in range(self.L):
                look = self.e2e_parts[(step * self.L + l + 1) % self.n_inst][0]
                look[0]()  # the next layer's lookup, on the main stream
                looked[l + 1].record(main)
                with torch.cuda.stream(side):
                    side.wait_event(looked[l + 1])
                    for call in look[1:]:  # its fill, beside this layer's attention
                        call()
                    filled[l + 1].record(side)
                if l >= 1:
                    main.wait_event(filled[l])
                for call in self.e2e_parts[(step * self.L + l) % self.n_inst][1]:
                    call()
            main.wait_stream(side)
            return
        if self.schedule == "stream":  # the same two-stream order as launch()
            torch = self.torch
            main, side = torch.cuda.current_stream(), self.side
            looked, attn_done, fork_l = self.e2e_ev
            fork = fork_l[0]
            fork.record(main)
            side.wait_event(fork)
            with torch.cuda.stream(side):
                self.e2e_tau()
            for l in range(self.L):
                look, _ = self.e2e_parts[(step * self.L + l + 1) % self.n_inst]
                with torch.cuda.stream(side):
                    if l >= 1:
                        side.wait_event(attn_done[l - 1])
                    for call in look:
                        call()
                    looked[l + 1].record(side)
                if l >= 1:
                    main.wait_event(looked[l])
                for call in self.e2e_parts[(step * self.L + l) % self.n_inst][1]:
                    call()
                attn_done[l].record(main)
            main.wait_stream(side)
            return
        self.e2e_tau()
        for l in range(self.L):
            for call in self.e2e_layer[(step * self.L + l) % self.n_inst]:
                call()

    def e2e_finish(self):
        self.e2e_pipe.finish()

    def lookup_stats(self, reps: int = 50) -> dict:
        """The lookup on its own, after the timed region: hit rate and
        near-threshold count of one lookup per buffer set against the
        generator's labels (the timed steps overwrite the labels of missed
        heads with the same queries, so later lookups of a set all hit), and
        the standalone time of clo_lookup_update (CUDA events around a graph
        of `reps` back-to-back calls on fresh label copies)."""
        torch, clo, cfg = self.torch, self.clo, self.cfg
        hits = misses = near = 0
        for j, it in enumerate(self.inst):
            lab = it["labels0"].clone()
            clo.clo_lookup_update(it["q"], lab, it["w"], self.tau[j * cfg.Hkv:(j + 1) * cfg.Hkv],
                                  it["pmask"], it["flag"], it["sim"], it["miss"], it["nmiss"])
            flag = it["flag"].cpu().numpy()
            sim = it["sim"].cpu().numpy().reshape(cfg.B, cfg.Hkv)
            tau = self.tau[j * cfg.Hkv:(j + 1) * cfg.Hkv].cpu().numpy()
            looked = flag != 2
            hits += int(((flag == 0) & looked).sum())
            misses += int(((flag == 1) & looked).sum())
            near += int((np.abs(sim - tau[None, :]).ravel()[looked] < 1e-4).sum())
        n = hits + misses
        labs = [it["labels0"].clone() for it in self.inst]

        def calls():
            for r in range(reps):
                j = r % self.n_inst
                it = self.inst[j]
                clo.clo_lookup_update(it["q"], labs[j], it["w"],
                                      self.tau[j * cfg.Hkv:(j + 1) * cfg.Hkv], it["pmask"],
                                      it["flag"], it["sim"], it["miss"], it["nmiss"])

        # Captured as one graph, so the host's launch rate does not set the time.
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return {"hit_rate": hits / n if n else None, "looked_up_heads": n,
                "near_tau_groups": near, "standalone_us_per_call": a.elapsed_time(b) * 1e3 / reps}

    def config(self) -> dict:
        c = self.cfg
        return {"workload": c.name, "batch": c.B, "layers": c.L, "q_heads": c.Hq,
                "kv_heads": c.Hkv, "head_dim": c.d, "context": c.T, "top_k": c.k,
                "persistent_heads": c.Np, "cache_buffer": c.addressing,
                "lookup_schedule": {
                    "fused": "next layer's lookup carried in each attention launch",
                    "stream": "one layer ahead on a second stream" + (
                        ", the miss-path fill after it on that stream" if c.miss_fill else ""),
                    "overlap": "one layer ahead on the main stream; the next layer's miss-path "
                               "fill on a second stream beside this layer's attention",
                    "serial": "before each layer's attention, same stream",
                    "pipelined": "one call a layer on one stream: attention l, the miss-path "
                                 "fill of layer l+1 beside it, the lookup of layer l+2 carried "
                                 "after it"}[self.schedule],
                "attention_ctas": self.main_ctas or "one full wave",
                "physical_buffer_sets": self.n_inst,
                "l2": f"inputs larger than L2: a buffer is re-read after "
                      f"{self.reuse_distance() / 2**30:.2f} GiB of other reads"} | (
            {"importance": "s = 1 on every head (tau = eta)",
             "query_label_cosine": f"U({c.c_lo}, {c.c_hi})",
             "label_reset": "each step first copies the drawn labels back (one libclo copy "
                            "launch, in the timed step; its bytes are not counted), so the "
                            "same groups miss every step",
             "misses_per_step": self.misses_per_step,
             "miss_bytes_per_step": self.miss_bytes_per_step(),
             "miss_fill": ({"host": "after each lookup, the missed heads' k rows from the full "
                                    "KV copy in pinned host memory (read over NVLink-C2C) into "
                                    "the Cache Buffer rows the next attention reads",
                            "device": "after each lookup, the missed heads' k rows from a full "
                                      "KV copy in HBM into the Cache Buffer"}
                           .get(c.miss_fill, "none"))}
            if c.label_reset else {})

    def reuse_distance(self) -> int:
        per = hybrid_attn_bytes(self.cfg)
        return per * max(1, self.n_inst)


class PagedWorkload:
    kind = "paged"
    e2e_path = PIPELINED_E2E

    def __init__(self, pc, dev, rank: int):
        import torch
        import offloaded_kv_decode_gb300 as clo

        self.clo, self.torch = clo, torch
        self.cfg = pc if rank == 0 else dataclasses.replace(pc, seed=pc.seed + 1000 * rank)
        self.L = 1
        self.q, self.kc, self.vc, self.bt, self.ctx = wl.paged_inputs(self.cfg, dev)
        self.ctx_np = self.ctx.cpu().numpy()
        self.out = torch.empty_like(self.q)
        self.ws = torch.empty(clo.clo_paged_workspace_size(pc.B, pc.Hq, pc.Hkv, pc.d),
                              dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.phases = 1
        self.n_inst = 1

    def bytes_per_step(self) -> int:
        return paged_bytes(self.cfg, self.ctx_np)

    def attn_bytes_per_launch(self) -> int:
        return paged_bytes(self.cfg, self.ctx_np)

    def launches_per_step(self) -> int:
        return 3  # empty-request zeroing, main kernel, partial merge

    def launch(self, step: int, attn_events=None):
        self.clo.clo_paged_decode_attn(self.q, self.kc, self.vc, self.bt, self.ctx, self.out,
                                       self.ws, err_flag=self.err,
                                       events=None if attn_events is None else attn_events[0])

    def e2e_setup(self):
        torch, clo = self.torch, self.clo
        self.h_q = self.q.cpu().pin_memory()
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        self.e2e_h2d = self.q.numel() * HALF
        self.e2e_d2h = self.out.numel() * HALF
        self.e2e_pipe = E2ECopies(clo, [(self.q, self.h_q)], [(self.h_out, self.out)])
        self.e2e_call = clo.prepare_paged_decode_attn(self.q, self.kc, self.vc, self.bt, self.ctx,
                                                      self.out, self.ws, err_flag=self.err)

    def e2e_step(self, step: int):
        self.e2e_pipe.step_in()
        self.e2e_call()

    def e2e_finish(self):
        self.e2e_pipe.finish()

    def config(self) -> dict:
        c = self.cfg
        return {"workload": c.name, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv,
                "head_dim": c.d, "context": f"U[{c.ctx_lo},{c.ctx_hi}]",
                "block_size": c.block_size, "tokens": int(self.ctx_np.sum()),
                "l2": f"inputs larger than L2: {self.bytes_per_step() / 2**30:.2f} GiB read per step"}


class FillWorkload:
    """Miss-path fill: every non-persistent KV head of the base layer missed,
    its top-k rows copied from the full KV copy (pinned host memory or HBM)
    into the Cache Buffer.  Two buffer sets (source, selection, destination)
    alternate, so consecutive steps touch disjoint rows."""
    kind = "fill"
    kernel = "fill_kernel"
    kernel_src = "clo_fill.cu"

    def __init__(self, name, dev, rank: int, batch: int = 0):
        import torch
        import offloaded_kv_decode_gb300 as clo

        base, self.src_where = wl.FILL_CONFIGS[name]
        self.name = name
        self.clo, self.torch = clo, torch
        cfg = wl.CONFIGS[base]
        if batch:
            cfg = dataclasses.replace(cfg, B=batch)
        self.cfg = cfg if rank == 0 else dataclasses.replace(cfg, seed=cfg.seed + 1000 * rank)
        self.L = 1
        self.n_inst = 2
        self.phases = 2
        pm = wl.persist_mask(self.cfg, 0)
        miss = [b * cfg.Hkv + g for b in range(cfg.B) for g in range(cfg.Hkv) if not pm[g]]
        self.n_miss = len(miss)
        self.miss = torch.tensor(miss, dtype=torch.int32, device=dev)
        self.count = torch.tensor([len(miss)], dtype=torch.int32, device=dev)
        self.inst = []
        for i in range(self.n_inst):
            li = i + 1000 * rank
            sK, sV = wl.full_kv(self.cfg, li, dev)
            if self.src_where == "host":
                sK, sV = sK.cpu().pin_memory(), sV.cpu().pin_memory()
            tok, slot = wl.fill_selection(self.cfg, li, dev)
            shape = (cfg.B, cfg.Hkv, cfg.C, cfg.d)
            self.inst.append(dict(srcK=sK, srcV=sV, tok=tok, slot=slot,
                                  cbK=torch.zeros(shape, dtype=torch.float16, device=dev),
                                  cbV=torch.zeros(shape, dtype=torch.float16, device=dev)))
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.row_bytes = cfg.d * HALF

    def link_bytes(self) -> int:
        """K and V rows read from the full copy by one call."""
        return self.n_miss * self.cfg.k * 2 * self.row_bytes

    def bytes_per_step(self) -> int:
        return self.link_bytes()

    def attn_bytes_per_launch(self) -> int:
        """Bytes the kernel moves through its bound: the rows read over the
        host link, or read and written in HBM (plus the token and slot ids)."""
        ids = self.n_miss * self.cfg.k * 8
        if self.src_where == "host":
            return self.link_bytes()
        return 2 * self.link_bytes() + ids

    def launches_per_step(self) -> int:
        return 1

    def launch(self, step: int, attn_events=None):
        it = self.inst[step % self.n_inst]
        self.clo.clo_fill_cache_buffer(it["srcK"], it["srcV"], it["tok"], it["slot"], it["cbK"],
                                       it["cbV"], self.miss, self.count, err_flag=self.err,
                                       events=None if attn_events is None else attn_events[0])

    def roofline_peak(self):
        """(peak GB/s, source, bound)."""
        if self.src_where == "device":
            p, src = peak_hbm()
            return p, src, "hbm"
        return measure_h2d_gbs(self.torch), "measured in this run: pinned host-to-device " \
            "cudaMemcpyAsync of 512 MiB, best of 5", "c2c"

    def e2e_setup(self):
        torch, clo = self.torch, self.clo
        self.h_miss = self.miss.cpu().pin_memory()
        self.h_count = self.count.cpu().pin_memory()
        self.h_err = torch.zeros(1, dtype=torch.int32).pin_memory()
        self.e2e_h2d = (self.miss.numel() + 1) * 4
        self.e2e_d2h = 4
        self.e2e_in = clo.prepare_copies([(self.miss, self.h_miss), (self.count, self.h_count)])
        self.e2e_fill = [clo.prepare_fill_cache_buffer(it["srcK"], it["srcV"], it["tok"],
                                                       it["slot"], it["cbK"], it["cbV"], self.miss,
                                                       self.count, err_flag=self.err)
                         for it in self.inst]
        self.e2e_out = clo.prepare_copies([(self.h_err, self.err)])

    def e2e_step(self, step: int):
        self.e2e_in()
        self.e2e_fill[step % self.n_inst]()
        self.e2e_out()

    def config(self) -> dict:
        c = self.cfg
        return {"workload": self.name, "base": c.name, "batch": c.B, "kv_heads": c.Hkv,
                "head_dim": c.d, "context": c.T, "top_k": c.k, "missed_heads": self.n_miss,
                "source": ("full KV copy in pinned host memory, read by the GPU over the host link"
                           if self.src_where == "host" else "full KV copy in HBM"),
                "rows_per_call": self.n_miss * c.k,
                "l2": "two buffer sets alternate; consecutive calls read and write disjoint rows"}


class TopkWorkload:
    """Top-k retrieval: every KV head ranks all T keys of the base layer
    against its query group and keeps the top k.  Two buffer sets alternate
    (each set's keys are larger than L2)."""
    kind = "topk"
    kernel = "topk_score_kernel"
    kernel_src = "clo_topk.cu"
    # Steps chained inside one graph measured slower here (103.5 us a step with
    # one graph a step, 109-114 us with 2-16 steps a graph), so each step is
    # its own graph.
    chain_steps = False

    def __init__(self, name, dev, rank: int, batch: int = 0):
        import torch
        import offloaded_kv_decode_gb300 as clo

        self.name = name
        self.clo, self.torch = clo, torch
        cfg = wl.CONFIGS[wl.TOPK_CONFIGS[name]]
        if batch:
            cfg = dataclasses.replace(cfg, B=batch)
        self.cfg = cfg if rank == 0 else dataclasses.replace(cfg, seed=cfg.seed + 1000 * rank)
        self.L, self.n_inst, self.phases = 1, 2, 2
        self.inst = []
        for i in range(self.n_inst):
            li = i + 1000 * rank
            q, _ = wl.queries_and_labels(self.cfg, li, dev)
            K, V = wl.full_kv(self.cfg, li, dev)
            del V
            self.inst.append(dict(q=q, K=K, idx=torch.empty((cfg.B, cfg.Hkv, cfg.k),
                                                            dtype=torch.int32, device=dev)))
        self.ws = torch.empty(clo.clo_topk_workspace_size(cfg.B, cfg.Hkv, cfg.T),
                              dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def attn_bytes_per_launch(self) -> int:
        """The scoring kernel's algorithmic reads: every key and the queries."""
        c = self.cfg
        return c.B * c.Hkv * c.T * c.d * HALF + c.B * c.Hq * c.d * HALF

    def bytes_per_step(self) -> int:
        c = self.cfg
        return self.attn_bytes_per_launch() + c.B * c.Hkv * c.k * 4

    def launches_per_step(self) -> int:
        return 2  # scoring, selection

    def launch(self, step: int, attn_events=None):
        it = self.inst[step % self.n_inst]
        self.clo.clo_topk_retrieve(it["q"], it["K"], self.cfg.k, it["idx"], self.ws,
                                   events=None if attn_events is None else attn_events[0])

    def e2e_setup(self):
        torch, clo = self.torch, self.clo
        self.h_q = [it["q"].cpu().pin_memory() for it in self.inst]
        self.h_idx = [torch.empty_like(it["idx"], device="cpu").pin_memory() for it in self.inst]
        c = self.cfg
        self.e2e_h2d = c.B * c.Hq * c.d * HALF
        self.e2e_d2h = c.B * c.Hkv * c.k * 4
        self.e2e_calls = [(clo.prepare_copies([(it["q"], self.h_q[j])]),
                           clo.prepare_topk_retrieve(it["q"], it["K"], c.k, it["idx"], self.ws),
                           clo.prepare_copies([(self.h_idx[j], it["idx"])]))
                          for j, it in enumerate(self.inst)]

    def e2e_step(self, step: int):
        for call in self.e2e_calls[step % self.n_inst]:
            call()

    def config(self) -> dict:
        c = self.cfg
        return {"workload": self.name, "base": c.name, "batch": c.B, "q_heads": c.Hq,
                "kv_heads": c.Hkv, "head_dim": c.d, "keys_per_head": c.T, "top_k": c.k,
                "score": "sum of the group's queries . K_t, fp32",
                "l2": f"two buffer sets of {c.B * c.Hkv * c.T * c.d * HALF / 2**20:.0f} MiB of keys alternate"}


def measure_h2d_gbs(torch, nbytes: int = 512 * 2 ** 20, reps: int = 5) -> float:
    """Pinned host-to-device copy bandwidth (GB/s), best of reps."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(reps + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        d.copy_(h, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    return best


# ---------------------------------------------------------------- CPU oracle sample

def oracle_sample(name: str):
    """A bounded CPU sample of the workload for the oracle: returns a list of
    jobs (callables) and the algorithmic bytes each job covers."""
    import torch  # noqa: F401  (workload generators use torch on the CPU)
    import oracle

    orc = oracle.get()
    scale = 1.0 / math.sqrt(wl.HEAD_DIM)
    jobs = []
    if name in wl.CONFIGS:
        cfg = wl.CONFIGS[name]
        small = wl.HybridConfig(cfg.name, B=2, L=1, Hq=cfg.Hq, Hkv=cfg.Hkv, T=cfg.T, Np=cfg.Np,
                                qmode=cfg.qmode, c_lo=cfg.c_lo, c_hi=cfg.c_hi,
                                low_frac=cfg.low_frac, smode=cfg.smode, seed=cfg.seed)
        q, lab = wl.queries_and_labels(small, 0)
        cbK, cbV, idx = wl.cache_buffer(small, 0)
        pK, pV = wl.persistent_cache(small, 0)
        pid = wl.persist_ids(small, 0).tolist()
        s = wl.importance(small, 0).astype(np.float64)
        tau = orc.thresholds(s, small.Hkv, small.G, wl.ETA, wl.N_EXP)
        qn, labn = q.numpy(), lab.numpy()
        pm = wl.persist_mask(small, 0)
        G = small.G
        jobs.append((lambda: orc.lookup_update(qn, labn, s, tau, pm),
                     hybrid_lookup_bytes(small)))
        for b in range(small.B):
            for g in range(small.Hkv):
                qg = qn[b, g * G:(g + 1) * G]
                if g in pid:
                    j = pid.index(g)
                    K, V = pK[b, j].numpy(), pV[b, j].numpy()
                    n = small.T
                    extra = 0
                else:
                    rows = idx[b, g].numpy()
                    K, V = cbK[b, g].numpy()[rows], cbV[b, g].numpy()[rows]
                    n = small.k
                    extra = n * 4
                jobs.append((lambda qg=qg, K=K, V=V: orc.attention_dense(qg, K, V, scale),
                             n * small.d * HALF * 2 + extra + 2 * G * small.d * HALF))
        desc = (f"two batch rows of {cfg.name} (the lookup, then every KV head's attention: "
                f"{cfg.Np} persistent x {cfg.T} and {cfg.Hkv - cfg.Np} x {cfg.k} indexed rows a "
                f"row)")
    elif name in wl.TOPK_CONFIGS:
        cfg = wl.CONFIGS[wl.TOPK_CONFIGS[name]]
        small = dataclasses.replace(cfg, B=1)
        q, _ = wl.queries_and_labels(small, 0)
        K, _ = wl.full_kv(small, 0)
        qn, Kn = q.numpy(), K.numpy()
        for g in range(small.Hkv):
            G = small.G
            jobs.append((lambda g=g: orc.topk_retrieve(qn[:, g * G:(g + 1) * G], Kn[:, g:g + 1],
                                                        small.k),
                         small.T * small.d * HALF + G * small.d * HALF))
        desc = (f"one batch row of {name} ({small.Hkv} KV heads x {small.T} keys, k = {small.k}, "
                f"fp64 scores and a full sort)")
    elif name in wl.FILL_CONFIGS:
        base, _ = wl.FILL_CONFIGS[name]
        cfg = wl.CONFIGS[base]
        small = dataclasses.replace(cfg, B=2)
        srcK, srcV = wl.full_kv(small, 0)
        tok, slot = wl.fill_selection(small, 0)
        # Written once so the timed fills do not pay first-touch page faults.
        cbK = np.full((small.B, small.Hkv, small.C, small.d), 1.0, np.float16)
        cbV = np.full_like(cbK, 1.0)
        pm = wl.persist_mask(small, 0)
        sK, sV, tk, sl = srcK.numpy(), srcV.numpy(), tok.numpy(), slot.numpy()
        for b in range(small.B):
            for g in range(small.Hkv):
                if pm[g]:
                    continue
                e = b * small.Hkv + g
                jobs.append((lambda e=e: orc.fill_cache_buffer(sK, sV, tk, sl, cbK, cbV, [e],
                                                               inplace=True),
                             small.k * small.d * HALF * 2))
        desc = (f"two batch rows of {name} ({int((pm == 0).sum())} missed KV heads a row x "
                f"{small.k} rows, full KV copy in host memory)")
    else:
        pc = wl.PAGED_CONFIGS[name]
        small = wl.PagedConfig(pc.name, B=4, Hq=pc.Hq, Hkv=pc.Hkv, ctx_lo=pc.ctx_lo,
                               ctx_hi=pc.ctx_hi, seed=pc.seed)
        q, kc, vc, bt, ctx = wl.paged_inputs(small)
        qn, ktn, vtn, btn, cln = q.numpy(), kc.numpy(), vc.numpy(), bt.numpy(), ctx.numpy()
        G = small.G
        for r in range(small.B):
            n = int(cln[r])
            nb = -(-n // 16)
            for h in range(small.Hkv):
                K = ktn[btn[r, :nb], h].reshape(-1, small.d)[:n]
                V = vtn[btn[r, :nb], h].reshape(-1, small.d)[:n]
                qg = qn[r, h * G:(h + 1) * G]
                jobs.append((lambda qg=qg, K=K, V=V: orc.attention_dense(qg, K, V, scale),
                             n * small.d * HALF * 2 + nb * 4 + 2 * G * small.d * HALF))
        desc = (f"4 requests of {pc.name} (all {pc.Hkv} heads each, context drawn from "
                f"U[{pc.ctx_lo},{pc.ctx_hi}])")
    return jobs, desc


def oracle_threads(name: str, jobs) -> int:
    """Host threads for the oracle sample: one a core, at most one a job (a
    thread runs its own share of the jobs, so no job runs twice at once); one
    for top-k, whose oracle routine is not reentrant."""
    if name in wl.TOPK_CONFIGS:
        return 1
    return max(1, min(os.cpu_count() or 1, len(jobs)))


def run_oracle_jobs(jobs, budget_s: float, threads: int = 1):
    """Runs the jobs until budget_s has elapsed (each thread at least one
    job): thread t takes jobs t, t + threads, ... round-robin; the oracle's C
    routines run outside the GIL.  Returns (bytes, seconds)."""
    t0 = time.perf_counter()

    def worker(t):
        mine = jobs[t::threads]
        done, i = 0, 0
        while True:
            fn, nb = mine[i % len(mine)]
            fn()
            done += nb
            i += 1
            if time.perf_counter() - t0 >= budget_s:
                return done

    if threads <= 1:
        done = worker(0)
    else:
        from concurrent.futures import ThreadPoolExecutor

        with ThreadPoolExecutor(max_workers=threads) as ex:
            done = sum(ex.map(worker, range(threads)))
    return done, time.perf_counter() - t0


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", gpu_id], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                pw.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------- main paths

def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def code_digest(path: str) -> str:
    """sha256 (first 16 hex digits) of a source file's code: comments removed
    and whitespace collapsed, so only a change to the code itself changes it."""
    import hashlib
    import re

    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = re.sub(r"\s+", " ", src).strip()
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def traffic_from_profiles(kernel_file: str, kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel code; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    got, traffic = None, None
    for line in text.splitlines():
        if line.startswith("code_sha256_16:"):
            got = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            try:
                traffic = float(line.split(":", 1)[1].split()[0])
            except (IndexError, ValueError):
                traffic = None
    return traffic if (got == code_digest(kernel_file) and traffic is not None) else None


def dist_setup(gpus: int):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if gpus > 1 and world == 1:
        raise SystemExit("--gpus N > 1 needs torchrun (one process per GPU)")
    pg = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    return rank, world, local, pg


def max_over_ranks(value: float, pg, device) -> float:
    if pg is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg):
    if pg is not None:
        pg.barrier()


def aggregate_value(step_bytes: int, world: int, ms_step_max: float) -> float:
    """Whole-job GB/s: every rank processes step_bytes per step (weak scaling);
    the job's step time is the slowest rank's."""
    return step_bytes * world / (ms_step_max * 1e-3) / 1e9


def run_ours(args):
    import torch

    rank, world, local, pg = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import offloaded_kv_decode_gb300 as clo

    clo.lib()
    if args.workload in wl.CONFIGS:
        cfg = wl.CONFIGS[args.workload]
        if args.batch:
            cfg = dataclasses.replace(cfg, B=args.batch)
        if args.ring and cfg.L > 1:
            cfg = dataclasses.replace(cfg, ring=args.ring)
        W = HybridWorkload(cfg, dev, rank, args.replicas, schedule=args.lookup_schedule,
                           side_ctas=args.side_ctas)
    elif args.workload in wl.FILL_CONFIGS:
        W = FillWorkload(args.workload, dev, rank, args.batch)
    elif args.workload in wl.TOPK_CONFIGS:
        W = TopkWorkload(args.workload, dev, rank, args.batch)
    else:
        pc = wl.PAGED_CONFIGS[args.workload]
        if args.batch:
            pc = dataclasses.replace(pc, B=args.batch)
        W = PagedWorkload(pc, dev, rank)
    stream = torch.cuda.current_stream(dev)

    # Eager warm-up (sets kernel attributes before capture).
    for i in range(max(1, W.phases)):
        W.launch(i)
    torch.cuda.synchronize(dev)
    assert int(W.err.item()) == 0, f"kernel error flag {int(W.err.item())}"

    # One graph per buffer phase for the timed steps, and a second copy with
    # timing events around each main attention kernel.  Event nodes serialise
    # the kernels around them (no programmatic overlap), so the value comes
    # from the plain graphs and the kernel duration from one replay of the
    # event graphs after every timed round.
    graphs, ev_graphs = [], []
    for ph in range(W.phases):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            W.launch(ph)
        graphs.append(g)
        evs = []
        for _ in range(W.L):
            b = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            b.record(stream)
            e.record(stream)
            evs.append((b, e))
        torch.cuda.synchronize(dev)
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge):
            W.launch(ph, attn_events=evs)
        ev_graphs.append((ge, evs))
    torch.cuda.synchronize(dev)

    def replay(step):
        graphs[step % W.phases].replay()

    for i in range(args.warmup):
        replay(i)
    torch.cuda.synchronize(dev)

    # The timed steps replay a graph of `chunk` consecutive steps (a multiple
    # of the buffer phases that divides K, at most 16), so the kernels chain
    # through programmatic dependent launch from one step to the next inside
    # a replay instead of stopping at a graph launch every step; K is still
    # timed exactly.  Without such a multiple, or for a workload that measured
    # slower chained (chain_steps = False), the per-step graphs are used.
    K = args.steps
    chunk = 1
    for c in range(16 // W.phases * W.phases, W.phases - 1, -W.phases):
        if c > 1 and K % c == 0 and getattr(W, "chain_steps", True):
            chunk = c
            break
    multi = None
    if chunk > 1:
        multi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(multi):
            for i in range(chunk):
                W.launch(i)
        torch.cuda.synchronize(dev)
        multi.replay()  # one untimed replay of the chunk graph itself
        torch.cuda.synchronize(dev)

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    rounds, attn_ms = [], []
    t_start = time.perf_counter()
    step = args.warmup
    while True:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        barrier(pg)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        if multi is not None:
            for _ in range(K // chunk):
                multi.replay()
            step += K
        else:
            for _ in range(K):
                replay(step)
                step += 1
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(pg)
        ms = max_over_ranks(ev0.elapsed_time(ev1), pg, dev)
        rounds.append(ms)
        for ph in range(W.phases):
            ev_graphs[ph][0].replay()
        torch.cuda.synchronize(dev)
        for ph in range(W.phases):
            for (b, e) in ev_graphs[ph][1]:
                attn_ms.append(b.elapsed_time(e))
        elapsed = time.perf_counter() - t_start
        if (sum(rounds) >= 1000.0 and elapsed >= 1.0) or len(rounds) >= args.max_rounds:
            break
    clocks = sampler.stop()
    assert int(W.err.item()) == 0, f"kernel error flag {int(W.err.item())}"

    ms_round = statistics.median(rounds)
    ms_step = ms_round / K
    step_bytes = W.bytes_per_step()
    value = aggregate_value(step_bytes, world, ms_step)

    attn_ms_mean = statistics.fmean(attn_ms)
    achieved = W.attn_bytes_per_launch() / (attn_ms_mean * 1e-3) / 1e9
    if hasattr(W, "roofline_peak"):
        peak, peak_src, bound = W.roofline_peak()
    else:
        (peak, peak_src), bound = peak_hbm(), "hbm"
    kernel = getattr(W, "kernel", "attn_split_kernel")
    kernel_src = os.path.join(ROOT, "offloaded_kv_decode_gb300", "csrc",
                              getattr(W, "kernel_src", "clo_attention.cu"))
    traffic = traffic_from_profiles(kernel_src, kernel, args.workload)

    # End to end through the public API with host buffers.
    e2e = None
    if not args.no_e2e:
        W.e2e_setup()
        finish = getattr(W, "e2e_finish", lambda: None)
        for i in range(args.warmup):
            W.e2e_step(i)
        finish()
        torch.cuda.synchronize(dev)
        barrier(pg)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            W.e2e_step(i)
        finish()  # the last step's results out, inside the timed region
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(pg)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), pg, dev) / K
        e2e = {"value": aggregate_value(step_bytes, world, e2e_ms), "unit": "GB/s",
               "h2d_bytes_per_step": W.e2e_h2d, "d2h_bytes_per_step": W.e2e_d2h,
               "ms_per_step": e2e_ms,
               "path": getattr(W, "e2e_path", "public API: prepared calls and clo_copy_async "
                               "to and from pinned host buffers, issued from Python each step")}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        jobs, desc = oracle_sample(args.workload)
        threads = oracle_threads(args.workload, jobs)
        nbytes, secs = run_oracle_jobs(jobs, args.cpu_budget, threads)
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{desc}; {secs:.1f} s of fp64 on {threads} host thread(s), one job "
                         f"(KV head or request) at a time each"}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "us_per_layer_step": ms_step * 1e3 / W.L,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded; shapes of the pages' workloads)",
        "config": W.config(),
        "step_frac_of_peak": value / world / peak,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kernel, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": W.attn_bytes_per_launch(),
                     "launch_ms_mean": attn_ms_mean, "launch_samples": len(attn_ms),
                     "launch_ms_source": getattr(
                         W, "launch_ms_source",
                         "CUDA events recorded around the kernel in a second copy of the step "
                         "graph, replayed after each timed round; the event nodes serialise the "
                         "launches next to the kernel (no programmatic overlap), so the duration "
                         "is a little longer than the kernel's share of a chained step"),
                     "layer_step_ms": ms_step / W.L},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": W.launches_per_step() * K,
        "timing": {"rounds": len(rounds), "round_ms_median": ms_round,
                   "round_ms_min": min(rounds), "round_ms_max": max(rounds),
                   "graph_phases": W.phases, "graph_steps": chunk},
        "clocks": clocks,
    }
    line["peaks"] = {"measured_hbm_gbs": peak_hbm()[0], "nominal_hbm_gbs": NOMINAL_HBM_GBS,
                     "step_frac_of_nominal": value / world / NOMINAL_HBM_GBS}
    if W.kind == "hybrid":
        line["tokens_per_s"] = W.cfg.B * world / (ms_step * 1e-3)
        line["lookup"] = W.lookup_stats()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def shape_config(name: str) -> dict:
    """The workload's name and shape, from its configuration alone (no device
    memory): the keys the reference arm reports, as the GPU arm's `config`
    reports them."""
    if name in wl.CONFIGS:
        c = wl.CONFIGS[name]
        return {"workload": c.name, "batch": c.B, "layers": c.L, "q_heads": c.Hq,
                "kv_heads": c.Hkv, "head_dim": c.d, "context": c.T, "top_k": c.k,
                "persistent_heads": c.Np, "cache_buffer": c.addressing}
    if name in wl.PAGED_CONFIGS:
        c = wl.PAGED_CONFIGS[name]
        return {"workload": c.name, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv,
                "head_dim": c.d, "context": f"U[{c.ctx_lo},{c.ctx_hi}]",
                "block_size": c.block_size,
                "tokens": int(wl.paged_context_lengths(c).sum())}
    base = wl.FILL_CONFIGS[name][0] if name in wl.FILL_CONFIGS else wl.TOPK_CONFIGS[name]
    c = wl.CONFIGS[base]
    return {"workload": name, "base": base, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv,
            "head_dim": c.d, "context": c.T, "top_k": c.k}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    jobs, desc = oracle_sample(args.workload)
    threads = oracle_threads(args.workload, jobs)
    per_step = max(0.5, min(5.0, args.cpu_budget / max(1, args.steps)))
    for _ in range(args.warmup):
        run_oracle_jobs(jobs[:1], 0.0)
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b, s = run_oracle_jobs(jobs, per_step, threads)
        tot_b += b
        tot_s += s
    value = tot_b / tot_s / 1e9
    cores = threads
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot_s / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; shapes of the pages' workloads)",
        "config": shape_config(args.workload),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {desc}, run for {per_step:.1f} s on {cores} host "
                                   f"thread(s)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(list(wl.CONFIGS) + list(wl.PAGED_CONFIGS) +
                                   list(wl.FILL_CONFIGS) + list(wl.TOPK_CONFIGS)))
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--max-rounds", type=int, default=2000)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--lookup-schedule",
                    choices=["fused", "stream", "serial", "overlap", "pipelined"],
                    default="fused",
                    help="fused: the next layer's lookup rides in each attention launch; "
                         "stream: it runs one layer ahead on a second stream; serial: lookup "
                         "then attention for every layer on one stream; overlap: the next "
                         "layer's lookup on the main stream, then its miss-path fill on a second "
                         "stream beside this layer's attention; pipelined: one "
                         "clo_hybrid_decode_layer call a layer on one stream (attention l, the "
                         "fill of layer l+1 beside it, the lookup of layer l+2 carried after "
                         "it)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller profiling cases)")
    ap.add_argument("--side-ctas", type=int, default=None,
                    help="--lookup-schedule overlap or pipelined: CTAs of the fill beside the "
                         "attention (the attention grid leaves as many of its slots free)")
    ap.add_argument("--ring", type=int, default=0,
                    help="physical layer buffers of a multi-layer workload (0 = the workload's "
                         "own: one per layer, or its ring); smaller device footprints for "
                         "profiling")
    ap.add_argument("--replicas", type=int, default=0,
                    help="physical buffer sets of a one-layer workload (0 = auto, >1 GB apart)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
