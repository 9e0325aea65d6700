"""Python binding of libclo (include/clo.h): argument marshalling only.

Every function here checks the tensors it is given (device, dtype,
contiguity, shapes), passes their pointers and the CUDA stream to the C ABI of
``libclo.so`` and raises ``CloError`` on a non-OK status.  All computation
happens inside libclo: in its CUDA kernels, and for the offline
persistent-head plan in the library's host code; there is no Python or torch
fallback.  If the library has not been built, the first call raises
``CloError``.

Torch is used for device memory, streams and events only.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libclo.so")

CLO_OK = 0
CLO_ERR_INVALID_ARG = 1
CLO_ERR_UNSUPPORTED = 2
CLO_ERR_CUDA = 3
CLO_ERR_BAD_INDEX = 4
CLO_ERR_WORKSPACE = 5
CLO_ERR_TIMEOUT = 6

FLAG_BAD_INDEX = 0x1
FLAG_BAD_PERSIST = 0x2
FLAG_BAD_CTX = 0x4
FLAG_TIMEOUT = 0x8

HEAD_DIM = 128


class CloError(RuntimeError):
    """A libclo call returned a non-OK status (or the library is missing)."""

    def __init__(self, msg: str, status: Optional[int] = None):
        super().__init__(msg)
        self.status = status


class AttnOpts(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int), ("ev_begin", ctypes.c_void_p),
                ("ev_end", ctypes.c_void_p)]


_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "clo_status_string": ([_I], ctypes.c_char_p),
    "clo_version": ([], _I),
    "clo_check_error_flag": ([ctypes.c_int32], _I),
    "clo_copy_async": ([_P, _I, _P], _I),
    "clo_wait_ready": ([_P, ctypes.c_uint32, ctypes.c_uint32, _P, _P], _I),
    "clo_signal_ready": ([_P, ctypes.c_uint32], _I),
    "clo_thresholds": ([_P, _I, _I, _F, _F, _P, _P], _I),
    "clo_thresholds_host": ([_P, _I, _I, _F, _F, _P], _I),
    "clo_lookup_update": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "clo_fill_cache_buffer": ([_P, _P, _I, _P, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P,
                               _P], _I),
    "clo_plan_persistent": ([_P, _P, _I, _I, _F, ctypes.c_double, ctypes.c_double,
                             ctypes.c_double, _P, _P, _P, _P], _I),
    "clo_topk_workspace_size": ([_I, _I, _I], _SZ),
    "clo_topk_retrieve": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P], _I),
    "clo_hybrid_workspace_size": ([_I, _I, _I, _I, _I], _SZ),
    "clo_hybrid_decode_attn": ([_P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                _F, _P, _P, _P, _SZ, _P, _P, _P], _I),
    "clo_hybrid_decode_attn_noalloc": ([_P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I,
                                        _I, _F, _P, _P, _P, _P, _P], _I),
    "clo_hybrid_noalloc_max_scratch": ([], _SZ),
    "clo_hybrid_decode_attn_lookup": ([_P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                       _F, _P, _P, _P, _SZ, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P], _I),
    "clo_hybrid_decode_layer": ([_P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                 _F, _P, _P, _P, _SZ, _P, _P, _P, _P, _P], _I),
    "clo_paged_workspace_size": ([_I, _I, _I, _I, _I], _SZ),
    "clo_paged_decode_attn": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                               _P, _SZ, _P, _P, _P], _I),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libclo.so (raises CloError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise CloError(f"{LIB_PATH} is missing: build it with "
                           "`python -m offloaded_kv_decode_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().clo_status_string(int(status)).decode()


def version() -> int:
    return int(lib().clo_version())


def check_error_flag(host_value: int) -> int:
    return int(lib().clo_check_error_flag(int(host_value)))


def _check(status: int, what: str):
    if status != CLO_OK:
        raise CloError(f"{what}: {status_string(status)}", status)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: Optional[torch.Tensor], name: str, dtype, ndim=None, optional=False) -> int:
    if t is None:
        if optional:
            return 0
        raise CloError(f"{name} is required", CLO_ERR_INVALID_ARG)
    if not t.is_cuda:
        raise CloError(f"{name} must be a CUDA tensor", CLO_ERR_INVALID_ARG)
    if t.dtype != dtype:
        raise CloError(f"{name} must be {dtype}, got {t.dtype}", CLO_ERR_INVALID_ARG)
    if not t.is_contiguous():
        raise CloError(f"{name} must be contiguous", CLO_ERR_INVALID_ARG)
    if ndim is not None and t.dim() != ndim:
        raise CloError(f"{name} must have {ndim} dims, got {tuple(t.shape)}", CLO_ERR_INVALID_ARG)
    return t.data_ptr()


def _dev_or_pinned(t: torch.Tensor, name: str, dtype, ndim) -> int:
    """A CUDA tensor, or a pinned host tensor the device reads in place."""
    if t is not None and not t.is_cuda:
        if not t.is_pinned():
            raise CloError(f"{name} must be a CUDA tensor or pinned host memory",
                           CLO_ERR_INVALID_ARG)
        if t.dtype != dtype or not t.is_contiguous() or t.dim() != ndim:
            raise CloError(f"{name} must be a contiguous {ndim}-d {dtype} tensor",
                           CLO_ERR_INVALID_ARG)
        return t.data_ptr()
    return _dev(t, name, dtype, ndim)


def _events(events) -> tuple:
    if events is None:
        return 0, 0
    b, e = events
    return int(b.cuda_event), int(e.cuda_event)


def _opts(num_ctas: int, events) -> Optional[AttnOpts]:
    if not num_ctas and events is None:
        return None
    eb, ee = _events(events)
    return AttnOpts(int(num_ctas), eb or None, ee or None)


_BYREF = type(ctypes.byref(ctypes.c_int()))


class PreparedCall:
    """One libclo call whose arguments were checked and marshalled once.

    Calling it issues the same C call again (same buffers; their contents may
    change between calls) without redoing the Python-side checks, for loops
    that re-run a decode step on fixed buffers.  It holds references to its
    tensors, so they stay alive as long as the object does.  The stream is
    the one given to the ``prepare_*`` function, else the current stream at
    each call.
    """

    __slots__ = ("_fn", "_args", "_what", "_keep", "_stream")

    def __init__(self, what: str, args: tuple, keep: tuple, stream=None):
        fn = getattr(lib(), what)
        types = fn.argtypes[:-1]  # the last argument is the stream
        if len(types) != len(args):
            raise CloError(f"{what}: {len(args)} arguments for {len(types)}", CLO_ERR_INVALID_ARG)
        self._fn = fn
        self._args = tuple(a if isinstance(a, _BYREF) else t(a) for t, a in zip(types, args))
        self._what = what
        self._keep = keep
        self._stream = None if stream is None else _stream(stream)

    def __call__(self):
        st = self._stream
        if st is None:
            st = torch.cuda.current_stream().cuda_stream
        status = self._fn(*self._args, st)
        if status != CLO_OK:
            _check(status, self._what)


def _run(call, stream):
    """Issues a (what, args, keep) call once on `stream`."""
    what, args, _ = call
    _check(getattr(lib(), what)(*args, _stream(stream)), what)


# ---------------------------------------------------------------- host-buffer copies

class CloCopy(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


def _copies_call(pairs):
    """pairs: (dst, src) tensors, contiguous, with the same number of bytes; each
    on the GPU or in pinned host memory, at least one of the two on the GPU."""
    pairs = list(pairs)
    arr = (CloCopy * max(len(pairs), 1))()
    for i, (dst, src) in enumerate(pairs):
        if isinstance(dst, torch.Tensor) and isinstance(src, torch.Tensor) and \
                dst.numel() == 0 and src.numel() == 0:
            arr[i] = CloCopy(None, None, 0)  # nothing to move
            continue
        for t, name in ((dst, "dst"), (src, "src")):
            if not isinstance(t, torch.Tensor) or not t.is_contiguous():
                raise CloError(f"copy {i}: {name} must be a contiguous tensor", CLO_ERR_INVALID_ARG)
            if not t.is_cuda and not t.is_pinned():
                raise CloError(f"copy {i}: {name} must be a CUDA tensor or pinned host memory",
                               CLO_ERR_INVALID_ARG)
        if not dst.is_cuda and not src.is_cuda:
            raise CloError(f"copy {i}: host-to-host copies are not made here",
                           CLO_ERR_INVALID_ARG)
        nb = dst.numel() * dst.element_size()
        if nb != src.numel() * src.element_size():
            raise CloError(f"copy {i}: dst and src sizes differ", CLO_ERR_INVALID_ARG)
        arr[i] = CloCopy(dst.data_ptr(), src.data_ptr(), nb)
    return "clo_copy_async", (ctypes.addressof(arr), len(pairs)), (arr, pairs)


def clo_copy_async(pairs: Sequence, stream=None):
    """Issues the copies (dst, src) on the stream (pinned host <-> CUDA, or CUDA <-> CUDA)."""
    _run(_copies_call(pairs), stream)


def prepare_copies(pairs: Sequence, stream=None) -> PreparedCall:
    """clo_copy_async on fixed buffers, checked once (see PreparedCall)."""
    what, args, keep = _copies_call(pairs)
    return PreparedCall(what, args, keep, stream)


# ---------------------------------------------------------------- data-ready sync

def _flag_ptr(ready: torch.Tensor) -> int:
    if not isinstance(ready, torch.Tensor) or ready.dtype not in (torch.int32, torch.uint32) or \
            ready.numel() < 1 or not ready.is_contiguous():
        raise CloError("ready must be a contiguous 32-bit integer tensor", CLO_ERR_INVALID_ARG)
    if not ready.is_cuda and not ready.is_pinned():
        raise CloError("ready must be pinned host memory or a CUDA tensor", CLO_ERR_INVALID_ARG)
    return ready.data_ptr()


def clo_wait_ready(ready: torch.Tensor, expected: int, timeout_us: int,
                   err_flag: Optional[torch.Tensor] = None, stream=None):
    """Queues a bounded GPU wait until ready[0] reaches `expected` (sequence
    numbers); on timeout FLAG_TIMEOUT is ORed into err_flag."""
    pe = _dev(err_flag, "err_flag", torch.int32, optional=True)
    _check(lib().clo_wait_ready(_flag_ptr(ready), int(expected) & 0xFFFFFFFF,
                                int(timeout_us) & 0xFFFFFFFF, pe, _stream(stream)),
           "clo_wait_ready")


def clo_signal_ready(ready: torch.Tensor, value: int):
    """Publishes `value` to ready[0] (pinned host memory) with release
    ordering, from the calling host thread."""
    if ready.is_cuda:
        raise CloError("clo_signal_ready writes host memory", CLO_ERR_INVALID_ARG)
    _check(lib().clo_signal_ready(_flag_ptr(ready), int(value) & 0xFFFFFFFF),
           "clo_signal_ready")


# ---------------------------------------------------------------- thresholds

def clo_thresholds(s: torch.Tensor, tau: torch.Tensor, group: int = 1, eta: float = 0.8,
                   n_exp: float = 3.0, stream=None) -> torch.Tensor:
    """tau[g] = cos(lambda*arccos(eta) + (1-lambda)*pi), lambda = mean(s of group g)^n."""
    _run(_thresholds_call(s, tau, group, eta, n_exp), stream)
    return tau


def prepare_thresholds(s, tau, group: int = 1, eta: float = 0.8, n_exp: float = 3.0,
                       stream=None) -> PreparedCall:
    """clo_thresholds on fixed buffers, checked once (see PreparedCall)."""
    return PreparedCall(*_thresholds_call(s, tau, group, eta, n_exp), stream)


def clo_thresholds_host(s, n_kv: int, group: int = 1, eta: float = 0.8, n_exp: float = 3.0):
    """The same thresholds computed by the library on the host (no GPU):
    s is an array-like of n_kv*group fp32 scores; returns tau as a float32
    numpy array [n_kv]."""
    import numpy as np

    sv = np.ascontiguousarray(np.asarray(s, dtype=np.float32).ravel())
    if sv.size != n_kv * group:
        raise CloError("s must hold n_kv*group scores", CLO_ERR_INVALID_ARG)
    tau = np.zeros(max(int(n_kv), 1), dtype=np.float32)
    _check(lib().clo_thresholds_host(sv.ctypes.data if sv.size else None, int(n_kv), int(group),
                                     float(eta), float(n_exp), tau.ctypes.data),
           "clo_thresholds_host")
    return tau[:n_kv].copy()


def _thresholds_call(s, tau, group, eta, n_exp):
    ps = _dev(s, "s", torch.float32)
    pt = _dev(tau, "tau", torch.float32)
    n_kv = tau.numel()
    if s.numel() != n_kv * group:
        raise CloError("s must hold tau.numel()*group scores", CLO_ERR_INVALID_ARG)
    return ("clo_thresholds", (ps, n_kv, int(group), float(eta), float(n_exp), pt), (s, tau))


# ---------------------------------------------------------------- lookup

def _lookup_args(q, labels, w_q, tau_kv, persist_mask, flag, sim, miss_list, miss_count):
    pq = _dev(q, "q", torch.float16, 3)
    pl = _dev(labels, "labels", torch.float16, 3)
    if labels.shape != q.shape:
        raise CloError("labels must match q", CLO_ERR_INVALID_ARG)
    B, Hq, d = q.shape
    Hkv = tau_kv.numel()
    pw = _dev(w_q, "w_q", torch.float32)
    pt = _dev(tau_kv, "tau_kv", torch.float32)
    pm = _dev(persist_mask, "persist_mask", torch.uint8, optional=True)
    pf = _dev(flag, "flag", torch.uint8)
    psim = _dev(sim, "sim", torch.float32)
    pml = _dev(miss_list, "miss_list", torch.int32)
    pmc = _dev(miss_count, "miss_count", torch.int32)
    if w_q.numel() != Hq or flag.numel() != B * Hkv or sim.numel() != B * Hkv or \
            miss_list.numel() < B * Hkv or miss_count.numel() < 1 or \
            (persist_mask is not None and persist_mask.numel() != Hkv):
        raise CloError("lookup buffer sizes do not match q / tau_kv", CLO_ERR_INVALID_ARG)
    return (pq, pl, pw, pt, pm, B, Hq, Hkv, d, pf, psim, pml, pmc)


def clo_lookup_update(q: torch.Tensor, labels: torch.Tensor, w_q: torch.Tensor,
                      tau_kv: torch.Tensor, persist_mask: Optional[torch.Tensor],
                      flag: torch.Tensor, sim: torch.Tensor, miss_list: torch.Tensor,
                      miss_count: torch.Tensor, stream=None):
    """Fused head-wise cache lookup + Eq. 10 + label update (labels updated in place)."""
    _run(_lookup_call(q, labels, w_q, tau_kv, persist_mask, flag, sim, miss_list, miss_count),
         stream)


def prepare_lookup_update(q, labels, w_q, tau_kv, persist_mask, flag, sim, miss_list,
                          miss_count, stream=None) -> PreparedCall:
    """clo_lookup_update on fixed buffers, checked once (see PreparedCall)."""
    return PreparedCall(*_lookup_call(q, labels, w_q, tau_kv, persist_mask, flag, sim, miss_list,
                                      miss_count), stream)


def _lookup_call(q, labels, w_q, tau_kv, persist_mask, flag, sim, miss_list, miss_count):
    a = _lookup_args(q, labels, w_q, tau_kv, persist_mask, flag, sim, miss_list, miss_count)
    return ("clo_lookup_update", a,
            (q, labels, w_q, tau_kv, persist_mask, flag, sim, miss_list, miss_count))


# ---------------------------------------------------------------- offline plan

def clo_plan_persistent(tau, s_hat, eps: float, t_comp_s: float, link_bytes_per_s: float,
                        head_bytes: float) -> dict:
    """Eqs. 11-13 on the host: tau, s_hat [L][Hkv] (array-likes, fp32) ->
    dict(D [L][Hkv] fp64, n_p, n_persist [L] int32, persist_ids [L][Hkv] int32,
    -1 padded)."""
    import numpy as np

    t = np.ascontiguousarray(np.asarray(tau, dtype=np.float32))
    s = np.ascontiguousarray(np.asarray(s_hat, dtype=np.float32))
    if t.ndim != 2 or s.shape != t.shape:
        raise CloError("tau and s_hat must be [L][Hkv]", CLO_ERR_INVALID_ARG)
    L, Hkv = t.shape
    D = np.zeros((L, Hkv), dtype=np.float64)
    n_p = np.zeros(1, dtype=np.int32)
    n_persist = np.zeros(max(L, 1), dtype=np.int32)
    ids = np.zeros((max(L, 1), Hkv), dtype=np.int32)
    _check(lib().clo_plan_persistent(t.ctypes.data, s.ctypes.data, L, Hkv, float(eps),
                                     float(t_comp_s), float(link_bytes_per_s), float(head_bytes),
                                     D.ctypes.data, n_p.ctypes.data, n_persist.ctypes.data,
                                     ids.ctypes.data), "clo_plan_persistent")
    return dict(D=D, n_p=int(n_p[0]), n_persist=n_persist[:L].copy(), persist_ids=ids[:L].copy())


# ---------------------------------------------------------------- top-k retrieval

def clo_topk_workspace_size(B: int, Hkv: int, T: int) -> int:
    return int(lib().clo_topk_workspace_size(B, Hkv, T))


def clo_topk_retrieve(q: torch.Tensor, K: torch.Tensor, k: int, idx: torch.Tensor,
                      workspace: torch.Tensor, num_ctas: int = 0, events=None, stream=None):
    """Per KV head, the k keys with the largest (sum of the group's queries) . K_t,
    ties to the lower token, ascending: q [B][Hq][d], K [B][Hkv][T][d] fp16,
    idx [B][Hkv][k] int32 output."""
    _run(_topk_call(q, K, k, idx, workspace, num_ctas, events), stream)


def prepare_topk_retrieve(q, K, k: int, idx, workspace, num_ctas: int = 0, events=None,
                          stream=None) -> PreparedCall:
    """clo_topk_retrieve on fixed buffers, checked once (see PreparedCall)."""
    return PreparedCall(*_topk_call(q, K, k, idx, workspace, num_ctas, events), stream)


def _topk_call(q, K, k, idx, workspace, num_ctas, events):
    pq = _dev(q, "q", torch.float16, 3)
    pk = _dev(K, "K", torch.float16, 4)
    pi = _dev(idx, "idx", torch.int32, 3)
    pw = _dev(workspace, "workspace", torch.uint8)
    B, Hq, d = q.shape
    Hkv, T = K.shape[1], K.shape[2]
    if K.shape[0] != B or K.shape[3] != d or tuple(idx.shape) != (B, Hkv, k):
        raise CloError("top-k shapes do not match", CLO_ERR_INVALID_ARG)
    opts = _opts(num_ctas, events)
    return ("clo_topk_retrieve",
            (pq, pk, B, Hq, Hkv, T, d, int(k), pi, pw, workspace.numel(),
             ctypes.byref(opts) if opts is not None else None),
            (q, K, idx, workspace, opts))


# ---------------------------------------------------------------- miss-path fill

def clo_fill_cache_buffer(srcK: torch.Tensor, srcV: torch.Tensor, tok: torch.Tensor,
                          slot: Optional[torch.Tensor], cbK: torch.Tensor, cbV: torch.Tensor,
                          miss_list: torch.Tensor, miss_count: torch.Tensor,
                          err_flag: Optional[torch.Tensor] = None, num_ctas: int = 0,
                          events: Optional[Sequence] = None, stream=None):
    """Copies the new top-k rows of every missed KV head from the full KV copy
    (srcK/srcV [B][Hkv][T][d], CUDA or pinned host memory) into the Cache
    Buffer (cbK/cbV [B][Hkv][C][d]) at slot[b][g][j] (tok itself when slot is
    None); tok/slot [B][Hkv][k] int32, miss_list/miss_count as written by
    clo_lookup_update."""
    _run(_fill_call(srcK, srcV, tok, slot, cbK, cbV, miss_list, miss_count, err_flag, num_ctas,
                    events), stream)


def prepare_fill_cache_buffer(srcK, srcV, tok, slot, cbK, cbV, miss_list, miss_count,
                              err_flag=None, num_ctas: int = 0, events=None,
                              stream=None) -> PreparedCall:
    """clo_fill_cache_buffer on fixed buffers, checked once (see PreparedCall)."""
    return PreparedCall(*_fill_call(srcK, srcV, tok, slot, cbK, cbV, miss_list, miss_count,
                                    err_flag, num_ctas, events), stream)


def _fill_call(srcK, srcV, tok, slot, cbK, cbV, miss_list, miss_count, err_flag, num_ctas,
               events):
    a = _fill_args(srcK, srcV, tok, slot, cbK, cbV, miss_list, miss_count)
    pe = _dev(err_flag, "err_flag", torch.int32, optional=True)
    opts = _opts(num_ctas, events)
    return ("clo_fill_cache_buffer",
            a + (pe, None if opts is None else ctypes.byref(opts)),
            (srcK, srcV, tok, slot, cbK, cbV, miss_list, miss_count, err_flag, opts))


def _fill_args(srcK, srcV, tok, slot, cbK, cbV, miss_list, miss_count):
    ps = _dev_or_pinned(srcK, "srcK", torch.float16, 4)
    pv = _dev_or_pinned(srcV, "srcV", torch.float16, 4)
    B, Hkv, T, d = srcK.shape
    if srcV.shape != srcK.shape:
        raise CloError("srcV must match srcK", CLO_ERR_INVALID_ARG)
    pt = _dev(tok, "tok", torch.int32, 3)
    k = tok.shape[2]
    psl = _dev(slot, "slot", torch.int32, 3, optional=True)
    pk = _dev(cbK, "cbK", torch.float16, 4)
    pcv = _dev(cbV, "cbV", torch.float16, 4)
    C = cbK.shape[2]
    if cbV.shape != cbK.shape or cbK.shape[:2] != (B, Hkv) or cbK.shape[3] != d or \
            tok.shape[:2] != (B, Hkv) or (slot is not None and slot.shape != tok.shape):
        raise CloError("fill shapes do not match", CLO_ERR_INVALID_ARG)
    pml = _dev(miss_list, "miss_list", torch.int32)
    pmc = _dev(miss_count, "miss_count", torch.int32)
    return (ps, pv, T, pt, psl, k, pk, pcv, C, pml, pmc, B, Hkv, d)


# ---------------------------------------------------------------- attention

def clo_hybrid_workspace_size(B: int, Hq: int, Hkv: int, d: int = HEAD_DIM,
                              num_ctas: int = 0) -> int:
    return int(lib().clo_hybrid_workspace_size(B, Hq, Hkv, d, num_ctas))


def clo_paged_workspace_size(B: int, Hq: int, Hkv: int, d: int = HEAD_DIM,
                             num_ctas: int = 0) -> int:
    return int(lib().clo_paged_workspace_size(B, Hq, Hkv, d, num_ctas))


def clo_hybrid_decode_attn(q: torch.Tensor, cbK: Optional[torch.Tensor],
                           cbV: Optional[torch.Tensor], idx: Optional[torch.Tensor],
                           pK: Optional[torch.Tensor], pV: Optional[torch.Tensor],
                           persist_ids: Optional[torch.Tensor], out: torch.Tensor,
                           workspace: torch.Tensor, lse: Optional[torch.Tensor] = None,
                           err_flag: Optional[torch.Tensor] = None,
                           scale: Optional[float] = None, num_ctas: int = 0,
                           events: Optional[Sequence] = None, stream=None):
    """Hybrid Cache Buffer / Persistent Cache GQA decode attention.

    q [B][Hq][d]; cbK/cbV [B][Hkv][C][d]; idx [B][Hkv][k] int32; pK/pV
    [B][Np][T][d]; persist_ids [Np] int32; out [B][Hq][d] fp16; lse [B][Hq]
    fp32 (optional); workspace: a CUDA uint8 tensor of at least
    clo_hybrid_workspace_size(...) bytes.
    """
    _run(_hybrid_call(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse, err_flag, scale,
                      num_ctas, events), stream)


def prepare_hybrid_decode_attn(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse=None,
                               err_flag=None, scale=None, num_ctas: int = 0, events=None,
                               stream=None) -> PreparedCall:
    """clo_hybrid_decode_attn on fixed buffers, checked once (see PreparedCall)."""
    return PreparedCall(*_hybrid_call(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse,
                                      err_flag, scale, num_ctas, events), stream)


def _hybrid_call(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse, err_flag, scale,
                 num_ctas, events):
    a = _hybrid_args(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse, err_flag, scale)
    opts = _opts(num_ctas, events)
    return ("clo_hybrid_decode_attn", a + (ctypes.byref(opts) if opts is not None else None,),
            (q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse, err_flag, opts))


def clo_hybrid_decode_attn_lookup(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace,
                                  q_next, labels_next, w_q_next, tau_next, persist_mask_next,
                                  flag_next, sim_next, miss_list_next, miss_count_next,
                                  lse=None, err_flag=None, scale=None, num_ctas: int = 0,
                                  events=None, stream=None):
    """clo_hybrid_decode_attn for this layer and clo_lookup_update for the next
    layer (same B, Hq, Hkv) in one launch sequence; the results equal the two
    separate calls."""
    _run(_hybrid_lookup_call(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, q_next,
                             labels_next, w_q_next, tau_next, persist_mask_next, flag_next,
                             sim_next, miss_list_next, miss_count_next, lse, err_flag, scale,
                             num_ctas, events), stream)


def prepare_hybrid_decode_attn_lookup(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace,
                                      q_next, labels_next, w_q_next, tau_next, persist_mask_next,
                                      flag_next, sim_next, miss_list_next, miss_count_next,
                                      lse=None, err_flag=None, scale=None, num_ctas: int = 0,
                                      events=None, stream=None) -> PreparedCall:
    """clo_hybrid_decode_attn_lookup on fixed buffers, checked once (see PreparedCall)."""
    return PreparedCall(*_hybrid_lookup_call(
        q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, q_next, labels_next, w_q_next,
        tau_next, persist_mask_next, flag_next, sim_next, miss_list_next, miss_count_next, lse,
        err_flag, scale, num_ctas, events), stream)


def _hybrid_lookup_call(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, q_next,
                        labels_next, w_q_next, tau_next, persist_mask_next, flag_next, sim_next,
                        miss_list_next, miss_count_next, lse, err_flag, scale, num_ctas, events):
    a = _hybrid_args(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse, err_flag, scale)
    b = _lookup_args(q_next, labels_next, w_q_next, tau_next, persist_mask_next, flag_next,
                     sim_next, miss_list_next, miss_count_next)
    if b[5:9] != a[11:15]:
        raise CloError("the next layer's lookup must have this layer's B, Hq, Hkv, d",
                       CLO_ERR_INVALID_ARG)
    opts = _opts(num_ctas, events)
    return ("clo_hybrid_decode_attn_lookup",
            a + (b[0], b[1], b[2], b[3], b[4], b[9], b[10], b[11], b[12],
                 ctypes.byref(opts) if opts is not None else None),
            (q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, q_next, labels_next, w_q_next,
             tau_next, persist_mask_next, flag_next, sim_next, miss_list_next, miss_count_next,
             lse, err_flag, opts))


class FillArgs(ctypes.Structure):
    _fields_ = [("srcK", ctypes.c_void_p), ("srcV", ctypes.c_void_p), ("T", ctypes.c_int),
                ("tok", ctypes.c_void_p), ("slot", ctypes.c_void_p), ("k", ctypes.c_int),
                ("cbK", ctypes.c_void_p), ("cbV", ctypes.c_void_p), ("C", ctypes.c_int),
                ("miss_list", ctypes.c_void_p), ("miss_count", ctypes.c_void_p),
                ("num_ctas", ctypes.c_int)]


class LookupArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("labels", ctypes.c_void_p), ("w_q", ctypes.c_void_p),
                ("tau", ctypes.c_void_p), ("persist_mask", ctypes.c_void_p),
                ("flag", ctypes.c_void_p), ("sim", ctypes.c_void_p),
                ("miss_list", ctypes.c_void_p), ("miss_count", ctypes.c_void_p)]


def clo_hybrid_decode_layer(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, fill=None,
                            lookup=None, lse=None, err_flag=None, scale=None, num_ctas: int = 0,
                            fill_ctas: int = 0, events=None, stream=None):
    """One layer of the decode flow on one stream: clo_hybrid_decode_attn for
    this layer, the next layer's fill beside it and a later layer's lookup in
    its merge launch.

    fill: None or the tensors of clo_fill_cache_buffer, (srcK, srcV, tok,
    slot, cbK, cbV, miss_list, miss_count), for the next layer; fill_ctas its
    CTAs (0: the library's share).  lookup: None or the tensors of
    clo_lookup_update, (q, labels, w_q, tau_kv, persist_mask, flag, sim,
    miss_list, miss_count), for the layer after.  The results equal the
    separate calls; the three must use disjoint buffers."""
    _run(_layer_call(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, fill, lookup, lse,
                     err_flag, scale, num_ctas, fill_ctas, events), stream)


def prepare_hybrid_decode_layer(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace,
                                fill=None, lookup=None, lse=None, err_flag=None, scale=None,
                                num_ctas: int = 0, fill_ctas: int = 0, events=None,
                                stream=None) -> PreparedCall:
    """clo_hybrid_decode_layer on fixed buffers, checked once (see PreparedCall)."""
    return PreparedCall(*_layer_call(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, fill,
                                     lookup, lse, err_flag, scale, num_ctas, fill_ctas, events),
                        stream)


def _layer_call(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, fill, lookup, lse,
                err_flag, scale, num_ctas, fill_ctas, events):
    a = _hybrid_args(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse, err_flag, scale)
    fa = la = None
    if fill is not None:
        if len(fill) != 8:
            raise CloError("fill: (srcK, srcV, tok, slot, cbK, cbV, miss_list, miss_count)",
                           CLO_ERR_INVALID_ARG)
        f = _fill_args(*fill)
        if (f[11], f[12], f[13]) != (a[11], a[13], a[14]):
            raise CloError("the fill must have this layer's B, Hkv, d", CLO_ERR_INVALID_ARG)
        fa = FillArgs(f[0], f[1], f[2], f[3], f[4] or None, f[5], f[6], f[7], f[8], f[9], f[10],
                      int(fill_ctas))
    if lookup is not None:
        if len(lookup) != 9:
            raise CloError("lookup: (q, labels, w_q, tau_kv, persist_mask, flag, sim, "
                           "miss_list, miss_count)", CLO_ERR_INVALID_ARG)
        b = _lookup_args(*lookup)
        if b[5:9] != a[11:15]:
            raise CloError("the lookup must have this layer's B, Hq, Hkv, d", CLO_ERR_INVALID_ARG)
        la = LookupArgs(b[0], b[1], b[2], b[3], b[4] or None, b[9], b[10], b[11], b[12])
    opts = _opts(num_ctas, events)
    return ("clo_hybrid_decode_layer",
            a + (None if fa is None else ctypes.byref(fa), None if la is None else ctypes.byref(la),
                 None if opts is None else ctypes.byref(opts)),
            (q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, fill, lookup, lse, err_flag,
             fa, la, opts))


def _hybrid_args(q, cbK, cbV, idx, pK, pV, persist_ids, out, workspace, lse, err_flag, scale):
    pq = _dev(q, "q", torch.float16, 3)
    B, Hq, d = q.shape
    Np = 0 if persist_ids is None else persist_ids.numel()
    if cbK is not None:
        Hkv, C = cbK.shape[1], cbK.shape[2]
        k = idx.shape[2] if idx is not None else 0
    else:
        Hkv, C, k = Np, 0, 0
    T = pK.shape[2] if (pK is not None and Np > 0) else 0
    pcbk = _dev(cbK, "cbK", torch.float16, 4, optional=True)
    pcbv = _dev(cbV, "cbV", torch.float16, 4, optional=True)
    pidx = _dev(idx, "idx", torch.int32, 3, optional=True)
    ppk = _dev(pK, "pK", torch.float16, 4, optional=True) if Np > 0 else 0
    ppv = _dev(pV, "pV", torch.float16, 4, optional=True) if Np > 0 else 0
    ppid = _dev(persist_ids, "persist_ids", torch.int32, optional=True) if Np > 0 else 0
    pout = _dev(out, "out", torch.float16, 3)
    plse = _dev(lse, "lse", torch.float32, optional=True)
    pws = _dev(workspace, "workspace", torch.uint8)
    perr = _dev(err_flag, "err_flag", torch.int32, optional=True)
    if out.shape != q.shape or (lse is not None and lse.numel() != B * Hq):
        raise CloError("out / lse shapes do not match q", CLO_ERR_INVALID_ARG)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return (pq, pcbk, pcbv, pidx, k, C, ppk, ppv, ppid, Np, T, B, Hq, Hkv, d, float(scale),
            pout, plse, pws, workspace.numel(), perr)


def clo_paged_decode_attn(q: torch.Tensor, kc: torch.Tensor, vc: torch.Tensor,
                          block_table: torch.Tensor, ctx_len: torch.Tensor, out: torch.Tensor,
                          workspace: torch.Tensor, lse: Optional[torch.Tensor] = None,
                          err_flag: Optional[torch.Tensor] = None,
                          scale: Optional[float] = None, num_ctas: int = 0,
                          events: Optional[Sequence] = None, stream=None):
    """Paged decode attention: q [B][Hq][d]; kc/vc [num_blocks][Hkv][16][d];
    block_table [B][max_blocks] int32; ctx_len [B] int32."""
    _run(_paged_call(q, kc, vc, block_table, ctx_len, out, workspace, lse, err_flag, scale,
                     num_ctas, events), stream)


def prepare_paged_decode_attn(q, kc, vc, block_table, ctx_len, out, workspace, lse=None,
                              err_flag=None, scale=None, num_ctas: int = 0, events=None,
                              stream=None) -> PreparedCall:
    """clo_paged_decode_attn on fixed buffers, checked once (see PreparedCall)."""
    return PreparedCall(*_paged_call(q, kc, vc, block_table, ctx_len, out, workspace, lse,
                                     err_flag, scale, num_ctas, events), stream)


def _paged_call(q, kc, vc, block_table, ctx_len, out, workspace, lse, err_flag, scale, num_ctas,
                events):
    pq = _dev(q, "q", torch.float16, 3)
    B, Hq, d = q.shape
    pk = _dev(kc, "kc", torch.float16, 4)
    pv = _dev(vc, "vc", torch.float16, 4)
    num_blocks, Hkv, bs = kc.shape[0], kc.shape[1], kc.shape[2]
    pbt = _dev(block_table, "block_table", torch.int32, 2)
    pcl = _dev(ctx_len, "ctx_len", torch.int32)
    pout = _dev(out, "out", torch.float16, 3)
    plse = _dev(lse, "lse", torch.float32, optional=True)
    pws = _dev(workspace, "workspace", torch.uint8)
    perr = _dev(err_flag, "err_flag", torch.int32, optional=True)
    if out.shape != q.shape or ctx_len.numel() != B or block_table.shape[0] != B or \
            vc.shape != kc.shape:
        raise CloError("paged buffer shapes do not match", CLO_ERR_INVALID_ARG)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    opts = _opts(num_ctas, events)
    return ("clo_paged_decode_attn",
            (pq, pk, pv, pbt, block_table.shape[1], pcl, num_blocks, B, Hq, Hkv, d, bs,
             float(scale), pout, plse, pws, workspace.numel(), perr,
             ctypes.byref(opts) if opts is not None else None),
            (q, kc, vc, block_table, ctx_len, out, workspace, lse, err_flag, opts))


def clo_hybrid_noalloc_max_scratch() -> int:
    """Bytes of the fixed scratch behind clo_hybrid_decode_attn_noalloc."""
    return int(lib().clo_hybrid_noalloc_max_scratch())


def clo_hybrid_decode_attn_noalloc(q: torch.Tensor, cbK: Optional[torch.Tensor],
                                   cbV: Optional[torch.Tensor], idx: Optional[torch.Tensor],
                                   pK: Optional[torch.Tensor], pV: Optional[torch.Tensor],
                                   persist_ids: Optional[torch.Tensor], out: torch.Tensor,
                                   lse: Optional[torch.Tensor] = None,
                                   err_flag: Optional[torch.Tensor] = None,
                                   scale: Optional[float] = None, num_ctas: int = 0,
                                   events: Optional[Sequence] = None, stream=None):
    """clo_hybrid_decode_attn without a caller workspace, for callers that
    cannot allocate device memory at call time (an engine whose own pool holds
    all free device memory, allocation frozen after start-up): the library's
    fixed 8 MiB scratch is used instead.  Raises CloError(CLO_ERR_WORKSPACE)
    for problems needing more; calls on one device that overlap on the GPU
    share that scratch and must be serialised."""
    pq = _dev(q, "q", torch.float16, 3)
    B, Hq, d = q.shape
    Np = 0 if persist_ids is None else persist_ids.numel()
    if cbK is not None:
        Hkv, C = cbK.shape[1], cbK.shape[2]
        k = idx.shape[2] if idx is not None else 0
    else:
        Hkv, C, k = Np, 0, 0
    T = pK.shape[2] if (pK is not None and Np > 0) else 0
    pcbk = _dev(cbK, "cbK", torch.float16, 4, optional=True)
    pcbv = _dev(cbV, "cbV", torch.float16, 4, optional=True)
    pidx = _dev(idx, "idx", torch.int32, 3, optional=True)
    ppk = _dev(pK, "pK", torch.float16, 4, optional=True) if Np > 0 else 0
    ppv = _dev(pV, "pV", torch.float16, 4, optional=True) if Np > 0 else 0
    ppid = _dev(persist_ids, "persist_ids", torch.int32, optional=True) if Np > 0 else 0
    pout = _dev(out, "out", torch.float16, 3)
    plse = _dev(lse, "lse", torch.float32, optional=True)
    perr = _dev(err_flag, "err_flag", torch.int32, optional=True)
    if out.shape != q.shape or (lse is not None and lse.numel() != B * Hq):
        raise CloError("out / lse shapes do not match q", CLO_ERR_INVALID_ARG)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    opts = _opts(num_ctas, events)
    _check(lib().clo_hybrid_decode_attn_noalloc(
        pq, pcbk, pcbv, pidx, k, C, ppk, ppv, ppid, Np, T, B, Hq, Hkv, d, float(scale),
        pout, plse, perr, ctypes.byref(opts) if opts is not None else None, _stream(stream)),
        "clo_hybrid_decode_attn_noalloc")
