"""fp64 CPU oracle for the CLO decode hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (``offloaded_kv_decode_gb300``
and its CUDA library) never imports, links or runs it, and this package never
imports the product path.  The arithmetic lives in ``clo_oracle.c`` (plain C,
double precision); this module only builds that file with gcc, loads it with
ctypes and moves numpy arrays in and out.

fp16 tensors cross this boundary as their raw binary16 bit patterns
(``np.uint16``), so the oracle sees exactly the bits the GPU sees.

Pins: every routine is checked in ``tests/test_oracle_pins.py`` against what
the pages and the mathematics fix (limits of Eqs. 7-9, Eq. 10's equal-sims
rule, Eq. 6's norm invariance, library cosine / softmax / SDPA on small cases,
brute-force special cases), and ``tests/test_oracle_mutants.py`` checks that
planted mistakes in this C file are caught by those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "clo_oracle.c")
LIBRARY = os.path.join(HERE, "libclo_oracle.so")

_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double

OK, BAD_ARG, BAD_INDEX = 0, 1, 4


def build(source: str = SOURCE, out: str = LIBRARY) -> str:
    """Compiles the oracle with gcc (plain -O2, strict IEEE double math)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", out, source, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """ctypes handle on one compiled oracle library."""

    def __init__(self, path: str = LIBRARY):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = _D
        lib.oracle_thresholds.argtypes = [_P, _I, _I, _D, _D, _P]
        lib.oracle_thresholds.restype = None
        lib.oracle_lookup_update.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I,
                                             _P, _P, _P, _P, _P]
        lib.oracle_lookup_update.restype = _I
        lib.oracle_attention_dense.argtypes = [_P, _P, _P, _I, _I, _I, _D, _P, _P]
        lib.oracle_attention_dense.restype = _I
        lib.oracle_hybrid_attn.argtypes = [_P, _P, _P, _P, _I, _I, _P, _P, _P, _I,
                                           _I, _I, _I, _I, _I, _D, _P, _P]
        lib.oracle_hybrid_attn.restype = _I
        lib.oracle_paged_attn.argtypes = [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I,
                                          _I, _I, _D, _P, _P]
        lib.oracle_paged_attn.restype = _I
        lib.oracle_fill_cache_buffer.argtypes = [_P, _P, _I, _P, _P, _I, _P, _P, _I,
                                                 _P, _I, _I, _I, _I]
        lib.oracle_fill_cache_buffer.restype = _I
        lib.oracle_plan_persistent.argtypes = [_P, _P, _I, _I, _D, _D, _D, _D, _P, _P, _P, _P]
        lib.oracle_plan_persistent.restype = _I
        lib.oracle_topk_retrieve.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _P]
        lib.oracle_topk_retrieve.restype = _I
        self.lib = lib

    # -- helpers ----------------------------------------------------------
    @staticmethod
    def _u16(a) -> np.ndarray:
        a = np.asarray(a)
        if a.dtype == np.float16:
            a = a.view(np.uint16)
        if a.dtype != np.uint16:
            raise TypeError("fp16 data must be float16 or uint16 bit patterns")
        return np.ascontiguousarray(a)

    @staticmethod
    def _f64(a) -> np.ndarray:
        return np.ascontiguousarray(np.asarray(a, dtype=np.float64))

    @staticmethod
    def _i32(a) -> np.ndarray:
        return np.ascontiguousarray(np.asarray(a, dtype=np.int32))

    # -- routines ---------------------------------------------------------
    def half_to_double(self, bits) -> np.ndarray:
        bits = np.asarray(bits, dtype=np.uint16).ravel()
        f = self.lib.oracle_half_to_double
        return np.array([f(int(b)) for b in bits], dtype=np.float64)

    def thresholds(self, s, n_kv: int, group: int = 1, eta: float = 0.8,
                   n_exp: float = 3.0) -> np.ndarray:
        """Eqs. 7-9; s has n_kv*group entries, returns tau [n_kv] (fp64)."""
        s = self._f64(s)
        if s.size != n_kv * group:
            raise ValueError("s must hold n_kv*group scores")
        tau = np.empty(n_kv, dtype=np.float64)
        self.lib.oracle_thresholds(_ptr(s), n_kv, group, eta, n_exp, _ptr(tau))
        return tau

    def lookup_update(self, q, labels, w_q, tau_kv, persist_mask=None):
        """Head-wise cache lookup + Eq. 10 + label update.

        q, labels: [B][Hq][d] fp16 (labels is not modified; the updated copy
        is returned).  Returns dict(flag u8 [B][Hkv], sim f64 [B][Hkv],
        cos f64 [B][Hq], labels u16 [B][Hq][d], miss_list i32, miss_count).
        """
        q = self._u16(q)
        lab = self._u16(labels).copy()
        B, Hq, d = q.shape
        w = self._f64(w_q)
        tau = self._f64(tau_kv)
        Hkv = tau.size
        pm = None if persist_mask is None else np.ascontiguousarray(
            np.asarray(persist_mask, dtype=np.uint8))
        flag = np.zeros((B, Hkv), dtype=np.uint8)
        sim = np.zeros((B, Hkv), dtype=np.float64)
        cos = np.zeros((B, Hq), dtype=np.float64)
        miss = np.zeros(max(B * Hkv, 1), dtype=np.int32)
        cnt = np.zeros(1, dtype=np.int32)
        rc = self.lib.oracle_lookup_update(
            _ptr(q), _ptr(lab), _ptr(w), _ptr(tau),
            None if pm is None else _ptr(pm), B, Hq, Hkv, d, _ptr(flag),
            _ptr(sim), _ptr(cos), _ptr(miss), _ptr(cnt))
        if rc != OK:
            raise ValueError(f"oracle_lookup_update rc={rc}")
        n = int(cnt[0])
        return dict(flag=flag, sim=sim, cos=cos, labels=lab,
                    miss_list=miss[:n].copy(), miss_count=n)

    def attention_dense(self, q, K, V, scale: float):
        """q [G][d], K/V [n][d] fp16 -> (out f64 [G][d], lse f64 [G])."""
        q, K, V = self._u16(q), self._u16(K), self._u16(V)
        G, d = q.shape
        n = K.shape[0]
        out = np.zeros((G, d), dtype=np.float64)
        lse = np.zeros(G, dtype=np.float64)
        rc = self.lib.oracle_attention_dense(_ptr(q), _ptr(K), _ptr(V), G, n, d,
                                             float(scale), _ptr(out), _ptr(lse))
        if rc != OK:
            raise ValueError(f"oracle_attention_dense rc={rc}")
        return out, lse

    def hybrid_attn(self, q, cbK, cbV, idx, pK, pV, persist_ids, scale: float):
        """Hybrid Cache Buffer / Persistent Cache attention.

        q [B][Hq][d], cbK/cbV [B][Hkv][C][d], idx [B][Hkv][k],
        pK/pV [B][Np][T][d], persist_ids [Np] -> (out [B][Hq][d], lse [B][Hq]).
        """
        q, cbK, cbV = self._u16(q), self._u16(cbK), self._u16(cbV)
        pK, pV = self._u16(pK), self._u16(pV)
        idx, pid = self._i32(idx), self._i32(persist_ids)
        B, Hq, d = q.shape
        Hkv, C = cbK.shape[1], cbK.shape[2]
        k = idx.shape[2]
        Np, T = pK.shape[1], pK.shape[2]
        out = np.zeros((B, Hq, d), dtype=np.float64)
        lse = np.zeros((B, Hq), dtype=np.float64)
        rc = self.lib.oracle_hybrid_attn(
            _ptr(q), _ptr(cbK), _ptr(cbV), _ptr(idx), k, C, _ptr(pK), _ptr(pV),
            _ptr(pid) if pid.size else None, Np, T, B, Hq, Hkv, d, float(scale),
            _ptr(out), _ptr(lse))
        if rc != OK:
            raise ValueError(f"oracle_hybrid_attn rc={rc}")
        return out, lse

    def paged_attn(self, q, kc, vc, block_table, ctx_len, scale: float):
        """q [B][Hq][d], kc/vc [num_blocks][Hkv][bs][d], block_table [B][mb],
        ctx_len [B] -> (out [B][Hq][d], lse [B][Hq])."""
        q, kc, vc = self._u16(q), self._u16(kc), self._u16(vc)
        bt, cl = self._i32(block_table), self._i32(ctx_len)
        B, Hq, d = q.shape
        nb, Hkv, bs = kc.shape[0], kc.shape[1], kc.shape[2]
        mb = bt.shape[1]
        out = np.zeros((B, Hq, d), dtype=np.float64)
        lse = np.zeros((B, Hq), dtype=np.float64)
        rc = self.lib.oracle_paged_attn(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), mb,
                                        _ptr(cl), nb, B, Hq, Hkv, d, bs,
                                        float(scale), _ptr(out), _ptr(lse))
        if rc != OK:
            raise ValueError(f"oracle_paged_attn rc={rc}")
        return out, lse

    def fill_cache_buffer(self, srcK, srcV, tok, slot, cbK, cbV, miss_list, inplace=False):
        """Miss-path fill.  srcK/srcV [B][Hkv][T][d], tok/slot [B][Hkv][k]
        (slot None: token-addressed), cbK/cbV [B][Hkv][C][d] (copied unless
        inplace, in which case they must be contiguous and are written),
        miss_list [n] -> (cbK, cbV, rc) with rc 0 or BAD_INDEX."""
        srcK, srcV = self._u16(srcK), self._u16(srcV)
        if inplace:
            outK, outV = self._u16(cbK), self._u16(cbV)
            if outK.ctypes.data != np.asarray(cbK).ctypes.data or \
                    outV.ctypes.data != np.asarray(cbV).ctypes.data:
                raise ValueError("inplace fill needs contiguous fp16 Cache Buffer arrays")
        else:
            outK, outV = self._u16(cbK).copy(), self._u16(cbV).copy()
        tok = self._i32(tok)
        sl = None if slot is None else self._i32(slot)
        ml = self._i32(miss_list).ravel()
        B, Hkv, T, d = srcK.shape
        C = outK.shape[2]
        k = tok.shape[2]
        rc = self.lib.oracle_fill_cache_buffer(
            _ptr(srcK), _ptr(srcV), T, _ptr(tok), None if sl is None else _ptr(sl), k,
            _ptr(outK), _ptr(outV), C, _ptr(ml) if ml.size else None, int(ml.size),
            B, Hkv, d)
        if rc not in (OK, BAD_INDEX):
            raise ValueError(f"oracle_fill_cache_buffer rc={rc}")
        return outK, outV, rc

    def plan_persistent(self, tau, s_hat, eps: float, t_comp: float, b_link: float,
                        mem_head: float):
        """Eqs. 11-13.  tau, s_hat [L][Hkv] -> dict(D [L][Hkv] f64, n_p int,
        n_persist [L] int32, persist_ids [L][Hkv] int32, -1 padded)."""
        tau, sh = self._f64(tau), self._f64(s_hat)
        if tau.ndim != 2 or sh.shape != tau.shape:
            raise ValueError("tau and s_hat must be [L][Hkv]")
        L, Hkv = tau.shape
        D = np.zeros((L, Hkv), dtype=np.float64)
        n_p = np.zeros(1, dtype=np.int32)
        n_persist = np.zeros(max(L, 1), dtype=np.int32)
        ids = np.zeros((max(L, 1), Hkv), dtype=np.int32)
        rc = self.lib.oracle_plan_persistent(_ptr(tau), _ptr(sh), L, Hkv, float(eps),
                                             float(t_comp), float(b_link), float(mem_head),
                                             _ptr(D), _ptr(n_p), _ptr(n_persist), _ptr(ids))
        if rc != OK:
            raise ValueError(f"oracle_plan_persistent rc={rc}")
        return dict(D=D, n_p=int(n_p[0]), n_persist=n_persist[:L].copy(), persist_ids=ids[:L].copy())

    def topk_retrieve(self, q, K, k: int) -> np.ndarray:
        """q [B][Hq][d], K [B][Hkv][T][d] fp16 -> idx int32 [B][Hkv][k]: per KV
        head the k tokens with the largest (sum of the group's q) . K_t,
        ties to the lower token, ascending.  Not reentrant (the C sort's
        comparator reads a file-level pointer): call it from one thread."""
        q, K = self._u16(q), self._u16(K)
        B, Hq, d = q.shape
        Hkv, T = K.shape[1], K.shape[2]
        idx = np.zeros((B, Hkv, max(k, 1)), dtype=np.int32)
        rc = self.lib.oracle_topk_retrieve(_ptr(q), _ptr(K), B, Hq, Hkv, T, d, int(k), _ptr(idx))
        if rc != OK:
            raise ValueError(f"oracle_topk_retrieve rc={rc}")
        return idx[:, :, :k].copy()


_default = None
_lock = threading.Lock()


def get() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            if (not os.path.exists(LIBRARY)
                    or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
                build()
            _default = Oracle(LIBRARY)
        return _default
