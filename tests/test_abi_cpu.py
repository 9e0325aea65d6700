"""libclo loads, exports every declared entry point, and rejects bad arguments
on the host before launching anything (CPU only: no kernel is launched)."""
import ctypes
import os
import re

import pytest
import torch

import offloaded_kv_decode_gb300 as clo
from offloaded_kv_decode_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "clo.h")
FAKE = 1 << 20  # aligned non-null stand-in pointer: never dereferenced on these paths


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return clo.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(clo_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) == 21, names
    for n in names:
        assert hasattr(L, n), f"{n} declared in clo.h but not exported"


def test_status_helpers(L):
    assert clo.status_string(0) == "CLO_OK"
    assert clo.status_string(4) == "CLO_ERR_BAD_INDEX"
    assert clo.version() >= 100
    assert clo.check_error_flag(0) == clo.CLO_OK
    assert clo.check_error_flag(clo.FLAG_BAD_INDEX | clo.FLAG_BAD_PERSIST) == clo.CLO_ERR_BAD_INDEX
    assert clo.check_error_flag(clo.FLAG_TIMEOUT) == clo.CLO_ERR_TIMEOUT
    assert clo.check_error_flag(clo.FLAG_TIMEOUT | clo.FLAG_BAD_INDEX) == clo.CLO_ERR_TIMEOUT
    assert clo.status_string(clo.CLO_ERR_TIMEOUT) == "CLO_ERR_TIMEOUT"


def test_copy_async_validates_before_issuing(L):
    """clo_copy_async rejects bad lists before any CUDA call (none is made here)."""
    assert L.clo_copy_async(None, 0, None) == clo.CLO_OK
    assert L.clo_copy_async(None, 1, None) == clo.CLO_ERR_INVALID_ARG
    arr = (clo.CloCopy * 2)(clo.CloCopy(None, None, 0), clo.CloCopy(None, 16, 8))
    assert L.clo_copy_async(ctypes.addressof(arr), -1, None) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_copy_async(ctypes.addressof(arr), 2, None) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_copy_async(ctypes.addressof(arr), 1, None) == clo.CLO_OK  # empty copy skipped
    # overlapping copies in one list are refused before anything is issued
    for a, b in [((FAKE, FAKE + 64, 64), (FAKE + 32, FAKE + 4096, 64)),   # dst / dst
                 ((FAKE, FAKE + 64, 64), (FAKE + 4096, FAKE + 16, 32)),   # dst / src
                 ((FAKE, FAKE + 64, 64), (FAKE + 64, FAKE + 4096, 16))]:  # src / dst
        arr = (clo.CloCopy * 2)(clo.CloCopy(*a), clo.CloCopy(*b))
        assert L.clo_copy_async(ctypes.addressof(arr), 2, None) == clo.CLO_ERR_INVALID_ARG
    self_copy = (clo.CloCopy * 1)(clo.CloCopy(FAKE, FAKE + 8, 16))
    assert L.clo_copy_async(ctypes.addressof(self_copy), 1, None) == clo.CLO_ERR_INVALID_ARG
    # a long list whose only conflict is between its first and last copy
    n = 3000
    arr = (clo.CloCopy * n)(*[clo.CloCopy(FAKE + 64 * i, FAKE + (1 << 24) + 64 * i, 32)
                              for i in range(n)])
    arr[n - 1] = clo.CloCopy(FAKE + (1 << 24) + 16, FAKE + (1 << 25), 8)  # writes copy 0's source
    assert L.clo_copy_async(ctypes.addressof(arr), n, None) == clo.CLO_ERR_INVALID_ARG


def test_copy_pairs_checked_in_python():
    a = torch.zeros(4)
    with pytest.raises(clo.CloError):  # pageable host memory on both sides
        clo.prepare_copies([(a, torch.zeros(4))])
    what, args, _ = clo._copies_call([(torch.empty(0), torch.empty(0))])  # empty: skipped
    assert what == "clo_copy_async" and args[1] == 1


def test_workspace_size_formula(L):
    # (2 * CTAs + B*Hkv) partial slots (one per part, CTA and token set) of
    # G*(128 floats + 1 lse), each array padded to 256 B.
    def expect(B, Hq, Hkv, C):
        slots = 2 * C + B * Hkv
        G = Hq // Hkv
        o = slots * G * 128 * 4
        l = slots * G * 4
        return -(-o // 256) * 256 + -(-l // 256) * 256
    for (B, Hq, Hkv, C) in [(1, 32, 8, 152), (8, 32, 8, 152), (16, 40, 8, 7), (256, 32, 32, 152)]:
        assert clo.clo_hybrid_workspace_size(B, Hq, Hkv, 128, C) == expect(B, Hq, Hkv, C)
        assert clo.clo_paged_workspace_size(B, Hq, Hkv, 128, C) == expect(B, Hq, Hkv, C)
    assert clo.clo_hybrid_workspace_size(1, 30, 8, 128, 4) == 0   # Hq % Hkv
    assert clo.clo_hybrid_workspace_size(1, 32, 8, 64, 4) == 0    # d != 128
    assert clo.clo_hybrid_workspace_size(1, 72, 8, 128, 4) == 0   # G > 8


def test_thresholds_rejects(L):
    assert L.clo_thresholds(None, 4, 1, 0.8, 3.0, FAKE, None) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_thresholds(FAKE, 4, 0, 0.8, 3.0, FAKE, None) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_thresholds(FAKE, 4, 1, 1.5, 3.0, FAKE, None) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_thresholds(FAKE, 0, 1, 0.8, 3.0, FAKE, None) == clo.CLO_OK  # empty: no launch


def _lookup(L, q=FAKE, B=1, Hq=32, Hkv=8, d=128, miss=FAKE):
    return L.clo_lookup_update(q, FAKE, FAKE, FAKE, None, B, Hq, Hkv, d, FAKE, FAKE, miss,
                               FAKE, None)


def test_lookup_rejects(L):
    assert _lookup(L, q=None) == clo.CLO_ERR_INVALID_ARG
    assert _lookup(L, miss=None) == clo.CLO_ERR_INVALID_ARG
    assert _lookup(L, Hq=30) == clo.CLO_ERR_INVALID_ARG
    assert _lookup(L, B=-1) == clo.CLO_ERR_INVALID_ARG
    assert _lookup(L, q=FAKE + 2) == clo.CLO_ERR_INVALID_ARG     # misaligned fp16 tensor
    assert _lookup(L, d=64) == clo.CLO_ERR_UNSUPPORTED
    assert _lookup(L, Hq=72) == clo.CLO_ERR_UNSUPPORTED           # G = 9
    assert _lookup(L, B=9000) == clo.CLO_ERR_UNSUPPORTED          # > 65536 groups


def _hybrid(L, k=10, C=100, Np=2, T=50, B=1, Hq=32, Hkv=8, d=128, scale=0.088, ws=FAKE,
            wsb=1 << 30, idx=FAKE, pK=FAKE, pid=FAKE):
    return L.clo_hybrid_decode_attn(FAKE, FAKE, FAKE, idx, k, C, pK, FAKE, pid, Np, T, B, Hq,
                                    Hkv, d, scale, FAKE, None, ws, wsb, None, None, None)


def test_hybrid_rejects(L):
    assert _hybrid(L, k=0) == clo.CLO_ERR_INVALID_ARG          # Cache Buffer heads need k >= 1
    assert _hybrid(L, k=101) == clo.CLO_ERR_INVALID_ARG        # k > C
    assert _hybrid(L, Np=9) == clo.CLO_ERR_INVALID_ARG         # Np > Hkv
    assert _hybrid(L, T=0) == clo.CLO_ERR_INVALID_ARG          # persistent heads need T >= 1
    assert _hybrid(L, idx=None) == clo.CLO_ERR_INVALID_ARG
    assert _hybrid(L, pK=None) == clo.CLO_ERR_INVALID_ARG
    assert _hybrid(L, pid=None) == clo.CLO_ERR_INVALID_ARG
    assert _hybrid(L, scale=0.0) == clo.CLO_ERR_INVALID_ARG
    assert _hybrid(L, scale=float("nan")) == clo.CLO_ERR_INVALID_ARG
    assert _hybrid(L, d=96) == clo.CLO_ERR_UNSUPPORTED
    assert _hybrid(L, Hq=80, Hkv=8) == clo.CLO_ERR_UNSUPPORTED  # G = 10
    assert _hybrid(L, Hq=65, Hkv=65) == clo.CLO_ERR_UNSUPPORTED  # more KV heads than the limit (64)
    assert _hybrid(L, B=0) == clo.CLO_OK                        # empty batch: nothing to do
    # All heads persistent: no Cache Buffer pointers needed, k may be 0.
    assert L.clo_hybrid_decode_attn(FAKE, None, None, None, 0, 0, FAKE, FAKE, FAKE, 8, 5, 0,
                                    32, 8, 128, 0.1, FAKE, None, FAKE, 1 << 20, None, None,
                                    None) == clo.CLO_OK


def _paged(L, B=4, Hq=32, Hkv=32, d=128, bs=16, mb=8, nb=64, bt=FAKE):
    return L.clo_paged_decode_attn(FAKE, FAKE, FAKE, bt, mb, FAKE, nb, B, Hq, Hkv, d, bs, 0.088,
                                   FAKE, None, FAKE, 1 << 30, None, None, None)


def test_paged_rejects(L):
    assert _paged(L, bt=None) == clo.CLO_ERR_INVALID_ARG
    assert _paged(L, mb=0) == clo.CLO_ERR_INVALID_ARG
    assert _paged(L, bs=32) == clo.CLO_ERR_UNSUPPORTED
    assert _paged(L, B=5000) == clo.CLO_ERR_UNSUPPORTED
    assert _paged(L, B=4096, Hkv=64, Hq=64, mb=1 << 14) == clo.CLO_ERR_UNSUPPORTED  # tile ids overflow
    assert _paged(L, B=0) == clo.CLO_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(clo, "_lib", None)
    monkeypatch.setattr(clo, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(clo.CloError):
        clo.lib()


def _fill(L, srcK=FAKE, T=64, tok=FAKE, slot=FAKE, k=8, C=64, ml=FAKE, mc=FAKE, B=1, Hkv=8, d=128):
    return L.clo_fill_cache_buffer(srcK, FAKE, T, tok, slot, k, FAKE, FAKE, C, ml, mc, B, Hkv, d,
                                   None, None, None)


def test_fill_rejects(L):
    assert _fill(L, srcK=None) == clo.CLO_ERR_INVALID_ARG
    assert _fill(L, tok=None) == clo.CLO_ERR_INVALID_ARG
    assert _fill(L, ml=None) == clo.CLO_ERR_INVALID_ARG
    assert _fill(L, mc=None) == clo.CLO_ERR_INVALID_ARG
    assert _fill(L, slot=None, C=32) == clo.CLO_ERR_INVALID_ARG  # token rows need C >= T
    assert _fill(L, srcK=FAKE + 2) == clo.CLO_ERR_INVALID_ARG    # misaligned fp16 rows
    assert _fill(L, B=-1) == clo.CLO_ERR_INVALID_ARG
    assert _fill(L, d=64) == clo.CLO_ERR_UNSUPPORTED
    assert _fill(L, k=0) == clo.CLO_OK                           # nothing to move: no launch
    assert _fill(L, B=0) == clo.CLO_OK


def test_fused_lookup_rejects(L):
    # The next layer's lookup arguments are checked before anything launches.
    def fused(q_next=FAKE, miss_count=FAKE, B=1, Hq=32, Hkv=8):
        return L.clo_hybrid_decode_attn_lookup(
            FAKE, FAKE, FAKE, FAKE, 10, 100, FAKE, FAKE, FAKE, 2, 50, B, Hq, Hkv, 128, 0.088,
            FAKE, None, FAKE, 1 << 30, None,
            q_next, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, miss_count, None, None)
    assert fused(q_next=None) == clo.CLO_ERR_INVALID_ARG
    assert fused(q_next=FAKE + 2) == clo.CLO_ERR_INVALID_ARG
    assert fused(miss_count=None) == clo.CLO_ERR_INVALID_ARG
    assert fused(Hq=30) == clo.CLO_ERR_INVALID_ARG
    assert fused(B=9000) == clo.CLO_ERR_UNSUPPORTED


def test_layer_rejects(L):
    """clo_hybrid_decode_layer checks its carried fill and lookup before
    anything launches (none of these cases reaches the device)."""
    def layer(B=1, Hq=32, Hkv=8, fill=None, lookup=None):
        return L.clo_hybrid_decode_layer(
            FAKE, FAKE, FAKE, FAKE, 10, 100, FAKE, FAKE, FAKE, 2, 50, B, Hq, Hkv, 128, 0.088,
            FAKE, None, FAKE, 1 << 30, None,
            None if fill is None else ctypes.byref(fill),
            None if lookup is None else ctypes.byref(lookup), None, None)

    def fill(**kw):
        a = dict(srcK=FAKE, srcV=FAKE, T=64, tok=FAKE, slot=FAKE, k=8, cbK=FAKE + 4096,
                 cbV=FAKE + 8192, C=64, miss_list=FAKE, miss_count=FAKE, num_ctas=0)
        a.update(kw)
        return clo.FillArgs(**a)

    def lookup(**kw):
        a = dict(q=FAKE, labels=FAKE, w_q=FAKE, tau=FAKE, persist_mask=None, flag=FAKE,
                 sim=FAKE, miss_list=FAKE + 256, miss_count=FAKE + 256)
        a.update(kw)
        return clo.LookupArgs(**a)

    assert layer(B=-1) == clo.CLO_ERR_INVALID_ARG
    assert layer(Hq=30) == clo.CLO_ERR_INVALID_ARG
    assert layer(fill=fill(num_ctas=-1)) == clo.CLO_ERR_INVALID_ARG
    assert layer(fill=fill(tok=None)) == clo.CLO_ERR_INVALID_ARG
    assert layer(fill=fill(miss_count=None)) == clo.CLO_ERR_INVALID_ARG
    assert layer(fill=fill(slot=None, C=32)) == clo.CLO_ERR_INVALID_ARG  # token rows need C >= T
    assert layer(fill=fill(srcK=FAKE + 2)) == clo.CLO_ERR_INVALID_ARG   # misaligned rows
    assert layer(lookup=lookup(q=None)) == clo.CLO_ERR_INVALID_ARG
    assert layer(lookup=lookup(miss_count=None)) == clo.CLO_ERR_INVALID_ARG
    assert layer(lookup=lookup(q=FAKE + 2)) == clo.CLO_ERR_INVALID_ARG
    assert layer(B=0, fill=fill()) == clo.CLO_OK  # empty batch, no lookup: nothing to do


def test_topk_rejects(L):
    def topk(q=FAKE, K=FAKE, B=1, Hq=32, Hkv=8, T=100, d=128, k=10, ws=FAKE, wsb=1 << 30):
        return L.clo_topk_retrieve(q, K, B, Hq, Hkv, T, d, k, FAKE, ws, wsb, None, None)
    assert topk(k=101) == clo.CLO_ERR_INVALID_ARG        # k > T
    assert topk(q=None) == clo.CLO_ERR_INVALID_ARG
    assert topk(K=FAKE + 2) == clo.CLO_ERR_INVALID_ARG   # misaligned rows
    assert topk(Hq=30) == clo.CLO_ERR_INVALID_ARG
    assert topk(d=64) == clo.CLO_ERR_UNSUPPORTED
    assert topk(Hq=72) == clo.CLO_ERR_UNSUPPORTED         # G = 9
    assert topk(wsb=10) == clo.CLO_ERR_WORKSPACE
    assert topk(k=0) == clo.CLO_OK and topk(B=0) == clo.CLO_OK
    assert clo.clo_topk_workspace_size(2, 8, 100) == 2 * 8 * 100 * 4


def test_header_is_plain_c_and_links(L, tmp_path):
    """clo.h compiles as C99 and a C program links against libclo.so and calls
    it through the header's declarations alone (no torch, no GPU work)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    src = tmp_path / "use_clo.c"
    src.write_text(
        '#include <stdio.h>\n#include <string.h>\n#include "clo.h"\n'
        "int main(void) {\n"
        "    if (clo_version() < 10000) return 1;\n"
        '    if (strcmp(clo_status_string(CLO_ERR_WORKSPACE), "CLO_ERR_WORKSPACE") != 0) return 2;\n'
        "    if (clo_check_error_flag(CLO_FLAG_BAD_PERSIST) != CLO_ERR_BAD_INDEX) return 3;\n"
        "    if (clo_copy_async(NULL, -1, 0) != CLO_ERR_INVALID_ARG) return 4;\n"
        "    if (clo_hybrid_workspace_size(1, 32, 8, 128, 152) == 0) return 5;\n"
        "    /* the host-only planner, called from C: one layer of 4 heads */\n"
        "    float tau[4] = {0.8f, -0.5f, 0.6f, 0.0f}, sh[4] = {0.1f, 0.9f, 0.3f, 0.95f};\n"
        "    double D[4]; int32_t np_, npers[1], ids[4];\n"
        "    if (clo_plan_persistent(tau, sh, 1, 4, 0.1f, 1e-4, 5e9, 5e5, D, &np_, npers, ids)\n"
        "        != CLO_OK) return 6;\n"
        "    /* host thresholds, Eqs. 7-9: s = 1 gives eta, s = 0 gives -1 */\n"
        "    float s3[3] = {1.0f, 0.0f, 0.5f}, t3[3];\n"
        "    if (clo_thresholds_host(s3, 3, 1, 0.8f, 3.0f, t3) != CLO_OK) return 7;\n"
        "    if (t3[0] < 0.799999f || t3[0] > 0.800001f || t3[1] > -0.999999f) return 8;\n"
        "    /* the host side of the data-ready sync */\n"
        "    uint32_t ready = 0;\n"
        "    if (clo_signal_ready(&ready, 42u) != CLO_OK || ready != 42u) return 9;\n"
        "    if (clo_wait_ready(&ready, 42u, 0u, NULL, 0) != CLO_ERR_INVALID_ARG) return 10;\n"
        "    /* the layer call's carried fill, declared in C */\n"
        "    clo_fill_args f;\n"
        "    memset(&f, 0, sizeof f);\n"
        "    f.k = 8; f.T = 64; f.C = 64;\n"
        "    if (clo_hybrid_decode_layer(NULL, NULL, NULL, NULL, 10, 100, NULL, NULL, NULL, 2, 50,\n"
        "                                1, 32, 8, 128, 0.088f, NULL, NULL, NULL, 0, NULL, &f, NULL,\n"
        "                                NULL, 0) != CLO_ERR_INVALID_ARG) return 11;\n"
        '    printf("%d %d %d %d %d\\n", np_, npers[0], ids[0], ids[1], ids[2]);\n'
        "    return 0;\n}\n")
    exe = tmp_path / "use_clo"
    libdir = os.path.dirname(clo.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, str(src), "-o", str(exe), "-L", libdir, "-lclo",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    # the same plan through the Python binding
    ref = clo.clo_plan_persistent([[0.8, -0.5, 0.6, 0.0]], [[0.1, 0.9, 0.3, 0.95]], 0.1, 1e-4,
                                  5e9, 5e5)
    want = [ref["n_p"], int(ref["n_persist"][0])] + [int(x) for x in ref["persist_ids"][0][:3]]
    assert [int(x) for x in r.stdout.split()] == want, (r.stdout, want)


def test_wait_ready_rejects_bad_arguments_and_signal_publishes(L):
    """clo_wait_ready checks its arguments before touching the GPU (on this
    machine every pointer is refused: no device can read it);
    clo_signal_ready is host code and stores the value."""
    import numpy as np

    flag = np.zeros(4, dtype=np.uint32)
    p = flag.ctypes.data
    assert L.clo_wait_ready(None, 1, 1000, None, None) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_wait_ready(p + 2, 1, 1000, None, None) == clo.CLO_ERR_INVALID_ARG  # misaligned
    assert L.clo_wait_ready(p, 1, 0, None, None) == clo.CLO_ERR_INVALID_ARG         # no limit
    assert L.clo_wait_ready(p, 1, 10_000_001, None, None) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_wait_ready(p, 1, 1000, None, None) == clo.CLO_ERR_INVALID_ARG      # pageable
    assert L.clo_signal_ready(None, 1) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_signal_ready(p, 0xFFFFFFF7) == clo.CLO_OK and flag[0] == 0xFFFFFFF7
    assert L.clo_signal_ready(p + 4, 3) == clo.CLO_OK and flag[1] == 3

