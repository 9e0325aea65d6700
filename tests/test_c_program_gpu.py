"""libclo from a plain C host program on the GPU: tests/c/layer_call.c links
against include/clo.h, libclo.so and the CUDA runtime only (no Python, no
torch), runs one clo_hybrid_decode_layer call and checks it against the fp64
oracle, which it links directly (oracle/libclo_oracle.so)."""
import glob
import os
import shutil
import subprocess

import pytest

import oracle
import offloaded_kv_decode_gb300 as clo

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cudart_dir(cuda_home):
    for pat in ("lib64", "lib", "targets/*/lib"):
        for d in glob.glob(os.path.join(cuda_home, pat)):
            if os.path.exists(os.path.join(d, "libcudart.so")):
                return d
    return None


def test_layer_call_from_a_c_program(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc is not None, "no C compiler"
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cudart = _cudart_dir(cuda_home)
    assert cudart is not None, f"libcudart.so not found under {cuda_home}"
    clo.lib()  # the library is built
    orc_dir = os.path.dirname(oracle.get().path)
    lib_dir = os.path.dirname(clo.LIB_PATH)
    exe = tmp_path / "layer_call"
    r = subprocess.run(
        [cc, "-std=c99", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
         "-I", os.path.join(cuda_home, "include"), os.path.join(ROOT, "tests", "c", "layer_call.c"),
         "-o", str(exe), "-L", lib_dir, "-lclo", "-L", orc_dir, "-lclo_oracle", "-L", cudart,
         "-lcudart", "-lm", f"-Wl,-rpath,{lib_dir}:{orc_dir}:{cudart}"],
        capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    print(r.stdout.strip())
