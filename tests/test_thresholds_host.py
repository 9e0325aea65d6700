"""clo_thresholds_host (CLO Eqs. 7-9 computed by the library on the host, fp32)
against the fp64 oracle, on the CPU: no GPU is touched."""
import numpy as np
import pytest

import oracle
import offloaded_kv_decode_gb300 as clo
from offloaded_kv_decode_gb300 import build as libbuild


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    clo.lib()


@pytest.mark.parametrize("group", [1, 4, 5, 8])
@pytest.mark.parametrize("eta,n", [(0.8, 3.0), (0.5, 1.0), (0.95, 5.0), (-0.3, 0.0)])
def test_host_thresholds_vs_oracle(group, eta, n):
    rng = np.random.Generator(np.random.PCG64(200 + group))
    n_kv = 384
    s = rng.uniform(0, 1, n_kv * group).astype(np.float32)
    s[:group] = 1.0           # the eta end of the chain (CLO section 4, check 2)
    s[group:2 * group] = 0.0  # the -1 end
    got = clo.clo_thresholds_host(s, n_kv, group, eta, n).astype(np.float64)
    ref = oracle.get().thresholds(s.astype(np.float64), n_kv, group, eta, n)
    assert got.dtype == np.float64 and got.shape == (n_kv,)
    assert np.max(np.abs(got - ref)) < 1e-6
    assert abs(got[0] - eta) < 1e-6
    if n > 0:
        assert abs(got[1] + 1.0) < 1e-6


def test_host_thresholds_beta_importance_tail():
    """The configured importance draws (Beta(0.5, 2), GQA-4 group means) sit
    at the steep end of the chain near s = 0 and s = 1: still within 1e-6."""
    rng = np.random.Generator(np.random.PCG64(7))
    s = rng.beta(0.5, 2.0, 8 * 4 * 64).astype(np.float32)
    s[-8:] = np.float32(1.0) - np.float32(2.0 ** -20) * np.arange(8, dtype=np.float32)
    got = clo.clo_thresholds_host(s, s.size // 4, 4)
    ref = oracle.get().thresholds(s.astype(np.float64), s.size // 4, 4, 0.8, 3.0)
    assert np.max(np.abs(got.astype(np.float64) - ref)) < 1e-6


def test_host_thresholds_rejects_bad_arguments():
    L = clo.lib()
    tau = np.zeros(4, np.float32)
    s = np.zeros(4, np.float32)
    assert L.clo_thresholds_host(None, 4, 1, 0.8, 3.0, tau.ctypes.data) == clo.CLO_ERR_INVALID_ARG
    assert L.clo_thresholds_host(s.ctypes.data, 4, 0, 0.8, 3.0, tau.ctypes.data) == \
        clo.CLO_ERR_INVALID_ARG
    assert L.clo_thresholds_host(s.ctypes.data, 4, 1, 1.5, 3.0, tau.ctypes.data) == \
        clo.CLO_ERR_INVALID_ARG
    assert L.clo_thresholds_host(s.ctypes.data, 4, 1, 0.8, -1.0, tau.ctypes.data) == \
        clo.CLO_ERR_INVALID_ARG
    assert L.clo_thresholds_host(None, 0, 1, 0.8, 3.0, None) == clo.CLO_OK  # empty: no-op
    with pytest.raises(clo.CloError):
        clo.clo_thresholds_host(np.zeros(5, np.float32), 2, 2)
