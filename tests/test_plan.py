"""clo_plan_persistent (host code in libclo) against the fp64 oracle: the
offline persistent-head plan of Eqs. 11-13 must match exactly (same fp32
inputs, the same fp64 arithmetic for D and N_p; integer outputs bit-exact).
Runs on the CPU: the plan is host code and launches nothing."""
import numpy as np
import pytest

import oracle
import offloaded_kv_decode_gb300 as clo
from offloaded_kv_decode_gb300 import build as libbuild


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    clo.lib()


def _both(tau, sh, eps, t, bw, mem):
    got = clo.clo_plan_persistent(tau, sh, eps, t, bw, mem)
    t32, s32 = np.asarray(tau, np.float32), np.asarray(sh, np.float32)
    ref = oracle.get().plan_persistent(t32.astype(np.float64), s32.astype(np.float64),
                                       float(np.float32(eps)), t, bw, mem)
    assert np.array_equal(got["D"], ref["D"]), "Eq. 11 differs"
    assert got["n_p"] == ref["n_p"], "Eq. 12 differs"
    assert np.array_equal(got["n_persist"], ref["n_persist"]), "Eq. 13 differs"
    assert np.array_equal(got["persist_ids"], ref["persist_ids"]), "resident heads differ"
    return got


@pytest.mark.parametrize("seed", range(6))
def test_plan_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    L, Hkv = (32, 8) if seed % 2 else (48, 8)
    tau = rng.uniform(-1.0, 0.8, (L, Hkv)).astype(np.float32)
    sh = rng.uniform(0.2, 1.0, (L, Hkv)).astype(np.float32)
    # Ties and D = 0 exactly in a few places.
    tau[3, 4], sh[3, 4] = tau[3, 2], sh[3, 2]
    tau[5, 1], sh[5, 1] = np.float32(0.5), np.float32(0.75)
    for bw in (0.0, 21.21e9, 206e9, 1e12):
        _both(tau, sh, 0.25 if seed == 0 else 0.1, 100e-6, bw, 13107 * 128 * 4)


def test_plan_edges():
    _both(np.zeros((0, 8), np.float32), np.zeros((0, 8), np.float32), 0.1, 1e-4, 1e9, 1e6)
    r = _both([[0.8] * 8], [[0.1] * 8], 0.05, 0.0, 1e9, 1e6)        # no time to prefetch
    assert r["n_p"] == 0 and r["n_persist"].tolist() == [8]
    r = _both([[0.8] * 8], [[0.1] * 8], 0.05, 1.0, 1e12, 1.0)       # huge capacity
    assert r["n_persist"].tolist() == [0]


def test_plan_rejects():
    t = np.zeros((2, 8), np.float32)
    for args in ((0.1, 1e-4, 1e9, 0.0), (0.1, -1.0, 1e9, 1e6), (0.1, 1e-4, -1.0, 1e6),
                 (float("nan"), 1e-4, 1e9, 1e6), (0.1, float("inf"), 1e9, 1e6)):
        with pytest.raises(clo.CloError):
            clo.clo_plan_persistent(t, t, *args)
