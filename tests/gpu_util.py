"""Helpers shared by the GPU parity tests: running libclo on seeded inputs and
comparing with the fp64 oracle at the tolerances the parity bar states."""
import math

import numpy as np
import pytest
import torch

# Attention outputs vs the fp64 oracle: max |err| and relative L2 error.
ATOL = 2e-3
REL_L2 = 1e-3
# lse is accumulated in fp32 from the same scores: absolute tolerance.
LSE_ATOL = 1e-4
# Lookup: groups whose fp64 similarity lies within this of tau are counted
# and excluded from the bit-exact mask comparison.
NEAR_TAU = 1e-4

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def dev():
    return torch.device("cuda:0")


def rel_l2(got, ref):
    num = np.linalg.norm((got - ref).ravel())
    den = np.linalg.norm(ref.ravel())
    return num / den if den > 0 else num


def assert_close(got16, ref64, what=""):
    got = np.asarray(got16, dtype=np.float64)
    err = np.abs(got - ref64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= ATOL, f"{what}: max abs err {err.max():.3e} > {ATOL}"
    r = rel_l2(got, ref64)
    assert r <= REL_L2, f"{what}: rel L2 {r:.3e} > {REL_L2}"
    return err.max(), r


def scale_for(d=128):
    return 1.0 / math.sqrt(d)
