"""Helpers shared by the GPU parity tests: running libclo on seeded inputs and
comparing with the fp64 oracle at the tolerances the parity bar states."""
import math
import os
from concurrent.futures import ThreadPoolExecutor

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


def assert_lookup_matches(ref, got, tau32, pm, G):
    """Lookup outputs from libclo (`got`: flag [B][Hkv], sim, labels fp16
    [B][Hq][d], miss_list, miss_count) against the oracle's (`ref`), as the
    parity bar states: flags, label bits and the miss list bit-exact except
    the groups whose fp64 similarity lies within NEAR_TAU of tau (counted,
    and excluded), similarities within 1e-5.  Returns the near-tau count."""
    B, Hkv = ref["flag"].shape
    near = np.abs(ref["sim"] - np.asarray(tau32, dtype=np.float64)[None, :]) < NEAR_TAU
    if pm is not None:
        near &= np.asarray(pm)[None, :] == 0
    ok = ~near
    gf = np.asarray(got["flag"]).reshape(B, Hkv)
    assert np.array_equal(gf[ok], ref["flag"][ok]), "hit/miss flags differ"
    gs = np.asarray(got["sim"], dtype=np.float64).reshape(B, Hkv)
    assert np.max(np.abs(gs - ref["sim"])) < 1e-5
    labg = np.asarray(got["labels"]).view(np.uint16).reshape(B, Hkv, G, -1)
    labr = ref["labels"].reshape(B, Hkv, G, -1)
    assert np.array_equal(labg[ok], labr[ok]), "label updates differ"
    near_ids = set(np.flatnonzero(near.ravel()).tolist())
    gl = [x for x in list(got["miss_list"]) if x not in near_ids]
    rl = [x for x in ref["miss_list"].tolist() if x not in near_ids]
    assert gl == rl, "miss list differs"
    ml = [int(x) for x in got["miss_list"]]
    assert ml == sorted(ml), "miss list not ascending"
    assert got["miss_count"] == int((gf == 1).sum())
    return int(near.sum())


def parallel_map(fn, items):
    """fn over items on the host cores (the oracle's C routines run outside
    the GIL), results in input order.  For the oracle's attention and lookup
    routines, which keep no state between calls; not for topk_retrieve."""
    items = list(items)
    workers = max(1, min(len(items), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, items))

