"""clo_thresholds (Eqs. 7-9) on the GPU vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import offloaded_kv_decode_gb300 as clo
from gpu_util import dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("group", [1, 4, 5])
@pytest.mark.parametrize("eta,n", [(0.8, 3.0), (0.5, 1.0), (0.95, 5.0)])
def test_thresholds_vs_oracle(group, eta, n):
    rng = np.random.Generator(np.random.PCG64(100 + group))
    n_kv = 384
    s = rng.uniform(0, 1, n_kv * group).astype(np.float32)
    s[:group] = 1.0          # tau = eta end of the chain
    s[group:2 * group] = 0.0  # tau = -1 end
    tau = torch.empty(n_kv, dtype=torch.float32, device=dev())
    clo.clo_thresholds(torch.from_numpy(s).to(dev()), tau, group, eta, n)
    torch.cuda.synchronize()
    ref = oracle.get().thresholds(s.astype(np.float64), n_kv, group, eta, n)
    got = tau.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) < 1e-6
    assert abs(got[0] - eta) < 1e-6 and abs(got[1] + 1.0) < 1e-6
    # and the library's host variant of the same map
    host = clo.clo_thresholds_host(s, n_kv, group, eta, n).astype(np.float64)
    assert np.max(np.abs(got - host)) < 1e-6
