"""kda_gate against the oracle's gate, every element."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_46_gb300 import gate, inputs
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid", [0, 1])
def test_gate_matches_oracle(wid):
    dev = need_gpu()
    w = inputs.workload(wid)
    d = inputs.prefill_inputs(w)
    g = gate(d["z"].to(dev), d["A"].to(dev))
    torch.cuda.synchronize()
    ref = oracle.gate(d["z"], d["A"])
    got = g.cpu().double().numpy()
    # float32 evaluation of exp/sigmoid: a few ulp of |g| <= 5
    assert np.max(np.abs(got - ref)) <= 2e-6
    assert np.all(got < 0) and np.all(got >= -5.0)


def test_gate_slab_of_large_workload_and_saturation():
    dev = need_gpu()
    w = inputs.workload(3)
    d = inputs.prefill_inputs(w, t0=70000, t1=74096)
    z = d["z"].clone()
    z[0, 0, :4] = torch.tensor([100.0, -100.0, 0.0, 1e-3])    # saturation and the exact midpoint
    g = gate(z.to(dev), d["A"].to(dev)).cpu().double().numpy()
    ref = oracle.gate(z, d["A"])
    assert np.max(np.abs(g - ref)) <= 2e-6
    # in float32 the sigmoid rounds to 1 for large arguments: g reaches -5 exactly
    assert g[0, 0, 0] == -5.0 and -1e-5 < g[0, 0, 1] <= 0.0
    assert abs(g[0, 0, 2] - (-2.5)) == 0.0
    assert np.all(g >= -5.0) and np.all(g < 0.0 + 1e-30)


def test_gate_empty_and_rejects_bad_dims():
    dev = need_gpu()
    z = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device=dev)
    A = torch.zeros((2, 64), dtype=torch.float32, device=dev)
    assert gate(z, A).shape == (0, 2, 64)
    from gated_delta_rule_46_gb300 import KDAError
    with pytest.raises(KDAError):
        gate(torch.zeros((4, 2, 48), dtype=torch.bfloat16, device=dev),
             torch.zeros((2, 48), dtype=torch.float32, device=dev))
