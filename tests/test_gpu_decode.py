"""kda_decode_step against the oracle: the 128-step decode workload, float32
inputs, odd head sizes, and the prefill -> decode handoff."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_46_gb300 import chunk_prefill, decode_step, inputs
from gpu_util import assert_close, errors, need_gpu, to_device

pytestmark = pytest.mark.gpu


def test_decode_workload_128_steps():
    """256 sequences x 32 heads, dk = dv = 128, bf16 inputs, float32 state
    (537 MB) updated in place for 128 consecutive steps."""
    dev = need_gpu()
    w = inputs.workload(4)
    A = inputs.decode_A(w)
    s0 = inputs.initial_state(w)
    state = s0.to(dev)
    A_dev = A.to(dev)
    ref_state = s0.double().numpy()
    worst_out = (0.0, 0.0)
    sq_diff = sq_ref = 0.0
    for step in range(w.decode_steps):
        d = inputs.decode_inputs(w, step)
        g = to_device(d, dev)
        o = decode_step(g["q"], g["k"], g["v"], g["z"], A_dev, g["beta"], state)
        ro, ref_state = oracle.decode_step(d["q"], d["k"], d["v"], d["z"], A, d["beta"], ref_state)
        got = o.double().cpu().numpy()
        sq_diff += float(np.sum((got - ro) ** 2))
        sq_ref += float(np.sum(ro ** 2))
        worst_out = (0.0, max(worst_out[1], float(np.max(np.abs(got - ro)))))
    torch.cuda.synchronize()
    rel_out = (sq_diff / sq_ref) ** 0.5
    assert rel_out <= 1e-2 and worst_out[1] <= 5e-2, (rel_out, worst_out[1])
    assert_close("state after 128 steps", state, ref_state, torch.bfloat16)


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128), (32, 128)])
def test_decode_float32_inputs(dk, dv):
    dev = need_gpu()
    rng = np.random.default_rng(dk * 1000 + dv)
    N, H = 5, 3
    st = torch.from_numpy((0.1 * rng.standard_normal((N, H, dk, dv))).astype(np.float32))
    A = torch.from_numpy(rng.uniform(-1, 1, (H, dk)).astype(np.float32))
    state = st.to(dev)
    ref = st.double().numpy()
    for _ in range(6):
        q = torch.nn.functional.normalize(torch.from_numpy(rng.standard_normal((N, H, dk)).astype(np.float32)), dim=-1)
        k = torch.nn.functional.normalize(torch.from_numpy(rng.standard_normal((N, H, dk)).astype(np.float32)), dim=-1)
        v = torch.from_numpy(rng.standard_normal((N, H, dv)).astype(np.float32))
        z = torch.from_numpy(rng.standard_normal((N, H, dk)).astype(np.float32))
        b = torch.sigmoid(torch.from_numpy(rng.standard_normal((N, H)).astype(np.float32)))
        o = decode_step(q.to(dev), k.to(dev), v.to(dev), z.to(dev), A.to(dev), b.to(dev), state)
        ro, ref = oracle.decode_step(q, k, v, z, A, b, ref)
        assert_close("decode out", o, ro, torch.float32)
    assert_close("decode state", state, ref, torch.float32)


def test_prefill_then_decode_handoff():
    """A prefill over T tokens then decode steps continue from its final state:
    equals one prefill over all the tokens (and the oracle)."""
    dev = need_gpu()
    N, H, T0, steps = 4, 2, 100, 5
    w = inputs.custom([T0 + steps] * N, H=H, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=41)
    d = inputs.prefill_inputs(w)
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"], d["initial_state"])
    L = T0 + steps
    head_idx = torch.cat([torch.arange(i * L, i * L + T0) for i in range(N)])
    sub = {n: d[n][head_idx] for n in ("q", "k", "v", "z", "beta")}
    cu = torch.arange(0, N + 1, dtype=torch.int32) * T0
    g = to_device(sub, dev)
    out, fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], d["A"].to(dev), g["beta"], cu.to(dev),
                             d["initial_state"].to(dev))
    for s in range(steps):
        idx = torch.tensor([i * L + T0 + s for i in range(N)])
        gs = to_device({n: d[n][idx] for n in ("q", "k", "v", "z", "beta")}, dev)
        o = decode_step(gs["q"], gs["k"], gs["v"], gs["z"], d["A"].to(dev), gs["beta"], fin)
        assert_close(f"decode step {s}", o, ro[idx.numpy()], torch.bfloat16)
    assert_close("state after handoff", fin, rf, torch.bfloat16)


def test_decode_empty_batch_and_bad_dims():
    dev = need_gpu()
    from gated_delta_rule_46_gb300 import KDAError
    z = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device=dev)
    st = torch.zeros((0, 2, 64, 64), dtype=torch.float32, device=dev)
    o = decode_step(z, z, z, z, torch.zeros((2, 64), device=dev), torch.zeros((0, 2), device=dev), st)
    assert o.shape == (0, 2, 64)
    z = torch.zeros((1, 2, 80), dtype=torch.bfloat16, device=dev)
    with pytest.raises(KDAError):
        decode_step(z, z, z, z, torch.zeros((2, 80), device=dev), torch.zeros((1, 2), device=dev),
                    torch.zeros((1, 2, 80, 80), device=dev))
