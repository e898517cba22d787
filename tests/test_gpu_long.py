"""The 1,048,576-token single-sequence prefill (H = 32, bf16), in one call.

Checked against the oracle on: the outputs of the first 8192 tokens; the final
state; and a 4096-token window at a random, chunk-unaligned position p,
recomputed by the oracle from the state the GPU carried to p (a GPU prefix call
over [0, p)), compared both with the single call's outputs in that window and
with a GPU call resumed from the same state.

Final state: the oracle runs the last W tokens from a zero state.  The state's
dependence on anything before the window is bounded by the product over the
window of ||(I - beta k k^T) Diag(alpha_t)||_2 <= prod_t max_c alpha_{t,c}
(the first factor has norm <= 1 because 0 < beta ||k||^2 <= 2), and the test
computes that bound from the window's gates and requires it below 1e-20, so the
truncation is invisible next to the tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_46_gb300 import chunk_prefill, inputs
from gpu_util import assert_close, device_prefill_inputs, need_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_long_context_prefill():
    dev = need_gpu()
    w = inputs.workload(3)
    T = w.total_tokens
    g = device_prefill_inputs(w, dev)
    out, fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], None)
    torch.cuda.synchronize()

    # (1) outputs of the first 8192 tokens
    d0 = inputs.prefill_inputs(w, 0, 0, 8192)
    ro, _ = oracle.prefill(d0["q"], d0["k"], d0["v"], d0["z"], d0["A"], d0["beta"], [0, 8192], None)
    assert_close("out[0:8192]", out[:8192], ro, torch.bfloat16)
    del d0, ro

    # (2) final state, from the last W tokens with a computed truncation bound
    W = 16384
    dw = inputs.prefill_inputs(w, 0, T - W, T)
    gw = oracle.gate(dw["z"], dw["A"])                       # [W, H, dk] float64
    log_bound = np.max(np.sum(np.max(gw, axis=2), axis=0))   # worst head: sum_t max_c g
    assert log_bound < np.log(1e-20), log_bound
    _, rf = oracle.prefill(dw["q"], dw["k"], dw["v"], dw["z"], dw["A"], dw["beta"], [0, W], None)
    assert_close("final state", fin, rf, torch.bfloat16)
    del dw, gw

    # (3) a window resumed from the GPU's carried state
    rng = np.random.default_rng(3)
    p = int(rng.integers(8192, T - 4096))
    if p % 64 == 0:
        p += 37
    cu_p = torch.tensor([0, p], dtype=torch.int32, device=dev)
    _, sp = chunk_prefill(g["q"][:p], g["k"][:p], g["v"][:p], g["z"][:p], g["A"], g["beta"][:p], cu_p, None)
    n = 4096
    cu_n = torch.tensor([0, n], dtype=torch.int32, device=dev)
    ow, _ = chunk_prefill(g["q"][p:p + n], g["k"][p:p + n], g["v"][p:p + n], g["z"][p:p + n], g["A"],
                          g["beta"][p:p + n], cu_n, sp)
    torch.cuda.synchronize()
    dwin = inputs.prefill_inputs(w, 0, p, p + n)
    rw, _ = oracle.prefill(dwin["q"], dwin["k"], dwin["v"], dwin["z"], dwin["A"], dwin["beta"], [0, n],
                           sp.cpu().double().numpy())
    assert_close(f"window [{p}, {p + n}) single call", out[p:p + n], rw, torch.bfloat16)
    assert_close(f"window [{p}, {p + n}) resumed call", ow, rw, torch.bfloat16)
