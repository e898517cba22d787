"""kda_chunk_prefill_logdecay: the log-decay given directly, unbounded below
(decays far stronger than the bounded gate's e^-5 per token, and channels
with almost none), against the oracle fed the same g; and, on the bounded
gate's own g, against kda_chunk_prefill."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_46_gb300 import KDAError, chunk_prefill, chunk_prefill_logdecay, gate, inputs
from gpu_util import assert_close, need_gpu, to_device

pytestmark = pytest.mark.gpu


def _unbounded_g(T, H, dk, seed):
    """Seeded log-decays: per channel a rate exp(U(-6, 4.5)) (from ~0.0025 up
    to ~90 per token) times softplus of a normal draw, so that within one
    16-token tile the cumulative log-decay reaches -1000 and below in some
    channels while others barely decay."""
    rng = np.random.default_rng(seed)
    rate = np.exp(rng.uniform(-6.0, 4.5, size=(1, H, dk)))
    x = rng.standard_normal((T, H, dk))
    return (-rate * np.log1p(np.exp(x))).astype(np.float32)


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 128),
                                         (torch.bfloat16, 32, 64)])
def test_unbounded_decay_against_oracle(dtype, dk, dv):
    dev = need_gpu()
    w = inputs.custom([300, 1, 77, 160], H=3, dk=dk, dv=dv, dtype=dtype, init="randn0.1", wid=61)
    d = inputs.prefill_inputs(w)
    g = torch.from_numpy(_unbounded_g(w.total_tokens, w.H, dk, 61))
    assert float(g.min()) < -60.0 and float(g.max()) > -0.01
    x = to_device(d, dev)
    out, fin = chunk_prefill_logdecay(x["q"], x["k"], x["v"], g.to(dev), x["beta"], x["cu_seqlens"],
                                      x["initial_state"])
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], None, None, d["beta"], d["cu_seqlens"],
                            d["initial_state"], g=g.numpy())
    assert_close("outputs", out, ro, dtype)
    assert_close("states", fin, rf, dtype)


def test_bounded_gate_matches_chunked_path():
    """On g from the bounded gate the unbounded entry point and the chunked
    tensor-core prefill compute the same layer."""
    dev = need_gpu()
    w = inputs.custom([1000, 129, 64], H=4, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1",
                      wid=62)
    x = to_device(inputs.prefill_inputs(w), dev)
    g = gate(x["z"], x["A"])
    ref_out, ref_fin = chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["A"], x["beta"],
                                     x["cu_seqlens"], x["initial_state"])
    out, fin = chunk_prefill_logdecay(x["q"], x["k"], x["v"], g, x["beta"], x["cu_seqlens"],
                                      x["initial_state"])
    torch.cuda.synchronize()
    assert_close("outputs", out, ref_out.double().cpu().numpy(), torch.bfloat16)
    assert_close("states", fin, ref_fin.double().cpu().numpy(), torch.bfloat16)


def test_logdecay_invalid_arguments():
    dev = need_gpu()
    w = inputs.custom([8], H=1, dk=32, dv=32, dtype=torch.float32, wid=63)
    x = to_device(inputs.prefill_inputs(w), dev)
    g = torch.zeros((8, 1, 32), dtype=torch.float32, device=dev)
    with pytest.raises(KDAError):          # a workspace without room for the status word
        chunk_prefill_logdecay(x["q"], x["k"], x["v"], g, x["beta"], x["cu_seqlens"],
                               workspace=torch.zeros(0, dtype=torch.uint8, device=dev))


def test_serial_kernel_few_and_many_chains():
    """The token-serial kernel on few (sequence, head) chains and on many (one
    CTA per chain and 32 value channels), against the oracle (float32)."""
    dev = need_gpu()
    for lens, H in (([40, 7, 90], 2), ([23] * 96, 4)):   # 24 and 1536 (chain, 32-column) blocks
        w = inputs.custom(lens, H=H, dk=128, dv=128, dtype=torch.float32, init="randn0.1", wid=64)
        d = inputs.prefill_inputs(w)
        g = torch.from_numpy(_unbounded_g(w.total_tokens, w.H, 128, 64))
        x = to_device(d, dev)
        out, fin = chunk_prefill_logdecay(x["q"], x["k"], x["v"], g.to(dev), x["beta"], x["cu_seqlens"],
                                          x["initial_state"])
        torch.cuda.synchronize()
        ro, rf = oracle.prefill(d["q"], d["k"], d["v"], None, None, d["beta"], d["cu_seqlens"],
                                d["initial_state"], g=g.numpy())
        assert_close("outputs", out, ro, torch.float32)
        assert_close("states", fin, rf, torch.float32)


def test_chunked_unbounded_path_against_oracle():
    """bf16, 128 x 128 heads, few long sequences: the chunked path (diagonal
    tiles pair by pair, every other factor with a non-positive exponent) and the
    token-serial kernel (a 256-byte workspace), both against the oracle."""
    from gated_delta_rule_46_gb300 import logdecay_workspace_size
    dev = need_gpu()
    w = inputs.custom([3000, 1100], H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=65)
    d = inputs.prefill_inputs(w)
    g = torch.from_numpy(_unbounded_g(w.total_tokens, w.H, 128, 65))
    x = to_device(d, dev)
    big = logdecay_workspace_size(w.total_tokens, 2, 2, 128, 128)
    assert big > 1 << 20                     # the chunked plan applies to this batch
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], None, None, d["beta"], d["cu_seqlens"],
                            d["initial_state"], g=g.numpy())
    for ws_bytes in (big, 256):
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        out, fin = chunk_prefill_logdecay(x["q"], x["k"], x["v"], g.to(dev), x["beta"], x["cu_seqlens"],
                                          x["initial_state"], workspace=ws)
        torch.cuda.synchronize()
        assert_close(f"outputs ({ws_bytes} B workspace)", out, ro, torch.bfloat16)
        assert_close(f"states ({ws_bytes} B workspace)", fin, rf, torch.bfloat16)


def test_chunked_unbounded_path_on_bounded_gate():
    """On the bounded gate's own g the chunked unbounded path equals the bounded
    chunked prefill (same layer, same tolerance)."""
    dev = need_gpu()
    w = inputs.custom([4096], H=4, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=66)
    x = to_device(inputs.prefill_inputs(w), dev)
    g = gate(x["z"], x["A"])
    ref_out, ref_fin = chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["A"], x["beta"],
                                     x["cu_seqlens"], x["initial_state"])
    out, fin = chunk_prefill_logdecay(x["q"], x["k"], x["v"], g, x["beta"], x["cu_seqlens"],
                                      x["initial_state"])
    torch.cuda.synchronize()
    assert_close("outputs", out, ref_out.double().cpu().numpy(), torch.bfloat16)
    assert_close("states", fin, ref_fin.double().cpu().numpy(), torch.bfloat16)


def test_chunked_unbounded_many_chains_against_oracle():
    """Many (sequence, head) chains: the fused kernel in its unbounded mode
    (diagonal tiles from the pre-pass, g in four float32 boxes), against the
    oracle, with a nonzero initial state and ragged lengths."""
    dev = need_gpu()
    rng = np.random.default_rng(67)
    lens = [int(x) for x in rng.integers(1, 300, size=30)]
    w = inputs.custom(lens, H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=67)
    d = inputs.prefill_inputs(w)
    g = torch.from_numpy(_unbounded_g(w.total_tokens, w.H, 128, 67))
    x = to_device(d, dev)
    out, fin = chunk_prefill_logdecay(x["q"], x["k"], x["v"], g.to(dev), x["beta"], x["cu_seqlens"],
                                      x["initial_state"])
    torch.cuda.synchronize()
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], None, None, d["beta"], d["cu_seqlens"],
                            d["initial_state"], g=g.numpy())
    assert_close("outputs", out, ro, torch.bfloat16)
    assert_close("states", fin, rf, torch.bfloat16)
