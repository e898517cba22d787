"""kda_chunk_prefill against the oracle: the tiny float32 workload, the
4096-token prefill, the packed variable-length batch, and edge cases
(ragged tails, empty sequences, every head size, null states, split/resume,
packing, determinism, malformed offsets)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_46_gb300 import KDAError, check_device_status, chunk_prefill, inputs
from gpu_util import assert_close, device_prefill_inputs, errors, need_gpu, to_device

pytestmark = pytest.mark.gpu


def _run_gpu(d, dev, **kw):
    g = to_device(d, dev)
    out, fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"],
                             g["initial_state"], **kw)
    torch.cuda.synchronize()
    return out, fin


def _run_oracle(d):
    return oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                          d["initial_state"])


@pytest.mark.parametrize("wid", [0, 1])
def test_workload_full(wid):
    """Tiny float32 workload (tolerance 1e-4) and the 4096-token bf16 prefill
    with a random initial state, every output and the final state."""
    dev = need_gpu()
    w = inputs.workload(wid)
    d = inputs.prefill_inputs(w)
    out, fin = _run_gpu(d, dev)
    ro, rf = _run_oracle(d)
    assert_close("out", out, ro, w.dtype)
    assert_close("final state", fin, rf, w.dtype)


def test_varlen_workload_sampled_sequences():
    """The packed 64-sequence batch in one call; the oracle recomputes a sample
    of whole sequences (longest, shortest and six more) for every head."""
    dev = need_gpu()
    w = inputs.workload(2)
    g = device_prefill_inputs(w, dev)
    out, fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], None)
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    out2, _ = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], None,
                            workspace=ws)
    assert check_device_status(ws) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, out2), "two identical calls differ"
    lens = np.array(w.seq_lens)
    rng = np.random.default_rng(2024)
    pick = sorted({int(np.argmax(lens)), int(np.argmin(lens))} |
                  set(int(i) for i in rng.choice(len(lens), 6, replace=False)))
    cu = np.concatenate([[0], np.cumsum(lens)])
    for i in pick:
        b, e = int(cu[i]), int(cu[i + 1])
        d = inputs.prefill_inputs(w, 0, b, e)
        ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], [0, e - b], None)
        assert_close(f"out seq {i} (len {e - b})", out[b:e], ro, w.dtype)
        assert_close(f"final seq {i}", fin[i:i + 1], rf, w.dtype)


EDGE_LENS = [1, 15, 16, 17, 63, 64, 65, 0, 127, 128, 129, 200]


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.bfloat16, 64, 64),
                                         (torch.bfloat16, 32, 128), (torch.float32, 32, 32),
                                         (torch.float32, 64, 128), (torch.float32, 128, 128)])
@pytest.mark.parametrize("init", ["zero", "randn0.1"])
def test_edge_lengths_all_head_sizes(dtype, dk, dv, init):
    dev = need_gpu()
    w = inputs.custom(EDGE_LENS, H=3, dk=dk, dv=dv, dtype=dtype, init=init, wid=11)
    d = inputs.prefill_inputs(w)
    out, fin = _run_gpu(d, dev)
    ro, rf = _run_oracle(d)
    assert_close("out", out, ro, dtype)
    assert_close("final state", fin, rf, dtype)
    if init == "zero":   # the empty sequence passes its (zero) start state through
        assert torch.count_nonzero(fin[EDGE_LENS.index(0)]) == 0


def test_null_final_state_and_in_place_state():
    dev = need_gpu()
    w = inputs.custom([300, 77], H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=12)
    d = inputs.prefill_inputs(w)
    g = to_device(d, dev)
    out_a, none = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"],
                                g["initial_state"], want_final_state=False)
    assert none is None
    state = g["initial_state"].clone()
    out_b, fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"],
                               state, final_state=state)
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()
    assert torch.equal(out_a, out_b)
    ro, rf = _run_oracle(d)
    assert_close("out", out_b, ro, torch.bfloat16)
    assert_close("in-place final state", state, rf, torch.bfloat16)


@pytest.mark.parametrize("cut", [1, 64, 100, 333])
def test_split_and_resume(cut):
    """[0, cut) then [cut, T) from the carried state equals one call (and the oracle)."""
    dev = need_gpu()
    T = 500
    w = inputs.custom([T], H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=13)
    d = inputs.prefill_inputs(w)
    g = to_device(d, dev)
    out, fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"],
                             g["initial_state"])
    cu1 = torch.tensor([0, cut], dtype=torch.int32, device=dev)
    cu2 = torch.tensor([0, T - cut], dtype=torch.int32, device=dev)
    o1, f1 = chunk_prefill(g["q"][:cut], g["k"][:cut], g["v"][:cut], g["z"][:cut], g["A"],
                           g["beta"][:cut], cu1, g["initial_state"])
    o2, f2 = chunk_prefill(g["q"][cut:].contiguous(), g["k"][cut:].contiguous(),
                           g["v"][cut:].contiguous(), g["z"][cut:].contiguous(), g["A"],
                           g["beta"][cut:].contiguous(), cu2, f1)
    torch.cuda.synchronize()
    ro, rf = _run_oracle(d)
    both = torch.cat([o1, o2])
    assert_close("resumed out", both, ro, torch.bfloat16)
    assert_close("resumed final", f2, rf, torch.bfloat16)
    assert_close("single vs resumed", both, out.double().cpu().numpy(), torch.bfloat16)


def test_packed_equals_separate_calls_bitwise():
    """Chunks restart at every sequence start, so a packed call computes each
    (sequence, head) chain exactly as a call on that sequence alone."""
    dev = need_gpu()
    lens = [70, 1, 190, 64]
    w = inputs.custom(lens, H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=14)
    d = inputs.prefill_inputs(w)
    out, fin = _run_gpu(d, dev)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for i in range(len(lens)):
        b, e = int(cu[i]), int(cu[i + 1])
        sub = {n: d[n][b:e].contiguous() for n in ("q", "k", "v", "z", "beta")}
        sub.update(A=d["A"], cu_seqlens=torch.tensor([0, e - b], dtype=torch.int32),
                   initial_state=d["initial_state"][i:i + 1].contiguous())
        o, f = _run_gpu(sub, dev)
        assert torch.equal(o, out[b:e]) and torch.equal(f[0], fin[i]), f"sequence {i}"


def test_deterministic_bitwise():
    dev = need_gpu()
    w = inputs.custom([1000, 33, 700], H=4, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=15)
    d = inputs.prefill_inputs(w)
    a = _run_gpu(d, dev)
    b = _run_gpu(d, dev)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_malformed_offsets_are_reported_not_faulted():
    """A decreasing offset pair is caught by the kernel's own bounds check: the
    sequence is treated as empty and the device status records the error."""
    dev = need_gpu()
    w = inputs.custom([100, 100], H=2, dk=128, dv=128, dtype=torch.bfloat16, wid=16)
    d = to_device(inputs.prefill_inputs(w), dev)
    cu = torch.tensor([0, 150, 120, 200], dtype=torch.int32, device=dev)   # sequence 1 ends before it starts
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    chunk_prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], cu, None, workspace=ws)
    assert check_device_status(ws) == 1      # KDA_ERR_INVALID_ARG recorded on the device


def test_unsupported_and_invalid_arguments():
    dev = need_gpu()
    q = torch.zeros((8, 2, 96), dtype=torch.bfloat16, device=dev)
    cu = torch.tensor([0, 8], dtype=torch.int32, device=dev)
    with pytest.raises(KDAError):
        chunk_prefill(q, q, q, q, torch.zeros((2, 96), device=dev), torch.zeros((8, 2), device=dev), cu)
    q = torch.zeros((8, 2, 128), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(16, dtype=torch.uint8, device=dev)
    with pytest.raises(KDAError):
        chunk_prefill(q, q, q, q, torch.zeros((2, 128), device=dev), torch.zeros((8, 2), device=dev), cu,
                      workspace=ws)


def _run_both_paths(d, dev):
    """The same call with a minimal workspace (the fused kernel) and with the
    workspace the library asks for (the split path when the batch has few
    chains)."""
    from gated_delta_rule_46_gb300 import workspace_size
    g = to_device(d, dev)
    T, H, dk = g["q"].shape
    N = g["cu_seqlens"].shape[0] - 1
    small = torch.zeros(4096 + 4 * N, dtype=torch.uint8, device=dev)
    big = torch.zeros(workspace_size(T, N, H, dk, dk), dtype=torch.uint8, device=dev)
    assert big.numel() > small.numel(), "this batch should plan the split path"
    args = (g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], g["initial_state"])
    of, ff = chunk_prefill(*args, workspace=small)
    os_, fs = chunk_prefill(*args, workspace=big)
    torch.cuda.synchronize()
    assert check_device_status(big) == 0 and check_device_status(small) == 0
    return (of, ff), (os_, fs)


def test_split_path_matches_fused_and_oracle():
    """Few chains, ragged sequences (one empty): the chunk-parallel split path
    agrees with the oracle and with the fused kernel."""
    dev = need_gpu()
    w = inputs.custom([1500, 33, 900, 0, 640, 129], H=4, dk=128, dv=128, dtype=torch.bfloat16,
                      init="randn0.1", wid=21)
    d = inputs.prefill_inputs(w)
    (of, ff), (os_, fs) = _run_both_paths(d, dev)
    ro, rf = _run_oracle(d)
    assert_close("split out", os_, ro, torch.bfloat16)
    assert_close("split final", fs, rf, torch.bfloat16)
    assert_close("fused out", of, ro, torch.bfloat16)
    assert_close("split vs fused out", os_, of.double().cpu().numpy(), torch.bfloat16)
    assert torch.equal(fs[3], d["initial_state"][3].to(dev))   # empty sequence passes its state


def test_split_path_several_windows():
    """A sequence long enough for the split path to run several windows of
    chunks, carrying the state between them."""
    dev = need_gpu()
    w = inputs.custom([20000, 3000], H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=22)
    d = inputs.prefill_inputs(w)
    (of, ff), (os_, fs) = _run_both_paths(d, dev)
    ro, rf = _run_oracle(d)
    assert_close("split out", os_, ro, torch.bfloat16)
    assert_close("split final", fs, rf, torch.bfloat16)
    assert_close("fused final", ff, rf, torch.bfloat16)
