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


def test_varlen_workload_every_sequence():
    """The packed 64-sequence batch in one call (the fused plan, 2,048 chains);
    the oracle recomputes every sequence for every head, outputs and final
    states.  The sequences are compared one by one so that host memory stays
    at one sequence's inputs."""
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
    del g, out2
    lens = np.array(w.seq_lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    worst = (0.0, 0.0)
    for i in range(len(lens)):
        b, e = int(cu[i]), int(cu[i + 1])
        d = inputs.prefill_inputs(w, 0, b, e)
        ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], [0, e - b], None)
        r1 = assert_close(f"out seq {i} (len {e - b})", out[b:e], ro, w.dtype)
        r2 = assert_close(f"final seq {i}", fin[i:i + 1], rf, w.dtype)
        worst = (max(worst[0], r1[0], r2[0]), max(worst[1], r1[1], r2[1]))
    print(f"varlen, all {len(lens)} sequences: worst rel-L2 {worst[0]:.2e}, max-abs {worst[1]:.2e}")


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


@pytest.mark.parametrize("dtype,dk,dv,slow", [(torch.float32, 128, 128, False), (torch.float32, 128, 128, True),
                                              (torch.float32, 32, 64, True), (torch.bfloat16, 64, 32, True),
                                              (torch.bfloat16, 32, 128, False)])
def test_chunked_float32_path_long_sequences(dtype, dk, dv, slow):
    """The chunkwise float32 kernel (float32 inputs, head sizes 32 and 64) over
    sequences of many 16-token chunks, the state carried from chunk to chunk;
    with gates near 0 (z shifted down by 10) the carried state dominates the
    outputs.  Tolerance 1e-4 for float32, the bf16 one otherwise."""
    dev = need_gpu()
    w = inputs.custom([1200, 301, 16], H=2, dk=dk, dv=dv, dtype=dtype, init="randn0.1", wid=17)
    d = inputs.prefill_inputs(w)
    if slow:
        d["z"] = (d["z"].float() - 10.0).to(dtype)
    out, fin = _run_gpu(d, dev)
    ro, rf = _run_oracle(d)
    assert_close("out", out, ro, dtype)
    assert_close("final state", fin, rf, dtype)


@pytest.mark.parametrize("n_seqs,dtype,dk,dv", [(160, torch.float32, 32, 32), (100, torch.float32, 32, 32),
                                                 (8, torch.bfloat16, 64, 64)])
def test_chunked_float32_path_value_blocks(n_seqs, dtype, dk, dv):
    """The chunkwise float32 kernel's value blocks: 32 channels per CTA when a
    batch gives at least two CTAs per SM, else 16 or 8 (on a 152-SM GPU: 320
    chains of 32 channels take the 32-channel block, 200 the 16-channel one,
    16 chains of 64 the 8-channel one).  Ragged lengths, a random start state,
    against the oracle."""
    dev = need_gpu()
    rng = np.random.default_rng(23 + n_seqs)
    lens = [int(x) for x in rng.integers(1, 60, n_seqs)]
    w = inputs.custom(lens, H=2, dk=dk, dv=dv, dtype=dtype, init="randn0.1", wid=23)
    d = inputs.prefill_inputs(w)
    out, fin = _run_gpu(d, dev)
    ro, rf = _run_oracle(d)
    assert_close("out", out, ro, dtype)
    assert_close("final state", fin, rf, dtype)


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


def _plan_workspaces(T, N, H):
    """Workspace sizes that select each tensor-core plan for this batch: the
    minimum (one fused kernel), the smallest size that leaves it (the windowed
    split plan) and the size the library asks for (the segment scan, for few
    chains).  The plan a size selects is read from the launch count."""
    from gated_delta_rule_46_gb300 import prefill_kernel_launches, workspace_size
    n = lambda ws: prefill_kernel_launches(T, N, H, 128, 128, torch.bfloat16, ws)
    small, big = 4096 + 4 * N, workspace_size(T, N, H, 128, 128)
    assert n(small) == 2 and n(big) == 5, (n(small), n(big))
    lo, hi = small, big
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if n(mid) == 2:
            lo = mid
        else:
            hi = mid
    hi = (hi + 255) // 256 * 256
    assert n(hi) not in (2, 5), "the windowed plan should sit between the other two"
    return small, hi, big


def _run_plans(d, dev):
    """The same call under each plan; returns {plan: (out, final)}."""
    g = to_device(d, dev)
    T, H, dk = g["q"].shape
    N = g["cu_seqlens"].shape[0] - 1
    sizes = dict(zip(("fused", "windows", "scan"), _plan_workspaces(T, N, H)))
    args = (g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], g["initial_state"])
    res = {}
    for plan, size in sizes.items():
        ws = torch.zeros(size, dtype=torch.uint8, device=dev)
        res[plan] = chunk_prefill(*args, workspace=ws)
        torch.cuda.synchronize()
        assert check_device_status(ws) == 0, plan
    return res


def test_split_plans_match_fused_and_oracle():
    """Few chains, ragged sequences (one empty, one shorter than a segment):
    the windowed split plan and the segment scan agree with the oracle and
    with the fused kernel."""
    dev = need_gpu()
    w = inputs.custom([1500, 33, 900, 0, 640, 129], H=4, dk=128, dv=128, dtype=torch.bfloat16,
                      init="randn0.1", wid=21)
    d = inputs.prefill_inputs(w)
    res = _run_plans(d, dev)
    ro, rf = _run_oracle(d)
    for plan, (o, f) in res.items():
        assert_close(f"{plan} out", o, ro, torch.bfloat16)
        assert_close(f"{plan} final", f, rf, torch.bfloat16)
        assert torch.equal(f[3], d["initial_state"][3].to(dev)), plan   # empty sequence passes its state
    for plan in ("windows", "scan"):
        assert_close(f"{plan} vs fused out", res[plan][0], res["fused"][0].double().cpu().numpy(),
                     torch.bfloat16)


def test_split_plans_long_sequence():
    """A sequence long enough for several windows (state carried between them)
    and for a few dozen scan segments, next to a shorter one."""
    dev = need_gpu()
    w = inputs.custom([20000, 3000], H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=22)
    d = inputs.prefill_inputs(w)
    res = _run_plans(d, dev)
    ro, rf = _run_oracle(d)
    for plan, (o, f) in res.items():
        assert_close(f"{plan} out", o, ro, torch.bfloat16)
        assert_close(f"{plan} final", f, rf, torch.bfloat16)


def test_slow_decay_all_plans():
    """Gates close to 0 (z shifted down by 10, so exp(A) z is far below 0 and
    g = -5 sigmoid(.) is small): the state keeps its memory over many chunks,
    so the carried state, the W S correction and the segment maps of the scan
    carry the result instead of decaying away within a chunk.  Every plan
    against the oracle."""
    dev = need_gpu()
    w = inputs.custom([3000, 1100, 700], H=4, dk=128, dv=128, dtype=torch.bfloat16,
                      init="randn0.1", wid=23)
    d = inputs.prefill_inputs(w)
    d["z"] = (d["z"].float() - 10.0).to(torch.bfloat16)
    g = oracle.gate(d["z"][:256], d["A"])
    assert (g.mean(axis=0) > -0.01).mean() > 0.3    # a third of the channels barely decay
    res = _run_plans(d, dev)
    ro, rf = _run_oracle(d)
    for plan, (o, f) in res.items():
        assert_close(f"{plan} out", o, ro, torch.bfloat16)
        assert_close(f"{plan} final", f, rf, torch.bfloat16)
