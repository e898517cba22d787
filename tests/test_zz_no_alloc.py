"""kda_chunk_prefill_noalloc: the prefill for callers that cannot allocate.

Some callers cannot call cudaMalloc when they run a prefill (plugin code whose
host application owns all device memory, serving loops with a memory budget
fixed at start-up, code that must not take the allocator's implicit device
synchronisation).  The no-alloc entry point takes no workspace and uses a
fixed scratch array inside the library instead.  These tests call it through
the C ABI, twice in a row on the same inputs (the second call reuses the
scratch the first one left behind), and check both results against the
regular kda_chunk_prefill within the parity tolerance.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

from gated_delta_rule_46_gb300 import chunk_prefill, chunk_prefill_noalloc, inputs, kda
from gpu_util import assert_close, need_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 64)])
def test_noalloc_matches_regular_entry_point_twice(dtype, dk, dv):
    dev = need_gpu()
    lens = [1, 63, 64, 65, 0, 300, 129]
    w = inputs.custom(lens, H=3, dk=dk, dv=dv, dtype=dtype, init="randn0.1", wid=91)
    g = to_device(inputs.prefill_inputs(w), dev)
    ref_out, ref_fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"],
                                     g["cu_seqlens"], g["initial_state"])
    # a caller that cannot allocate passes its own output buffers
    out = torch.empty_like(ref_out)
    fin = torch.empty_like(ref_fin)
    for call in range(2):
        out.fill_(float("nan"))
        fin.fill_(float("nan"))
        chunk_prefill_noalloc(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"],
                              g["initial_state"], final_state=fin, out=out)
        torch.cuda.synchronize()
        assert_close(f"call {call} output", out, ref_out.double().cpu().numpy(), dtype)
        assert_close(f"call {call} final state", fin, ref_fin.double().cpu().numpy(), dtype)


def test_noalloc_rejects_too_many_sequences_before_launch():
    need_gpu()
    L = kda.lib()
    fn = L.kda_chunk_prefill_noalloc
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.argtypes = [P, P, P, P, P, P, P, I, I64, I, I, I, I, P, P, P, P]
    fn.restype = I
    fake = P(4096)   # never dereferenced: the size check comes first
    too_many = 16384 + 1
    st = fn(fake, fake, fake, fake, fake, fake, fake, too_many, 10, 2, 128, 128, kda.KDA_BF16,
            None, None, fake, None)
    assert st == kda.KDA_ERR_UNSUPPORTED


def _min_workspace(N, dev):
    """The smallest workspace kda_chunk_prefill accepts: the fused plan only."""
    return torch.zeros((256 + 4 * N + 255) // 256 * 256, dtype=torch.uint8, device=dev)


def test_noalloc_is_bitwise_the_fused_plan_and_matches_the_oracle():
    """With the minimum workspace kda_chunk_prefill runs the same one-kernel plan
    as the no-alloc call, so the two agree bit for bit; both are checked
    against the oracle directly."""
    import oracle
    from gated_delta_rule_46_gb300 import check_device_status
    dev = need_gpu()
    lens = [1, 63, 64, 65, 0, 300, 129, 1000]
    w = inputs.custom(lens, H=3, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=92)
    d = inputs.prefill_inputs(w)
    g = to_device(d, dev)
    ws = _min_workspace(len(lens), dev)
    ref_out, ref_fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"],
                                     g["cu_seqlens"], g["initial_state"], workspace=ws)
    assert check_device_status(ws) == 0
    out, fin = chunk_prefill_noalloc(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"],
                                     g["cu_seqlens"], g["initial_state"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                            d["initial_state"])
    assert_close("no-alloc output vs oracle", out, ro, torch.bfloat16)
    assert_close("no-alloc final state vs oracle", fin, rf, torch.bfloat16)


def test_noalloc_few_long_chains_match_the_segment_scan_plan():
    """One sequence of 2048 tokens with two heads: kda_chunk_prefill with its
    full workspace runs the segment-scan plan, the no-alloc call the fused
    kernel; they sum in different orders and agree within the tolerance, and
    both match the oracle."""
    import oracle
    from gated_delta_rule_46_gb300 import prefill_kernel_launches, workspace_size
    dev = need_gpu()
    w = inputs.custom([2048], H=2, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=93)
    d = inputs.prefill_inputs(w)
    g = to_device(d, dev)
    full = workspace_size(2048, 1, 2, 128, 128)
    assert prefill_kernel_launches(2048, 1, 2, 128, 128, torch.bfloat16, full) == 5
    ref_out, ref_fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"],
                                     g["cu_seqlens"], g["initial_state"])
    out, fin = chunk_prefill_noalloc(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"],
                                     g["cu_seqlens"], g["initial_state"])
    torch.cuda.synchronize()
    assert_close("no-alloc vs segment scan output", out, ref_out.double().cpu().numpy(), torch.bfloat16)
    assert_close("no-alloc vs segment scan state", fin, ref_fin.double().cpu().numpy(), torch.bfloat16)
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                            d["initial_state"])
    assert_close("no-alloc output vs oracle", out, ro, torch.bfloat16)
    assert_close("no-alloc final state vs oracle", fin, rf, torch.bfloat16)


def test_noalloc_at_the_largest_accepted_batch():
    """num_seqs == KDA_NOALLOC_MAX_SEQS: the longest-first schedule fills the
    fixed scratch exactly.  Very short sequences (0 to 3 tokens), one head;
    bit for bit against kda_chunk_prefill's fused plan, whose status word must
    stay clear, and against the oracle."""
    import numpy as np
    import oracle
    from gated_delta_rule_46_gb300 import check_device_status
    dev = need_gpu()
    n = 16384
    lens = [int(x) for x in np.random.default_rng(7).integers(0, 4, n)]
    w = inputs.custom(lens, H=1, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=94)
    d = inputs.prefill_inputs(w)
    g = to_device(d, dev)
    ws = _min_workspace(n, dev)
    ref_out, ref_fin = chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"],
                                     g["cu_seqlens"], g["initial_state"], workspace=ws)
    assert check_device_status(ws) == 0
    for call in range(2):
        out, fin = chunk_prefill_noalloc(g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"],
                                         g["cu_seqlens"], g["initial_state"])
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin), f"call {call}"
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                            d["initial_state"])
    assert_close("output vs oracle", out, ro, torch.bfloat16)
    assert_close("final state vs oracle", fin, rf, torch.bfloat16)
