"""The bounded-wait expiry path of the tensor-core prefill, exercised without
faulting or hanging anything.

Every mbarrier wait in the prefill kernels has a cycle budget; when one runs
out the kernel records KDA_ERR_DEVICE_TIMEOUT in the call's status word, lets
its copies and tensor-core operations in flight land, frees its tensor memory
and returns.  kda_testing_expire_next_wait() makes CTA 0 of the named kernels
wait once on a barrier that nothing arrives at, with a budget of about a
millisecond, so that this path runs for real.  Each case checks that the call
returns, that the status word reports the timeout, that no CUDA error is left
behind, and that the next ordinary call on the same buffers matches the
oracle.
"""
import pytest
import torch

import oracle
from gated_delta_rule_46_gb300 import (check_device_status, chunk_prefill,
                                       chunk_prefill_logdecay, gate, inputs,
                                       logdecay_workspace_size, prefill_kernel_launches,
                                       workspace_size)
from gated_delta_rule_46_gb300 import kda as K
from gpu_util import assert_close, need_gpu, to_device

KDA_ERR_DEVICE_TIMEOUT = K.KDA_ERR_DEVICE_TIMEOUT
expire_next_wait = K.testing_expire_next_wait   # (a name pytest does not collect)

pytestmark = pytest.mark.gpu


def _inputs(lens, H, dev):
    w = inputs.custom(lens, H=H, dk=128, dv=128, dtype=torch.bfloat16, init="randn0.1", wid=41)
    d = inputs.prefill_inputs(w)
    return d, to_device(d, dev)


def _windowed_size(T, N, H):
    """The smallest workspace that selects the windowed split plan (between the
    fused plan's minimum and the segment scan's full size)."""
    n = lambda ws: prefill_kernel_launches(T, N, H, 128, 128, torch.bfloat16, ws)
    lo, hi = 4096 + 4 * N, workspace_size(T, N, H, 128, 128)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if n(mid) == 2:
            lo = mid
        else:
            hi = mid
    hi = (hi + 255) // 256 * 256
    assert n(hi) not in (2, 5)
    return hi


# (plan, kernels to expire); the few-chain batch below selects the scan plan
# with the full workspace, the windowed plan with a middle-sized one and the
# fused kernel with the minimum.
CASES = [
    ("fused", K.KDA_TESTING_FUSED),
    ("scan", K.KDA_TESTING_INTRA),
    ("scan", K.KDA_TESTING_SEGMENT),
    ("scan", K.KDA_TESTING_SCAN),
    ("scan", K.KDA_TESTING_STATE),
    ("scan", K.KDA_TESTING_INTRA | K.KDA_TESTING_SEGMENT | K.KDA_TESTING_SCAN | K.KDA_TESTING_STATE),
    ("windows", K.KDA_TESTING_INTRA | K.KDA_TESTING_STATE),
]


@pytest.mark.parametrize("plan,kernels", CASES)
def test_expired_wait_is_reported_and_the_next_call_is_exact(plan, kernels):
    dev = need_gpu()
    lens = [1500, 900]
    H = 2
    d, g = _inputs(lens, H, dev)
    T, N = sum(lens), len(lens)
    size = {"fused": 4096 + 4 * N, "windows": _windowed_size(T, N, H),
            "scan": workspace_size(T, N, H, 128, 128)}[plan]
    launches = prefill_kernel_launches(T, N, H, 128, 128, torch.bfloat16, size)
    assert (plan == "fused") == (launches == 2) and (plan == "scan") == (launches == 5)
    ws = torch.zeros(size, dtype=torch.uint8, device=dev)
    args = (g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], g["initial_state"])
    out = torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev)

    expire_next_wait(kernels)
    chunk_prefill(*args, final_state=fin, out=out, workspace=ws)
    assert check_device_status(ws) == KDA_ERR_DEVICE_TIMEOUT
    torch.cuda.synchronize()                 # raises if the context had an error

    chunk_prefill(*args, final_state=fin, out=out, workspace=ws)   # disarmed: ordinary call
    assert check_device_status(ws) == 0
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                            d["initial_state"])
    assert_close("output after recovery", out, ro, torch.bfloat16)
    assert_close("final state after recovery", fin, rf, torch.bfloat16)


@pytest.mark.parametrize("lens", [[1500, 900], [130, 70, 200, 64] * 40])
def test_expired_wait_in_the_unbounded_decay_path(lens):
    """The same through kda_chunk_prefill_logdecay: the segment-scan plan for
    few long sequences, the fused kernel's unbounded mode for many chains."""
    dev = need_gpu()
    H = 2
    d, g = _inputs(lens, H, dev)
    T, N = sum(lens), len(lens)
    gd = gate(g["z"], g["A"])
    ws = torch.zeros(logdecay_workspace_size(T, N, H, 128, 128), dtype=torch.uint8, device=dev)
    args = (g["q"], g["k"], g["v"], gd, g["beta"], g["cu_seqlens"], g["initial_state"])
    expire_next_wait(K.KDA_TESTING_FUSED | K.KDA_TESTING_INTRA | K.KDA_TESTING_STATE)
    out, fin = chunk_prefill_logdecay(*args, workspace=ws)
    assert check_device_status(ws) == KDA_ERR_DEVICE_TIMEOUT
    torch.cuda.synchronize()
    out, fin = chunk_prefill_logdecay(*args, workspace=ws)
    assert check_device_status(ws) == 0
    ro, rf = oracle.prefill(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], d["cu_seqlens"],
                            d["initial_state"])
    assert_close("output after recovery", out, ro, torch.bfloat16)
    assert_close("final state after recovery", fin, rf, torch.bfloat16)


def test_disarmed_mask_changes_nothing():
    """Arming with 0 leaves the next prefill untouched: the status word stays
    clear and the results equal an unarmed call's bit for bit."""
    dev = need_gpu()
    d, g = _inputs([300, 77], 2, dev)
    args = (g["q"], g["k"], g["v"], g["z"], g["A"], g["beta"], g["cu_seqlens"], g["initial_state"])
    ws = torch.zeros(workspace_size(377, 2, 2, 128, 128), dtype=torch.uint8, device=dev)
    a = chunk_prefill(*args, workspace=ws)
    expire_next_wait(0)
    b = chunk_prefill(*args, workspace=ws)
    assert check_device_status(ws) == 0
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
