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
