"""The C ABI library builds, loads without a GPU, exports every entry point
that the headers under include/ declare, and rejects bad arguments on the
host."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def _declared_functions():
    names = []
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kda_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_46_gb300 import kda
    return kda.lib()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("kda_gate", "kda_chunk_prefill", "kda_decode_step", "kda_prefill_workspace_size",
              "kda_check_device_status", "kda_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib._name)
    for n in _declared_functions():
        assert hasattr(raw, n), f"{n} declared under include/ but not exported"


def test_status_strings(lib):
    for code in range(5):
        assert lib.kda_status_string(code).startswith(b"KDA_")


def test_host_side_validation(lib):
    from gated_delta_rule_46_gb300 import kda
    P = ctypes.c_void_p
    fake = P(4096)
    # negative sizes / unsupported head dims are rejected before any launch
    assert lib.kda_gate(fake, kda.KDA_BF16, fake, fake, -1, 2, 128, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_gate(fake, kda.KDA_BF16, fake, fake, 4, 2, 48, None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_gate(fake, 7, fake, fake, 4, 2, 128, None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_decode_step(fake, fake, fake, fake, fake, fake, fake, fake, 2, 2, 128, 96,
                               kda.KDA_BF16, None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_decode_step(None, fake, fake, fake, fake, fake, fake, fake, 2, 2, 128, 128,
                               kda.KDA_BF16, None) == kda.KDA_ERR_INVALID_ARG
    ws = lib.kda_prefill_workspace_size(1000, 3, 2, 128, 128, kda.KDA_BF16)
    assert ws >= 256 + 12 and ws % 256 == 0
    # workspace too small
    assert lib.kda_chunk_prefill(fake, fake, fake, fake, fake, fake, fake, 3, 1000, 2, 128, 128,
                                 kda.KDA_BF16, None, None, fake, fake, 16, None) == kda.KDA_ERR_INVALID_ARG
    # zero sequences: nothing to do
    assert lib.kda_chunk_prefill(None, None, None, None, None, None, None, 0, 0, 2, 128, 128,
                                 kda.KDA_BF16, None, None, None, fake, 256, None) == kda.KDA_OK
    # zero-length decode batch
    assert lib.kda_decode_step(None, None, None, None, None, None, None, None, 0, 2, 128, 128,
                               kda.KDA_BF16, None) == kda.KDA_OK
    # the unbounded-decay prefill: status word needs 4 bytes; dk outside {32, 64, 128}
    assert lib.kda_chunk_prefill_logdecay(fake, fake, fake, fake, fake, fake, 3, 1000, 2, 128, 128,
                                          kda.KDA_BF16, None, None, fake, fake, 2,
                                          None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_chunk_prefill_logdecay(fake, fake, fake, fake, fake, fake, 3, 1000, 2, 96, 128,
                                          kda.KDA_BF16, None, None, fake, fake, 256,
                                          None) == kda.KDA_ERR_UNSUPPORTED
    # the pool handoff copy: null slot ids, misaligned pool, unsupported head size
    assert lib.kda_state_slots_copy(fake, 4, None, fake, 2, 2, 128, 128, 1, None,
                                    None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_state_slots_copy(P(4100), 4, fake, fake, 2, 2, 128, 128, 1, None,
                                    None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_state_slots_copy(fake, 4, fake, fake, 2, 2, 96, 128, 0, None,
                                    None) == kda.KDA_ERR_UNSUPPORTED


def test_logdecay_workspace_sizes(lib):
    """Host-side plan sizes of the unbounded-decay path: the bounded plan's
    workspace plus 8 KB of diagonal tiles per (head, chunk slot), slots
    S = T/64 + N + 1 per head; the minimum for shapes the chunked path skips."""
    from gated_delta_rule_46_gb300 import kda
    bf, f32 = kda.KDA_BF16, kda.KDA_F32
    for T, N, H in ((4096, 1, 16), (611958, 64, 32), (538, 4, 3)):
        unb = lib.kda_prefill_logdecay_workspace_size(T, N, H, 128, 128, bf)
        bounded = lib.kda_prefill_workspace_size(T, N, H, 128, 128, bf)
        diag = H * ((T >> 6) + N + 1) * 8192
        assert unb >= diag and unb % 256 == 0
        assert unb >= diag + min(bounded, 256)
    # float32 or other head sizes: the token-serial kernel, the bounded minimum
    assert lib.kda_prefill_logdecay_workspace_size(4096, 1, 16, 128, 128, f32) == \
        lib.kda_prefill_workspace_size(4096, 1, 16, 128, 128, f32)
    assert lib.kda_prefill_logdecay_workspace_size(4096, 1, 16, 64, 64, bf) == \
        lib.kda_prefill_workspace_size(4096, 1, 16, 64, 64, bf)


def test_bindings_reject_host_tensors():
    """The product path has no CPU fallback: host tensors are refused before
    any library call."""
    import torch
    from gated_delta_rule_46_gb300 import chunk_prefill_logdecay, state_slots_copy
    q = torch.zeros(8, 1, 32, dtype=torch.float32)
    with pytest.raises(ValueError):
        chunk_prefill_logdecay(q, q, q, q, torch.zeros(8, 1), torch.tensor([0, 8], dtype=torch.int32))
    with pytest.raises(ValueError):
        state_slots_copy(torch.zeros(2, 1, 32, 32), torch.zeros(1, dtype=torch.int32), torch.zeros(1, 1, 32, 32))
