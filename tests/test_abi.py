"""The C ABI library builds, loads without a GPU, exports every entry point
that include/kda.h declares, and rejects bad arguments on the host."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kda_\w+)\s*\(", src, flags=re.M)
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
        assert hasattr(raw, n), f"{n} declared in include/kda.h but not exported"


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
