"""The seeded input generator: deterministic, slab-independent, right shapes."""
import numpy as np
import torch

from gated_delta_rule_46_gb300 import inputs


def test_token_ranges_match_full_draw():
    w = inputs.custom([70000, 3000], H=2, dk=8, dv=4, dtype=torch.bfloat16, init="randn0.1", wid=7)
    full = inputs.prefill_inputs(w)
    part = inputs.prefill_inputs(w, t0=65000, t1=70500)
    for n in ("q", "k", "v", "z", "beta"):
        assert torch.equal(full[n][65000:70500], part[n]), n
    assert torch.equal(full["A"], part["A"])
    assert torch.equal(full["initial_state"], part["initial_state"])
    again = inputs.prefill_inputs(w)
    assert all(torch.equal(full[n], again[n]) for n in ("q", "k", "v", "z", "beta"))


def test_shapes_dtypes_and_distributions():
    w = inputs.workload(1)
    d = inputs.prefill_inputs(w)
    assert d["q"].shape == (4096, 16, 128) and d["q"].dtype == torch.bfloat16
    assert d["v"].shape == (4096, 16, 128) and d["beta"].shape == (4096, 16)
    assert d["A"].shape == (16, 128) and d["initial_state"].shape == (1, 16, 128, 128)
    assert d["cu_seqlens"].tolist() == [0, 4096]
    nq = d["q"].float().norm(dim=-1)
    assert torch.all((nq - 1).abs() < 1e-2)
    assert 0 < d["beta"].min() and d["beta"].max() < 1
    assert -1 <= d["A"].min() and d["A"].max() <= 1
    assert abs(d["initial_state"].std().item() - 0.1) < 2e-3
    w0 = inputs.workload(0)
    d0 = inputs.prefill_inputs(w0)
    assert d0["q"].dtype == torch.float32 and d0["initial_state"] is None


def test_varlen_lengths_and_decode():
    w = inputs.workload(2)
    assert len(w.seq_lens) == 64 and min(w.seq_lens) >= 256 and max(w.seq_lens) <= 16384
    w4 = inputs.workload(4)
    a = inputs.decode_inputs(w4, 3)
    b = inputs.decode_inputs(w4, 3)
    c = inputs.decode_inputs(w4, 4)
    assert torch.equal(a["q"], b["q"]) and not torch.equal(a["q"], c["q"])
    assert a["q"].shape == (256, 32, 128) and a["beta"].shape == (256, 32)
