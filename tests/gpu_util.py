"""Helpers shared by the GPU parity tests (no KDA arithmetic here)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_46_gb300 import inputs

# Tolerances of the parity target: bf16 inputs with float32 accumulation, and
# the float32 workload.  rel-L2 = ||x - y|| / ||y|| over the tensor compared,
# max-abs = max |x - y|; outputs and states are compared separately.
BF16_REL, BF16_ABS = 1e-2, 5e-2
F32_REL, F32_ABS = 1e-4, 1e-4


def tol_for(dtype):
    return (BF16_REL, BF16_ABS) if dtype == torch.bfloat16 else (F32_REL, F32_ABS)


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch.device("cuda:0")


def errors(got, ref):
    g = got.detach().double().cpu().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite values"
    diff = g - r
    den = np.linalg.norm(r)
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    mx = float(np.max(np.abs(diff))) if diff.size else 0.0
    return rel, mx


def assert_close(name, got, ref, dtype):
    rel_tol, abs_tol = tol_for(dtype)
    rel, mx = errors(got, ref)
    assert rel <= rel_tol and mx <= abs_tol, f"{name}: rel-L2 {rel:.3e} (<= {rel_tol}), max-abs {mx:.3e} (<= {abs_tol})"
    return rel, mx


def to_device(d, dev):
    return {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in d.items()}


def device_prefill_inputs(w, dev, seed=0, slab=8 * inputs.SLAB):
    """The whole workload on the device, generated slab by slab (host memory
    stays at one slab)."""
    T, H = w.total_tokens, w.H
    out = {
        "q": torch.empty((T, H, w.dk), dtype=w.dtype, device=dev),
        "k": torch.empty((T, H, w.dk), dtype=w.dtype, device=dev),
        "v": torch.empty((T, H, w.dv), dtype=w.dtype, device=dev),
        "z": torch.empty((T, H, w.dk), dtype=w.dtype, device=dev),
        "beta": torch.empty((T, H), dtype=torch.float32, device=dev),
    }
    for t0 in range(0, T, slab):
        t1 = min(T, t0 + slab)
        d = inputs.prefill_inputs(w, seed, t0, t1)
        for n in ("q", "k", "v", "z", "beta"):
            out[n][t0:t1].copy_(d[n])
    d = inputs.prefill_inputs(w, seed, 0, 0)
    out["A"] = d["A"].to(dev)
    out["cu_seqlens"] = d["cu_seqlens"].to(dev)
    out["initial_state"] = None if d["initial_state"] is None else d["initial_state"].to(dev)
    return out
