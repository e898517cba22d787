"""fp64 CPU oracle for Kimi Delta Attention (KDA).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline arm of ``bench.py`` may import this package.  The product path
(``gated_delta_rule_46_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision, token by
token); this module only builds that file with gcc, loads it with ctypes and
marshals numpy arrays.  Its definitions follow "Kimi K3 internals analysis"
(molayo1419.me), section "Sequence mixing": the bounded gate
g = -5 * sigmoid(exp(A) * z), alpha = exp(g), and the delta-rule write into a
fixed-size state whose old contents decay channel-wise before the write.

Every function of the oracle is pinned by ``tests/test_oracle_pins.py``
against closed forms and independently derived formulations (see the test
module's docstring for the list).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into oracle/_build/libkda_oracle.so with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
               "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.kda_oracle_gate.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
            lib.kda_oracle_gate.restype = None
            lib.kda_oracle_prefill.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               P, P, P, ctypes.c_int]
            lib.kda_oracle_prefill.restype = ctypes.c_int
            lib.kda_oracle_decode_step.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int]
            lib.kda_oracle_decode_step.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(x):
    """Contiguous float32 numpy view/copy of a numpy array or CPU torch tensor.

    bf16 and fp32 values are exactly representable in float32, so this
    conversion loses nothing."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def gate(z, A) -> np.ndarray:
    """g[t, h, c] = -5 * sigmoid(exp(A[h, c]) * z[t, h, c]) in float64."""
    z32, A32 = _f32(z), _f32(A)
    T, H, dk = z32.shape
    assert A32.shape == (H, dk)
    g = np.empty((T, H, dk), dtype=np.float64)
    _load().kda_oracle_gate(_ptr(z32), _ptr(A32), _ptr(g), T, H, dk)
    return g


def prefill(q, k, v, z, A, beta, cu_seqlens, initial_state=None, g=None,
            threads: int | None = None):
    """Token-by-token KDA over packed sequences.

    q, k, z: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; A: [H, dk];
    cu_seqlens: [N + 1] offsets; initial_state: [N, H, dk, dv] or None (zeros);
    g: optional log-decay [T, H, dk] used instead of (z, A).
    Returns (out [T, H, dv] float64, final_state [N, H, dk, dv] float64).
    """
    q32, k32, v32 = _f32(q), _f32(k), _f32(v)
    T, H, dk = q32.shape
    dv = v32.shape[2]
    b32 = _f32(beta)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens if not hasattr(cu_seqlens, "numpy")
                                         else cu_seqlens.cpu().numpy()), dtype=np.int64)
    N = cu.shape[0] - 1
    z32 = _f32(z) if g is None else None
    A32 = _f32(A) if g is None else None
    g64 = _f64(g)
    s0 = _f64(initial_state)
    out = np.empty((T, H, dv), dtype=np.float64)
    fin = np.empty((N, H, dk, dv), dtype=np.float64)
    rc = _load().kda_oracle_prefill(_ptr(q32), _ptr(k32), _ptr(v32), _ptr(z32), _ptr(A32),
                                    _ptr(g64), _ptr(b32), _ptr(cu), N, H, dk, dv, _ptr(s0),
                                    _ptr(fin), _ptr(out), threads or default_threads())
    if rc != 0:
        raise ValueError("kda_oracle_prefill rejected its arguments")
    return out, fin


def decode_step(q, k, v, z, A, beta, state, threads: int | None = None):
    """One token per sequence: q, k, z [N, H, dk]; v [N, H, dv]; beta [N, H];
    state [N, H, dk, dv] (float64, updated copy returned).
    Returns (out [N, H, dv] float64, new_state float64)."""
    q32, k32, v32, z32, A32, b32 = map(_f32, (q, k, v, z, A, beta))
    N, H, dk = q32.shape
    dv = v32.shape[2]
    st = np.array(_f64(state), dtype=np.float64, copy=True, order="C")
    out = np.empty((N, H, dv), dtype=np.float64)
    rc = _load().kda_oracle_decode_step(_ptr(q32), _ptr(k32), _ptr(v32), _ptr(z32), _ptr(A32),
                                        _ptr(b32), _ptr(st), _ptr(out), N, H, dk, dv,
                                        threads or default_threads())
    if rc != 0:
        raise ValueError("kda_oracle_decode_step rejected its arguments")
    return out, st
