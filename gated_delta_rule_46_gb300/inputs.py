"""Seeded synthetic inputs for KDA prefill and decode.

This module only draws random numbers and lays them out; it holds none of the
KDA arithmetic.  The tests feed the same tensors to the CUDA library and to the
CPU oracle, and the benchmark uses the same recipe.

Recipe (every workload):
  * q, k ~ N(0, 1), L2-normalised over the key dimension per (token, head) in
    float32, then rounded to the input dtype (round-to-nearest-even for bf16);
  * v, z ~ N(0, 1), rounded to the input dtype;
  * beta = sigmoid(N(0, 1)), float32, one scalar per (token, head);
  * A ~ U(-1, 1), float32, one per (head, key channel);
  * initial state: zeros, or 0.1 * N(0, 1) float32 where the workload asks.

Every tensor is drawn in slabs of ``SLAB`` tokens.  Each (tensor, slab) pair has
its own numpy PCG64 stream keyed by (seed, workload id, tensor id, slab index),
so any token range can be produced on its own, in any order, on any number of
threads, and always comes out the same.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass, field

import numpy as np
import torch

SLAB = 16384

# tensor ids for the per-stream seeds
_Q, _K, _V, _Z, _BETA, _A, _STATE, _LENS = 1, 2, 3, 4, 5, 6, 7, 8


@dataclass(frozen=True)
class Workload:
    """One benchmark/parity workload (the five sizes the KDA pages' target asks for)."""
    wid: int
    name: str
    H: int
    dk: int
    dv: int
    dtype: torch.dtype
    seq_lens: tuple = ()
    init: str = "zero"          # "zero" or "randn0.1"
    decode_N: int = 0           # decode workloads: sequences per step
    decode_steps: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_lens))


def _varlen_lengths(seed: int, wid: int, n: int, lo: int, hi: int) -> tuple:
    rng = np.random.default_rng([seed, wid, _LENS, 0])
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


def workload(wid: int, seed: int = 0) -> Workload:
    """The five workloads.

    0 tiny:    1 x 64 tokens, H=2, dk=dv=32, float32, zero initial state.
    1 prefill: 1 x 4096 tokens, H=16, dk=dv=128, bf16, initial state 0.1*N(0,1).
    2 varlen:  64 packed sequences, lengths U[256, 16384], H=32, bf16, zero state.
    3 long:    1 x 1,048,576 tokens, H=32, bf16, zero state.
    4 decode:  256 sequences x 1 token per step, 128 steps, H=32, bf16 inputs,
               float32 state 0.1*N(0,1).
    """
    if wid == 0:
        return Workload(0, "tiny", 2, 32, 32, torch.float32, (64,), "zero")
    if wid == 1:
        return Workload(1, "prefill", 16, 128, 128, torch.bfloat16, (4096,), "randn0.1")
    if wid == 2:
        return Workload(2, "varlen", 32, 128, 128, torch.bfloat16,
                        _varlen_lengths(seed, 2, 64, 256, 16384), "zero")
    if wid == 3:
        return Workload(3, "long", 32, 128, 128, torch.bfloat16, (1 << 20,), "zero")
    if wid == 4:
        return Workload(4, "decode", 32, 128, 128, torch.bfloat16, (), "randn0.1",
                        decode_N=256, decode_steps=128)
    raise ValueError(f"unknown workload {wid}")


def custom(seq_lens, H, dk, dv, dtype=torch.bfloat16, init="zero", wid=100) -> Workload:
    """An ad-hoc workload for edge-case tests (any lengths, including 0)."""
    return Workload(wid, "custom", H, dk, dv, dtype, tuple(int(x) for x in seq_lens), init)


def _rng(seed, wid, tid, slab):
    return np.random.default_rng([seed, wid, tid, slab])


def _normal(seed, wid, tid, slab, shape):
    return _rng(seed, wid, tid, slab).standard_normal(shape, dtype=np.float32)


def _l2norm_lastdim(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return x / n


def _to(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t if dtype == torch.float32 else t.to(dtype)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _slab_tensor(w: Workload, seed: int, tid: int, t0: int, t1: int, inner: int,
                 normalize: bool, out: torch.Tensor):
    """Fill out[0:t1-t0] with tokens [t0, t1) of one per-token tensor."""
    H = w.H
    s_first, s_last = t0 // SLAB, (t1 - 1) // SLAB

    def one(s):
        a, b = s * SLAB, min((s + 1) * SLAB, w.total_tokens)
        x = _normal(seed, w.wid, tid, s, (b - a, H, inner))
        lo, hi = max(a, t0), min(b, t1)
        x = x[lo - a:hi - a]
        if normalize:
            x = _l2norm_lastdim(x)
        out[lo - t0:hi - t0] = _to(x, out.dtype)

    slabs = list(range(s_first, s_last + 1))
    if len(slabs) == 1:
        one(slabs[0])
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, slabs))


def prefill_inputs(w: Workload, seed: int = 0, t0: int = 0, t1: int | None = None) -> dict:
    """Host (CPU) tensors for tokens [t0, t1) of a prefill workload.

    Returns q, k, z [n, H, dk] and v [n, H, dv] in the workload dtype, beta [n, H]
    float32, A [H, dk] float32, cu_seqlens int32 for the whole workload and,
    when the workload has one, the initial state [N, H, dk, dv] float32.
    """
    T = w.total_tokens
    t1 = T if t1 is None else t1
    assert 0 <= t0 <= t1 <= T
    n = t1 - t0
    H, dk, dv = w.H, w.dk, w.dv
    res = {}
    for name, tid, inner, norm in (("q", _Q, dk, True), ("k", _K, dk, True),
                                   ("v", _V, dv, False), ("z", _Z, dk, False)):
        buf = torch.empty((n, H, inner), dtype=w.dtype)
        if n:
            _slab_tensor(w, seed, tid, t0, t1, inner, norm, buf)
        res[name] = buf
    beta = torch.empty((n, H), dtype=torch.float32)
    if n:
        s_first, s_last = t0 // SLAB, (t1 - 1) // SLAB
        for s in range(s_first, s_last + 1):
            a, b = s * SLAB, min((s + 1) * SLAB, T)
            x = _normal(seed, w.wid, _BETA, s, (b - a, H))
            x = 1.0 / (1.0 + np.exp(-x))
            lo, hi = max(a, t0), min(b, t1)
            beta[lo - t0:hi - t0] = torch.from_numpy(x[lo - a:hi - a].astype(np.float32))
    res["beta"] = beta
    res["A"] = torch.from_numpy(
        _rng(seed, w.wid, _A, 0).uniform(-1.0, 1.0, (H, dk)).astype(np.float32))
    cu = np.zeros(len(w.seq_lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(w.seq_lens, dtype=np.int64))
    res["cu_seqlens"] = torch.from_numpy(cu.astype(np.int32))
    res["initial_state"] = initial_state(w, seed)
    return res


def initial_state(w: Workload, seed: int = 0, N: int | None = None):
    """[N, H, dk, dv] float32 state, or None for a zero-initialised workload."""
    if w.init == "zero":
        return None
    N = (w.decode_N if w.decode_N else len(w.seq_lens)) if N is None else N
    x = _normal(seed, w.wid, _STATE, 0, (N, w.H, w.dk, w.dv)) * np.float32(0.1)
    return torch.from_numpy(x)


def decode_inputs(w: Workload, step: int, seed: int = 0) -> dict:
    """Host tensors for one decode step: q, k, z [N, H, dk], v [N, H, dv], beta [N, H]
    (A is shared by every step: ``decode_A``)."""
    N, H, dk, dv = w.decode_N, w.H, w.dk, w.dv
    q = _l2norm_lastdim(_normal(seed, w.wid, _Q, step, (N, H, dk)))
    k = _l2norm_lastdim(_normal(seed, w.wid, _K, step, (N, H, dk)))
    v = _normal(seed, w.wid, _V, step, (N, H, dv))
    z = _normal(seed, w.wid, _Z, step, (N, H, dk))
    b = _normal(seed, w.wid, _BETA, step, (N, H))
    b = (1.0 / (1.0 + np.exp(-b))).astype(np.float32)
    return {"q": _to(q, w.dtype), "k": _to(k, w.dtype), "v": _to(v, w.dtype),
            "z": _to(z, w.dtype), "beta": torch.from_numpy(b)}


def decode_A(w: Workload, seed: int = 0) -> torch.Tensor:
    return torch.from_numpy(
        _rng(seed, w.wid, _A, 0).uniform(-1.0, 1.0, (w.H, w.dk)).astype(np.float32))


def bytes_per_token_head(dk: int, dv: int, elem: int) -> int:
    """Algorithmic HBM bytes per (token, head) of a prefill: q, k, z, v read,
    beta read, o written."""
    return elem * (3 * dk + dv) + 4 + elem * dv


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["SLAB", "Workload", "workload", "custom", "prefill_inputs", "initial_state",
           "decode_inputs", "decode_A", "bytes_per_token_head", "ceil_div"]
