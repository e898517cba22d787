"""Python binding of the C ABI in include/kda.h (ctypes, argument marshalling only).

Every step of the KDA path runs in the CUDA library ``libkda_gb300.so``; this
module checks shapes, dtypes, devices and contiguity of torch tensors, passes
their device pointers and the current CUDA stream, and turns a non-OK status
into an exception.  There is no fallback: if the library is missing or was
not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_DEVICE_TIMEOUT = range(5)
KDA_F32, KDA_BF16 = 0, 1
# kernels of the tensor-core prefill, as named by include/kda_testing.h
KDA_TESTING_FUSED, KDA_TESTING_INTRA, KDA_TESTING_SEGMENT, KDA_TESTING_SCAN, KDA_TESTING_STATE = (
    1, 2, 4, 8, 16)

_lock = threading.Lock()
_lib = None


class KDAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib().kda_status_string(status).decode()}")


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded CUDA library (built on first use if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not found at {path}")
            L = ctypes.CDLL(path)
            P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            L.kda_status_string.argtypes = [I]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_gate.argtypes = [P, I, P, P, I64, I, I, P]
            L.kda_gate.restype = I
            L.kda_prefill_workspace_size.argtypes = [I64, I, I, I, I, I]
            L.kda_prefill_workspace_size.restype = SZ
            L.kda_chunk_prefill.argtypes = [P, P, P, P, P, P, P, I, I64, I, I, I, I, P, P, P, P,
                                            SZ, P]
            L.kda_chunk_prefill.restype = I
            L.kda_decode_step.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P]
            L.kda_decode_step.restype = I
            L.kda_chunk_prefill_logdecay.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, I, P, P,
                                                     P, P, SZ, P]
            L.kda_chunk_prefill_logdecay.restype = I
            L.kda_prefill_logdecay_workspace_size.argtypes = [I64, I, I, I, I, I]
            L.kda_prefill_logdecay_workspace_size.restype = SZ
            L.kda_state_slots_copy.argtypes = [P, I, P, P, I, I, I, I, I, P, P]
            L.kda_state_slots_copy.restype = I
            L.kda_decode_tokens.argtypes = [P, P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, P, P]
            L.kda_decode_tokens.restype = I
            L.kda_prefill_kernel_launches.argtypes = [I64, I, I, I, I, I, SZ]
            L.kda_prefill_kernel_launches.restype = I
            L.kda_check_device_status.argtypes = [P, P]
            L.kda_check_device_status.restype = I
            L.kda_segment_map_workspace_size.argtypes = [I64, I, I, I, I, I]
            L.kda_segment_map_workspace_size.restype = SZ
            L.kda_segment_map.argtypes = [P, P, P, P, P, P, P, I, I64, I, I, I, I, P, P, P, SZ, P]
            L.kda_segment_map.restype = I
            L.kda_state_compose.argtypes = [P, P, I, I, I, I, I, P, P, P]
            L.kda_state_compose.restype = I
            L.kda_testing_expire_next_wait.argtypes = [I]
            L.kda_testing_expire_next_wait.restype = None
            _lib = L
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(t, name, shape=None, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _on(device):
    """Makes `device` current for a call: the library launches on the current
    device and takes torch's current stream of that device."""
    return torch.cuda.device(device)


def _raise(status, what):
    if status != KDA_OK:
        raise KDAError(status, what)


def gate(z: torch.Tensor, A: torch.Tensor, g_out: torch.Tensor | None = None, stream=None):
    """g = -5 sigmoid(exp(A) z) for z [T, H, dk] (bf16 or f32), A [H, dk] f32."""
    _check(z, "z")
    T, H, dk = z.shape
    _check(A, "A", (H, dk), torch.float32, z.device)
    if g_out is None:
        g_out = torch.empty((T, H, dk), dtype=torch.float32, device=z.device)
    _check(g_out, "g_out", (T, H, dk), torch.float32, z.device)
    with _on(z.device):
        _raise(lib().kda_gate(_ptr(z), _dtype_code(z), _ptr(A), _ptr(g_out), T, H, dk,
                              _stream(stream)), "kda_gate")
    return g_out


def workspace_size(total_tokens: int, num_seqs: int, H: int, dk: int, dv: int,
                   dtype: torch.dtype = torch.bfloat16) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib().kda_prefill_workspace_size(total_tokens, num_seqs, H, dk, dv, code))


def chunk_prefill(q, k, v, z, A, beta, cu_seqlens, initial_state=None, final_state=None,
                  out=None, workspace=None, want_final_state=True, stream=None):
    """KDA prefill over packed sequences.

    q, k, z [T, H, dk]; v [T, H, dv] (bf16 or f32, all the same); A [H, dk] f32;
    beta [T, H] f32; cu_seqlens [N + 1] int32 (device); initial_state
    [N, H, dk, dv] f32 or None.  Returns (out [T, H, dv], final_state or None).
    """
    _check(q, "q")
    T, H, dk = q.shape
    dv = v.shape[2] if v.dim() == 3 else -1
    dev = q.device
    for name, t in (("k", k), ("z", z)):
        _check(t, name, (T, H, dk), q.dtype, dev)
    _check(v, "v", (T, H, dv), q.dtype, dev)
    _check(A, "A", (H, dk), torch.float32, dev)
    _check(beta, "beta", (T, H), torch.float32, dev)
    _check(cu_seqlens, "cu_seqlens", None, torch.int32, dev)
    N = cu_seqlens.shape[0] - 1
    if initial_state is not None:
        _check(initial_state, "initial_state", (N, H, dk, dv), torch.float32, dev)
    if final_state is None and want_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if final_state is not None:
        _check(final_state, "final_state", (N, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _check(out, "out", (T, H, dv), q.dtype, dev)
    wsb = workspace_size(T, N, H, dk, dv, q.dtype)
    if workspace is None:
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    _check(workspace, "workspace", None, torch.uint8, dev)
    with _on(dev):
        st = lib().kda_chunk_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta),
                                     _ptr(cu_seqlens), N, T, H, dk, dv, _dtype_code(q),
                                     _ptr(initial_state), _ptr(final_state), _ptr(out),
                                     _ptr(workspace), workspace.numel(), _stream(stream))
    _raise(st, "kda_chunk_prefill")
    return out, final_state


def logdecay_workspace_size(total_tokens: int, num_seqs: int, H: int, dk: int, dv: int,
                            dtype=torch.bfloat16) -> int:
    """Workspace bytes for chunk_prefill_logdecay's chunked path."""
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib().kda_prefill_logdecay_workspace_size(total_tokens, num_seqs, H, dk, dv, code))


def chunk_prefill_logdecay(q, k, v, g, beta, cu_seqlens, initial_state=None, final_state=None,
                           out=None, workspace=None, want_final_state=True, stream=None):
    """Prefill with the log-decay g [T, H, dk] f32 given directly (no lower bound);
    the token-serial kernel.  Other arguments as chunk_prefill."""
    _check(q, "q")
    T, H, dk = q.shape
    dv = v.shape[2] if v.dim() == 3 else -1
    dev = q.device
    _check(k, "k", (T, H, dk), q.dtype, dev)
    _check(v, "v", (T, H, dv), q.dtype, dev)
    _check(g, "g", (T, H, dk), torch.float32, dev)
    _check(beta, "beta", (T, H), torch.float32, dev)
    _check(cu_seqlens, "cu_seqlens", None, torch.int32, dev)
    N = cu_seqlens.shape[0] - 1
    if initial_state is not None:
        _check(initial_state, "initial_state", (N, H, dk, dv), torch.float32, dev)
    if final_state is None and want_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    if final_state is not None:
        _check(final_state, "final_state", (N, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _check(out, "out", (T, H, dv), q.dtype, dev)
    if workspace is None:
        workspace = torch.zeros(logdecay_workspace_size(T, N, H, dk, dv, q.dtype), dtype=torch.uint8,
                                device=dev)
    _check(workspace, "workspace", None, torch.uint8, dev)
    with _on(dev):
        st = lib().kda_chunk_prefill_logdecay(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                              _ptr(cu_seqlens), N, T, H, dk, dv, _dtype_code(q),
                                              _ptr(initial_state), _ptr(final_state), _ptr(out),
                                              _ptr(workspace), workspace.numel(), _stream(stream))
    _raise(st, "kda_chunk_prefill_logdecay")
    return out, final_state


def decode_tokens(q, k, v, z, A, beta, state_pool, slot_ids=None, out=None, status=None,
                  stream=None):
    """n new tokens for each of N sequences, states in a pool (updated in place).

    q, k, z [N, n, H, dk]; v [N, n, H, dv]; beta [N, n, H] f32; state_pool
    [P, H, dk, dv] f32; slot_ids [N] int32 (device) or None for slot i = i;
    a negative slot is a padding row.  status: optional device uint32 tensor
    (e.g. a prefill workspace) that records ids >= P.  Returns out [N, n, H, dv].
    """
    _check(q, "q")
    N, n, H, dk = q.shape
    dv = v.shape[3] if v.dim() == 4 else -1
    dev = q.device
    for name, t in (("k", k), ("z", z)):
        _check(t, name, (N, n, H, dk), q.dtype, dev)
    _check(v, "v", (N, n, H, dv), q.dtype, dev)
    _check(A, "A", (H, dk), torch.float32, dev)
    _check(beta, "beta", (N, n, H), torch.float32, dev)
    _check(state_pool, "state_pool", None, torch.float32, dev)
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError(f"state_pool must be [P, {H}, {dk}, {dv}], got {tuple(state_pool.shape)}")
    if slot_ids is not None:
        _check(slot_ids, "slot_ids", (N,), torch.int32, dev)
    if out is None:
        out = torch.empty((N, n, H, dv), dtype=q.dtype, device=dev)
    _check(out, "out", (N, n, H, dv), q.dtype, dev)
    if status is not None:
        _check(status, "status", None, None, dev)
    with _on(dev):
        st = lib().kda_decode_tokens(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta),
                                     _ptr(state_pool), state_pool.shape[0], _ptr(slot_ids), _ptr(out),
                                     N, n, H, dk, dv, _dtype_code(q), _ptr(status), _stream(stream))
    _raise(st, "kda_decode_tokens")
    return out


def state_slots_copy(state_pool, slot_ids, states, to_pool=True, status=None, stream=None):
    """Copy states [N, H, dk, dv] f32 into (to_pool) or out of the pool slots
    slot_ids [N] int32 of state_pool [P, H, dk, dv] f32 (the prefill -> decode
    handoff).  Returns states."""
    _check(state_pool, "state_pool")
    P, H, dk, dv = state_pool.shape
    dev = state_pool.device
    _check(state_pool, "state_pool", (P, H, dk, dv), torch.float32, dev)
    _check(slot_ids, "slot_ids", None, torch.int32, dev)
    N = slot_ids.shape[0]
    _check(states, "states", (N, H, dk, dv), torch.float32, dev)
    if status is not None:
        _check(status, "status", None, None, dev)
    with _on(dev):
        st = lib().kda_state_slots_copy(_ptr(state_pool), P, _ptr(slot_ids), _ptr(states), N, H, dk,
                                        dv, 1 if to_pool else 0, _ptr(status), _stream(stream))
    _raise(st, "kda_state_slots_copy")
    return states


def prefill_kernel_launches(total_tokens, num_seqs, H, dk, dv, dtype, workspace_bytes) -> int:
    """Kernels one chunk_prefill call with these sizes launches (see the C header)."""
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib().kda_prefill_kernel_launches(total_tokens, num_seqs, H, dk, dv, code,
                                                 workspace_bytes))


def check_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the status word kept in the workspace."""
    _check(workspace, "workspace")
    with _on(workspace.device):
        return int(lib().kda_check_device_status(_ptr(workspace), _stream(stream)))


def decode_step(q, k, v, z, A, beta, state, out=None, stream=None):
    """One token per sequence; ``state`` [N, H, dk, dv] f32 is updated in place."""
    _check(q, "q")
    N, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    for name, t in (("k", k), ("z", z)):
        _check(t, name, (N, H, dk), q.dtype, dev)
    _check(v, "v", (N, H, dv), q.dtype, dev)
    _check(A, "A", (H, dk), torch.float32, dev)
    _check(beta, "beta", (N, H), torch.float32, dev)
    _check(state, "state", (N, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=dev)
    _check(out, "out", (N, H, dv), q.dtype, dev)
    with _on(dev):
        st = lib().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta),
                                   _ptr(state), _ptr(out), N, H, dk, dv, _dtype_code(q),
                                   _stream(stream))
    _raise(st, "kda_decode_step")
    return out


def chunk_prefill_noalloc(q, k, v, z, A, beta, cu_seqlens, initial_state=None, final_state=None,
                          out=None, stream=None):
    """kda_chunk_prefill_noalloc: the same prefill without a caller workspace
    (the library's fixed scratch is used; see include/kda.h).  ``out`` and
    ``final_state`` must be given by callers that cannot allocate; when they
    are None this wrapper allocates them with torch for convenience."""
    L = lib()
    fn = L.kda_chunk_prefill_noalloc
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    fn.argtypes = [P, P, P, P, P, P, P, I, I64, I, I, I, I, P, P, P, P]
    fn.restype = I
    _check(q, "q")
    T, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    for name, t in (("k", k), ("z", z)):
        _check(t, name, (T, H, dk), q.dtype, dev)
    _check(v, "v", (T, H, dv), q.dtype, dev)
    _check(A, "A", (H, dk), torch.float32, dev)
    _check(beta, "beta", (T, H), torch.float32, dev)
    _check(cu_seqlens, "cu_seqlens", None, torch.int32, dev)
    N = cu_seqlens.shape[0] - 1
    if initial_state is not None:
        _check(initial_state, "initial_state", (N, H, dk, dv), torch.float32, dev)
    if final_state is None:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check(final_state, "final_state", (N, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
    _check(out, "out", (T, H, dv), q.dtype, dev)
    with _on(dev):   # the scratch address and the stream are the current device's
        st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta), _ptr(cu_seqlens), N, T,
                H, dk, dv, _dtype_code(q), _ptr(initial_state), _ptr(final_state), _ptr(out),
                _stream(stream))
    _raise(st, "kda_chunk_prefill_noalloc")
    return out, final_state


def testing_expire_next_wait(kernels: int) -> None:
    """Test support (include/kda_testing.h): the next bf16 d=128 prefill call's
    kernels named by the KDA_TESTING_* mask `kernels` see one bounded wait in
    their first CTA run out, and take their timeout path."""
    lib().kda_testing_expire_next_wait(int(kernels))


def segment_map_workspace_size(total_tokens: int, num_seqs: int, H: int, dk: int, dv: int,
                               dtype: torch.dtype = torch.bfloat16) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib().kda_segment_map_workspace_size(total_tokens, num_seqs, H, dk, dv, code))


def segment_map(q, k, v, z, A, beta, cu_seqlens, M=None, b=None, workspace=None, stream=None):
    """The affine state map S_out = M S_in + b of every (sequence, head) of a
    packed batch (kda_segment_map).  Returns (M [N, H, dk, dk], b [N, H, dk, dv])."""
    _check(q, "q")
    T, H, dk = q.shape
    dv = v.shape[2] if v.dim() == 3 else -1
    dev = q.device
    for name, t in (("k", k), ("z", z)):
        _check(t, name, (T, H, dk), q.dtype, dev)
    _check(v, "v", (T, H, dv), q.dtype, dev)
    _check(A, "A", (H, dk), torch.float32, dev)
    _check(beta, "beta", (T, H), torch.float32, dev)
    _check(cu_seqlens, "cu_seqlens", None, torch.int32, dev)
    N = cu_seqlens.shape[0] - 1
    if M is None:
        M = torch.empty((N, H, dk, dk), dtype=torch.float32, device=dev)
    if b is None:
        b = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    _check(M, "M", (N, H, dk, dk), torch.float32, dev)
    _check(b, "b", (N, H, dk, dv), torch.float32, dev)
    if workspace is None:
        workspace = torch.empty(segment_map_workspace_size(T, N, H, dk, dv, q.dtype), dtype=torch.uint8,
                                device=dev)
    _check(workspace, "workspace", None, torch.uint8, dev)
    with _on(dev):
        st = lib().kda_segment_map(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(beta),
                                   _ptr(cu_seqlens), N, T, H, dk, dv, _dtype_code(q), _ptr(M), _ptr(b),
                                   _ptr(workspace), workspace.numel(), _stream(stream))
    _raise(st, "kda_segment_map")
    return M, b


def state_compose(M, b, initial_state=None, states=None, stream=None):
    """states[0] = initial_state (or zeros), states[r + 1] = M[r] states[r] + b[r]
    (kda_state_compose).  M [R, N, H, dk, dk], b [R, N, H, dk, dv] f32; returns
    states [R + 1, N, H, dk, dv]."""
    _check(M, "M", None, torch.float32)
    R, N, H, dk, dk2 = M.shape
    if dk2 != dk:
        raise ValueError("M must be [R, N, H, dk, dk]")
    dev = M.device
    _check(b, "b", None, torch.float32, dev)
    if b.dim() != 5 or tuple(b.shape[:4]) != (R, N, H, dk):
        raise ValueError(f"b must be [{R}, {N}, {H}, {dk}, dv], got {tuple(b.shape)}")
    dv = b.shape[4]
    if initial_state is not None:
        _check(initial_state, "initial_state", (N, H, dk, dv), torch.float32, dev)
    if states is None:
        states = torch.empty((R + 1, N, H, dk, dv), dtype=torch.float32, device=dev)
    _check(states, "states", (R + 1, N, H, dk, dv), torch.float32, dev)
    with _on(dev):
        st = lib().kda_state_compose(_ptr(M), _ptr(b), R, N, H, dk, dv, _ptr(initial_state),
                                     _ptr(states), _stream(stream))
    _raise(st, "kda_state_compose")
    return states
