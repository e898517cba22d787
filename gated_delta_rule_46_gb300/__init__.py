"""GB300 (sm_103a) Kimi Delta Attention: gate, chunkwise prefill, decode step.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/kda.h``); ``kda`` is its thin ctypes binding and ``inputs`` the
seeded synthetic workloads.
"""
from . import inputs  # noqa: F401
from .kda import (KDAError, check_device_status, chunk_prefill, chunk_prefill_logdecay,  # noqa: F401
                  chunk_prefill_noalloc, decode_step, decode_tokens, gate, lib, library_path,
                  logdecay_workspace_size, prefill_kernel_launches, segment_map,
                  segment_map_workspace_size, state_compose, state_slots_copy,
                  testing_expire_next_wait, workspace_size)

__all__ = ["inputs", "KDAError", "chunk_prefill", "check_device_status", "decode_step", "gate",
           "lib", "library_path", "workspace_size", "chunk_prefill_noalloc", "prefill_kernel_launches",
           "decode_tokens", "chunk_prefill_logdecay", "state_slots_copy",
           "logdecay_workspace_size", "testing_expire_next_wait", "segment_map",
           "segment_map_workspace_size", "state_compose"]
