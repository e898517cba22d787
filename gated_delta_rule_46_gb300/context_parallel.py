"""Context-parallel KDA prefill: long sequences split over several ranks.

"Kimi K3 internals analysis" (molayo1419.me), section "3T급 MoE를 위한 인프라"
(infrastructure for the 3T-class MoE), the KDA context-parallelism paragraph:
the state map of a segment of tokens is affine, S_out = M S_in + b, the maps of
consecutive segments compose associatively, and so each worker can run its own
segment, exchange a fixed-size summary of it and then finish from its true
incoming state.

Rank r holds, for every sequence of the batch, segment r of that sequence
(segments in rank order, any lengths, also zero).  One call:

  1. maps: (M, b) of this rank's segment of every (sequence, head), from the
     library (kda_segment_map);
  2. exchange: one all_gather of the maps, N x H x dk x (dk + dv) float32 per
     rank whatever the segment lengths; every rank receives them into buffers
     of its own device memory (no kernel reads another rank's memory);
  3. local exclusive scan: the maps of the ranks before this one, composed in
     order from the sequences' initial state (kda_state_compose), give this
     rank's incoming state;
  4. rerun: this rank's segment from that state (kda_chunk_prefill), which
     writes its outputs and the state after its segment; on the last rank that
     is each sequence's final state.

Every arithmetic step runs in the CUDA library; this module only orders the
calls and the collective.  `ops` lets a caller substitute the three compute
steps (the CPU tests of the exchange logic do, on gloo ranks).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import kda


class LibraryOps:
    """The three compute steps on the CUDA library."""

    def segment_map(self, q, k, v, z, A, beta, cu_seqlens):
        return kda.segment_map(q, k, v, z, A, beta, cu_seqlens)

    def state_compose(self, M, b, initial_state):
        return kda.state_compose(M, b, initial_state)

    def chunk_prefill(self, q, k, v, z, A, beta, cu_seqlens, initial_state):
        return kda.chunk_prefill(q, k, v, z, A, beta, cu_seqlens, initial_state)


def all_gather_maps(flat: torch.Tensor, group=None) -> list:
    """Every rank's `flat` (same size everywhere), in rank order, each copied
    into `flat`'s own device.  Under gloo a CUDA tensor travels through host
    memory."""
    world = dist.get_world_size(group)
    backend = dist.get_backend(group)
    src = flat if (backend == "nccl" or not flat.is_cuda) else flat.cpu()
    out = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(out, src.contiguous(), group=group)
    return [o.to(flat.device) for o in out]


def context_parallel_prefill(q, k, v, z, A, beta, cu_seqlens, initial_state=None, group=None,
                             ops=None):
    """This rank's part of a context-parallel prefill (see the module docstring).

    q, k, z [T_r, H, dk], v [T_r, H, dv], beta [T_r, H], cu_seqlens [N + 1]: this
    rank's segment of each of the N sequences, packed; A [H, dk];
    initial_state [N, H, dk, dv] or None: the start state of every sequence,
    the same on every rank.  Returns (out [T_r, H, dv], state after this
    rank's segments [N, H, dk, dv], incoming state [N, H, dk, dv]).
    """
    ops = ops or LibraryOps()
    rank = dist.get_rank(group)
    M, b = ops.segment_map(q, k, v, z, A, beta, cu_seqlens)
    flat = torch.cat([M.reshape(-1), b.reshape(-1)])
    gathered = all_gather_maps(flat, group)
    nm = M.numel()
    prior = gathered[:rank]
    if prior:
        Ms = torch.stack([g[:nm].view(M.shape) for g in prior])
        bs = torch.stack([g[nm:].view(b.shape) for g in prior])
    else:
        Ms = M.new_empty((0,) + tuple(M.shape))
        bs = b.new_empty((0,) + tuple(b.shape))
    states = ops.state_compose(Ms, bs, initial_state)
    s_in = states[rank].contiguous()
    out, s_out = ops.chunk_prefill(q, k, v, z, A, beta, cu_seqlens, s_in)
    return out, s_out, s_in
