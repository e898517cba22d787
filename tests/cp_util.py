"""Helpers of the context-parallel tests (no KDA arithmetic here): splitting a
packed batch into per-rank segments, and running a function on gloo ranks."""
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_segments(d, lens, cuts):
    """Per rank, the packed inputs of its segment of every sequence.

    d: full packed inputs (q, k, v, z, beta [T, ...], A, cu_seqlens);
    cuts[i]: the split points of sequence i (len(cuts[i]) = world - 1).
    Returns a list over ranks of dicts with q, k, v, z, beta, A, cu_seqlens and
    `spans` (the (start, end) token range of each segment in the full batch)."""
    world = len(cuts[0]) + 1
    cu = np.concatenate([[0], np.cumsum(lens)])
    out = []
    for r in range(world):
        spans = []
        for i, L in enumerate(lens):
            edges = [0] + list(cuts[i]) + [L]
            spans.append((int(cu[i] + edges[r]), int(cu[i] + edges[r + 1])))
        seg = {}
        for n in ("q", "k", "v", "z", "beta"):
            parts = [d[n][a:b] for a, b in spans]
            seg[n] = torch.cat(parts).contiguous()
        seg["A"] = d["A"]
        seg["cu_seqlens"] = torch.tensor(np.concatenate([[0], np.cumsum([b - a for a, b in spans])]),
                                         dtype=torch.int32)
        seg["spans"] = spans
        out.append(seg)
    return out


def _entry(rank, world, port, fn, args, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, HERE)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        results[rank] = fn(rank, world, *args)
    finally:
        dist.destroy_process_group()


def run_ranks(world, fn, *args, timeout=600):
    """Runs fn(rank, world, *args) on `world` spawned gloo ranks; returns the
    results by rank (fn must be importable by the children)."""
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    port = free_port()
    procs = [ctx.Process(target=_entry, args=(r, world, port, fn, args, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=timeout)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0] * world, codes
    return [results[r] for r in range(world)]
