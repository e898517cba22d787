"""The multi-rank paths of bench.py on the CPU: two gloo ranks on 127.0.0.1.

bench.py --gpus N runs one process per GPU under torchrun; every rank works
on its own seeded copy of the workloads (no collective on the data path) and
the timed result is the slowest rank's, taken with one all-reduce.  These
tests run that host logic with the gloo backend: the max over ranks, the
per-rank seeds giving different inputs, and the reference arm letting rank 0
alone do the work.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from gated_delta_rule_46_gb300 import inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the slowest rank's time wins on every rank
        t = bench.max_over_ranks(1.5 + rank, world, "cpu")
        # bench seeds each rank's workload by its rank: different inputs
        d = inputs.prefill_inputs(inputs.workload(0), seed=rank)
        first = float(d["q"].flatten()[0])
        gathered = [None] * world
        dist.all_gather_object(gathered, first)
        # the reference arm: ranks other than 0 return at once
        class Args:
            steps, warmup, gpus = 1, 3, world
        rc = bench.run_reference(Args()) if rank != 0 else None
        results[rank] = (t, gathered, rc, bench._dist())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0, p.exitcode
    for r in range(world):
        t, gathered, rc, d = results[r]
        assert t == 1.5 + (world - 1)                       # max over ranks, same on every rank
        assert gathered[0] != gathered[1]                   # rank-seeded inputs differ
        assert d == (r, world, r)
        if r != 0:
            assert rc == 0                                  # no work off rank 0


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
