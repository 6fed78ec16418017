"""The bench's multi-rank host logic on two CPU processes (gloo).

With --gpus N every rank runs its own replica of the block (the path has no
collective across GPUs); the ranks meet only to agree on the timing: the job
is as slow as its slowest rank, and `value` counts every replica's FLOPs.
The reference arm runs on rank 0 alone; the other ranks exit without work.
"""

import io
import multiprocessing as mp
import os
import socket
from contextlib import redirect_stdout

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    args = bench.parse_args(["--impl", "reference", "--gpus", "2"])
    world, r, local = bench.dist_setup(args)
    ms = bench.slowest_rank_ms(10.0 + 5.0 * r, world, "cpu")
    out = io.StringIO()
    if r == 1:   # rank 0 would time the oracle; the others must not
        with redirect_stdout(out):
            bench.reference_arm(args, bench.workload_cfg("layer_bf16", 0),
                                world, r)
    q.put((r, world, local, ms, bench.job_tflops(3e12, world, ms),
           out.getvalue()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_both_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in (0, 1)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, ms, val, out) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert ms == 15.0                       # max(10, 15) on both ranks
        assert val == pytest.approx(2 * 3e12 / 0.015 / 1e12)
    assert res[1][5] == ""                      # rank 1: no reference line


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.slowest_rank_ms(12.5, 1, "cpu") == 12.5
    assert bench.job_tflops(4.5e13, 1, 30.0) == pytest.approx(1500.0)
