"""bench.py's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Under torchrun every rank runs its own replica; the timings are max-reduced
and the unit counts sum-reduced over ranks, and only rank 0 prints.  The GPU
work itself needs a GPU per rank and is not exercised here.
"""
import argparse
import contextlib
import io
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        # rank r: times (r + 1, 10 r), units (r + 1, 2)
        mx, sm = bench.reduce_max_sum([rank + 1.0, 10.0 * rank], [rank + 1.0, 2.0], ws)
        bench.barrier(ws)
        q.put((rank, mx, sm))
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, sm in got:
        assert mx == [2.0, 10.0], (rank, mx)   # max over ranks
        assert sm == [3.0, 4.0], (rank, sm)    # sum over ranks


def test_single_rank_reduction_is_identity():
    assert bench.reduce_max_sum([1.5, 2.5], [3.0], 1) == ([1.5, 2.5], [3.0])


def test_reference_arm_runs_on_rank_zero_only():
    args = argparse.Namespace(steps=2, warmup=3, gpus=2)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        rc = bench.run_reference(args, ws=2, rank=1)
    assert rc == 0 and out.getvalue() == ""
