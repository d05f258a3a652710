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


def test_reference_arm_prints_one_contract_line():
    # rank 0 runs the oracle on bounded samples of the workloads and prints the
    # same JSON line as the GPU arm, marked as the reference
    import json
    args = argparse.Namespace(steps=1, warmup=3, gpus=1)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        rc = bench.run_reference(args, ws=1, rank=0)
    lines = [l for l in out.getvalue().splitlines() if l.strip()]
    assert rc == 0 and len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]
