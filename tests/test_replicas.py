"""The multi-GPU path is replicas only: each rank runs the whole step on its
own GPU and the job reports the units of all ranks over the slowest rank's
time.  Covered here on the CPU with two gloo ranks: the max-over-ranks
reduction the bench uses, the barrier, and that only rank 0 runs and prints
the reference arm."""

import contextlib
import io
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, q):
    import bench
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank], ws)
        dist.barrier()
        ws_env, rank_env, _ = bench.dist_env()
        out = io.StringIO()
        if rank != 0:  # the reference arm does no work on other ranks
            with contextlib.redirect_stdout(out):
                bench.run_reference(type("A", (), {"batch": 4, "cpu_sample": 1, "warmup": 3, "steps": 1})())
        q.put((rank, got, ws_env, rank_env, out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_and_only_rank0_reports():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(ws):
        rank, got, ws_env, rank_env, out = q.get(timeout=120)
        res[rank] = (got, ws_env, rank_env, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (got, ws_env, rank_env, out) in res.items():
        assert got == [2.0, 10.0, 0.5], got          # element-wise max over both ranks
        assert (ws_env, rank_env) == (ws, rank)
    assert res[1][3] == ""                            # rank 1 printed nothing for the reference arm
