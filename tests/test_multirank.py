"""The multi-process path of bench.py on CPU: two gloo ranks, as torchrun
launches them (127.0.0.1 rendezvous).  Covers the host logic only: the
replicas share no data, the job time is the slowest rank's, the job value
counts every rank's tokens, and only rank 0 of the reference arm runs."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as WL  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.rank_env()
        ms = [3.0, 5.5][rank]  # the second rank is slower
        slowest = bench.max_over_ranks(torch, ms, w, torch.device("cpu"))
        value = bench.job_throughput(128, w, slowest)
        # Each replica draws its own requests (seed = rank).
        idx = WL.row_adapters(WL.LLAMA8B_R16, "verify", k=1, seed=r)
        # Reference arm: only rank 0 times the oracle; the others exit 0 silently.
        out = io.StringIO()
        rc = None
        if r != 0:
            with redirect_stdout(out):
                rc = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "gpus": w})())
        q.put((r, w, lr, slowest, value, idx.tolist(), rc, out.getvalue()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.start_processes(_rank_main, args=(world, port, q), nprocs=world, join=True, start_method="spawn")
    res = sorted(q.get(timeout=60) for _ in range(world))
    for r, (rank, w, local, slowest, value, _, rc, out) in enumerate(res):
        assert (rank, w, local) == (r, world, r)
        assert slowest == 5.5                                  # max over ranks
        assert value == pytest.approx(128 * world / 5.5e-3)    # whole-job tokens/s
        if rank != 0:
            assert rc == 0 and out == ""
    assert res[0][5] != res[1][5]                              # disjoint request draws per replica


def test_single_rank_helpers():
    assert bench.max_over_ranks(torch, 2.5, 1, torch.device("cpu")) == 2.5
    assert bench.job_throughput(128, 1, 0.25) == pytest.approx(512000.0)
    assert np.isfinite(bench.job_throughput(1, 8, 1e-3))
