"""world_size-2 checks of the multi-GPU bookkeeping on CPU (gloo): the step
time is the max over ranks and the rate counts every rank's replica; the
reference arm runs on rank 0 only.  No GPU and no NCCL are involved."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank                   # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms, world)
    rate = bench.whole_job_rate(65536, world, ms)
    dist.barrier()
    dist.destroy_process_group()
    out[rank] = (ms, rate)


def test_max_over_ranks_and_whole_job_rate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]                         # every rank sees the same numbers
    ms, rate = res[0]
    assert ms == 15.0                               # the slowest rank
    assert abs(rate - 2 * 65536 / 0.015) < 1e-6     # both replicas' tokens over the slowest time


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(100, 1, 10.0) == 10000.0


def test_reference_arm_skips_nonzero_ranks(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        cpu_tokens, steps, warmup, gpus = 64, 1, 0, 2
    bench.run_reference(A(), rank=1, world=2)      # returns at once, prints nothing
    assert capsys.readouterr().out == ""
