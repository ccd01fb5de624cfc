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


def _shard_worker(rank, world, port, out):
    """Each rank runs the fp64 oracle on its contiguous key-head group and the
    value heads that group owns; rank 0 gathers the slices over gloo."""
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from gated_deltanet_chunked_chunk_gb300 import workloads as W
    from gated_deltanet_chunked_chunk_gb300.sharding import shard_prefill_inputs
    case = W.prefill_case("shard", 5, 2, 150, 4, 8, 64, 64, init="all")
    g, beta = oracle.gating(case.A_log, case.a, case.b, case.dt_bias)
    g = torch.from_numpy(g).float().reshape(case.B, case.T, case.HV)
    beta = torch.from_numpy(beta).float().reshape(case.B, case.T, case.HV)
    q, k, v, gg, bb, h0 = shard_prefill_inputs(case.q, case.k, case.v, g, beta, case.initial_state, rank, world)
    o, ht = oracle.recurrent(q, k, v, gg, bb, initial_state=h0, nthreads=2)
    o_t, ht_t = torch.from_numpy(o), torch.from_numpy(ht)
    o_all = [torch.empty_like(o_t) for _ in range(world)]
    h_all = [torch.empty_like(ht_t) for _ in range(world)]
    dist.all_gather(o_all, o_t)
    dist.all_gather(h_all, ht_t)
    dist.destroy_process_group()
    if rank == 0:
        out["o"] = torch.cat(o_all, dim=2).numpy()
        out["ht"] = torch.cat(h_all, dim=1).numpy()
        o_ref, ht_ref = oracle.recurrent(case.q, case.k, case.v, g, beta, initial_state=case.initial_state,
                                         nthreads=2)
        out["o_ref"], out["ht_ref"] = o_ref, ht_ref


def test_head_group_sharding_reproduces_unsharded_result_gloo():
    import numpy as np
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_shard_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    # every (sequence, value head) is computed on its own, so the concatenation
    # of the ranks' slices is the unsharded result bit for bit
    np.testing.assert_array_equal(res["o"], res["o_ref"])
    np.testing.assert_array_equal(res["ht"], res["ht_ref"])


def test_head_shard_bounds():
    sys.path.insert(0, ROOT)
    from gated_deltanet_chunked_chunk_gb300.sharding import head_shard
    assert head_shard(16, 32, 0, 4) == (0, 4, 0, 8)
    assert head_shard(16, 32, 3, 4) == (12, 16, 24, 32)
    with pytest.raises(ValueError):
        head_shard(16, 32, 0, 3)       # 16 key heads do not split over 3 ranks
    with pytest.raises(ValueError):
        head_shard(16, 24, 0, 2)       # HV not a multiple of H
