"""The bench's multi-GPU path is replicas only (no data-path collective): each
rank runs its own batch, and the job's time is the max over ranks. This runs
that host logic as two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_verify_topk_gb300 import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        local_ms = [120.0, 175.5][rank]          # rank 1 is the slow replica
        job_ms = bench.max_over_ranks(local_ms, w, torch.device("cpu"))
        rate = bench.job_rate(w, 50, job_ms)
        wl = synth.WORKLOADS["llama8b_gqa"]
        lens = synth.draw_lengths(wl, seed=bench.replica_seed(wl, r))[0].tolist()
        results[rank] = (w, r, local, job_ms, rate, lens)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_the_slowest_replica():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    assert sorted(res) == [0, 1]
    for rank, (w, r, local, job_ms, rate, _) in res.items():
        assert (w, r, local) == (world, rank, rank)
        assert job_ms == 175.5                   # max over ranks, seen by every rank
        assert rate == pytest.approx(world * 50 / 0.1755)
    assert res[0][5] != res[1][5]                # each replica draws its own batch


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_rate(1, 10, 1000.0) == 10.0
