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


def _torchrun(args, timeout=300):
    import subprocess
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py")] + args
    env = {**os.environ, "PYTHONPATH": ROOT}
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


@pytest.fixture(scope="module")
def built_library():
    sys.path.insert(0, ROOT)
    from speculative_decoding_verify_topk_gb300 import build
    build.build()


def test_multi_rank_run_refuses_the_mla_workload(built_library):
    """Two ranks of `bench.py --workload dsv3_mla` (the absorbed-MLA kernel,
    whose cluster-multicast loads are kept to single-GPU runs) stop with a
    nonzero status and say why, before either rank touches a GPU."""
    res = _torchrun(["--gpus", "2", "--workload", "dsv3_mla", "--steps", "2", "--warmup", "3"])
    assert res.returncode != 0
    assert "single-GPU runs only" in res.stdout + res.stderr


def test_refusal_covers_only_the_mla_path(built_library):
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_verify_topk_gb300 import synth
    mla = [n for n in synth.WORKLOADS if bench.single_gpu_only(n)]
    assert mla == ["dsv3_mla"]
    args = bench.parse(["--workload", "dsv3_mla"])
    assert bench.multi_rank_refusal(args, 1) is None          # one GPU: allowed
    assert "single-GPU" in bench.multi_rank_refusal(args, 2)
    assert bench.multi_rank_refusal(bench.parse([]), 2) is None   # the default line is GQA
