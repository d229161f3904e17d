"""The multi-rank host logic of bench.py on CPU: two gloo ranks (the replicas of a run with
--gpus 2) agree on the slowest rank's time, the job throughput counts every rank's bytes, and
the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    el = 1.5 + rank  # rank 1 is the slow one
    got = bench.max_over_ranks(torch, dist, el, torch.device("cpu"))
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp

    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    # 2 ranks x 3 steps x 4 GB in 2 s (the slowest rank's time) = 12 GB/s
    assert bench.job_gbps(4e9, 2, 3, 2.0) == pytest.approx(12.0)
    assert bench.job_gbps(4e9, 1, 3, 2.0) == pytest.approx(6.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
