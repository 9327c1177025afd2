"""The benchmark's multi-rank logic on CPU: two gloo ranks (no GPU).

Each GPU is an independent replica (no collective on the data path); ranks only
agree on the slowest rank's time, and the job's throughput is every rank's
bytes over that time.  The reference arm prints from rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.dist_max(1.0 + rank, dist)          # rank 1 took 2 s
    gbs = bench.job_gbs(10**9, 4, world, slowest)       # 1 GB per rank per step, 4 steps
    out[rank] = (slowest, gbs)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    slowest, gbs = out[0]
    assert slowest == 2.0
    assert gbs == pytest.approx(2 * 4 * 1.0 / 2.0)      # 8 GB over the slowest 2 s


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
