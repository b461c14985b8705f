"""The multi-GPU bench path on CPU: replicas aggregated over two gloo ranks
(max over ranks, all ranks' particles), and the reference arm's rank-0-only
behaviour. No GPU and no collective in the data path."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 2.0 * rank
    value, ms = bench.aggregate_over_ranks(local_ms, 1000, world, dist, device="cpu")
    out[rank] = (value, ms)
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, 29517, out), nprocs=2, join=True)
    for rank in (0, 1):
        value, ms = out[rank]
        assert ms == 12.0
        assert value == pytest.approx(2 * 1000 / 0.012)


def test_single_rank_aggregate():
    sys.path.insert(0, ROOT)
    import bench

    value, ms = bench.aggregate_over_ranks(4.0, 1 << 20, 1)
    assert ms == 4.0 and value == pytest.approx((1 << 20) / 0.004)


def test_reference_arm_runs_the_oracle_on_cpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--cpu-sample", "4000"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--cpu-sample", "4000"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
