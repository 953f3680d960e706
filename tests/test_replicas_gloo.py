"""The several-GPU form of the benchmark, on the CPU.

The layer does not shard: with N GPUs the benchmark runs N independent
replicas of the same step, and the only exchange is host-side bookkeeping
(the job's time is the slowest rank's; the job's rate is N replicas' bytes
over that time; rank 0 alone prints).  These tests run that bookkeeping as
two gloo ranks on 127.0.0.1, with no GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, out_dir):
    # environment as torch.distributed.run sets it
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench

    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        # each rank times a different figure; the job's time is the largest
        ms = 2.5 + 1.25 * rank
        job_ms = bench.max_over_ranks(ms, w, "cpu")
        rate = bench.whole_job_gbs(w, 3.0e9, job_ms)
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"job_ms": job_ms, "rate": rate}, f)


def test_max_over_ranks_and_whole_job_rate_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_rank_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    slowest = 2.5 + 1.25 * (world - 1)
    for g in got:
        assert g["job_ms"] == slowest                      # every rank agrees on the max
        # 2 replicas x 3 GB in 3.75 ms
        assert g["rate"] == pytest.approx(world * 3.0 / (slowest * 1e-3), rel=1e-12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench

    assert not dist.is_initialized()
    assert bench.max_over_ranks(4, 1, "cpu") == 4.0
    assert bench.whole_job_gbs(1, 2.0e9, 2.0) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched the way several GPUs are: rank 0
    alone times the oracle and prints one JSON line, rank 1 exits 0 without
    work."""
    env = dict(os.environ)
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
