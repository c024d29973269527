"""The multi-process bench path on CPU: two gloo ranks on 127.0.0.1 (no GPU).

Every rank of `bench.py` runs its own independent windows (replicas, no exchange on the data path).
What the ranks share is bookkeeping: the timed region's time is the maximum over ranks, and the
whole-job rate counts every rank's tokens. The reference arm runs on rank 0 only; the other ranks
exit without work or output.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_dir):
    import bench
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_env()
        assert (w, r, l) == (world, rank, rank)
        ms = bench.max_over_ranks(times[rank], w, "cpu")
        rate = bench.job_rate(w, 4, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(1.5, 2.5), (3.0, 0.25)])
def test_max_over_ranks_and_job_rate_gloo(tmp_path, times):
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), times, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    slow = max(times)
    for r in res:
        assert r["ms"] == slow                               # every rank reports the slowest time
        assert r["rate"] == pytest.approx(world * 4 / (slow * 1e-3))


def test_single_process_bookkeeping():
    import bench
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.job_rate(1, 4, 0.5) == pytest.approx(8000.0)


def test_reference_arm_other_ranks_exit_silently():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_under_torchrun_prints_one_line():
    """Two processes launched as the driver launches them; rank 0 alone times the oracle."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--layers", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
