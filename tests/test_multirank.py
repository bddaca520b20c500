"""The N > 1 path of bench.py on the CPU: world-size-2 gloo ranks on
127.0.0.1.

With N GPUs the benchmark runs N independent replicas (the step has no
data-path exchange on one GPU per process); the only cross-rank steps are the
barriers and taking the slowest rank's time, from which the whole-job
throughput is formed.  Those are exercised here with real process groups; the
reference arm's non-zero ranks must exit without output.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    sys.path.insert(0, ROOT)
    import bench
    dist.barrier()
    ms = bench.max_over_ranks(10.0 + 7.5 * rank, world, "cpu")          # the slowest rank's time
    v = bench.replica_throughput(world, 65536, 4, ms)
    dist.barrier()
    with open(os.path.join(outdir, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": v}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_throughput(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    assert res[0] == res[1]
    assert res[0]["ms"] == 17.5
    assert res[0]["value"] == pytest.approx(2 * 65536 * 4 / 0.0175)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.replica_throughput(1, 1000, 10, 500.0) == pytest.approx(20000.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
