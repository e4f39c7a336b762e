"""The N > 1 path of bench.py on CPU: world_size-2 gloo process groups (127.0.0.1).

Replicas only: each rank runs its own GEMM, the only exchange is the MAX of
the ranks' timed regions; the reference arm runs on rank 0 alone.
"""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out_dir):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.max_over_ranks(values[rank], dist, "cpu")
        value = bench.whole_job_value(2.0e12, 10, world, slowest)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world, values = 2, [0.25, 0.5]
    mp.spawn(_worker, args=(world, _free_port(), values, str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    # both ranks see the slowest time; the job's TOPS count both replicas' work over it
    assert all(r["slowest"] == 0.5 for r in res)
    assert all(abs(r["value"] - 2.0e12 * 10 * 2 / 0.5 / 1e12) < 1e-9 for r in res)


def _run_reference(rank: int):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                           "i4i4_256", "--steps", "2", "--warmup", "3"], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


def test_reference_arm_runs_on_rank0_only():
    other = _run_reference(1)
    assert other.returncode == 0 and other.stdout.strip() == ""
    first = _run_reference(0)
    assert first.returncode == 0, first.stderr
    line = json.loads(first.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
