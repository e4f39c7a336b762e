"""bench.py is a one-GPU benchmark: it refuses --gpus other than 1 and any
launch with WORLD_SIZE above 1 (a torchrun job) before touching a GPU, and
its reference arm (the CPU oracle) runs at N = 1.  All of this runs on CPU."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, **env):
    full_env = dict(os.environ, **env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=full_env,
                          capture_output=True, text=True, timeout=600)


def test_more_than_one_gpu_is_refused():
    for args, env in ((["--gpus", "2"], {}), (["--gpus", "8", "--impl", "reference"], {}),
                      ([], {"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1", "MASTER_ADDR": "127.0.0.1"}),
                      (["--impl", "reference"], {"WORLD_SIZE": "4", "RANK": "0"})):
        r = _bench(args, **env)
        assert r.returncode == 2, (args, env, r.stdout, r.stderr)
        assert r.stdout.strip() == ""
        msg = r.stderr.strip().splitlines()
        assert len(msg) == 1 and "one GPU only" in msg[0], r.stderr


def test_reference_arm_runs_at_one_gpu():
    r = _bench(["--impl", "reference", "--workload", "i4i4_256", "--steps", "2", "--warmup", "3"],
               WORLD_SIZE="1")
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
