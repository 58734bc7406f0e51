"""The benchmark's multi-process path on CPU (gloo, world size 2): the barrier,
the max over ranks of the timed region and the whole-job aggregation, and the
reference arm's rule that only rank 0 runs and prints."""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent

CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import bench
d = bench.Dist("gloo")
d.barrier()
ms = 10.0 * (d.rank + 1)                  # rank 1 is the slow one
worst = d.max(ms)
print(json.dumps({"rank": d.rank, "world": d.world, "max_ms": worst,
                  "value": bench.whole_job_gbs(d.world, 1000, 5, worst)}), flush=True)
d.barrier()
d.close()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, world: int, port: int) -> dict:
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), ROOT=str(ROOT))
    env.pop("CUDA_VISIBLE_DEVICES", None)
    return env


def test_two_ranks_take_the_max_time_and_aggregate():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", CHILD], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2 and o["max_ms"] == 20.0
        # 2 ranks x 1000 bytes x 5 steps over the slowest rank's 20 ms.
        assert o["value"] == pytest.approx(2 * 1000 * 5 / 0.020 / 1e9)


def test_reference_arm_runs_on_rank_zero_only():
    port = _free_port()
    p = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=_env(1, 2, port), capture_output=True, text=True,
                       timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_whole_job_rate_is_weak_scaling():
    import bench
    one = bench.whole_job_gbs(1, 859_758_592, 100, 31.9)
    assert bench.whole_job_gbs(4, 859_758_592, 100, 31.9) == pytest.approx(4 * one)
    assert bench.whole_job_gbs(2, 1, 1, 1.0) == pytest.approx(2e-6)
