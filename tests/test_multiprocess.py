"""The replica path of bench.py on the CPU: two gloo ranks (127.0.0.1), the
slowest rank's time, the whole-job throughput, and the reference arm printing
from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
total = bench.slowest_rank_ms(10.0 + 5.0 * rank, dist)   # rank 1 is slower
value = bench.job_tflops(world, 2.0e12, 4, total)
dist.barrier()
print(json.dumps({"rank": rank, "world": world, "total_ms": total, "value": value}), flush=True)
dist.destroy_process_group()
"""


def _launch(code, world, extra_env=None, args=()):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r), WORLD_SIZE=str(world),
                   LOCAL_RANK=str(r), ROOT=ROOT, **(extra_env or {}))
        cmd = [sys.executable, "-c", code] if code else [sys.executable, os.path.join(ROOT, "bench.py"), *args]
        procs.append(subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=240)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    outs = _launch(WORKER, 2)
    lines = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for ln in lines:
        assert ln["world"] == 2
        assert ln["total_ms"] == 15.0                       # max over ranks
        assert ln["value"] == pytest.approx(2 * 2.0e12 * 4 / 15e-3 / 1e12)  # both ranks' work


def test_reference_arm_prints_once_from_rank_zero():
    pytest.importorskip("numpy")
    outs = _launch(None, 2, args=("--impl", "reference", "--steps", "3", "--warmup", "3", "--workload", "gemm_128"))
    printed = [o.strip() for o in outs]
    assert printed[1] == ""
    line = json.loads(printed[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
