"""The bench's multi-rank path on CPU: two gloo ranks on 127.0.0.1.

Each rank of `bench.py --gpus N` runs its own replica of the workload (the
(sequence, head) units are independent, so there is no collective on the data
path); the ranks meet only in a barrier around the timed region and in the
max-over-ranks of the elapsed time.  These tests run those helpers as two real
processes, and check that the reference arm does its work on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import bench
ws, rank, local = bench.dist_setup()
import torch.distributed as dist
backend = dist.get_backend()
bench.barrier(ws)
# elapsed times differ per rank; the job's time is the slowest rank's
mx = bench.max_over_ranks(1.5 * (rank + 1), ws)
bench.barrier(ws)
dist.destroy_process_group()
print(json.dumps({"ws": ws, "rank": rank, "local": local, "backend": backend, "max": mx}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, ws, port):
    env = dict(os.environ)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(ws),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    return env


def test_gloo_two_ranks_barrier_and_max():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", WORKER, ROOT], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["ws"] == 2 and o["backend"] == "gloo"
        assert o["max"] == pytest.approx(3.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = _env(1, 2, _free_port())
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=180)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
