"""The benchmark's multi-process plumbing on the CPU: two ranks over gloo (127.0.0.1).

bench.py runs one independent replica per GPU; the only collectives are a barrier around
the timed region and the max over ranks of its elapsed time. These tests run bench.Dist
in two processes, as torchrun would launch them, and check both, plus that the
reference arm leaves every rank but 0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys, time
sys.path.insert(0, os.environ["AQ_ROOT"])
import torch
import bench

d = bench.Dist()
d.init("gloo")
t0 = time.perf_counter()
if d.rank == 1:
    time.sleep(0.5)          # the slower rank: the barrier makes rank 0 wait for it
d.barrier()
waited = time.perf_counter() - t0
elapsed = 1.25 + 2.0 * d.rank          # each rank's own "timed region"
worst = d.max(elapsed, torch.device("cpu"))
ref = bench.run_reference(None, d) if d.rank != 0 else "rank 0 runs the oracle"
d.close()
print(json.dumps({"rank": d.rank, "world": d.world, "waited": waited, "max": worst,
                  "reference_on_this_rank": ref}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_two_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                   RANK=str(rank), LOCAL_RANK=str(rank), AQ_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=180)
            assert p.returncode == 0, err[-2000:]
            outs.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    return sorted(outs, key=lambda o: o["rank"])


@pytest.fixture(scope="module")
def ranks():
    return _run_two_ranks()


def test_two_ranks_join_one_group(ranks):
    assert [o["rank"] for o in ranks] == [0, 1]
    assert all(o["world"] == 2 for o in ranks)


def test_barrier_holds_the_faster_rank(ranks):
    assert ranks[0]["waited"] >= 0.4          # rank 0 waited for the sleeping rank 1


def test_timing_is_the_max_over_ranks(ranks):
    assert all(o["max"] == 3.25 for o in ranks)


def test_reference_arm_runs_on_rank_zero_only(ranks):
    assert ranks[1]["reference_on_this_rank"] is None
