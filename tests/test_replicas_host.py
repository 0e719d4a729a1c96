"""The N > 1 path of bench.py on CPU (gloo, world size 2): process-group
setup from the launcher's environment, the barrier, the max-over-ranks of the
step time and the whole-job aggregate, and the reference arm under torchrun
(rank 0 alone prints one JSON line, the other rank exits without work).
Replicas only: no collective touches the data path."""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CHILD = r"""
import json, os, sys, types
sys.path.insert(0, os.environ["REPO"])
import bench
args = types.SimpleNamespace(impl="reference")
world, rank, local, pg = bench.dist_setup(args)
bench.barrier(pg)
ms = 10.0 + 5.0 * rank                      # per-rank step time (ms)
ms_max = bench.max_over_ranks(pg, ms)
flops_per_rank = 1.0e12
value = world * flops_per_rank / (ms_max * 1e-3) / 1e12
bench.barrier(pg)
print(json.dumps({"rank": rank, "world": world, "ms_max": ms_max, "value": value}))
pg.destroy_process_group()
"""


def test_two_gloo_ranks_agree_on_max_time_and_aggregate():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, REPO=ROOT, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["world"] == 2
        assert o["ms_max"] == 15.0                 # the slower rank's time
        assert abs(o["value"] - 2 * 1.0 / 0.015) < 1e-9   # whole-job aggregate over both ranks


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle"
