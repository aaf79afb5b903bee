"""Multi-process host logic of bench.py on CPU: two gloo ranks (no GPU).

The bench runs one replica per GPU; its timing takes a barrier and the max of
every rank's time, and the reference arm runs on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO_ROOT"])
import bench
d = bench.Dist(False)
assert d.on and d.ws == 2
d.barrier()
m = d.max(10.0 + d.rank)          # each rank reports its own time; all see the slowest
with open(os.path.join(os.environ["OUT_DIR"], "rank%d.json" % d.rank), "w") as f:
    json.dump({"rank": d.rank, "max": m}, f)
d.close()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch(args, timeout=120, out_dir=""):
    env = dict(os.environ, REPO_ROOT=ROOT, CUDA_VISIBLE_DEVICES="", OUT_DIR=str(out_dir))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=%d" % free_port()] + args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    script = tmp_path / "child.py"
    script.write_text(CHILD)
    r = launch([str(script)], out_dir=tmp_path)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads((tmp_path / ("rank%d.json" % i)).read_text()) for i in range(2)]
    assert sorted(x["rank"] for x in lines) == [0, 1]
    assert all(x["max"] == 11.0 for x in lines)


@pytest.mark.slow
def test_reference_arm_prints_once_under_torchrun():
    r = launch(["bench.py", "--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0"], 600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["value"] > 0
