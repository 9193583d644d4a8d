"""The N > 1 timing logic of the benchmark on CPU ranks (gloo, world size 2):
max over ranks, whole-job aggregation, and rank-0-only reference output."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:{port}", rank=int(sys.argv[1]), world_size=2)
import bench
rank = dist.get_rank()
secs = [1.5, 2.0][rank]
m = bench.max_over_ranks(secs)
gbs = bench.aggregate_gbs(1e9, 10, m, dist.get_world_size())
print(json.dumps({{"rank": rank, "max": m, "gbs": gbs}}))
dist.destroy_process_group()
"""


def _free_port():
    import socket

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_max_over_ranks_and_aggregate_on_two_gloo_ranks():
    pytest.importorskip("torch")
    import json

    code = WORKER.format(root=ROOT, port=_free_port())
    procs = [subprocess.Popen([sys.executable, "-c", code, str(r)], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                              text=True) for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["max"] == 2.0  # the slowest rank decides
        assert abs(o["gbs"] - 1e9 * 10 * 2 / 2.0 / 1e9) < 1e-9  # 2 replicas x 10 steps x 1 GB / 2 s


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--gpus", "2"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_single_process_max_is_identity():
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.aggregate_gbs(2e9, 4, 2.0, 1) == 4.0
