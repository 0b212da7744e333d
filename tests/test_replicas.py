"""The multi-GPU path of bench.py is N independent replicas (every (b, h) is
independent; there is no exchange on the hot path): each rank times its own
loop, the job's duration is the slowest rank's and its work the sum of the
ranks'.  Checked here with two gloo ranks on the CPU."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO_ROOT"])
import torch.distributed as dist
import bench
world, rank, local = bench.dist_setup()
dist.init_process_group("gloo", rank=rank, world_size=world)
ms, value = bench.aggregate_over_ranks(100.0 + 50.0 * rank, 10, 1e12, world, dist, "cpu")
print(json.dumps({"rank": rank, "local": local, "world": world, "ms": ms, "value": value}), flush=True)
dist.barrier()
dist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_report_the_slowest_rank_and_the_summed_work():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                   LOCAL_RANK=str(rank), REPO_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert (o["world"], o["local"]) == (2, o["rank"])
        assert o["ms"] == 150.0  # the slower rank's loop
        # 2 ranks x 10 steps x 1e12 FLOP in 0.15 s
        assert abs(o["value"] - 2 * 10 * 1e12 / 0.150 / 1e12) < 1e-9


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    ms, value = bench.aggregate_over_ranks(200.0, 4, 5e11, 1)
    assert ms == 200.0 and abs(value - 5e11 * 4 / 0.2 / 1e12) < 1e-12


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
