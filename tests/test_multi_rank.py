"""The benchmark's multi-process path on the CPU: two gloo ranks on 127.0.0.1.

bench.py runs one independent replica per rank (the layer has no exchange step), brackets
the timed steps with barriers, takes the slowest rank's time and reports the whole-job rate.
These tests run that plumbing with world_size 2 over gloo, and check that the reference
arm's other ranks exit without work.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, sys
sys.path.insert(0, {root!r})
import torch
import bench
world, rank = bench.dist_init(2)
ms = [12.0, 30.0][rank]                      # this rank's timed region
bench.barrier(world)
slowest = bench.max_over_ranks(ms, world)
rate = bench.replica_throughput(1000, world, slowest)
bench.barrier(world)
print(json.dumps({{"rank": rank, "world": world, "backend": torch.distributed.get_backend(),
                  "slowest": slowest, "rate": rate}}))
torch.distributed.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    return dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    code = WORKER.format(root=ROOT)
    procs = [subprocess.Popen([sys.executable, "-c", code], env=_env(r, 2, port), cwd=ROOT,
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
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
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["world"] == 2 and o["backend"] == "gloo"
        assert o["slowest"] == 30.0                   # max over ranks, seen by every rank
        assert abs(o["rate"] - 1000 * 2 / 0.030) < 1e-6  # all ranks' units / slowest time


def test_reference_arm_other_ranks_exit_without_work():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=_env(1, 2, _free_port()), cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_replica_throughput_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_throughput(2600 * 40, 1, 13.0) == 2600 * 40 / 0.013
