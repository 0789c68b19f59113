"""The benchmark's multi-process path on CPU: two gloo ranks run bench.py's rank set-up, barrier
and max-over-ranks timing reduction, and the reference arm's rank filter (only rank 0 works)."""

import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = textwrap.dedent("""
    import os, sys, time
    sys.path.insert(0, os.environ["ROOT"])
    import torch.distributed as dist
    import bench
    rank, world, local = bench.dist_setup(2)
    assert (rank, world) == (int(os.environ["RANK"]), 2) and dist.get_backend() == "gloo"
    bench.barrier(world)
    # each rank "times" a different duration; every rank must see the maximum
    v = bench.max_over_ranks(1.5 + rank, world)
    assert v == 2.5, v
    bench.barrier(world)
    print(f"rank {rank} ok {v}", flush=True)
    dist.destroy_process_group()
""")


def test_two_gloo_ranks_share_the_max_time():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, ROOT=ROOT, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = []
    for p in procs:
        out, _ = p.communicate(timeout=180)
        outs.append(out)
        assert p.returncode == 0, out
    assert "rank 0 ok 2.5" in outs[0] and "rank 1 ok 2.5" in outs[1]


REFERENCE_RANK = textwrap.dedent("""
    import os, sys
    sys.path.insert(0, os.environ["ROOT"])
    import bench
    called = []
    bench.time_oracle_for = lambda *a, **k: called.append(1) or (1.0, 1.0, 1, 1)
    class Args: gpus = 2; steps = 1; warmup = 0
    bench.run_reference(Args())
    print("worked" if called else "idle", flush=True)
""")


def test_reference_arm_runs_on_rank_zero_only():
    port = free_port()
    env = dict(os.environ, ROOT=ROOT, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    # rank 1 alone: it must return before any rendezvous or oracle work
    env["WORLD_SIZE"] = "1"
    out = subprocess.run([sys.executable, "-c", REFERENCE_RANK.replace(
        "import bench\n", "import bench\nbench.dist_setup = lambda n: (1, 2, 1)\n")],
        env=env, cwd=ROOT, capture_output=True, text=True, timeout=180)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "idle"
