"""The multi-rank path of bench.py on CPU: two gloo ranks, one process each, with
the environment torchrun gives them (RANK, WORLD_SIZE, LOCAL_RANK, MASTER_*), as
the benchmark runs with one GPU per rank; and the benchmark's host-side
bookkeeping.  No GPU is used."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(world)
    slowest = bench.dist_max(100.0 + 10.0 * rank)   # each rank's elapsed ms
    bench.barrier()
    q.put((r, w, dist.get_backend(), slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 and g[2] == "gloo" for g in got)
    assert all(g[3] == 110.0 for g in got)      # both ranks see the slowest rank's time


def test_weak_scaling_throughput():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 128 tokens x 10 steps in 20 ms (the slowest rank) = 128,000 tokens/s
    assert bench.job_throughput(2, 128, 10, 20.0) == pytest.approx(128000.0)
    assert bench.job_throughput(1, 128, 10, 20.0) == pytest.approx(64000.0)


def test_launch_count_thresholds_match_the_library():
    """bench.py counts a layer's kernels from the library's path choices: its copies
    of the thresholds must be the ones the CUDA source uses."""
    import re
    sys.path.insert(0, ROOT)
    import bench
    src = open(os.path.join(ROOT, "combine_softmax_top_expert_b300", "csrc", "layout.cu")).read()

    def const(name):
        return int(re.search(r"constexpr int " + name + r" = (\d+);", src).group(1))

    assert const("kChunk") == bench.LAYOUT_CHUNK_SLOTS
    assert const("kSmallP") == bench.SMALL_LAYOUT_EXPERTS
    assert const("kSmallRouteWork") == bench.SMALL_ROUTE_WORK


def test_reference_arm_under_torchrun_prints_once():
    """bench.py --impl reference launched like the driver launches it for N = 2:
    rank 0 times the oracle and prints one JSON line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_fp32"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
