"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one replica per rank (the product has no exchange step) and
reduces only its timings: a barrier around the timed region and the maximum
of the ranks' elapsed times.  Those pieces, and the launch of the reference
arm under torch.distributed.run (rank 0 prints the one JSON line, the other
ranks exit 0 without work), are exercised here without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # each rank's "elapsed time": the job's time is the slowest rank's
    got = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    out[rank] = got
    bench.barrier(w)
    dist.destroy_process_group()


def test_barrier_and_max_over_two_gloo_ranks():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "square_256_f16"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=280, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_roofline_bound_follows_arithmetic_intensity():
    """The bench's roofline is tensor-bound for 4096^3 + bias and HBM-bound
    for 16 x 16384^2, at the measured peaks of a GB300 (1951 TFLOP/s bf16,
    6791 GB/s copy)."""
    sys.path.insert(0, ROOT)
    import bench
    b, mem = bench.roofline_bound(4096, 4096, 4096, 4096, 4096, 1951.4, 6791.4)
    assert b == 2.0 * (3 * 4096 * 4096 + 4096) and not mem      # 14.8 us of bytes, 70 us of flops
    b, mem = bench.roofline_bound(16, 16384, 16384, 16384, 0, 1951.4, 6791.4)
    assert b == 2.0 * (16 * 16384 * 2 + 16384 * 16384) and mem  # 79 us of bytes, 4.4 us of flops
    # SwiGLU writes half the columns
    b, _ = bench.roofline_bound(8192, 28672, 4096, 14336, 0, 1951.4, 6791.4)
    assert b == 2.0 * (8192 * 4096 + 4096 * 28672 + 8192 * 14336)
    # no peaks known: never claims a memory bound
    assert bench.roofline_bound(16, 16384, 16384, 16384, 0, None, None)[1] is False
