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
