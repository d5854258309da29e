"""Benchmark of fgemm on the proj_4096_bf16_bias workload (and others).

Default run (N = 1): C = A @ B + bias, M = N = K = 4096, bf16, A ~ N(0,1),
B ~ N(0,1/K), bias ~ N(0, 0.02^2), algorithm picked by the decision model,
through the public binding (fgemm.matmul -> fgemm_matmul_ex).  Prints ONE
JSON line.  Four rotating input/output sets (384 MB, more than the L2) are
cycled so that every timed step streams its operands from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fgemm|reference]
                    [--workload NAME] [--algo auto|classical|strassen1|strassen2|winograd1]
                    [--tile 0|64|128|256]

The roofline object reports the kernel against the measured bf16 peak (TFLOP/s),
or against the measured copy bandwidth (GB/s of A, B, C and bias read or
written once) when those bytes at that bandwidth take longer than the flops at
the peak, as for the small-M shapes.

--impl reference times the fp64 CPU oracle on host cores (a bounded sample
of the same workload per step): the comparison arm; there is no installable
reference implementation of this method.

Under torchrun (N > 1) every rank runs its own replica of the workload on
its own GPU (the product has no exchange step); value = total FLOPs of all
ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "effective TFLOP/s (2*M*N*K/t) bf16 GEMM"
UNIT = "TFLOP/s"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=250)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fgemm", choices=["fgemm", "reference"])
    ap.add_argument("--workload", default="square_16384_bf16")
    ap.add_argument("--algo", default="auto")
    ap.add_argument("--tile", type=int, default=0, help="tile_n (0 = model)")
    ap.add_argument("--tile-m", type=int, default=0, help="tile_m: 128 one CTA, 256 CTA pair")
    ap.add_argument("--sets", type=int, default=0, help="rotating input sets (0 = auto)")
    ap.add_argument("--split", default="auto", choices=["off", "auto", "force"],
                    help="K split of the last wave of CTA-pair tiles")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-forms", action="store_true",
                    help="skip the same-run timing of the other forms and of the 256^3 case")
    ap.add_argument("--sweep", action="store_true",
                    help="decision-model check: every legal form/tile vs auto on the sweep shapes")
    ap.add_argument("--out", default=None, help="JSON-lines file for --sweep")
    ap.add_argument("--mx", default=None, choices=["e4m3", "e5m2"],
                    help="time the block-scaled 8-bit (MX) product on the workload's shape")
    return ap.parse_args()


# ----------------------------------------------------------- distributed

def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local % max(1, torch.cuda.device_count()))
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- workload

def workload_shape(name):
    from complexity_matmul_tcgen05_gb300 import inputs
    if name in inputs.WORKLOADS:
        w = inputs.WORKLOADS[name]
        return w["M"], w["N"], w["K"], w["dtype"], w["epi"]
    m = re.fullmatch(r"sweep_(\d+)x(\d+)x(\d+)", name)
    if m:
        M, N, K = map(int, m.groups())
        return M, N, K, "bf16", "none"
    raise SystemExit(f"unknown workload {name}")


def make_inputs(name, device):
    from complexity_matmul_tcgen05_gb300 import inputs
    if name in inputs.WORKLOADS:
        return inputs.workload_inputs(name, device)
    M, N, K, _, _ = workload_shape(name)
    A, B = inputs.sweep_inputs(M, N, K, device)
    return A, B, None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------- peaks / ncu

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), d.get("hbm_gbs"), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def roofline_bound(M, N, K, n_out, bias_elems, tflops, gbs):
    """(algorithmic bytes, memory-bound?) of one 16-bit product: A, B, C and
    the bias read or written once, against 2MNK flops; memory-bound when those
    bytes at `gbs` take longer than the flops at `tflops`."""
    alg_bytes = 2.0 * (M * K + K * N + M * n_out + bias_elems)
    flops = 2.0 * M * N * K
    return alg_bytes, bool(tflops and gbs) and alg_bytes / (gbs * 1e9) > flops / (tflops * 1e12)


# The device-code sources each form's kernels are built from.
COMMON_SOURCES = ("fgemm_internal.h", "fgemm_ptx.cuh", "fgemm_kernel.cuh")
FORM_SOURCES = {
    "classical_pair": ("fgemm_kernel_pair.cuh", "fgemm_kern_pair.cu"),
    "classical": ("fgemm_kern_classical.cu",),
    "classical_small_m": ("fgemm_kern_skinny.cu",),
    "lcma_pair": ("fgemm_kern_lcma.cu",),
    "strassen1": ("fgemm_kern_strassen1.cu",),
    "strassen2": ("fgemm_kern_strassen2.cu",),
    "winograd1": ("fgemm_kern_winograd1.cu",),
}


def form_key(algo, tile_m):
    if algo == "classical":
        return "classical_pair" if tile_m == 256 else ("classical_small_m" if tile_m < 128 else "classical")
    if tile_m == 256 and algo in ("strassen1", "strassen2", "winograd1"):
        return "lcma_pair"
    return algo


def kernel_source_hash(algo="classical", tile_m=256):
    """Hash of the device-code sources of one form's kernels: recorded ncu
    counters are used only while the kernels they were taken on are
    unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "complexity_matmul_tcgen05_gb300", "csrc")
    for f in COMMON_SOURCES + FORM_SOURCES[form_key(algo, tile_m)]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def ncu_traffic(workload, algo, tile_m, tile):
    """DRAM bytes per launch recorded under profiles/ for this workload, if
    the counters were taken on the current kernel sources."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    want = kernel_source_hash(algo, tile_m)
    pat = re.compile(r"traffic_bytes_per_launch\s*:\s*(\d+)\s+workload=(\S+)\s+algo=(\S+)\s+"
                     r"tile=(\d+)x(\d+)\s+sources=(\w+)")
    for f in sorted(os.listdir(pdir)):
        if not f.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, f)) as fh:
            for line in fh:
                m = pat.search(line)
                if m and m.group(2) == workload and m.group(3) == algo and \
                        int(m.group(4)) == tile_m and int(m.group(5)) == tile and \
                        m.group(6) == want:
                    return int(m.group(1))
    return None


# ----------------------------------------------------------- CPU oracle

def cpu_oracle_sample(name, target_s=10.0, device_inputs=None, entries=None):
    """Times the fp64 oracle on a bounded sample of the workload's output
    entries (each a K-long dot product of decoded 16-bit inputs): `entries`
    of them, or as many as take about target_s.  Returns (TFLOP/s, seconds,
    entries, threads)."""
    import numpy as np
    import oracle
    from complexity_matmul_tcgen05_gb300 import inputs
    M, N, K, dtype, epi = workload_shape(name)
    if device_inputs is None:
        A, B, bias = make_inputs(name, "cpu")
    else:
        A, B, bias = (None if t is None else t.cpu() for t in device_inputs)
    Ab, Bb = inputs.bits(A), inputs.bits(B)
    bb = None if bias is None else inputs.bits(bias)
    n_out = N // 2 if epi == "swiglu" else N
    per_entry = 2.0 * K * (2 if epi == "swiglu" else 1)
    n = entries if entries else 256
    elapsed = 0.0
    while True:
        rows, cols = inputs.sample_positions(M, n_out, n=n)
        t0 = time.perf_counter()
        oracle.reference_sampled(Ab, Bb, dtype, rows.numpy(), cols.numpy(), epi, 1.0, bb)
        elapsed = time.perf_counter() - t0
        if entries or elapsed >= target_s or n >= (1 << 26):
            break
        grow = max(2.0, min(16.0, target_s / max(elapsed, 1e-3)))
        n = int(n * grow)
    entries = rows.numel()
    return per_entry * entries / elapsed / 1e12, elapsed, entries, oracle.num_threads()


# --------------------------------------------------------------- arms

def workload_config(name):
    """The workload's identity, the same in both arms: what the numbers are on."""
    M, N, K, dtype, epi = workload_shape(name)
    return {"workload": name, "M": M, "N": N, "K": K, "dtype": dtype, "epilogue": epi}


def run_reference(args, rank, world):
    """The comparison arm: the fp64 CPU oracle, as it stands, on host cores."""
    if rank != 0:
        return
    M, N, K, dtype, epi = workload_shape(args.workload)
    # inputs drawn once; the sample size fixed in the warm-up so that each
    # step takes about per_step seconds and the whole run about two minutes
    per_step = min(3.0, 100.0 / max(1, args.steps))
    host_inputs = make_inputs(args.workload, "cpu")
    _, t_probe, n_probe, _ = cpu_oracle_sample(args.workload, target_s=per_step / 4,
                                               device_inputs=host_inputs)
    n_step = max(256, int(n_probe * per_step / max(t_probe, 1e-6)))
    for _ in range(max(0, args.warmup)):
        cpu_oracle_sample(args.workload, device_inputs=host_inputs, entries=max(256, n_step // 16))
    vals, secs, ents = [], 0.0, 0
    for _ in range(args.steps):
        v, s, e, thr = cpu_oracle_sample(args.workload, device_inputs=host_inputs, entries=n_step)
        vals.append(v)
        secs += s
        ents += e
    value = 2.0 * K * (2 if epi == "swiglu" else 1) * ents / secs / 1e12
    sample = (f"{ents} sampled output entries over {args.steps} steps, each a K={K} fp64 dot "
              f"product of decoded {dtype} inputs (stratified, seed 3)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(args.workload),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_calls(fn, n, stream):
    """Mean ms of n back-to-back calls of fn(i) (CUDA events around each on
    `stream`), and the ms of the whole run."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(n):
        ev[i][0].record(stream)
        fn(i)
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev), t0.elapsed_time(t1)


def time_forms(A, B, C, bias, epi, algos, handle, stream, target_ms=1500.0, max_rounds=60):
    """The given forms on the same inputs, each with the model's best tile of
    that form, timed round-robin: every round runs each form once (CUDA
    events around each call), so the forms see the same clocks and power
    state; rounds continue for about target_ms.  Returns {algo: (median ms,
    calls)}."""
    from complexity_matmul_tcgen05_gb300 import fgemm

    def call(algo):
        fgemm.matmul(A, B, out=C, epilogue=epi, bias=bias, algo=algo, handle=handle)

    for algo in algos:
        call(algo)
        call(algo)
    torch.cuda.synchronize()
    times = {a: [] for a in algos}
    elapsed = 0.0
    rounds = 0
    while rounds < 3 or (elapsed < target_ms and rounds < max_rounds):
        for algo in algos:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call(algo)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            times[algo].append(ms)
            elapsed += ms
        rounds += 1
    if handle.get_error() != fgemm.OK:
        raise SystemExit(f"device error timing {algos}: {handle.last_message()}")
    return {a: (statistics.median(t), len(t)) for a, t in times.items()}


def run_fgemm(args, rank, world):
    from complexity_matmul_tcgen05_gb300 import fgemm
    M, N, K, dtype, epi = workload_shape(args.workload)
    dev = torch.device("cuda", torch.cuda.current_device())
    A0, B0, bias0 = make_inputs(args.workload, dev)
    n_out = N // 2 if epi == "swiglu" else N
    set_bytes = 2 * (M * K + K * N + M * n_out)
    l2 = 126 * 2 ** 20
    sets = args.sets if args.sets > 0 else max(1, min(8, math.ceil(3 * l2 / set_bytes)))
    As, Bs, Cs, biases = [A0], [B0], [], [bias0]
    for i in range(1, sets):   # distinct copies so each step misses the L2
        As.append(A0.clone())
        Bs.append(B0.clone())
        biases.append(None if bias0 is None else bias0.clone())
    for i in range(sets):
        Cs.append(torch.empty((M, n_out), dtype=A0.dtype, device=dev))
    if sets == 1:
        l2_note = (f"inputs larger than the L2: A {M * K * 2 / 2 ** 20:.0f} MiB, "
                   f"B {K * N * 2 / 2 ** 20:.0f} MiB, C {M * n_out * 2 / 2 ** 20:.0f} MiB")
    else:
        l2_note = (f"{sets} rotating input/output sets ({sets * set_bytes / 2 ** 20:.0f} MiB) "
                   f"cycled between steps")
    handle = fgemm.default_handle()
    handle.set_split_mode(args.split)
    stream = torch.cuda.current_stream(dev)
    algo, tile, tile_m = args.algo, args.tile, args.tile_m
    # the form and tile the calls run (AUTO's choice, or the forced form with
    # the model's best tile of it where none is given), and the kernels each
    # call launches
    plan_algo, plan_tm, plan_tile, pred_us = handle.plan(M, N, K, fgemm._dtype_code(A0.dtype),
                                                         fgemm.make_epilogue(epi), algo=algo,
                                                         tile_m=tile_m, tile_n=tile)
    per_call = handle.call_launches(M, N, K, fgemm.make_epilogue(epi), algo=algo, tile_m=tile_m,
                                    tile_n=tile)

    def step(i):
        fgemm.matmul(As[i % sets], Bs[i % sets], out=Cs[i % sets], epilogue=epi,
                     bias=biases[i % sets], algo=algo, tile_n=tile, tile_m=tile_m, handle=handle)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    if handle.get_error() != fgemm.OK:
        raise SystemExit(f"device error during warm-up: {handle.last_message()}")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step(i)
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.25)  # at least one clock sample after the last step
    barrier(world)
    status = handle.get_error()
    if status != fgemm.OK:
        raise SystemExit(f"device error in the timed region: {handle.last_message()}")
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    kern_ms = [a.elapsed_time(b) for a, b in ev]
    kern_avg_ms = statistics.mean(kern_ms)
    flops = 2.0 * M * N * K
    value = flops * world * args.steps / (total_ms * 1e-3) / 1e12

    # The other forms on the same inputs in the same run (the classical
    # kernel and the Strassen-like forms, each with the model's best tile of
    # that form), after the timed region.
    depth = {"classical": 0, "strassen1": 1, "strassen2": 2, "winograd1": 1}
    burst, sustained, hbm, src = measured_peaks()
    long_step = total_ms >= 500.0
    peak = sustained if (long_step and sustained) else burst
    peak_kind = "sustained" if (long_step and sustained) else "burst"
    forms = {}
    if rank == 0 and not args.no_forms:
        w = inputs_mod().WORKLOADS.get(args.workload, {})
        legal, tiles = [], {}
        for form in ("classical", "strassen1", "strassen2", "winograd1"):
            if form not in w.get("algos", ()) and not (form == "classical"):
                continue
            if fgemm.validate(M, N, K, 16, K, 16, N, 16, n_out, fgemm._dtype_code(A0.dtype),
                              fgemm.make_epilogue(epi, 1.0, 16 if bias0 is not None else None),
                              form) != fgemm.OK:
                continue
            _, f_tm, f_tn, f_us = handle.plan(M, N, K, fgemm._dtype_code(A0.dtype),
                                              fgemm.make_epilogue(epi), algo=form)
            legal.append(form)
            tiles[form] = (f_tm, f_tn, f_us)
        # forms predicted within 1.5x of the fastest share the rounds; each
        # slower one (two Strassen levels) is timed in rounds of its own, so
        # that its long, DRAM-heavy calls do not sit between the calls of
        # the forms compared with each other
        fast = min(tiles[f][2] for f in legal) if legal else 0.0
        groups = [[f for f in legal if tiles[f][2] <= 1.5 * fast]] + \
            [[f] for f in legal if tiles[f][2] > 1.5 * fast]
        for g in groups:
            if not g:
                continue
            res = time_forms(As[0], Bs[0], Cs[0], biases[0], epi, g, handle, stream,
                             target_ms=1500.0 if len(g) > 1 else 400.0)
            for form, (ms, n) in res.items():
                eff = flops / (ms * 1e-3) / 1e12
                executed = eff * (7.0 / 8.0) ** depth[form]
                forms[form] = {"tile_m": tiles[form][0], "tile_n": tiles[form][1],
                               "ms_per_call": ms, "calls": n, "predicted_ms": tiles[form][2] / 1e3,
                               "effective_tflops": eff, "executed_tflops": executed,
                               "executed_frac_of_peak": executed / peak if peak else None,
                               "timing": "median of per-call CUDA events, " +
                                         ("forms round-robin" if len(g) > 1 else "in rounds of its own")}
        if "classical" in forms:
            for f, d in forms.items():
                d["vs_classical"] = d["effective_tflops"] / forms["classical"]["effective_tflops"]

    # The small fp16 case (256^3, classical and one-level Strassen): launch-
    # bound, so it is reported as time per call, back to back and as one
    # launch alone.
    small = None
    if rank == 0 and not args.no_forms and args.workload != "square_256_f16":
        sA, sB, _ = make_inputs("square_256_f16", dev)
        sC = torch.empty((256, 256), dtype=sA.dtype, device=dev)
        small = {"workload": "square_256_f16"}
        for form in ("classical", "strassen1"):
            def call(i, form=form):
                fgemm.matmul(sA, sB, out=sC, algo=form, handle=handle)
            for i in range(5):
                call(i)
            back_to_back, _ = time_calls(call, 200, stream)
            alone = statistics.median(time_calls(call, 1, stream)[0] for _ in range(20))
            f_algo, f_tm, f_tn, pred = handle.plan(256, 256, 256, fgemm.F16, None, algo=form)
            small[form] = {"tile_m": f_tm, "tile_n": f_tn, "us_back_to_back": back_to_back * 1e3,
                           "us_alone": alone * 1e3, "predicted_us": pred}
        if handle.get_error() != fgemm.OK:
            raise SystemExit(f"device error in the 256^3 case: {handle.last_message()}")

    # End to end through the library's host-buffer call: fgemm.matmul on
    # pinned CPU tensors (fgemm_matmul_host_ex) uploads B (and the bias), then
    # streams A's row blocks up while earlier blocks are multiplied and their
    # C blocks come down into a pinned host tensor.  Steps are issued without
    # waiting (blocking=False, two pinned outputs in turn), so a step's
    # uploads run under the previous step's products, as a serving loop
    # would; the timed region ends when the last step's C is on the host.
    e2e = None
    if not args.no_e2e:
        hA = A0.cpu().pin_memory()
        hB = B0.cpu().pin_memory()
        hbias = None if bias0 is None else bias0.cpu().pin_memory()
        hCs = [torch.empty((M, n_out), dtype=A0.dtype).pin_memory() for _ in range(2)]

        def e2e_step(i):
            fgemm.matmul(hA, hB, out=hCs[i % 2], epilogue=epi, bias=hbias, algo=algo, tile_n=tile,
                         tile_m=tile_m, handle=handle, blocking=False)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 40))
        barrier(world)
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - w0) * 1e3, world)
        if handle.get_error() != fgemm.OK:
            raise SystemExit(f"device error in the e2e steps: {handle.last_message()}")
        handle.set_stream(torch.cuda.current_stream(dev).cuda_stream)
        h2d = hA.numel() * 2 + hB.numel() * 2 + (0 if hbias is None else hbias.numel() * 2)
        e2e = {"value": flops * world * n_e2e / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hCs[0].numel() * 2,
               "steps": n_e2e, "path": "fgemm.matmul on pinned host tensors: fgemm_matmul_host_ex "
               "(B up, then A row blocks up / products / C blocks down, pipelined); steps issued "
               "without waiting, so a step's uploads overlap the previous step's products; host "
               "wall clock until the last C is on the host"}

    if rank != 0:
        return
    achieved = flops / (kern_avg_ms * 1e-3) / 1e12
    executed = achieved * (7.0 / 8.0) ** depth[plan_algo]
    alg_bytes, memory_bound = roofline_bound(M, N, K, n_out, 0 if bias0 is None else bias0.numel(),
                                             burst, hbm)
    traffic = ncu_traffic(args.workload, plan_algo, plan_tm, plan_tile)
    if memory_bound:
        gbs = alg_bytes / (kern_avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                "traffic": traffic, "algorithmic_bytes": alg_bytes,
                "peak_source": f"{src} copy bandwidth", "tflops": achieved, "kernel_ms": kern_avg_ms}
    else:
        roof = {"bound": "tensor", "achieved": executed, "peak": peak, "unit": UNIT,
                "frac": executed / peak if peak else None, "traffic": traffic,
                "peak_source": f"{src} bf16 dense ({peak_kind}: the timed region is "
                               f"{total_ms / 1e3:.2f} s of back-to-back launches)",
                "effective_tflops": achieved, "executed_tflops": executed,
                "algorithmic_flops": flops * (7.0 / 8.0) ** depth[plan_algo],
                "kernel_ms": kern_avg_ms}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if dtype == "bf16" else "f16",
        "data": "synthetic",
        "config": workload_config(args.workload),
        "plan": {"algo": plan_algo, "tile_m": plan_tm, "tile_n": plan_tile, "k_split": args.split,
                 "predicted_us": pred_us},
        "l2": l2_note,
        "parallelism": f"replicas x{world}",
        "roofline": roof,
        "forms": forms,
        "gpu_launches": args.steps * per_call,
        "clocks": clk.summary(),
    }
    if forms and algo == "auto" and plan_algo in forms:
        # AUTO's pick against the fastest form timed in the same run (a pick
        # inside the model's margin of a faster form shows here as < 1)
        fastest = max(forms, key=lambda f: forms[f]["effective_tflops"])
        line["decision"] = {"auto": plan_algo, "fastest_form": fastest,
                            "auto_vs_fastest": forms[plan_algo]["effective_tflops"] /
                            forms[fastest]["effective_tflops"]}
    if small is not None:
        line["small_case"] = small
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline and world == 1:
        v, s, e, thr = cpu_oracle_sample(args.workload, target_s=10.0,
                                         device_inputs=(A0, B0, bias0))
        line["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"{e} stratified output entries (seed 3) of the same workload, each a "
                      f"K={K} fp64 dot product of decoded inputs, {s:.1f} s"}
    print(json.dumps(line), flush=True)


def inputs_mod():
    from complexity_matmul_tcgen05_gb300 import inputs
    return inputs


CANDIDATES = [("classical", 16, 128), ("classical", 32, 128), ("classical", 64, 128),
              ("classical", 128, 64), ("classical", 128, 128), ("classical", 128, 256),
              ("classical", 256, 128), ("classical", 256, 256), ("strassen1", 128, 128),
              ("strassen1", 128, 256), ("strassen1", 256, 128), ("strassen1", 256, 256),
              ("strassen2", 128, 128), ("strassen2", 128, 256), ("strassen2", 256, 128),
              ("strassen2", 256, 256), ("winograd1", 128, 128),
              ("winograd1", 128, 256), ("winograd1", 256, 128), ("winograd1", 256, 256)]


def run_sweep(args):
    """Times every legal (form, tile) and AUTO on each sweep shape (CUDA
    events, median of 5 after 2 warm-ups, a 512 MiB buffer written between
    runs to flush the L2) and the host cost of the decision (a fresh model
    evaluation, and a whole cached call).  One JSON line per shape."""
    from complexity_matmul_tcgen05_gb300 import fgemm, inputs
    dev = torch.device("cuda", torch.cuda.current_device())
    handle = fgemm.default_handle()
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    out = open(args.out, "w") if args.out else None
    model = handle.device_model()
    L = fgemm.lib()
    import ctypes

    def time_one(A, B, C, algo, tm, tn):
        ts = []
        for r in range(7):
            flush.fill_(r & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fgemm.matmul(A, B, out=C, algo=algo, tile_m=tm, tile_n=tn, handle=handle)
            e1.record()
            torch.cuda.synchronize()
            if r >= 2:
                ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    for (M, N, K) in inputs.SWEEP_SHAPES:
        A, B = inputs.sweep_inputs(M, N, K, dev)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        times = {}
        for algo, tm, tn in CANDIDATES:
            if fgemm.validate(M, N, K, 16, K, 16, N, 16, N, fgemm.BF16, None, algo, tn, tm) != fgemm.OK:
                continue
            times[f"{algo}:{tm}x{tn}"] = time_one(A, B, C, algo, tm, tn)
        a_algo, a_tm, a_tn, pred = handle.plan(M, N, K)
        t_auto = time_one(A, B, C, "auto", 0, 0)
        best = min(times, key=times.get)
        # host cost of one fresh model evaluation (every form and tile)
        a = ctypes.c_int()
        x, y, us = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
        t0 = time.perf_counter()
        for _ in range(1000):
            L.fgemm_model_plan(ctypes.byref(model), M, N, K, 0, ctypes.byref(a), ctypes.byref(x),
                               ctypes.byref(y), ctypes.byref(us))
        plan_us = (time.perf_counter() - t0) * 1e3
        # host cost of a whole cached call (checks, plan lookup, launch)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(50):
            handle.matmul_raw(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                              fgemm.BF16, None, "auto", 0, 0)
        call_us = (time.perf_counter() - t0) / 50 * 1e6
        torch.cuda.synchronize()
        rec = {"M": M, "N": N, "K": K, "times_us": times, "best": best, "best_us": times[best],
               "auto": f"{a_algo}:{a_tm}x{a_tn}", "auto_us": t_auto, "predicted_us": pred,
               "regret": t_auto / times[best] - 1.0,
               "auto_tflops": 2.0 * M * N * K / (t_auto * 1e-6) / 1e12,
               "model_eval_us": plan_us, "host_call_us": call_us,
               "decision_share": plan_us / t_auto}
        line = json.dumps(rec)
        print(line, flush=True)
        if out:
            out.write(line + "\n")
            out.flush()
        del A, B, C
    if handle.get_error() != fgemm.OK:
        raise SystemExit(f"device error: {handle.last_message()}")


def run_mx(args):
    """Times fgemm_matmul_mx (8-bit elements, E8M0 scales per 32 values of
    K) on the workload's shape: the whole call, its 8-bit-to-bf16 step alone
    and the bf16 product alone.  Each is captured `steps` times in a CUDA
    graph over four rotating input sets and timed by CUDA events around a
    replay, so host launch costs do not count.  One JSON line."""
    from complexity_matmul_tcgen05_gb300 import fgemm
    dev = torch.device("cuda", torch.cuda.current_device())
    M, N, K, _, _ = workload_shape(args.workload)
    kb = (K + 31) // 32
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    sets = 4
    # Elements as block-scaled quantisation leaves them: Gaussian values whose
    # block maxima sit near the top of the 8-bit range (sigma 64 of E4M3's
    # 448, 8192 of E5M2's 57344), cast by torch; scales spread around 2^0.
    sigma, f8 = (64.0, torch.float8_e4m3fn) if args.mx == "e4m3" else (8192.0, torch.float8_e5m2)
    def fp8(rows, cols):
        x = torch.randn((rows, cols), generator=g, device=dev) * sigma
        return x.to(f8).view(torch.uint8)
    def scales(rows, cols):
        return torch.randint(120, 135, (rows, cols), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    As = [fp8(M, K) for _ in range(sets)]
    Bs = [fp8(K, N) for _ in range(sets)]
    SA = scales(M, kb)
    SB = scales(kb, N)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    Ab = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    Bb = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
    h = fgemm.default_handle()

    def timed(fn):
        for i in range(max(3, args.warmup)):
            fn(i)  # allocations and launch set-up happen before the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                fn(i)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / args.steps

    full = timed(lambda i: fgemm.matmul_mx(As[i % sets], SA, Bs[i % sets], SB, a_format=args.mx,
                                           b_format=args.mx, out=C, handle=h))
    conv = timed(lambda i: (fgemm.mx_to_bf16(As[i % sets], SA, args.mx, "row", handle=h, out=Ab),
                            fgemm.mx_to_bf16(Bs[i % sets], SB, args.mx, "col", handle=h, out=Bb)))
    prod = timed(lambda i: fgemm.matmul(Ab, Bb, out=C, handle=h))
    if h.get_error() != fgemm.OK:
        raise SystemExit(f"device error: {h.last_message()}")
    flops = 2.0 * M * N * K
    mx_bytes = M * K + K * N + M * kb + kb * N
    print(json.dumps({
        "metric": METRIC, "value": flops / (full * 1e-6) / 1e12, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": full / 1e3,
        "higher_is_better": True, "dtype": f"mx-{args.mx} -> bf16", "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K, "mx_format": args.mx,
                   "l2": f"{sets} rotating 8-bit input sets", "timing": "CUDA graph replay"},
        "mx_to_bf16_us": conv, "mx_to_bf16_gbs": (mx_bytes + 2 * (M * K + K * N)) / (conv * 1e3),
        "bf16_product_us": prod, "whole_call_us": full}), flush=True)


def main():
    args = parse()
    if args.sweep:
        run_sweep(args)
        return
    if args.mx:
        run_mx(args)
        return
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py --impl fgemm needs a CUDA device")
        run_fgemm(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
