"""GPU parity at the full workload sizes, on 4096 stratified sampled output
entries that the oracle computes one by one (K-long fp64 dot products of the
decoded inputs), through the same binding call the benchmark times."""
import numpy as np
import pytest
import torch

import oracle
from complexity_matmul_tcgen05_gb300 import fgemm, inputs
from parity_util import (TOL_NORMWISE, elementwise_act_ok, elementwise_ok, gpu_bits, preact_bound,
                         record, run)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


def _picked(M, N, K, epi):
    return fgemm.plan(M, N, K, epilogue=epi)[0]


def _sampled_check(name, A, B, bias, run_algo, epi, dtype, tile=0, tile_m=0):
    """Runs `run_algo` and checks sampled entries against the oracle with the
    tolerance of the form that actually ran: its normwise budget, bare, and
    for classical the per-entry rule (carried through SwiGLU to first order).
    A rounded-operand form through SwiGLU has its activated output held to
    the budget times the activation's condition number at the samples, and
    its pre-activation product (the same form, no activation) to the bare
    budget."""
    M, K = A.shape
    N = B.shape[1]
    n_out = N // 2 if epi == "swiglu" else N
    algo = _picked(M, N, K, epi) if run_algo == "auto" else run_algo
    depth_blocks = {"classical": 1, "strassen1": 2, "strassen2": 4, "winograd1": 2}[algo]
    C = run(A, B, algo=run_algo, epilogue=epi, bias=bias, tile_n=tile, tile_m=tile_m)
    # Strassen forms sit within a few percent of their normwise budgets (the
    # rounded operand sums alone give 4.7e-3 and 9.7e-3 on these inputs), so
    # they get 8x more samples: the sampled estimate's relative noise drops
    # from about 1.6% to about 0.6%.
    n_samples = 4096 if algo == "classical" else 32768
    rows, cols = inputs.sample_positions(M, n_out, n=n_samples, row_blocks=depth_blocks,
                                         col_blocks=depth_blocks)
    rows, cols = rows.numpy(), cols.numpy()
    Ab, Bb = gpu_bits(A), gpu_bits(B)
    bb = None if bias is None else gpu_bits(bias)
    ref = oracle.reference_sampled(Ab, Bb, dtype, rows, cols, epi, 1.0, bb)
    ridx, cidx = torch.as_tensor(rows, device=DEV), torch.as_tensor(cols, device=DEV)
    got = oracle.decode(gpu_bits(C[ridx, cidx]), dtype)
    err = float(np.linalg.norm(got - oracle.round_to(ref, dtype)) / np.linalg.norm(ref))
    tol = TOL_NORMWISE[algo]
    if epi != "swiglu":
        record(f"{name} normwise ({algo})", err, tol)
        assert err <= tol, (name, algo, err)
        if algo == "classical":
            absdot = oracle.gemm_sampled(Ab & np.uint16(0x7FFF), Bb & np.uint16(0x7FFF), dtype, rows, cols)
            ok, frac = elementwise_ok(got, ref, absdot, K, dtype)
            record(f"{name} entries on the dot-product branch", frac, 1.0)
            assert ok, name
        return err
    # SwiGLU: the gate and up pre-activation values at the samples
    bv = None if bb is None else oracle.decode(bb, dtype)
    g = oracle.gemm_sampled(Ab, Bb, dtype, rows, cols)
    u = oracle.gemm_sampled(Ab, Bb, dtype, rows, cols + n_out)
    bg = 0.0 if bv is None else bv[cols]
    bu = 0.0 if bv is None else bv[cols + n_out]
    vg, vu = g + bg, u + bu
    if algo == "classical":
        record(f"{name} normwise swiglu ({algo})", err, tol)
        assert err <= tol, (name, algo, err)
        absA, absB = Ab & np.uint16(0x7FFF), Bb & np.uint16(0x7FFF)
        dg = preact_bound(g, oracle.gemm_sampled(absA, absB, dtype, rows, cols), K, 1.0, bg)
        du = preact_bound(u, oracle.gemm_sampled(absA, absB, dtype, rows, cols + n_out), K, 1.0, bu)
        ok, frac = elementwise_act_ok(got, "swiglu", vg, dg, vu, du, dtype)
        record(f"{name} swiglu entries on the propagated branch", frac, 1.0)
        assert ok, name
        return err
    sig = 1 / (1 + np.exp(-vg))
    silu = vg * sig
    ds = sig * (1 + vg * (1 - sig))
    kappa = float(np.linalg.norm(np.abs(ds * vu * vg) + np.abs(silu * vu)) / np.linalg.norm(silu * vu))
    record(f"{name} normwise swiglu ({algo}, x kappa {kappa:.2f})", err, tol * max(1.0, kappa))
    assert err <= tol * max(1.0, kappa), (name, algo, err, kappa)
    # the same form's pre-activation product, gate | up, against the bare budget
    del C
    P = run(A, B, algo=run_algo, epilogue="scale_bias" if bias is not None else "none", bias=bias,
            tile_n=tile, tile_m=tile_m)
    both_r = np.concatenate([rows, rows])
    both_c = np.concatenate([cols, cols + n_out])
    pref = np.concatenate([vg, vu])
    pgot = oracle.decode(gpu_bits(P[torch.as_tensor(both_r, device=DEV),
                                    torch.as_tensor(both_c, device=DEV)]), dtype)
    e_pre = float(np.linalg.norm(pgot - oracle.round_to(pref, dtype)) / np.linalg.norm(pref))
    record(f"{name} normwise pre-activation ({algo})", e_pre, tol)
    assert e_pre <= tol, (name, algo, e_pre)
    return err


@pytest.mark.parametrize("algo", ["auto", "classical"])
def test_proj_4096_bias(algo):
    A, B, bias = inputs.workload_inputs("proj_4096_bf16_bias", DEV)
    _sampled_check("proj_4096", A, B, bias, algo, "scale_bias", "bf16")


@pytest.mark.parametrize("algo,tile_m", [("classical", 0), ("strassen1", 256), ("strassen1", 128),
                                         ("winograd1", 256), ("auto", 0)])
def test_ffn_up_swiglu(algo, tile_m):
    A, B, _ = inputs.workload_inputs("ffn_up_swiglu_bf16", DEV)
    _sampled_check("ffn_up", A, B, None, algo, "swiglu", "bf16", tile_m=tile_m)


@pytest.mark.parametrize("algo,tile_m", [("classical", 0), ("strassen1", 256), ("strassen1", 128),
                                         ("strassen2", 128), ("strassen2", 256), ("winograd1", 256),
                                         ("winograd1", 128), ("auto", 0)])
def test_square_16384(algo, tile_m):
    A, B, _ = inputs.workload_inputs("square_16384_bf16", DEV)
    _sampled_check("square_16384", A, B, None, algo, "none", "bf16", tile_m=tile_m)


@pytest.mark.parametrize("algo,tile_m", [("winograd1", 256), ("auto", 0)])
def test_square_20480(algo, tile_m):
    """The smallest cube on which AUTO takes one Winograd level on CTA pairs:
    21 whole waves of output positions plus 4 positions as product units
    shared out over the pairs."""
    A, B, _ = inputs.workload_inputs("square_20480_bf16", DEV)
    _sampled_check("square_20480", A, B, None, algo, "none", "bf16", tile_m=tile_m)


@pytest.mark.parametrize("algo,tile_m", [("classical", 0), ("winograd1", 256), ("strassen1", 256),
                                         ("auto", 0)])
def test_square_24576(algo, tile_m):
    """The largest square workload the benchmark names: 30 whole waves of
    output positions on the pairs plus a partial one, Winograd's sums formed
    inside its product kernel."""
    A, B, _ = inputs.workload_inputs("square_24576_bf16", DEV)
    _sampled_check("square_24576", A, B, None, algo, "none", "bf16", tile_m=tile_m)


@pytest.mark.parametrize("shape", inputs.SWEEP_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_sweep_shapes_every_legal_form(shape):
    M, N, K = shape
    A, B = inputs.sweep_inputs(M, N, K, DEV)
    for algo in ("classical", "strassen1", "strassen2", "winograd1", "auto"):
        s = fgemm.validate(M, N, K, 16, K, 16, N, 16, N, fgemm.BF16, None, algo)
        if s == fgemm.ERR_UNSUPPORTED:
            continue
        _sampled_check(f"sweep {shape}", A, B, None, algo, "none", "bf16")
    for tm in (16, 32, 64):  # the small-M kernel, where M fits
        if M <= tm:
            _sampled_check(f"sweep {shape} small-M {tm}", A, B, None, "classical", "none", "bf16",
                           tile=128, tile_m=tm)


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2")])
def test_mx_4096_sampled(fa, fb):
    """The block-scaled 8-bit product at the size `bench.py --mx` times, on its
    input recipe (Gaussian values cast to 8 bits by torch, scales around 2^0):
    4096 sampled entries against the oracle's decoded values (every entry a
    K-long fp64 dot product), with the classical normwise and per-entry
    bounds."""
    n = 4096
    kb = n // 32
    g = torch.Generator().manual_seed(7)
    def fp8(fmt):
        sigma, f8 = (64.0, torch.float8_e4m3fn) if fmt == "e4m3" else (8192.0, torch.float8_e5m2)
        return (torch.randn((n, n), generator=g) * sigma).to(f8).view(torch.uint8)
    A, B = fp8(fa), fp8(fb)
    SA = torch.randint(120, 135, (n, kb), generator=g, dtype=torch.int32).to(torch.uint8)
    SB = torch.randint(120, 135, (kb, n), generator=g, dtype=torch.int32).to(torch.uint8)
    C = fgemm.matmul_mx(A.to(DEV), SA.to(DEV), B.to(DEV), SB.to(DEV), a_format=fa, b_format=fb)
    torch.cuda.synchronize()
    assert fgemm.default_handle().get_error() == fgemm.OK
    rows, cols = inputs.sample_positions(n, n, n=4096, tile_m=256, tile_n=256)
    rows, cols = rows.numpy(), cols.numpy()
    Av = oracle.mx_values(A.numpy(), SA.numpy(), fa, "row")[rows]          # sampled rows of A
    Bv = oracle.mx_values(B.numpy(), SB.numpy(), fb, "col")[:, cols]       # sampled columns of B
    ref = np.einsum("ik,ki->i", Av, Bv)
    absdot = np.einsum("ik,ki->i", np.abs(Av), np.abs(Bv))
    got = oracle.decode(gpu_bits(C[torch.as_tensor(rows, device=DEV), torch.as_tensor(cols, device=DEV)]),
                        "bf16")
    err = float(np.linalg.norm(got - oracle.round_to(ref, "bf16")) / np.linalg.norm(ref))
    assert err <= TOL_NORMWISE["classical"], err
    ok, _ = elementwise_ok(got, ref, absdot, n, "bf16")
    assert ok
