"""Pins for the fp64 CPU oracle, against things other than itself.

Each test ties one oracle function to an independent fact: a library routine
(torch / numpy / scipy conversions and products), brute force in plain
Python, a closed form, or an algebraic identity of the exact product.  The
set is chosen so that a dropped term, a wrong sign or index, or a transposed
operand anywhere in the oracle fails at least one test.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from complexity_matmul_tcgen05_gb300 import inputs

ALL16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def _torch_values(bits, tdtype):
    t = torch.from_numpy(bits.view(np.int16).copy()).view(tdtype)
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------- decoding

@pytest.mark.parametrize("dtype,tdtype", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_decode_all_patterns_match_torch(dtype, tdtype):
    ours = oracle.decode(ALL16, dtype)
    ref = _torch_values(ALL16, tdtype)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_special_values():
    assert oracle.decode(np.array([0x3C00], np.uint16), "f16")[0] == 1.0
    assert oracle.decode(np.array([0x0001], np.uint16), "f16")[0] == 2.0 ** -24
    assert oracle.decode(np.array([0x7BFF], np.uint16), "f16")[0] == 65504.0
    assert oracle.decode(np.array([0x3F80], np.uint16), "bf16")[0] == 1.0
    assert oracle.decode(np.array([0x0001], np.uint16), "bf16")[0] == 2.0 ** -133
    assert oracle.decode(np.array([0xC000], np.uint16), "bf16")[0] == -2.0


# ---------------------------------------------------------------- encoding

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_encode_roundtrips_every_non_nan_pattern(dtype):
    vals = oracle.decode(ALL16, dtype)
    keep = ~np.isnan(vals)
    back = oracle.encode(vals[keep], dtype)
    assert np.array_equal(back, ALL16[keep])


def test_encode_f16_matches_numpy_rne_from_double():
    rng = np.random.default_rng(7)
    mant = rng.random(200000) + 0.5
    expo = rng.integers(-30, 18, 200000)
    x = np.ldexp(mant, expo) * np.where(rng.random(200000) < 0.5, -1, 1)
    # exact ties: midpoints between neighbouring fp16 values
    base = oracle.decode(ALL16[(ALL16 & 0x7C00) != 0x7C00], "f16")
    base = np.sort(base[np.isfinite(base)])
    mids = (base[:-1] + base[1:]) / 2
    x = np.concatenate([x, mids, [65519.0, 65520.0, 65536.0, 1e-9, -1e-9]])
    ours = oracle.encode(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_encode_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(8)
    mant = rng.random(200000) + 0.5
    expo = rng.integers(-140, 120, 200000)
    x = (np.ldexp(mant, expo) * np.where(rng.random(200000) < 0.5, -1, 1)).astype(np.float32)
    x = x[np.isfinite(x)]
    ours = oracle.encode(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_encode_bf16_ties_go_to_even():
    one = 1.0
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even is 1.0
    assert oracle.encode(np.array([one + 2.0 ** -8]), "bf16")[0] == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert oracle.encode(np.array([one + 3 * 2.0 ** -8]), "bf16")[0] == 0x3F82
    # just above a tie rounds up
    assert oracle.encode(np.array([one + 2.0 ** -8 + 2.0 ** -30]), "bf16")[0] == 0x3F81


# ----------------------------------------------------------- classical gemm

def _brute(A, B):
    M, K = len(A), len(A[0])
    N = len(B[0])
    C = [[0.0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s += A[i][k] * B[k][j]
            C[i][j] = s
    return C


def test_gemm_equals_brute_force_bitwise():
    rng = np.random.default_rng(1)
    for (M, N, K) in [(1, 1, 1), (3, 5, 4), (7, 2, 9), (4, 4, 16)]:
        A = rng.standard_normal((M, K))
        B = rng.standard_normal((K, N))
        ref = np.array(_brute(A.tolist(), B.tolist()))
        assert np.array_equal(oracle.gemm(A, B), ref)


@pytest.mark.parametrize("shape", [(17, 33, 65), (64, 1, 128), (1, 96, 31), (130, 70, 257)])
def test_gemm_matches_numpy(shape):
    M, N, K = shape
    rng = np.random.default_rng(M * N + K)
    A = rng.uniform(-1, 1, (M, K))
    B = rng.uniform(-1, 1, (K, N))
    C = oracle.gemm(A, B)
    ref = A @ B
    assert np.max(np.abs(C - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_gemm_identity_zero_permutation_exact():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((12, 12))
    I = np.eye(12)
    assert np.array_equal(oracle.gemm(I, X), X)
    assert np.array_equal(oracle.gemm(X, I), X)
    assert np.array_equal(oracle.gemm(np.zeros((12, 12)), X), np.zeros((12, 12)))
    perm = rng.permutation(12)
    P = I[perm]
    assert np.array_equal(oracle.gemm(P, X), X[perm])
    assert np.array_equal(oracle.gemm(X, P.T), X[:, perm])


def test_gemm_transpose_identity():
    rng = np.random.default_rng(3)
    A = rng.standard_normal((9, 13))
    B = rng.standard_normal((13, 6))
    assert np.array_equal(oracle.gemm(A, B).T, oracle.gemm(B.T, A.T))


def test_gemm_not_transposed_operand():
    # a non-square case where A@B and A@B.T-like mistakes differ in shape/value
    A = np.array([[1.0, 2.0, 3.0]])
    B = np.array([[1.0, 0.0], [0.0, 10.0], [0.0, 100.0]])
    assert np.array_equal(oracle.gemm(A, B), np.array([[1.0, 320.0]]))


# ---------------------------------------------------------------- epilogue

def test_epilogue_alpha_bias_closed_form():
    X = np.array([[1.0, -2.0, 3.0], [0.5, 0.0, -4.0]])
    bias = np.array([10.0, 20.0, 30.0])
    out = oracle.epilogue(X, "scale_bias", 2.0, bias)
    assert np.array_equal(out, 2.0 * X + bias[None, :])
    assert np.array_equal(oracle.epilogue(X, "none", 1.0, None), X)


def test_silu_against_scipy_and_limits():
    from scipy.special import expit
    xs = np.linspace(-30, 30, 1201)
    ours = oracle.epilogue(xs.reshape(1, -1), "silu")[0]
    ref = xs * expit(xs)
    assert np.max(np.abs(ours - ref) / np.maximum(1e-300, np.abs(ref) + 1e-300)) < 1e-14
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12          # -> x for large x
    assert abs(oracle.silu(-40.0)) < 1e-15                # -> 0 for very negative x
    assert abs(oracle.silu(1e-8) / 1e-8 - 0.5) < 1e-8     # slope 1/2 at the origin
    assert abs(oracle.silu(-1.0) - (-1.0 / (1.0 + math.e))) < 1e-16


def test_swiglu_pairs_gate_with_up():
    from scipy.special import expit
    g = np.array([[1.0, -2.0]])
    u = np.array([[3.0, 5.0]])
    acc = np.concatenate([g, u], axis=1)             # gate | up
    bias = np.array([0.5, 0.25, -1.0, 2.0])
    out = oracle.epilogue(acc, "swiglu", 1.5, bias)
    vg = 1.5 * g + bias[:2]
    vu = 1.5 * u + bias[2:]
    ref = vg * expit(vg) * vu
    assert out.shape == (1, 2)
    assert np.max(np.abs(out - ref)) < 1e-14


# ----------------------------------------------------------------- Strassen

@pytest.mark.parametrize("depth,shape", [(1, (2, 2, 2)), (1, (8, 6, 4)), (1, (34, 18, 50)),
                                         (2, (4, 4, 4)), (2, (16, 24, 8)), (2, (36, 20, 44))])
def test_strassen_equals_classical(depth, shape):
    M, N, K = shape
    rng = np.random.default_rng(M + 3 * N + 7 * K + depth)
    A = rng.uniform(-1, 1, (M, K))
    B = rng.uniform(-1, 1, (K, N))
    ref = oracle.gemm(A, B)
    S = oracle.strassen(A, B, depth)
    assert np.linalg.norm(S - ref) <= 1e-12 * np.linalg.norm(ref)


@pytest.mark.parametrize("depth", [1, 2])
def test_strassen_exact_on_integers(depth):
    rng = np.random.default_rng(11 + depth)
    A = rng.integers(-3, 4, (16, 12)).astype(np.float64)
    B = rng.integers(-3, 4, (12, 20)).astype(np.float64)
    assert np.array_equal(oracle.strassen(A, B, depth), A @ B)


def test_strassen_every_quadrant_depends_on_the_right_blocks():
    # One nonzero block at a time: C = A B has a known block structure, so a
    # wrong index or sign in any of the 7 products or 4 combinations shows.
    n = 2
    for ai in range(2):
        for ak in range(2):
            for bk in range(2):
                for bj in range(2):
                    A = np.zeros((2 * n, 2 * n))
                    B = np.zeros((2 * n, 2 * n))
                    A[ai * n:(ai + 1) * n, ak * n:(ak + 1) * n] = np.arange(1, n * n + 1).reshape(n, n)
                    B[bk * n:(bk + 1) * n, bj * n:(bj + 1) * n] = np.arange(2, n * n + 2).reshape(n, n)
                    assert np.array_equal(oracle.strassen(A, B, 1), A @ B)


def test_strassen_rejects_indivisible():
    with pytest.raises(ValueError):
        oracle.strassen(np.ones((3, 4)), np.ones((4, 4)), 1)
    with pytest.raises(ValueError):
        oracle.strassen(np.ones((6, 4)), np.ones((4, 4)), 2)


@pytest.mark.parametrize("depth", [1, 2])
def test_emulated_without_rounding_is_exact_strassen(depth):
    rng = np.random.default_rng(5)
    A = rng.uniform(-1, 1, (16, 8))
    B = rng.uniform(-1, 1, (8, 12))
    assert np.array_equal(oracle.strassen_emulated(A, B, depth, "f64"), oracle.strassen(A, B, depth))


@pytest.mark.parametrize("depth", [1, 2])
def test_emulated_on_ternary_inputs_is_exact(depth):
    # operand sums of {-1,0,1} values are small integers, exact in any 16-bit type
    rng = np.random.default_rng(6)
    A = rng.integers(-1, 2, (32, 16)).astype(np.float64)
    B = rng.integers(-1, 2, (16, 24)).astype(np.float64)
    assert np.array_equal(oracle.strassen_emulated(A, B, depth, "bf16"), A @ B)


# Textbook one-level Strassen as coefficient matrices over the 2 x 2 blocks
# [X11, X12, X21, X22]: product p multiplies (U[p] . A-blocks) by (V[p] .
# B-blocks), and output block q collects W[q] . (M1 .. M7).  Two levels are
# the Kronecker squares of U, V and W (written out independently of the
# oracle's recursion).
_U = np.array([[1, 0, 0, 1], [0, 0, 1, 1], [1, 0, 0, 0], [0, 0, 0, 1],
               [1, 1, 0, 0], [-1, 0, 1, 0], [0, 1, 0, -1]], dtype=np.float64)
_V = np.array([[1, 0, 0, 1], [1, 0, 0, 0], [0, 1, 0, -1], [-1, 0, 1, 0],
               [0, 0, 0, 1], [1, 1, 0, 0], [0, 0, 1, 1]], dtype=np.float64)
_W = np.array([[1, 0, 0, 1, -1, 0, 1], [0, 0, 1, 0, 1, 0, 0],
               [0, 1, 0, 1, 0, 0, 0], [1, -1, 1, 0, 0, 1, 0]], dtype=np.float64)


def _blocks2(X):
    """The 16 scalar entries of a 4 x 4 matrix in two-level block order:
    index 4 * outer + inner, each of outer / inner = 2 * row_half + col_half."""
    out = np.empty(16)
    for o in range(4):
        for i in range(4):
            r = 2 * (o >> 1) + (i >> 1)
            c = 2 * (o & 1) + (i & 1)
            out[4 * o + i] = X[r, c]
    return out


def _bf16_once(x):
    """fp64 -> fp32 -> bf16 (both round-to-nearest-even), as torch casts."""
    return torch.tensor(x, dtype=torch.float64).to(torch.float32).to(torch.bfloat16) \
        .to(torch.float64).numpy()


def test_strassen_coefficients_reproduce_the_product():
    # the coefficient matrices above are the textbook scheme: exact on random 2 x 2
    rng = np.random.default_rng(21)
    A, B = rng.uniform(-1, 1, (2, 2)), rng.uniform(-1, 1, (2, 2))
    m = (_U @ A.reshape(4)) * (_V @ B.reshape(4))
    assert np.allclose((_W @ m).reshape(2, 2), A @ B, rtol=0, atol=1e-15)
    assert np.allclose(oracle.strassen(A, B, 1), (_W @ m).reshape(2, 2), rtol=0, atol=1e-15)


def test_strassen_emulated_depth2_rounds_each_leaf_once_from_its_quarter_blocks():
    # 4 x 4 scalars, B = I: every leaf operand of the 49 products is a signed
    # sum of up to four scalar quarter blocks.  The leaf of (M1, M1) sums
    # A00 + A11 + A22 + A33 (outer A11 + A22, then inner X11 + X22).  With
    # A00 = 1, A22 = 2^-10, A11 = 2^-8, A33 = 0 the exact sum 1 + 2^-8 + 2^-10
    # is above the bf16 midpoint and rounds to 1 + 2^-7.  Rounding at the
    # outer level first (1 + 2^-10 -> 1, then 1 + 2^-8 is a tie -> 1) or
    # rounding the running sum would give 1, and that shows in C.
    A = np.zeros((4, 4))
    A[0, 0], A[2, 2], A[1, 1], A[3, 3] = 1.0, 2.0 ** -10, 2.0 ** -8, 0.0
    A[0, 3], A[3, 0], A[1, 2] = 0.375, -0.5, 0.25
    B = np.eye(4)
    U2, V2, W2 = np.kron(_U, _U), np.kron(_V, _V), np.kron(_W, _W)
    a, b = _blocks2(A), _blocks2(B)
    S = _bf16_once(U2 @ a)               # every leaf rounded once from its exact sum
    T = _bf16_once(V2 @ b)
    c = W2 @ (S * T)
    expect = np.empty((4, 4))
    for o in range(4):
        for i in range(4):
            expect[2 * (o >> 1) + (i >> 1), 2 * (o & 1) + (i & 1)] = c[4 * o + i]
    got = oracle.strassen_emulated(A, B, 2, "bf16")
    assert np.allclose(got, expect, rtol=0, atol=1e-15)
    # the wrong placement: round the outer sums first, then the leaf sums
    outer_a = _bf16_once(np.kron(_U, np.eye(4)) @ a)        # 7 outer sums x 4 inner entries
    wrong_S = _bf16_once(np.kron(np.eye(7), _U) @ outer_a)
    assert not np.allclose(wrong_S, S)
    wrong = W2 @ (wrong_S * T)
    assert not np.allclose(c, wrong, rtol=0, atol=1e-6)    # the tie is visible in C
    # no rounding at all gives A exactly (B = I), so the rounding shows too
    assert not np.allclose(got, A, rtol=0, atol=1e-6)


@pytest.mark.parametrize("dtype,depth,lo,hi", [("bf16", 1, 3e-4, 5e-3), ("bf16", 2, 6e-4, 1e-2),
                                               ("f16", 1, 4e-5, 1e-3)])
def test_emulated_rounding_error_is_in_the_expected_band(dtype, depth, lo, hi):
    rng = np.random.default_rng(9)
    n = 128
    A = oracle.round_to(rng.uniform(-1, 1, (n, n)), dtype)
    B = oracle.round_to(rng.uniform(-1, 1, (n, n)), dtype)
    ref = oracle.gemm(A, B)
    E = oracle.strassen_emulated(A, B, depth, dtype)
    rel = np.linalg.norm(E - ref) / np.linalg.norm(ref)
    assert lo < rel < hi, rel


# ----------------------------------------------------------------- Winograd

@pytest.mark.parametrize("depth,shape", [(1, (2, 2, 2)), (1, (8, 6, 4)), (1, (34, 18, 50)),
                                         (2, (4, 4, 4)), (2, (16, 24, 8)), (2, (36, 20, 44))])
def test_winograd_equals_classical(depth, shape):
    M, N, K = shape
    rng = np.random.default_rng(2 * M + 5 * N + 3 * K + depth)
    A = rng.uniform(-1, 1, (M, K))
    B = rng.uniform(-1, 1, (K, N))
    ref = oracle.gemm(A, B)
    W = oracle.winograd(A, B, depth)
    assert np.linalg.norm(W - ref) <= 1e-12 * np.linalg.norm(ref)


@pytest.mark.parametrize("depth", [1, 2])
def test_winograd_exact_on_integers(depth):
    rng = np.random.default_rng(21 + depth)
    A = rng.integers(-3, 4, (16, 12)).astype(np.float64)
    B = rng.integers(-3, 4, (12, 20)).astype(np.float64)
    assert np.array_equal(oracle.winograd(A, B, depth), A @ B)


def test_winograd_every_quadrant_depends_on_the_right_blocks():
    # one nonzero block of A and one of B at a time: any wrong block, sign or
    # partial sum in the seven products or the output sums shows
    n = 2
    for ai in range(2):
        for ak in range(2):
            for bk in range(2):
                for bj in range(2):
                    A = np.zeros((2 * n, 2 * n))
                    B = np.zeros((2 * n, 2 * n))
                    A[ai * n:(ai + 1) * n, ak * n:(ak + 1) * n] = np.arange(1, n * n + 1).reshape(n, n)
                    B[bk * n:(bk + 1) * n, bj * n:(bj + 1) * n] = np.arange(3, n * n + 3).reshape(n, n)
                    assert np.array_equal(oracle.winograd(A, B, 1), A @ B)


def test_winograd_rejects_indivisible():
    with pytest.raises(ValueError):
        oracle.winograd(np.ones((3, 4)), np.ones((4, 4)), 1)
    with pytest.raises(ValueError):
        oracle.winograd_emulated(np.ones((6, 4)), np.ones((4, 4)), 2, "bf16")


@pytest.mark.parametrize("depth", [1, 2])
def test_winograd_emulated_without_rounding_is_exact_winograd(depth):
    rng = np.random.default_rng(15)
    A = rng.uniform(-1, 1, (16, 8))
    B = rng.uniform(-1, 1, (8, 12))
    assert np.array_equal(oracle.winograd_emulated(A, B, depth, "f64"), oracle.winograd(A, B, depth))


def test_winograd_emulated_on_ternary_inputs_is_exact():
    # operands are signed sums of up to four {-1,0,1} values: exact in bf16
    rng = np.random.default_rng(16)
    A = rng.integers(-1, 2, (32, 16)).astype(np.float64)
    B = rng.integers(-1, 2, (16, 24)).astype(np.float64)
    assert np.array_equal(oracle.winograd_emulated(A, B, 1, "bf16"), A @ B)


def test_winograd_emulated_rounds_each_operand_once_from_its_blocks():
    # 2 x 2 scalars, B = I: the products' operands are the expanded sums
    #   P3: a + b - c - d   P5: (c + d) * (-1)   P6: (c + d - a) * 2
    #   P7: a - c           P4: d * 2             P1: a, P2: 0
    # and the emulation must round each of them once (fp32, then bf16), not
    # the partial sums they are built from.  With a = 1, c = 2^-9, d = 2^-10,
    # c + d - a is a bf16 tie (rounded to even), so the rounding shows in C.
    a, b, c, d = 1.0, 2.0 ** -8, 2.0 ** -9, 2.0 ** -10
    A = np.array([[a, b], [c, d]])
    B = np.eye(2)

    def r(x):  # fp32, then bf16, both round-to-nearest-even (torch casts)
        return float(torch.tensor(x, dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
                     .to(torch.float64))

    p1, p2 = r(a) * 1.0, r(b) * 0.0
    p3 = r(a + b - c - d) * 1.0
    p4 = r(d) * r(2.0)
    p5 = r(c + d) * r(-1.0)
    p6 = r(c + d - a) * r(2.0)
    p7 = r(a - c) * r(1.0)
    expect = np.array([[p1 + p2, p1 + p6 + p5 + p3],
                       [p1 + p6 + p7 - p4, p1 + p6 + p7 + p5]])
    got = oracle.winograd_emulated(A, B, 1, "bf16")
    assert np.allclose(got, expect, rtol=0, atol=1e-15)
    assert not np.allclose(got, A, rtol=0, atol=1e-6)  # the tie is visible


@pytest.mark.parametrize("dtype,depth,lo,hi", [("bf16", 1, 1e-3, 1e-2), ("bf16", 2, 3e-3, 3e-2),
                                               ("f16", 1, 1e-4, 2e-3)])
def test_winograd_emulated_rounding_error_is_in_the_expected_band(dtype, depth, lo, hi):
    # rounding up to four-term operand sums to an 8-bit (bf16) or 11-bit (f16)
    # significand: well above zero, and below 2^-7 / 2^-10 per level
    rng = np.random.default_rng(9)
    n = 128
    A = oracle.round_to(rng.uniform(-1, 1, (n, n)), dtype)
    B = oracle.round_to(rng.uniform(-1, 1, (n, n)), dtype)
    ref = oracle.gemm(A, B)
    E = oracle.winograd_emulated(A, B, depth, dtype)
    rel = np.linalg.norm(E - ref) / np.linalg.norm(ref)
    assert lo < rel < hi, rel


# ------------------------------------------------------- 8-bit MX inputs

@pytest.mark.parametrize("fmt,tdtype", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_decode_all_patterns_match_torch(fmt, tdtype):
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(tdtype).to(torch.float64).numpy()
    got = oracle.fp8_decode(bits, fmt)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_fp8_special_values():
    e4 = oracle.fp8_decode(np.array([0x38, 0x7E, 0x7F, 0x01, 0x80], dtype=np.uint8), "e4m3")
    assert e4[0] == 1.0 and e4[1] == 448.0 and np.isnan(e4[2]) and e4[3] == 2.0 ** -9
    assert e4[4] == 0.0 and np.signbit(e4[4])
    e5 = oracle.fp8_decode(np.array([0x3C, 0x7B, 0x7C, 0xFC, 0x7D, 0x01], dtype=np.uint8), "e5m2")
    assert e5[0] == 1.0 and e5[1] == 57344.0 and e5[2] == np.inf and e5[3] == -np.inf
    assert np.isnan(e5[4]) and e5[5] == 2.0 ** -16


def test_e8m0_decode_all_patterns_match_torch():
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = oracle.e8m0_decode(bits)
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def test_mx_values_blocks_along_rows_and_columns():
    rng = np.random.default_rng(40)
    X = rng.integers(0, 256, (40, 70)).astype(np.uint8)
    X[(X & 0x7F) == 0x7F] = 0x38                        # no NaN patterns
    Sr = rng.integers(120, 135, (40, 3)).astype(np.uint8)   # blocks of 32 along a row
    Sc = rng.integers(120, 135, (2, 70)).astype(np.uint8)   # blocks of 32 down a column
    v = oracle.fp8_decode(X, "e4m3")
    rowscale = 2.0 ** (np.repeat(Sr.astype(np.int64), 32, axis=1)[:, :70] - 127)
    colscale = 2.0 ** (np.repeat(Sc.astype(np.int64), 32, axis=0)[:40, :] - 127)
    assert np.array_equal(oracle.mx_values(X, Sr, "e4m3", "row"), v * rowscale)
    assert np.array_equal(oracle.mx_values(X, Sc, "e4m3", "col"), v * colscale)


def test_mx_product_closed_form():
    # A = 1.0 everywhere with row scales 2^1, B = 0.5 with column scales 2^-2:
    # every entry of the product is K * 2 * 0.5 * 0.25
    M, N, K = 4, 6, 64
    A = np.full((M, K), 0x38, dtype=np.uint8)              # E4M3 1.0
    B = np.full((K, N), 0x38, dtype=np.uint8)              # E5M2 0.5 is 0x38 as well
    SA = np.full((M, K // 32), 128, dtype=np.uint8)
    SB = np.full((K // 32, N), 125, dtype=np.uint8)
    C = oracle.gemm(oracle.mx_values(A, SA, "e4m3", "row"), oracle.mx_values(B, SB, "e5m2", "col"))
    assert np.array_equal(C, np.full((M, N), K * 2.0 * 0.5 * 0.25))


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(31)
    x = rng.normal(0, 3, (7, 300))
    g = rng.uniform(0.5, 1.5, 300)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (300,), torch.from_numpy(g), eps=1e-5)
    assert np.allclose(oracle.rmsnorm(x, g, 1e-5), ref.numpy(), rtol=1e-13, atol=0)


def test_rmsnorm_closed_forms_and_invariance():
    # a constant row c: mean(x^2) = c^2, so y = c / sqrt(c^2 + eps)
    x = np.full((3, 64), 2.5)
    assert np.allclose(oracle.rmsnorm(x, None, 0.25), 2.5 / np.sqrt(6.25 + 0.25), rtol=1e-15)
    # scaling a row by s leaves it unchanged when eps = 0; a row of +-1 is fixed
    rng = np.random.default_rng(32)
    x = rng.normal(size=(5, 96))
    assert np.allclose(oracle.rmsnorm(7.0 * x, None, 0.0), oracle.rmsnorm(x, None, 0.0), rtol=1e-13)
    pm = np.where(rng.normal(size=(4, 128)) > 0, 1.0, -1.0)
    assert np.array_equal(oracle.rmsnorm(pm, None, 0.0), pm)


def test_block_sumsq_and_row_scale():
    x = np.arange(1.0, 1 + 3 * 130).reshape(3, 130)   # last block has 2 columns
    s = oracle.block_sumsq(x)
    assert s.shape == (3, 3)
    for p, (a, b) in enumerate([(0, 64), (64, 128), (128, 130)]):
        assert np.array_equal(s[p], (x[:, a:b] ** 2).sum(axis=1))
    r = oracle.row_scale(s, 130, 1e-3)
    assert np.allclose(r, 1 / np.sqrt((x ** 2).mean(axis=1) + 1e-3), rtol=1e-15)


def test_rms_scale_folded_into_the_next_product():
    # RMSNorm(x) W == diag(r) x (diag(g) W): what the consumer's epilogue uses
    rng = np.random.default_rng(33)
    x = rng.normal(size=(6, 192))
    g = rng.uniform(0.5, 1.5, 192)
    W = rng.normal(size=(192, 40))
    r = oracle.row_scale(oracle.block_sumsq(x), 192, 1e-6)
    lhs = oracle.gemm(oracle.rmsnorm(x, g, 1e-6), W)
    rhs = r[:, None] * oracle.gemm(x, g[:, None] * W)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ sampled path

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_sampled_equals_full_bitwise(dtype):
    A = inputs.matrix(40, 70, "uniform", dtype, 0)
    B = inputs.matrix(70, 30, "uniform", dtype, 1)
    Ab, Bb = inputs.bits(A), inputs.bits(B)
    full = oracle.gemm(oracle.decode(Ab, dtype), oracle.decode(Bb, dtype))
    rows, cols = inputs.sample_positions(40, 30, n=64, tile_m=16, tile_n=8)
    rows, cols = rows.numpy(), cols.numpy()
    s = oracle.gemm_sampled(Ab, Bb, dtype, rows, cols)
    assert np.array_equal(s, full[rows, cols])


@pytest.mark.parametrize("kind", ["scale_bias", "silu", "swiglu"])
def test_reference_sampled_equals_full_reference(kind):
    A = inputs.matrix(24, 48, "normal", "bf16", 0)
    B = inputs.matrix(48, 32, "normal_inv_k", "bf16", 1, k=48)
    bias = inputs.matrix(1, 32, "normal_0.02", "bf16", 2)[0]
    Ab, Bb, bb = inputs.bits(A), inputs.bits(B), inputs.bits(bias)
    full = oracle.reference(Ab, Bb, "bf16", kind, 0.75, bb)
    Nout = full.shape[1]
    rows, cols = inputs.sample_positions(24, Nout, n=40, tile_m=8, tile_n=8)
    rows, cols = rows.numpy(), cols.numpy()
    s = oracle.reference_sampled(Ab, Bb, "bf16", rows, cols, kind, 0.75, bb)
    assert np.array_equal(s, full[rows, cols])


def test_inputs_are_seeded_and_shaped():
    a1 = inputs.matrix(8, 8, "uniform", "bf16", 0)
    a2 = inputs.matrix(8, 8, "uniform", "bf16", 0)
    a3 = inputs.matrix(8, 8, "uniform", "bf16", 1)
    assert torch.equal(a1, a2) and not torch.equal(a1, a3)
    assert a1.dtype == torch.bfloat16 and a1.abs().max() <= 1
    t = inputs.matrix(64, 64, "ternary", "f16", 0)
    assert set(torch.unique(t).tolist()) <= {-1.0, 0.0, 1.0}
