"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small and mid sizes are checked on every output entry; the full-size
workloads on 4096 stratified sampled entries computed one by one by the
oracle, in the same launch configuration the benchmark times.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from complexity_matmul_tcgen05_gb300 import fgemm, inputs
from parity_util import (TOL_EMULATED, TOL_NORMWISE, activation_condition, elementwise_act_ok,
                         elementwise_ok, gpu_bits, normwise, preact_bound, record, run, values)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ternary(M, N, K, dtype, seed=10):
    A = inputs.matrix(M, K, "ternary", dtype, seed, DEV)
    B = inputs.matrix(K, N, "ternary", dtype, seed + 1, DEV)
    bias = inputs.matrix(1, N, "ternary_bias", dtype, seed + 2, DEV)[0]
    return A, B, bias


def _exact_reference(A, B, bias, dtype):
    ref = oracle.reference(gpu_bits(A), gpu_bits(B), dtype, "scale_bias", 1.0, gpu_bits(bias))
    return oracle.encode(ref, dtype)


# ------------------------------------------------- exact ternary parity

EXACT_CASES = [
    # (algo, M, N, K, tile_n)
    ("classical", 128, 256, 64, 256),
    ("classical", 128, 128, 64, 128),
    ("classical", 128, 64, 64, 64),
    ("classical", 1, 8, 8, 0),
    ("classical", 200, 328, 136, 256),     # ragged M, N, K tails
    ("classical", 257, 520, 1032, 128),
    ("classical", 300, 72, 520, 64),
    ("classical", 1000, 1000, 1000, 0),
    ("strassen1", 256, 256, 128, 128),
    ("strassen1", 256, 512, 128, 256),
    ("strassen1", 512, 1024, 640, 256),
    ("strassen2", 512, 512, 256, 128),
    ("strassen2", 512, 1024, 512, 256),
    ("winograd1", 256, 256, 128, 128),
    ("winograd1", 256, 512, 128, 256),
    ("winograd1", 512, 1024, 640, 256),
    ("winograd1", 1024, 512, 384, 128),
]
# CTA-pair tiles (256 rows over two SMs): (M, N, K, tile_n)
EXACT_PAIR_CASES = [
    (256, 256, 64, 256),
    (256, 128, 64, 128),
    (100, 256, 128, 256),      # the odd CTA's rows are all past M
    (300, 520, 1032, 128),     # ragged M, N, K
    (1000, 1000, 1000, 256),
    (2048, 1024, 512, 128),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("algo,M,N,K,tile", EXACT_CASES)
def test_exact_ternary(algo, M, N, K, tile, dtype):
    """Inputs in {-1,0,1}, integer bias: every form must equal RNE(exact C) bit for bit."""
    A, B, bias = _ternary(M, N, K, dtype)
    C = run(A, B, algo=algo, epilogue="scale_bias", bias=bias, tile_n=tile)
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, dtype))


# One level on CTA pairs (summed operands streamed through HBM by a pre-pass,
# products on the pair mainloop).  Each shape's (position, product) units are
# shared out over the pairs: 512 x 512 x 128 has 1 position (7 units, one per
# pair, so all 7 pairs finish it together); 512 x 1024 has 2 (14 units);
# 2048^2 at 256 has 16 (112 units over 76 pairs); 4096 x 4096 x 512 has 64
# (448 units: about 6 per pair, positions shared at every range boundary).
LCMA_PAIR_CASES = [(512, 512, 128, 128), (512, 1024, 256, 256), (1024, 2048, 640, 256),
                   (1536, 768, 384, 128), (2048, 2048, 256, 256), (4096, 4096, 512, 256),
                   (8192, 8192, 128, 256)]  # one K block per product, 3 whole waves per pair


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("algo", ["strassen1", "winograd1"])
@pytest.mark.parametrize("M,N,K,tile", LCMA_PAIR_CASES)
def test_exact_ternary_lcma_cta_pair(M, N, K, tile, algo, dtype):
    """One Strassen / Winograd level on CTA pairs: RNE(exact C) bit for bit."""
    A, B, bias = _ternary(M, N, K, dtype)
    C = run(A, B, algo=algo, epilogue="scale_bias", bias=bias, tile_n=tile, tile_m=256)
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, dtype))


# Enough output positions for whole waves on the pairs (the positions every
# pair runs through all seven products, folding and finishing them itself)
# besides a partial last wave: 4096 x 5120 has 8 x 10 positions of 256 x 256
# in its 2048 x 2560 blocks (SwiGLU: 8 x 5), 8 x 20 at tile 128.
@pytest.mark.parametrize("algo", ["strassen1", "winograd1"])
@pytest.mark.parametrize("tile", [256, 128])
@pytest.mark.parametrize("epilogue,alpha", [("none", 1.0), ("scale_bias", 0.75), ("silu", 1.25),
                                            ("swiglu", 1.0)])
def test_lcma_cta_pair_whole_positions_every_entry(algo, tile, epilogue, alpha):
    M, N, K = 4096, 5120 if epilogue != "swiglu" else 10240, 128
    A = inputs.matrix(M, K, "uniform", "bf16", 72, DEV)
    B = inputs.matrix(K, N, "uniform", "bf16", 73, DEV)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 74, DEV)[0] if epilogue != "none" else None
    _full_check(A, B, algo, "bf16", epilogue, alpha, bias, tile, 1, tile_m=256)


@pytest.mark.parametrize("algo", ["strassen1", "winograd1"])
@pytest.mark.parametrize("epilogue", ["scale_bias", "swiglu"])
def test_exact_ternary_lcma_cta_pair_whole_positions(algo, epilogue):
    M, N, K = 4096, 5120 if epilogue != "swiglu" else 10240, 384
    A, B, bias = _ternary(M, N, K, "bf16", seed=75)
    C = run(A, B, algo=algo, epilogue=epilogue, bias=bias, tile_n=256, tile_m=256)
    if epilogue == "scale_bias":
        assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, "bf16"))
    else:
        # gate and up are exact integers, so silu(gate) * up is the classical
        # kernel's, evaluated by the same fp32 operations: the same bits; and
        # each entry within the per-entry rule of the oracle's
        C0 = run(A, B, algo="classical", epilogue="swiglu", bias=bias, tile_n=256, tile_m=256)
        assert torch.equal(C.view(torch.int16), C0.view(torch.int16))
        Av, Bv, bv = values(A), values(B), values(bias)
        _act_entries_ok(values(C), "swiglu", oracle.gemm(Av, Bv), oracle.gemm(np.abs(Av), np.abs(Bv)), K,
                        1.0, bv, "bf16")


@pytest.mark.parametrize("algo", ["strassen1", "winograd1"])
def test_lcma_cta_pair_deterministic_and_graph_replay(algo):
    """Positions shared by two pairs are summed in pair order: two launches
    give the same bits; a captured graph replays the launch (its arrival
    counters count from zero each time) with the same result."""
    M, N, K = 4096, 2048, 1024
    A = inputs.matrix(M, K, "uniform", "bf16", 70, DEV)
    B = inputs.matrix(K, N, "uniform", "bf16", 71, DEV)
    kw = dict(algo=algo, tile_n=256, tile_m=256)
    C1 = run(A, B, **kw)
    C2 = run(A, B, **kw)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    C = torch.empty_like(C1)
    fgemm.matmul(A, B, out=C, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fgemm.matmul(A, B, out=C, **kw)
    for _ in range(3):
        C.view(torch.int16).fill_(0x7F7B)
        g.replay()
        torch.cuda.synchronize()
        assert fgemm.default_handle().get_error() == fgemm.OK
        assert torch.equal(C.view(torch.int16), C1.view(torch.int16))


# Two Strassen levels on CTA pairs: the 49 leaf operands of each side formed
# by the pre-pass (each from the 16 quarter blocks, one rounding), 49
# quarter-size products per position, folded into 16 output blocks.
# 1024^2 x 256 at 256 has one position (49 units over 49 pairs); 2048 x 4096
# has 8 positions (392 units over the pairs); 8192^2 at tile 128 has 128
# positions: one whole wave over the pairs plus a partial one; 16384 x 8192
# at tile 128 has 256: three whole waves (each pair's positions run outer
# product by outer product, the seven inner products back to back).
LCMA2_PAIR_CASES = [(1024, 1024, 256, 256), (1024, 1024, 256, 128), (2048, 4096, 512, 256),
                    (4096, 4096, 1024, 256), (8192, 8192, 256, 128), (16384, 8192, 256, 128)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K,tile", LCMA2_PAIR_CASES)
def test_exact_ternary_strassen2_cta_pair(M, N, K, tile, dtype):
    """Two Strassen levels on CTA pairs: RNE(exact C) bit for bit (operand
    sums in [-4, 4], products and folds exact in fp32)."""
    A, B, bias = _ternary(M, N, K, dtype)
    C = run(A, B, algo="strassen2", epilogue="scale_bias", bias=bias, tile_n=tile, tile_m=256)
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, dtype))


@pytest.mark.parametrize("tile", [256, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("epilogue,alpha", [("none", 1.0), ("silu", 1.25)])
def test_strassen2_cta_pair_every_entry_and_emulation(tile, dtype, epilogue, alpha):
    """Every entry within the two-level budget, and the tight pin against the
    oracle's emulated two-level Strassen (leaf operands rounded once)."""
    M, N, K = 1024, 2048, 1024
    A = inputs.matrix(M, K, "uniform", dtype, 80, DEV)
    B = inputs.matrix(K, N, "uniform", dtype, 81, DEV)
    bias = inputs.matrix(1, N, "normal_0.02", dtype, 82, DEV)[0] if epilogue != "none" else None
    _full_check(A, B, "strassen2", dtype, epilogue, alpha, bias, tile, 2, tile_m=256)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_strassen2_cta_pair_whole_positions_emulation(dtype):
    """Three whole waves of positions (the two-stage fold) besides a partial
    one: every entry against the oracle's emulated two-level Strassen."""
    M, N, K = 16384, 8192, 256
    A = inputs.matrix(M, K, "uniform", dtype, 85, DEV)
    B = inputs.matrix(K, N, "uniform", dtype, 86, DEV)
    _full_check(A, B, "strassen2", dtype, "none", 1.0, None, 128, 2, tile_m=256)


def test_strassen2_cta_pair_deterministic_and_graph_replay():
    """Two launches give the same bits; a captured graph (pre-pass and
    product kernel) replays with the same result."""
    M, N, K = 4096, 4096, 1024
    A = inputs.matrix(M, K, "uniform", "bf16", 83, DEV)
    B = inputs.matrix(K, N, "uniform", "bf16", 84, DEV)
    kw = dict(algo="strassen2", tile_n=256, tile_m=256)
    assert fgemm.default_handle().call_launches(M, N, K, **kw) == 2
    C1 = run(A, B, **kw)
    C2 = run(A, B, **kw)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    C = torch.empty_like(C1)
    fgemm.matmul(A, B, out=C, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fgemm.matmul(A, B, out=C, **kw)
    for _ in range(3):
        C.view(torch.int16).fill_(0x7F7B)
        g.replay()
        torch.cuda.synchronize()
        assert fgemm.default_handle().get_error() == fgemm.OK
        assert torch.equal(C.view(torch.int16), C1.view(torch.int16))


@pytest.fixture
def formation():
    """Sets the default handle's operand-formation mode for one test, then
    restores auto."""
    h = fgemm.default_handle()
    yield h.set_lcma_formation
    h.set_lcma_formation("auto")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K,tile", LCMA_PAIR_CASES)
def test_exact_ternary_winograd_formed_in_kernel(M, N, K, tile, dtype, formation):
    """Winograd's temporaries formed by the product kernel's own warps while
    its first two products (A11 B11, A12 B21) run: RNE(exact C) bit for bit."""
    formation("in_kernel")
    A, B, bias = _ternary(M, N, K, dtype, seed=76)
    C = run(A, B, algo="winograd1", epilogue="scale_bias", bias=bias, tile_n=tile, tile_m=256)
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, dtype))


@pytest.mark.parametrize("algo", ["winograd1", "strassen1"])
@pytest.mark.parametrize("M,N,K,tile,epilogue", [
    (4096, 5120, 1024, 256, "none"),      # whole positions and a tail
    (4096, 10240, 512, 256, "swiglu"),
    (2048, 2048, 2048, 128, "silu"),      # tail units only
    (1536, 768, 384, 128, "scale_bias"),
])
def test_lcma_formation_modes_give_the_same_bits(M, N, K, tile, epilogue, algo, formation):
    """The temporaries hold the same values whoever forms them, and the
    products run in the same order, so the pre-pass and the in-kernel
    formation give the same C bit for bit (Winograd: both sides' sums in the
    kernel; Strassen: B's in the kernel while M2 and M5 run, A's by the
    pre-pass)."""
    A = inputs.matrix(M, K, "uniform", "bf16", 77, DEV)
    B = inputs.matrix(K, N, "uniform", "bf16", 78, DEV)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 79, DEV)[0] if epilogue != "none" else None
    kw = dict(algo=algo, epilogue=epilogue, bias=bias, tile_n=tile, tile_m=256)
    formation("prepass")
    C1 = run(A, B, **kw)
    formation("in_kernel")
    C2 = run(A, B, **kw)
    C3 = run(A, B, **kw)  # the band counters start from zero every launch
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    assert torch.equal(C2.view(torch.int16), C3.view(torch.int16))


def test_call_launches_follows_the_formation(formation):
    """The launch count a call reports: one kernel, except one level on CTA
    pairs whose operand sums a pre-pass forms (Strassen always; Winograd
    when its sum-free products span fewer than 16 waves, or when asked)."""
    h = fgemm.default_handle()
    assert h.call_launches(4096, 4096, 4096, algo="classical", tile_m=256, tile_n=256) == 1
    assert h.call_launches(16384, 16384, 16384, algo="strassen1", tile_m=256, tile_n=256) == 2
    assert h.call_launches(16384, 16384, 16384, algo="winograd1", tile_m=256, tile_n=256) == 1
    assert h.call_launches(4096, 4096, 4096, algo="winograd1", tile_m=256, tile_n=256) == 2
    assert h.call_launches(4096, 4096, 4096, algo="winograd1", tile_m=128, tile_n=256) == 1
    assert h.call_launches(4096, 4096, 0, algo="classical") == 1
    formation("prepass")
    assert h.call_launches(16384, 16384, 16384, algo="winograd1", tile_m=256, tile_n=256) == 2
    formation("in_kernel")
    assert h.call_launches(4096, 4096, 4096, algo="winograd1", tile_m=256, tile_n=256) == 1
    assert h.call_launches(16384, 16384, 16384, algo="strassen1", tile_m=256, tile_n=256) == 2
    with pytest.raises(fgemm.FgemmError):
        h.call_launches(384, 256, 128, algo="strassen1", tile_m=256, tile_n=256)


def test_winograd_formed_in_kernel_graph_replay(formation):
    """A captured launch with in-kernel formation replays with the same
    result: the clearing of its band counters is part of the graph."""
    formation("in_kernel")
    M, N, K = 4096, 5120, 1024
    A = inputs.matrix(M, K, "uniform", "bf16", 80, DEV)
    B = inputs.matrix(K, N, "uniform", "bf16", 81, DEV)
    kw = dict(algo="winograd1", tile_n=256, tile_m=256)
    C1 = run(A, B, **kw)
    C = torch.empty_like(C1)
    fgemm.matmul(A, B, out=C, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fgemm.matmul(A, B, out=C, **kw)
    for _ in range(3):
        C.view(torch.int16).fill_(0x7F7B)
        g.replay()
        torch.cuda.synchronize()
        assert fgemm.default_handle().get_error() == fgemm.OK
        assert torch.equal(C.view(torch.int16), C1.view(torch.int16))
    # the graph's B now changes: the replay forms the new temporaries
    B2 = inputs.matrix(K, N, "uniform", "bf16", 82, DEV)
    B.copy_(B2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), run(A, B2, **kw).view(torch.int16))


@pytest.mark.parametrize("M,N,K,tile", [
    (8192, 2048, 64, 256), (8192, 2048, 64, 128), (8192, 4096, 64, 256), (8192, 2048, 128, 256),
    (16384, 4096, 64, 256), (8192, 2048, 192, 256),
])
def test_exact_ternary_cta_pair_short_k_many_tiles(M, N, K, tile):
    """One or two K blocks and three to fourteen tiles per pair: the warps
    that help with a pair's last tile get there while the MMAs of its earlier
    tiles still run (they must wait for the last tile itself); five launches
    in a row, each bit for bit."""
    A, B, bias = _ternary(M, N, K, "bf16", seed=110)
    ref = _exact_reference(A, B, bias, "bf16")
    for _ in range(5):
        C = run(A, B, algo="classical", epilogue="scale_bias", bias=bias, tile_n=tile, tile_m=256)
        assert np.array_equal(gpu_bits(C), ref)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K,tile", EXACT_PAIR_CASES)
def test_exact_ternary_cta_pair(M, N, K, tile, dtype):
    A, B, bias = _ternary(M, N, K, dtype)
    C = run(A, B, algo="classical", epilogue="scale_bias", bias=bias, tile_n=tile, tile_m=256)
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, dtype))


@pytest.mark.parametrize("tile_m,tile_n", [(0, 128), (256, 128), (256, 256)])
def test_exact_ternary_strided_and_guard_band(tile_m, tile_n):
    """lda/ldb/ldc larger than the row length; C's padding and rows around it
    untouched (on CTA pairs C leaves by TMA stores, clipped at M and N)."""
    M, N, K = 130, 200, 136
    A0, B0, bias = _ternary(M, N, K, "bf16", seed=20)
    A = torch.zeros((M, K + 24), dtype=torch.bfloat16, device=DEV)[:, :K]
    A.copy_(A0)
    B = torch.zeros((K, N + 56), dtype=torch.bfloat16, device=DEV)[:, :N]
    B.copy_(B0)
    canary = 0x7F7B  # a bf16 NaN pattern never produced by the kernel
    big = torch.full((M + 2, N + 40), canary, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    C = big[1:M + 1, :N]
    run(A, B, epilogue="scale_bias", bias=bias, out=C, tile_n=tile_n, tile_m=tile_m)
    ref = _exact_reference(A0, B0, bias, "bf16")
    assert np.array_equal(gpu_bits(C), ref)
    raw = big.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (raw[0] == canary).all() and (raw[M + 1] == canary).all()
    assert (raw[1:M + 1, N:] == canary).all()


def test_pair_swiglu_padded_output_guard_band():
    """SwiGLU on CTA pairs into an output with a padded row pitch: every entry
    of the valid region within the classical bounds, the padding untouched."""
    M, N, K = 600, 1040, 520     # 3 x 5 pair tiles (128 output columns each), ragged
    A = inputs.matrix(M, K, "normal", "bf16", 21, DEV)
    B = inputs.matrix(K, N, "normal_inv_k", "bf16", 22, DEV, k=K)
    canary = 0x7F7B
    big = torch.full((M + 2, N // 2 + 24), canary, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    C = big[1:M + 1, :N // 2]
    run(A, B, epilogue="swiglu", out=C, tile_n=256, tile_m=256)
    raw = big.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (raw[0] == canary).all() and (raw[M + 1] == canary).all()
    assert (raw[1:M + 1, N // 2:] == canary).all()
    Av, Bv = oracle.decode(gpu_bits(A), "bf16"), oracle.decode(gpu_bits(B), "bf16")
    prod = oracle.gemm(Av, Bv)
    ref = oracle.epilogue(prod, "swiglu", 1.0, None)
    err = normwise(values(C), ref, "bf16")
    record("normwise swiglu (classical)", err, TOL_NORMWISE["classical"])
    assert err <= TOL_NORMWISE["classical"]
    _act_entries_ok(values(C), "swiglu", prod, oracle.gemm(np.abs(Av), np.abs(Bv)), K, 1.0, None,
                    "bf16")


# ----------------------------------------- full-entry tolerance parity

def _act_entries_ok(c, kind, raw, absdot, K, alpha, bias, dtype):
    """The per-entry classical rule through SiLU / SwiGLU (parity_util
    elementwise_act_ok) on full matrices: raw and absdot are the M x N
    pre-activation product and its sum of |a||b| (gate | up for SwiGLU)."""
    b = 0.0 if bias is None else bias[None, :]
    v = alpha * raw + b
    dv = preact_bound(raw, absdot, K, alpha, b)
    if kind == "silu":
        ok, frac = elementwise_act_ok(c, "silu", v, dv, None, None, dtype)
    else:
        h = raw.shape[1] // 2
        ok, frac = elementwise_act_ok(c, "swiglu", v[:, :h], dv[:, :h], v[:, h:], dv[:, h:], dtype)
    record(f"{kind} entries on the propagated branch", frac, 1.0)
    assert ok


def _full_check(A, B, algo, dtype, epilogue="none", alpha=1.0, bias=None, tile=0, depth=0,
                tile_m=0):
    """Every entry: the form's normwise budget; for classical the per-entry
    rule (8 ulp, or the dot-product bound carried through the activation);
    for the rounded-operand forms the tight pin against the oracle's emulated
    (rounded-operand) form through the same epilogue.

    The budgets are the forms' own, bare.  Through SiLU / SwiGLU a rounded-
    operand form's activated output is further held to its budget times the
    activation's condition number kappa at the reference (its product error
    is amplified by up to kappa), and the same form's pre-activation product
    (alpha and bias, no activation) is run and held to the bare budgets."""
    C = run(A, B, algo=algo, epilogue=epilogue, alpha=alpha, bias=bias, tile_n=tile, tile_m=tile_m)
    Ab, Bb = gpu_bits(A), gpu_bits(B)
    bb = None if bias is None else gpu_bits(bias)
    Av, Bv = oracle.decode(Ab, dtype), oracle.decode(Bb, dtype)
    bv = None if bb is None else oracle.decode(bb, dtype)
    raw = oracle.gemm(Av, Bv)
    ref = oracle.epilogue(raw, epilogue, alpha, bv)
    c = values(C)
    err = normwise(c, ref, dtype)
    activated = epilogue in ("silu", "swiglu")
    tol = TOL_NORMWISE[algo]
    if algo == "classical" or not activated:
        record(f"normwise {epilogue} ({algo})", err, tol)
        assert err <= tol, err
    else:
        kappa = activation_condition(raw, epilogue, alpha, bv)
        record(f"normwise {epilogue} ({algo}, x kappa {kappa:.2f})", err, tol * max(1.0, kappa))
        assert err <= tol * max(1.0, kappa), (err, kappa)
    if algo == "classical":
        absdot = oracle.gemm(np.abs(Av), np.abs(Bv))
        if activated:
            _act_entries_ok(c, epilogue, raw, absdot, A.shape[1], alpha, bv, dtype)
        else:
            ok, frac = elementwise_ok(c, ref, abs(alpha) * absdot, A.shape[1], dtype)
            record("entries on the dot-product branch", frac, 1.0)
            assert ok
    if depth > 0:
        emulated = oracle.winograd_emulated if algo == "winograd1" else oracle.strassen_emulated
        emu_raw = emulated(Av, Bv, depth, dtype)
        emu = oracle.epilogue(emu_raw, epilogue, alpha, bv)
        e2 = float(np.linalg.norm(c - oracle.round_to(emu, dtype)) / np.linalg.norm(emu))
        record(f"vs emulated, {epilogue} ({algo})", e2, TOL_EMULATED)
        assert e2 <= TOL_EMULATED, e2
        if activated:
            pre_epi = "scale_bias" if bias is not None else "none"
            P = run(A, B, algo=algo, epilogue=pre_epi, alpha=alpha, bias=bias, tile_n=tile,
                    tile_m=tile_m)
            p = values(P)
            e_pre = normwise(p, oracle.epilogue(raw, pre_epi, alpha, bv), dtype)
            record(f"normwise pre-activation ({algo})", e_pre, tol)
            assert e_pre <= tol, e_pre
            emu_pre = oracle.epilogue(emu_raw, pre_epi, alpha, bv)
            e2p = float(np.linalg.norm(p - oracle.round_to(emu_pre, dtype)) / np.linalg.norm(emu_pre))
            record(f"vs emulated, pre-activation ({algo})", e2p, TOL_EMULATED)
            assert e2p <= TOL_EMULATED, e2p
    return err


@pytest.mark.parametrize("algo,depth", [("classical", 0), ("strassen1", 1)])
def test_square_256_fp16_every_entry(algo, depth):
    """fp16 256^3, A,B ~ U[-1,1] (seeds 0,1): all 65536 entries."""
    A, B, _ = inputs.workload_inputs("square_256_f16", DEV)
    _full_check(A, B, algo, "f16", depth=depth)


@pytest.mark.parametrize("tile_m,tile", [(128, 64), (128, 128), (128, 256), (256, 128), (256, 256)])
@pytest.mark.parametrize("epilogue,alpha", [("none", 1.0), ("scale_bias", 0.5), ("silu", 1.25)])
def test_classical_epilogues_every_entry(epilogue, alpha, tile_m, tile):
    M, N, K = 384, 640, 320
    A = inputs.matrix(M, K, "normal", "bf16", 0, DEV)
    B = inputs.matrix(K, N, "normal_inv_k", "bf16", 1, DEV, k=K)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 2, DEV)[0] if epilogue != "none" else None
    _full_check(A, B, "classical", "bf16", epilogue, alpha, bias, tile, tile_m=tile_m)


@pytest.mark.parametrize("algo,tile_m,tile,depth", [
    ("classical", 128, 128, 0), ("classical", 128, 256, 0), ("classical", 256, 128, 0),
    ("classical", 256, 256, 0), ("strassen1", 128, 128, 1), ("strassen1", 128, 256, 1),
    ("strassen1", 256, 256, 1), ("strassen1", 256, 128, 1), ("strassen2", 128, 128, 2),
    ("winograd1", 128, 256, 1), ("winograd1", 256, 256, 1)])
def test_swiglu_every_entry(algo, tile_m, tile, depth):
    M, N, K = 512, 2048, 512
    A = inputs.matrix(M, K, "normal", "bf16", 0, DEV)
    B = inputs.matrix(K, N, "normal_inv_k", "bf16", 1, DEV, k=K)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 2, DEV)[0]
    _full_check(A, B, algo, "bf16", "swiglu", 1.0, bias, tile, depth, tile_m=tile_m)


@pytest.mark.parametrize("algo,tile_m,tile,depth", [
    ("strassen1", 128, 128, 1), ("strassen1", 128, 256, 1), ("strassen1", 256, 128, 1),
    ("strassen1", 256, 256, 1), ("strassen2", 128, 128, 2), ("strassen2", 128, 256, 2),
    ("winograd1", 128, 128, 1), ("winograd1", 128, 256, 1), ("winograd1", 256, 128, 1),
    ("winograd1", 256, 256, 1)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_strassen_every_entry_and_emulation(algo, tile_m, tile, depth, dtype):
    """Normwise bound and the tighter pin: GPU Strassen vs the emulated
    (rounded-operand) Strassen of the oracle."""
    M, N, K = 512, 1024, 768
    A = inputs.matrix(M, K, "uniform", dtype, 0, DEV)
    B = inputs.matrix(K, N, "uniform", dtype, 1, DEV)
    _full_check(A, B, algo, dtype, tile=tile, depth=depth, tile_m=tile_m)


# -------------------------------------------------------------- edge cases

def test_empty_and_k_zero():
    A = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    B = torch.ones((64, 32), dtype=torch.bfloat16, device=DEV)
    C = run(A, B)
    assert C.shape == (0, 32)
    A = torch.empty((5, 0), dtype=torch.bfloat16, device=DEV)
    B = torch.empty((0, 16), dtype=torch.bfloat16, device=DEV)
    bias = inputs.matrix(1, 16, "normal", "bf16", 3, DEV)[0]
    C = run(A, B, epilogue="scale_bias", bias=bias)
    ref = oracle.encode(np.tile(values(bias), (5, 1)), "bf16")
    assert np.array_equal(gpu_bits(C), ref)


def test_rejections_do_not_launch():
    h = fgemm.default_handle()
    A = torch.zeros((128, 72), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((72, 64), dtype=torch.bfloat16, device=DEV)
    C = torch.zeros((128, 64), dtype=torch.bfloat16, device=DEV)
    s = h.matmul_raw(128, 64, 72, A.data_ptr() + 2, 72, B.data_ptr(), 64, C.data_ptr(), 64, fgemm.BF16)
    assert s == fgemm.ERR_ALIGNMENT
    s = h.matmul_raw(128, 64, 72, A.data_ptr(), 72, B.data_ptr(), 64, C.data_ptr(), 64, fgemm.BF16,
                     None, "strassen1")
    assert s == fgemm.ERR_UNSUPPORTED
    s = h.matmul_raw(128, 64, 72, A.data_ptr(), 72, B.data_ptr(), 64, C.data_ptr(), 64, fgemm.BF16,
                     fgemm.make_epilogue("scale_bias"))
    assert s == fgemm.ERR_INVALID_ARG
    assert h.get_error() == fgemm.OK


def test_plan_is_legal_and_launchable():
    for (M, N, K) in [(256, 256, 256), (4096, 4096, 4096), (16, 2048, 2048), (16384, 16384, 16384)]:
        algo, tile_m, tile, us = fgemm.plan(M, N, K)
        assert algo in ("classical", "strassen1", "strassen2", "winograd1") and tile in (64, 128, 256)
        assert tile_m in (128, 256) or (tile_m in (16, 32, 64) and M <= tile_m and tile == 128)
        assert us > 0
        A = inputs.matrix(M, K, "ternary", "bf16", 32, DEV)
        B = inputs.matrix(K, N, "ternary", "bf16", 33, DEV)
        if M * N * K <= 2 ** 33:  # launch what the plan chose
            C = run(A, B, algo=algo, tile_n=tile, tile_m=tile_m)
            ref = A.float() @ B.float()
            assert torch.equal(C.float(), ref.to(torch.bfloat16).float())


def test_auto_takes_the_model_decision_with_its_margin():
    """A handle's AUTO is fgemm_model_plan on the handle's model: a
    low-complexity form only when predicted faster than the best classical
    form by the margin (on the planned cubes and the 17 sweep shapes), and
    never with a margin of 0.9; with a margin of 0 the fastest prediction."""
    L = fgemm.lib()
    h = fgemm.Handle()
    m = h.device_model()
    shapes = [(n, n, n) for n in (4096, 8192, 12288, 16384, 20480, 24576, 32768)] + \
        [(M, n, n) for M in (16, 128, 1024, 8192) for n in (2048, 4096, 8192, 16384)] + [(65536, 1024, 1024)]

    def model_pick(model, M, N, K):
        a, tm, tn, us = ctypes.c_int(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
        assert L.fgemm_model_plan(ctypes.byref(model), M, N, K, 0, ctypes.byref(a), ctypes.byref(tm),
                                  ctypes.byref(tn), ctypes.byref(us)) == fgemm.OK
        return fgemm.ALGO_NAMES[a.value], tm.value, tn.value, us.value

    try:
        for margin in (m.lcma_margin, 0.9, 0.0):
            m.lcma_margin = margin
            h.set_device_model(m)
            for (M, N, K) in shapes:
                got = h.plan(M, N, K)
                want = model_pick(m, M, N, K)
                assert got[:3] == want[:3] and abs(got[3] - want[3]) <= 1e-9 * want[3], (margin, M, N, K, got, want)
                if margin == 0.9:
                    assert got[0] == "classical", (M, N, K, got)
                if got[0] != "classical":
                    best_classical = h.plan(M, N, K, algo="classical")[3]
                    assert got[3] < (1.0 - margin) * best_classical, (margin, M, N, K, got, best_classical)
    finally:
        h.close()


def test_host_buffers_end_to_end():
    A = inputs.matrix(256, 128, "ternary", "bf16", 30)
    B = inputs.matrix(128, 192, "ternary", "bf16", 31)
    C = fgemm.matmul(A.pin_memory(), B.pin_memory(), algo="classical")
    assert C.device.type == "cpu"
    ref = oracle.encode(oracle.gemm(values(A), values(B)), "bf16")
    assert np.array_equal(gpu_bits(C), ref)


def test_two_handles_two_streams():
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    A, B, bias = _ternary(256, 256, 128, "bf16", seed=40)
    ref = _exact_reference(A, B, bias, "bf16")
    h2 = fgemm.Handle()
    with torch.cuda.stream(s1):
        C1 = fgemm.matmul(A, B, epilogue="scale_bias", bias=bias, algo="strassen1")
    with torch.cuda.stream(s2):
        C2 = fgemm.matmul(A, B, epilogue="scale_bias", bias=bias, algo="classical", handle=h2)
    torch.cuda.synchronize()
    assert np.array_equal(gpu_bits(C1), ref) and np.array_equal(gpu_bits(C2), ref)
    assert h2.get_error() == fgemm.OK
    h2.close()


# ------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout_and_handle_survives():
    """A wait that nothing will complete gives up after its limit, the kernel
    exits, fgemm_get_error reports the timeout (role and block), and the same
    handle then computes a correct product."""
    import time
    h = fgemm.Handle()
    assert h.get_error() == fgemm.OK
    t0 = time.perf_counter()
    assert fgemm.lib().fgemm_selftest_wait_timeout(h.ptr, 50) == fgemm.OK
    status = h.get_error()
    elapsed = time.perf_counter() - t0
    assert status == fgemm.ERR_TIMEOUT
    assert "producer" in h.last_message()
    assert 0.045 <= elapsed < 5.0
    assert h.get_error() == fgemm.OK            # the word was cleared
    A, B, bias = _ternary(256, 256, 128, "bf16", seed=80)
    C = fgemm.matmul(A, B, epilogue="scale_bias", bias=bias, algo="classical", handle=h)
    torch.cuda.synchronize()
    assert h.get_error() == fgemm.OK
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, "bf16"))
    h.close()


# ------------------------------------- K split of the last wave (CTA pairs)

@pytest.fixture
def split_mode():
    """Sets the default handle's K-split mode for one test, then restores auto."""
    h = fgemm.default_handle()
    yield h.set_split_mode
    h.set_split_mode("auto")


SPLIT_CASES = [
    # (M, N, K, tile_n): tiles on the pairs that fit, with a partial last wave
    (256, 256, 4096, 256),     # one tile shared by every pair
    (256, 256, 64, 256),       # one K block: too short to share, whole-tile path
    (2304, 2048, 1032, 256),   # 72 tiles (fewer than the pairs), ragged K
    (4096, 4096, 512, 256),    # 256 tiles: a full wave count plus a tail
    (300, 520, 1032, 128),     # ragged M, N, K
    (5000, 640, 776, 128),     # 20 x 5 = 100 tiles, ragged M and K
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K,tile", SPLIT_CASES)
def test_exact_ternary_cta_pair_split(M, N, K, tile, dtype, split_mode):
    """Split pieces summed by the last one: still RNE(exact C) bit for bit."""
    split_mode("force")
    A, B, bias = _ternary(M, N, K, dtype, seed=30)
    C = run(A, B, algo="classical", epilogue="scale_bias", bias=bias, tile_n=tile, tile_m=256)
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, dtype))


@pytest.mark.parametrize("epilogue,alpha,tile", [("scale_bias", 0.75, 256), ("silu", 1.0, 128),
                                                 ("swiglu", 1.0, 256), ("swiglu", 1.0, 128)])
def test_split_every_entry_and_deterministic(epilogue, alpha, tile, split_mode):
    """Forced split on random inputs: every entry within the classical bounds,
    and two runs give the same bits (the pieces are summed in a fixed order)."""
    split_mode("force")
    M, N, K = 1280, 2048, 2112  # 5 x 8 = 40 pair tiles (SwiGLU: 5 x 8 or 5 x 16), K ragged
    A = inputs.matrix(M, K, "normal", "bf16", 40, DEV)
    B = inputs.matrix(K, N, "normal_inv_k", "bf16", 41, DEV, k=K)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 42, DEV)[0] if epilogue != "swiglu" else None
    _full_check(A, B, "classical", "bf16", epilogue=epilogue, alpha=alpha, bias=bias, tile=tile,
                tile_m=256)
    C1 = run(A, B, algo="classical", epilogue=epilogue, alpha=alpha, bias=bias, tile_n=tile,
             tile_m=256)
    C2 = run(A, B, algo="classical", epilogue=epilogue, alpha=alpha, bias=bias, tile_n=tile,
             tile_m=256)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    # and the whole-wave form agrees within the classical tolerance
    split_mode("off")
    C0 = run(A, B, algo="classical", epilogue=epilogue, alpha=alpha, bias=bias, tile_n=tile,
             tile_m=256)
    d = values(C1) - values(C0)
    assert np.linalg.norm(d) <= 1e-3 * max(np.linalg.norm(values(C0)), 1e-30)


# --------------------------------------------- small-M kernel (C^T = B^T A^T)

SMALL_M_CASES = [
    # (M, N, K, tile_m)
    (1, 8, 64, 16),          # one row, one ragged column tile
    (16, 4096, 4096, 16),    # 32 tiles x 64 K blocks over every SM
    (7, 1000, 520, 16),      # ragged M, N, K
    (32, 520, 64, 32),       # one K block: whole tiles only
    (33, 2048, 1032, 64),
    (64, 4096, 8192, 64),
    (16, 16384, 256, 16),    # more tiles than SMs
    (16, 128, 32768, 16),    # one tile shared by 64 CTAs (64 pieces)
    (16, 16384, 4096, 16),   # 128 CTAs of one whole tile each
    (16, 4096, 16384, 16),   # 128 CTAs of a quarter tile: 4 pieces a tile
    (16, 28672, 4096, 16),   # 224 tiles on 128 CTAs: shares of 1.75 tiles cross tile ends
    (48, 16384, 8192, 64),   # ragged M in 64-row tiles, one whole tile per CTA
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K,tm", SMALL_M_CASES)
def test_exact_ternary_small_m(M, N, K, tm, dtype):
    A, B, bias = _ternary(M, N, K, dtype, seed=50)
    C = run(A, B, algo="classical", epilogue="scale_bias", bias=bias, tile_n=128, tile_m=tm)
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, dtype))


@pytest.mark.parametrize("tm", [16, 32, 64])
@pytest.mark.parametrize("epilogue,alpha", [("none", 1.0), ("scale_bias", 0.5), ("silu", 1.25)])
def test_small_m_every_entry_and_deterministic(tm, epilogue, alpha):
    M, N, K = tm - 3, 1536, 3080  # ragged M, N and K; 12 tiles shared over the SMs
    A = inputs.matrix(M, K, "normal", "bf16", 60, DEV)
    B = inputs.matrix(K, N, "normal_inv_k", "bf16", 61, DEV, k=K)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 62, DEV)[0]
    _full_check(A, B, "classical", "bf16", epilogue=epilogue, alpha=alpha, bias=bias, tile=128,
                tile_m=tm)
    C1 = run(A, B, algo="classical", epilogue=epilogue, alpha=alpha, bias=bias, tile_n=128, tile_m=tm)
    C2 = run(A, B, algo="classical", epilogue=epilogue, alpha=alpha, bias=bias, tile_n=128, tile_m=tm)
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


def test_small_m_strided_and_guard_band():
    """lda/ldb/ldc beyond the row length; rows past M and C's padding untouched."""
    M, N, K = 12, 300, 200
    A0, B0, bias = _ternary(M, N, K, "bf16", seed=70)
    A = torch.zeros((M, K + 40), dtype=torch.bfloat16, device=DEV)[:, :K]
    A.copy_(A0)
    B = torch.zeros((K, N + 20), dtype=torch.bfloat16, device=DEV)[:, :N]
    B.copy_(B0)
    canary = 0x7F7B
    big = torch.full((M + 2, N + 28), canary, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    C = big[1:M + 1, :N]
    run(A, B, epilogue="scale_bias", bias=bias, out=C, tile_n=128, tile_m=16)
    assert np.array_equal(gpu_bits(C), _exact_reference(A0, B0, bias, "bf16"))
    raw = big.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (raw[0] == canary).all() and (raw[M + 1] == canary).all()
    assert (raw[1:M + 1, N:] == canary).all()


@pytest.mark.parametrize("M,N,K,tm,tn", [(4096, 4096, 512, 256, 256),   # CTA pairs, split last wave
                                         (16, 4096, 4096, 16, 128),     # small-M stream-K
                                         (2560, 2048, 512, 256, 256)])  # 80 tiles: 4 split in 4
def test_graph_replays_recount_split_pieces(M, N, K, tm, tn, split_mode):
    """A CUDA graph replays the same launch parameters; the pieces' arrival
    counters must start from zero on every replay, or tiles go unwritten."""
    split_mode("force")
    A, B, bias = _ternary(M, N, K, "bf16", seed=80)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    kw = dict(out=C, epilogue="scale_bias", bias=bias, algo="classical", tile_n=tn, tile_m=tm)
    fgemm.matmul(A, B, **kw)  # allocations and launch set-up happen outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fgemm.matmul(A, B, **kw)
    ref = _exact_reference(A, B, bias, "bf16")
    for _ in range(3):
        C.view(torch.int16).fill_(0x7F7B)  # a NaN pattern the kernel never writes
        g.replay()
        torch.cuda.synchronize()
        assert fgemm.default_handle().get_error() == fgemm.OK
        assert np.array_equal(gpu_bits(C), ref)


# ------------------------------------------ RMSNorm statistics in the epilogue

@pytest.mark.parametrize("tm,tn,epilogue", [(128, 64, "none"), (128, 128, "scale_bias"),
                                            (128, 256, "silu"), (256, 128, "none"),
                                            (256, 256, "scale_bias"), (128, 256, "swiglu"),
                                            (256, 256, "swiglu")])
def test_rms_sums_of_squares_out(tm, tn, epilogue):
    """The producer's block sums of squares equal the oracle's over the values
    C actually holds (fp32 sums of 64 squares against fp64)."""
    M, N, K = 300, 1000, 520          # ragged rows, a partial last block
    if epilogue == "swiglu":
        N = 2064                      # output width 1032: 17 blocks, the last of 8 columns
    A = inputs.matrix(M, K, "normal", "bf16", 90, DEV)
    B = inputs.matrix(K, N, "normal_inv_k", "bf16", 91, DEV, k=K)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 92, DEV)[0] if epilogue == "scale_bias" else None
    n_out = N // 2 if epilogue == "swiglu" else N
    S = torch.full(((n_out + 63) // 64, M), float("nan"), dtype=torch.float32, device=DEV)
    C = fgemm.matmul(A, B, epilogue=epilogue, bias=bias, tile_m=tm, tile_n=tn, sumsq_out=S)
    torch.cuda.synchronize()
    assert fgemm.default_handle().get_error() == fgemm.OK
    ref = oracle.block_sumsq(values(C))
    got = S.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert np.allclose(got, ref, rtol=1e-5, atol=0), np.max(np.abs(got - ref) / np.maximum(ref, 1e-30))


@pytest.mark.parametrize("tm,tn", [(128, 128), (256, 256)])
def test_rms_scale_in_chain(tm, tn):
    """x = A W1 (+ its sums of squares); y = RMSNorm(x; g) W2 computed as
    diag(r) x (g W2) by the second product: against the oracle's chain on the
    same bf16 inputs (x as stored, g W2 as rounded), and against the plain
    definition RMSNorm(x) W2 within the rounding of g W2."""
    M, D, F, K = 512, 1024, 768, 640
    eps = 1e-5
    A = inputs.matrix(M, K, "normal", "bf16", 93, DEV)
    W1 = inputs.matrix(K, D, "normal_inv_k", "bf16", 94, DEV, k=K)
    W2 = inputs.matrix(D, F, "normal_inv_k", "bf16", 95, DEV, k=D)
    g = (1.0 + 0.1 * torch.randn(D, generator=torch.Generator().manual_seed(96))).to(torch.float64)
    S = torch.empty(((D + 63) // 64, M), dtype=torch.float32, device=DEV)
    X = fgemm.matmul(A, W1, tile_m=tm, tile_n=tn, sumsq_out=S)
    W2g = (g[:, None] * W2.double().cpu()).to(torch.bfloat16).to(DEV)   # g folded, rounded once
    Y = fgemm.matmul(X, W2g, tile_m=tm, tile_n=tn, sumsq_in=S, norm_width=D, rms_eps=eps)
    torch.cuda.synchronize()
    assert fgemm.default_handle().get_error() == fgemm.OK
    xv = values(X)
    r = oracle.row_scale(oracle.block_sumsq(xv), D, eps)
    acc = oracle.gemm(xv, values(W2g))
    ref = r[:, None] * acc
    y = values(Y)
    assert normwise(y, ref, "bf16") <= TOL_NORMWISE["classical"]
    absdot = r[:, None] * oracle.gemm(np.abs(xv), np.abs(values(W2g)))
    ok, _ = elementwise_ok(y, ref, absdot, D, "bf16")
    assert ok
    # the definition, with the exact gain: off only by the rounding of g W2
    defn = oracle.gemm(oracle.rmsnorm(xv, g.numpy(), eps), values(W2))
    assert float(np.linalg.norm(y - defn) / np.linalg.norm(defn)) <= 5e-3


def test_rms_rejections():
    A = torch.zeros((256, 128), dtype=torch.bfloat16, device=DEV)
    B = torch.zeros((128, 256), dtype=torch.bfloat16, device=DEV)
    S = torch.zeros((4, 256), dtype=torch.float32, device=DEV)
    with pytest.raises(fgemm.FgemmError):   # Strassen forms carry no statistics
        fgemm.matmul(A, B, algo="strassen1", sumsq_out=S)
    with pytest.raises(fgemm.FgemmError):   # nor does the small-M kernel
        fgemm.matmul(A[:16], B, tile_m=16, tile_n=128, sumsq_out=S[:, :16].contiguous())
    with pytest.raises(fgemm.FgemmError):   # eps must be finite and >= 0
        fgemm.matmul(A, B, sumsq_in=S, norm_width=256, rms_eps=-1.0)


# ----------------------------------------------- block-scaled 8-bit (MX) inputs

def _mx_random(rows, cols, fmt, along, seed, lo=118, hi=136):
    """Random 8-bit floats (no NaN or infinity patterns) and E8M0 scales in
    [lo, hi) (2^-9 .. 2^8): uint8 tensors on the device."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.int32).to(torch.uint8)
    special = (x & 0x7F) == 0x7F if fmt == "e4m3" else (x & 0x7C) == 0x7C
    x[special] = 0x38
    kb = (cols + 31) // 32 if along == "row" else (rows + 31) // 32
    shape = (rows, kb) if along == "row" else (kb, cols)
    s = torch.randint(lo, hi, shape, generator=g, dtype=torch.int32).to(torch.uint8)
    return x.to(DEV), s.to(DEV)


def _np(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("along", ["row", "col"])
def test_mx_to_bf16_every_pattern_and_scale(fmt, along):
    """Every 8-bit pattern (NaNs and infinities included) under every E8M0
    scale: the bf16 value equals the exact value rounded once (subnormal
    results, overflow to infinity, NaN scales)."""
    x = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    if along == "row":   # 256 rows = one per scale; each row is all 256 patterns
        X = x.repeat(256, 1).to(DEV)
        S = torch.arange(256, dtype=torch.int32).to(torch.uint8)[:, None].repeat(1, 8).to(DEV)
    else:                # 256 columns per pattern block, scales down each column
        X = x[:, None].repeat(1, 256).to(DEV)
        S = torch.arange(256, dtype=torch.int32).to(torch.uint8)[None, :].repeat(8, 1).to(DEV)
    Y = fgemm.mx_to_bf16(X, S, fmt, along)
    torch.cuda.synchronize()
    ref = oracle.mx_values(_np(X), _np(S), fmt, along)
    got = values(Y)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(gpu_bits(Y)[ok], oracle.encode(ref[ok], "bf16"))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("along", ["row", "col"])
@pytest.mark.parametrize("rows,cols,offset", [(96, 1024, 0), (70, 1000, 0), (65, 515, 1)])
def test_mx_to_bf16_quantised_data_with_planted_specials(fmt, along, rows, cols, offset):
    """Gaussian values cast to 8 bits (almost every 16-column group is plain
    normals and zeros) with a few planted subnormals, NaN / infinity patterns,
    zeros of both signs and out-of-range scales; ragged column counts and
    (offset 1) rows that are not 16-byte aligned.  Bit for bit against the
    oracle."""
    g = torch.Generator().manual_seed(105)
    sigma, f8 = (64.0, torch.float8_e4m3fn) if fmt == "e4m3" else (8192.0, torch.float8_e5m2)
    full = (torch.randn((rows, cols + offset), generator=g) * sigma).to(f8).view(torch.uint8)
    n = rows * (cols + offset)
    flat = full.view(-1)
    idx = torch.randint(0, n, (40,), generator=g)
    sub = 0x05 if fmt == "e4m3" else 0x02            # 8-bit subnormals
    nan = 0x7F if fmt == "e4m3" else 0x7E
    plant = torch.tensor([sub, sub | 0x80, nan, 0x00, 0x80] * 8, dtype=torch.uint8)
    flat[idx] = plant
    if fmt == "e5m2":
        flat[idx[:4]] = torch.tensor([0x7C, 0xFC, 0x7F, 0x01], dtype=torch.uint8)   # +-inf, NaN, subnormal
    X = full.to(DEV)[:, offset:]
    kb = (cols + 31) // 32 if along == "row" else (rows + 31) // 32
    shape = (rows, kb) if along == "row" else (kb, cols)
    S = torch.randint(100, 150, shape, generator=g, dtype=torch.int32).to(torch.uint8)
    sflat = S.view(-1)
    sidx = torch.randint(0, sflat.numel(), (6,), generator=g)
    sflat[sidx] = torch.tensor([0, 3, 250, 255, 254, 1], dtype=torch.uint8)
    S = S.to(DEV)
    Y = fgemm.mx_to_bf16(X, S, fmt, along)
    torch.cuda.synchronize()
    ref = oracle.mx_values(_np(X), _np(S), fmt, along)
    got = values(Y)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(gpu_bits(Y)[ok], oracle.encode(ref[ok], "bf16"))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_mx_values_exact_through_identity(fmt):
    """C = A x I through the whole MX product: every entry is A's value rounded
    once to bf16, bit for bit (scales that keep the values in bf16's normal
    range; how the tensor core treats subnormal inputs is not this test's)."""
    M, K = 130, 96
    A, SA = _mx_random(M, K, fmt, "row", 100, lo=20, hi=240)
    B = torch.zeros((K, K), dtype=torch.uint8, device=DEV)
    B.fill_diagonal_(0x38 if fmt == "e4m3" else 0x3C)         # 1.0
    SB = torch.full(((K + 31) // 32, K), 127, dtype=torch.uint8, device=DEV)
    C = fgemm.matmul_mx(A, SA, B, SB, a_format=fmt, b_format=fmt)
    torch.cuda.synchronize()
    assert fgemm.default_handle().get_error() == fgemm.OK
    ref = oracle.encode(oracle.mx_values(_np(A), _np(SA), fmt, "row"), "bf16")
    got = gpu_bits(C)
    # -0 in A meets +0 products from the rest of the row: the sum is +0
    zero = ((got & 0x7FFF) == 0) & ((ref & 0x7FFF) == 0)
    assert np.array_equal(np.where(zero, 0, got), np.where(zero, 0, ref))


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e5m2")])
@pytest.mark.parametrize("M,N,K,epilogue", [(256, 512, 1024, "none"), (300, 520, 1000, "scale_bias"),
                                            (1024, 1024, 2048, "silu")])
def test_mx_product_every_entry(fa, fb, M, N, K, epilogue):
    A, SA = _mx_random(M, K, fa, "row", 101)
    B, SB = _mx_random(K, N, fb, "col", 102)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 103, DEV)[0] if epilogue == "scale_bias" else None
    C = fgemm.matmul_mx(A, SA, B, SB, a_format=fa, b_format=fb, epilogue=epilogue, bias=bias)
    torch.cuda.synchronize()
    assert fgemm.default_handle().get_error() == fgemm.OK
    Av = oracle.mx_values(_np(A), _np(SA), fa, "row")
    Bv = oracle.mx_values(_np(B), _np(SB), fb, "col")
    bv = None if bias is None else values(bias)
    raw = oracle.gemm(Av, Bv)
    ref = oracle.epilogue(raw, epilogue, 1.0, bv)
    c = values(C)
    err = normwise(c, ref, "bf16")
    record(f"normwise MX {fa}/{fb} {epilogue}", err, TOL_NORMWISE["classical"])
    assert err <= TOL_NORMWISE["classical"]
    absdot = oracle.gemm(np.abs(Av), np.abs(Bv))
    if epilogue in ("none", "scale_bias"):
        ok, _ = elementwise_ok(c, ref, absdot, K, "bf16")
        assert ok
    else:
        _act_entries_ok(c, epilogue, raw, absdot, K, 1.0, bv, "bf16")


def test_mx_exact_ternary():
    """Elements in {-1, 0, 1} with unit scales: integer products, exact."""
    M, N, K = 256, 384, 520
    g = torch.Generator().manual_seed(104)
    pick = torch.tensor([0x00, 0x38, 0xB8], dtype=torch.uint8)     # 0, 1, -1 in E4M3
    A = pick[torch.randint(0, 3, (M, K), generator=g)].to(DEV)
    B = pick[torch.randint(0, 3, (K, N), generator=g)].to(DEV)
    SA = torch.full((M, (K + 31) // 32), 127, dtype=torch.uint8, device=DEV)
    SB = torch.full(((K + 31) // 32, N), 127, dtype=torch.uint8, device=DEV)
    C = fgemm.matmul_mx(A, SA, B, SB)
    ref = oracle.encode(oracle.gemm(oracle.fp8_decode(_np(A), "e4m3"), oracle.fp8_decode(_np(B), "e4m3")),
                        "bf16")
    assert np.array_equal(gpu_bits(C), ref)


# ------------------------------------------------------------ calibration

def test_calibrate_reduced_size_and_reload(tmp_path, monkeypatch):
    """fgemm_calibrate at 2048^3 on a handle of its own: every rate it
    measures is finite and positive, the JSON it writes reloads into a fresh
    handle (FGEMM_CALIB) as the same model, and AUTO's picks under it stay
    legal and compute the right product."""
    import json
    import math
    h = fgemm.Handle()
    path = tmp_path / "calib.json"
    h.calibrate(str(path), n=2048)
    m = h.device_model()
    effs = list(m.eff_classical) + list(m.eff_pair) + [x for row in m.eff_strassen for x in row] + \
        list(m.eff_strassen_pair) + list(m.eff_winograd)
    for e in effs:
        assert math.isfinite(e) and 0 < e < 2.0, effs
    assert 0.5 <= m.launch_us < 100 and 0.5 <= m.tile_fill_us < 200
    assert 1000 < m.hbm_gbs < 20000
    d = json.load(open(path))
    assert abs(d["eff_pair_256"] - m.eff_pair[1]) <= 1e-8 and abs(d["launch_us"] - m.launch_us) <= 1e-8
    monkeypatch.setenv("FGEMM_CALIB", str(path))
    h2 = fgemm.Handle()
    m2 = h2.device_model()
    assert abs(m2.eff_pair[1] - m.eff_pair[1]) <= 1e-8 and abs(m2.tile_fill_us - m.tile_fill_us) <= 1e-8
    for (M, N, K) in [(256, 256, 256), (4096, 4096, 1024), (16, 2048, 2048), (2048, 2048, 2048)]:
        algo, tm, tn, us = h2.plan(M, N, K)
        assert fgemm.validate(M, N, K, 16, K, 16, N, 16, N, fgemm.BF16, None, algo, tn, tm) == fgemm.OK
        assert math.isfinite(us) and us > 0
        A = inputs.matrix(M, K, "ternary", "bf16", 34, DEV)
        B = inputs.matrix(K, N, "ternary", "bf16", 35, DEV)
        C = fgemm.matmul(A, B, handle=h2)
        torch.cuda.synchronize()
        assert h2.get_error() == fgemm.OK
        assert torch.equal(C.float(), (A.float() @ B.float()).to(torch.bfloat16).float())
    monkeypatch.setenv("FGEMM_CALIB", str(tmp_path / "missing.json"))
    with pytest.raises(fgemm.FgemmError):
        fgemm.Handle()
    h.close()
    h2.close()


# ------------------------------------------- host buffers (fgemm_matmul_host)

def _host(t, pinned):
    h = t.cpu()
    return h.pin_memory() if pinned else h


@pytest.mark.parametrize("M,N,K,pinned", [
    (8192, 16384, 512, True),    # four row blocks of 2048, pipelined
    (4096, 16384, 256, True),    # two row blocks
    (300, 520, 100, False),      # one ragged block, K and N off the 8-element pitch, pageable
    (1, 1, 1, True),
])
def test_host_path_exact_ternary(M, N, K, pinned):
    """A, B, C and the bias in host memory: RNE(exact C) bit for bit."""
    A, B, bias = _ternary(M, N, K, "bf16", seed=90)
    hA, hB, hbias = _host(A, pinned), _host(B, pinned), _host(bias, pinned)
    C = fgemm.matmul(hA, hB, epilogue="scale_bias", bias=hbias)
    assert C.device.type == "cpu"
    assert np.array_equal(gpu_bits(C), _exact_reference(A, B, bias, "bf16"))


def test_host_path_strided_views_and_guard_band():
    """Host views with leading dimensions past the row (lda > K, ldb > N,
    ldc > N_out): the result lands in the view, the columns around it keep
    their values."""
    M, N, K = 4096, 16384, 136
    A, B, bias = _ternary(M, N, K, "bf16", seed=91)
    hA = torch.zeros(M, K + 40, dtype=torch.bfloat16).pin_memory()
    hA[:, 8:8 + K] = A.cpu()
    hB = torch.zeros(K, N + 24, dtype=torch.bfloat16).pin_memory()
    hB[:, :N] = B.cpu()
    hC = torch.full((M, N + 16), 7.0, dtype=torch.bfloat16).pin_memory()
    out = hC[:, 16:]
    fgemm.matmul(hA[:, 8:8 + K], hB[:, :N], out=out, epilogue="scale_bias", bias=bias.cpu())
    assert np.array_equal(gpu_bits(out), _exact_reference(A, B, bias, "bf16"))
    assert torch.all(hC[:, :16] == 7.0)


@pytest.mark.parametrize("algo,tile_m,epilogue", [("classical", 256, "swiglu"),
                                                  ("classical", 128, "silu"),
                                                  ("winograd1", 256, "none")])
def test_host_path_matches_the_device_path(algo, tile_m, epilogue, split_mode):
    """Uniform inputs: the host call's row blocks run the device path's kernel
    on the same rows; with the last-wave K split off every entry is summed in
    the same order, so C is the same bit for bit."""
    split_mode("off")
    M, N, K = 8192, 16384, 1024
    A = inputs.matrix(M, K, "uniform", "bf16", 92, DEV)
    B = inputs.matrix(K, N, "uniform", "bf16", 93, DEV)
    bias = inputs.matrix(1, N, "normal_0.02", "bf16", 94, DEV)[0] if epilogue != "none" else None
    kw = dict(epilogue=epilogue, algo=algo, tile_m=tile_m, tile_n=256)
    hC = fgemm.matmul(A.cpu().pin_memory(), B.cpu().pin_memory(),
                      bias=None if bias is None else bias.cpu(), **kw)
    # the device path on the same 2048-row blocks (the host call's blocks)
    Cd = torch.empty(M, hC.shape[1], dtype=torch.bfloat16, device=DEV)
    for i in range(0, M, 2048):
        fgemm.matmul(A[i:i + 2048], B, out=Cd[i:i + 2048], bias=bias, **kw)
    torch.cuda.synchronize()
    assert torch.equal(hC.view(torch.int16), Cd.cpu().view(torch.int16))


def test_host_path_rejects_bad_arguments():
    hA = torch.zeros(64, 64, dtype=torch.bfloat16)
    hB = torch.zeros(64, 64, dtype=torch.float16)
    with pytest.raises(fgemm.FgemmError):
        fgemm.matmul(hA, hB)
    with pytest.raises(fgemm.FgemmError):
        fgemm.matmul(hA, torch.zeros(32, 64, dtype=torch.bfloat16))
    with pytest.raises(fgemm.FgemmError):
        fgemm.matmul(hA, hA, out=torch.zeros(64, 32, dtype=torch.bfloat16))


def test_host_overlap_chained_calls_wait_for_their_inputs():
    """Non-blocking host calls whose input is an earlier call's output: the
    second call's upload waits for the first call's C to be on the host
    (ternary inputs keep C1 exact, so C2 = RNE(C1 B2) bit for bit)."""
    M, N, K = 8192, 2048, 64
    A, B, _ = _ternary(M, N, K, "bf16", seed=95)
    B2 = inputs.matrix(N, 512, "ternary", "bf16", 96, DEV)
    hA, hB, hB2 = A.cpu().pin_memory(), B.cpu().pin_memory(), B2.cpu().pin_memory()
    hC1 = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    hC2 = torch.empty(M, 512, dtype=torch.bfloat16).pin_memory()
    for _ in range(2):
        hC1.view(torch.int16).fill_(0x7F7B)
        fgemm.matmul(hA, hB, out=hC1, blocking=False)
        fgemm.matmul(hC1, hB2, out=hC2, blocking=False)
        torch.cuda.current_stream().synchronize()
        assert fgemm.default_handle().get_error() == fgemm.OK
        zero = torch.zeros(N, dtype=torch.bfloat16, device=DEV)
        assert np.array_equal(gpu_bits(hC1), _exact_reference(A, B, zero, "bf16"))
        C1 = hC1.to(DEV)
        assert np.array_equal(gpu_bits(hC2), _exact_reference(C1, B2, zero[:512], "bf16"))


@pytest.mark.parametrize("shapes", [
    [(4096, 16384, 256)] * 6,
    # shapes that change from call to call (the slots keep their places while
    # earlier calls still use them), and a larger one that makes them grow
    [(4096, 16384, 256), (8192, 2048, 64), (512, 4096, 1024), (4096, 16384, 256), (8192, 2048, 64),
     (8192, 16384, 512)],
], ids=["same", "mixed"])
def test_host_overlap_back_to_back_calls(shapes):
    """Six non-blocking host calls in a row over the handle's two slots of B,
    A blocks and C blocks (different inputs and outputs each): every C is the
    exact product."""
    calls = []
    for j, (M, N, K) in enumerate(shapes):
        A, B, bias = _ternary(M, N, K, "bf16", seed=100 + 3 * j)
        calls.append((A, B, bias, A.cpu().pin_memory(), B.cpu().pin_memory(), bias.cpu().pin_memory(),
                      torch.empty(M, N, dtype=torch.bfloat16).pin_memory()))
    for (_, _, _, hA, hB, hbias, hC) in calls:
        fgemm.matmul(hA, hB, out=hC, epilogue="scale_bias", bias=hbias, blocking=False)
    torch.cuda.current_stream().synchronize()
    assert fgemm.default_handle().get_error() == fgemm.OK
    for (A, B, bias, _, _, _, hC) in calls:
        assert np.array_equal(gpu_bits(hC), _exact_reference(A, B, bias, "bf16"))
