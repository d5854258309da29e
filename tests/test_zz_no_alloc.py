"""The Strassen entry point that allocates nothing (fgemm_strassen_matmul_static).

It is meant for callers that may not call cudaMalloc -- code under a framework
whose memory pool owns the device, serving loops that cannot afford
cudaMalloc's implicit synchronisation, plug-ins handed only buffers and a
stream.  Its scratch is an array built into the library, so these tests check
that consecutive calls (each finding the previous call's leftovers in that
array) give what the handle-based entry point gives for the same arguments
and tile, that each result matches the oracle's emulated Strassen, that a
product too large for the array is refused before anything runs, and that a
timeout inside its kernel is reported by fgemm_strassen_static_get_error.
The file is named so that pytest collects it last.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from complexity_matmul_tcgen05_gb300 import fgemm, inputs
from parity_util import TOL_EMULATED, TOL_NORMWISE, gpu_bits, normwise, record, values

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _static(A, B, C, depth, tile_n, epi=None):
    M, K = A.shape
    N = B.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    dt = fgemm.BF16 if A.dtype == torch.bfloat16 else fgemm.F16
    return fgemm.lib().fgemm_strassen_matmul_static(
        M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(), C.stride(0),
        dt, ctypes.byref(epi) if epi is not None else None, depth, tile_n,
        ctypes.c_void_p(stream))


def _static_error():
    return fgemm.lib().fgemm_strassen_static_get_error(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check(A, B, depth, tile_n, epilogue="none", bias=None, alpha=1.0):
    """One call of the static entry point against (1) the handle entry point
    with the same form and tile (128-row tiles: the same kernel and grid, so
    the same bits), and (2) the oracle: the emulated (rounded-operand)
    Strassen through the same epilogue within 1e-4, and the exact product
    within the form's budget (the pre-activation budget times the
    activation's condition number for SwiGLU)."""
    dtype = "bf16" if A.dtype == torch.bfloat16 else "f16"
    N = B.shape[1]
    n_out = N // 2 if epilogue == "swiglu" else N
    C = torch.full((A.shape[0], n_out), float("nan"), dtype=A.dtype, device=DEV)
    epi = fgemm.make_epilogue(epilogue, alpha, None if bias is None else bias.data_ptr())
    status = _static(A, B, C, depth, tile_n, epi)
    assert status == fgemm.OK, fgemm.lib().fgemm_last_message(None).decode()
    assert _static_error() == fgemm.OK
    ref = fgemm.matmul(A, B, epilogue=epilogue, bias=bias, alpha=alpha, algo=f"strassen{depth}",
                       tile_n=tile_n, tile_m=128)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    c = values(C)
    assert np.isfinite(c).all()
    Av, Bv = values(A), values(B)
    bv = None if bias is None else values(bias)
    emu = oracle.epilogue(oracle.strassen_emulated(Av, Bv, depth, dtype), epilogue, alpha, bv)
    e2 = float(np.linalg.norm(c - oracle.round_to(emu, dtype)) / np.linalg.norm(emu))
    record(f"static depth {depth} tile {tile_n} vs emulated", e2, TOL_EMULATED)
    assert e2 <= TOL_EMULATED, e2
    exact = oracle.epilogue(oracle.gemm(Av, Bv), epilogue, alpha, bv)
    err = normwise(c, exact, dtype)
    tol = TOL_NORMWISE[f"strassen{depth}"]
    if epilogue in ("silu", "swiglu"):
        from parity_util import activation_condition
        tol *= max(1.0, activation_condition(oracle.gemm(Av, Bv), epilogue, alpha, bv))
    record(f"static depth {depth} tile {tile_n} normwise", err, tol)
    assert err <= tol, err


@pytest.mark.parametrize("depth,tile_n", [(1, 128), (1, 256), (2, 128), (2, 256)])
def test_matches_the_handle_path_and_the_oracle(depth, tile_n):
    M, N, K = 512, 1024, 768 if depth == 1 else 512
    A = inputs.matrix(M, K, "uniform", "bf16", 50 + depth, DEV)
    B = inputs.matrix(K, N, "uniform", "bf16", 60 + tile_n, DEV)
    _check(A, B, depth, tile_n)


def test_three_calls_in_a_row_over_leftover_scratch():
    # depth 1 at tile 256, then depth 2 (SwiGLU with bias) over its leftover
    # partial tiles, then depth 1 at tile 128 in fp16 with alpha and bias:
    # a smaller slice of the larger stale layout the depth-2 call left
    A1 = inputs.matrix(512, 768, "uniform", "bf16", 50, DEV)
    B1 = inputs.matrix(768, 1024, "uniform", "bf16", 51, DEV)
    _check(A1, B1, depth=1, tile_n=256)
    A2 = inputs.matrix(512, 512, "normal", "bf16", 52, DEV)
    B2 = inputs.matrix(512, 2048, "normal_inv_k", "bf16", 53, DEV, k=512)
    bias2 = inputs.matrix(1, 2048, "normal_0.02", "bf16", 54, DEV)[0]
    _check(A2, B2, depth=2, tile_n=128, epilogue="swiglu", bias=bias2)
    A3 = inputs.matrix(768, 512, "uniform", "f16", 55, DEV)
    B3 = inputs.matrix(512, 1280, "uniform", "f16", 56, DEV)
    bias3 = inputs.matrix(1, 1280, "normal_0.02", "f16", 57, DEV)[0]
    _check(A3, B3, depth=1, tile_n=128, epilogue="scale_bias", bias=bias3, alpha=0.75)


def test_too_large_for_the_static_scratch_is_refused():
    # depth 2 at 8192^3: 256 tiles -> 152 CTAs x 1 MiB of partial tiles > 64 MiB
    L = fgemm.lib()
    s = L.fgemm_strassen_matmul_static(8192, 8192, 8192, 256, 8192, 256, 8192, 256, 8192,
                                       fgemm.BF16, None, 2, 128, None)
    assert s == fgemm.ERR_UNSUPPORTED
    assert "static scratch" in L.fgemm_last_message(None).decode()
    s = L.fgemm_strassen_matmul_static(256, 256, 128, 256, 128, 256, 256, 256, 256,
                                       fgemm.BF16, None, 3, 128, None)
    assert s == fgemm.ERR_INVALID_ARG


def test_a_timeout_is_reported_then_cleared():
    """A bounded wait that runs out latches a code in the static error word;
    the query returns FGEMM_ERR_TIMEOUT once (naming the role), clears it, and
    the next product is exact."""
    L = fgemm.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert _static_error() == fgemm.OK
    t0 = time.perf_counter()
    assert L.fgemm_strassen_static_selftest_timeout(50, stream) == fgemm.OK
    assert _static_error() == fgemm.ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.045
    assert "producer" in L.fgemm_last_message(None).decode()
    assert _static_error() == fgemm.OK
    A = inputs.matrix(256, 128, "ternary", "bf16", 58, DEV)
    B = inputs.matrix(128, 256, "ternary", "bf16", 59, DEV)
    C = torch.empty((256, 256), dtype=torch.bfloat16, device=DEV)
    assert _static(A, B, C, 1, 128) == fgemm.OK
    assert _static_error() == fgemm.OK
    ref = oracle.encode(oracle.gemm(values(A), values(B)), "bf16")
    assert np.array_equal(gpu_bits(C), ref)
