"""The Strassen entry point that allocates nothing (fgemm_strassen_matmul_static).

It is meant for callers that may not call cudaMalloc -- code under a framework
whose memory pool owns the device, serving loops that cannot afford
cudaMalloc's implicit synchronisation, plug-ins handed only buffers and a
stream.  Its scratch is an array built into the library, so this test checks
that two calls in a row (the second one finding the first one's leftovers in
that array) give what the handle-based entry point gives for the same
arguments, and that a product too large for the array is refused before
anything runs.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from complexity_matmul_tcgen05_gb300 import fgemm, inputs
from parity_util import TOL_EMULATED, values

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _static(A, B, C, depth, tile_n, epi=None):
    M, K = A.shape
    N = B.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return fgemm.lib().fgemm_strassen_matmul_static(
        M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(), C.stride(0),
        fgemm.BF16, ctypes.byref(epi) if epi is not None else None, depth, tile_n,
        ctypes.c_void_p(stream))


def _check_against_handle_path(A, B, depth, tile_n, epilogue="none", bias=None):
    N = B.shape[1]
    n_out = N // 2 if epilogue == "swiglu" else N
    C = torch.full((A.shape[0], n_out), float("nan"), dtype=torch.bfloat16, device=DEV)
    epi = fgemm.make_epilogue(epilogue, 1.0, None if bias is None else bias.data_ptr())
    status = _static(A, B, C, depth, tile_n, epi)
    assert status == fgemm.OK, fgemm.lib().fgemm_last_message(None).decode()
    torch.cuda.synchronize()
    ref = fgemm.matmul(A, B, epilogue=epilogue, bias=bias, algo=f"strassen{depth}", tile_n=tile_n)
    torch.cuda.synchronize()
    c, r = values(C), values(ref)
    assert np.isfinite(c).all()
    assert np.linalg.norm(c - r) <= TOL_EMULATED * np.linalg.norm(r)
    # same kernel, same launch shape: the results agree bit for bit
    assert torch.equal(C.view(torch.int16), ref.view(torch.int16))


def test_two_calls_in_a_row_match_the_handle_entry_point():
    M, N, K = 512, 1024, 768
    A1 = inputs.matrix(M, K, "uniform", "bf16", 50, DEV)
    B1 = inputs.matrix(K, N, "uniform", "bf16", 51, DEV)
    _check_against_handle_path(A1, B1, depth=1, tile_n=256)
    # second call: other inputs, depth 2, SwiGLU with bias, over the first
    # call's leftover partial tiles
    M2, N2, K2 = 512, 2048, 512
    A2 = inputs.matrix(M2, K2, "normal", "bf16", 52, DEV)
    B2 = inputs.matrix(K2, N2, "normal_inv_k", "bf16", 53, DEV, k=K2)
    bias = inputs.matrix(1, N2, "normal_0.02", "bf16", 54, DEV)[0]
    _check_against_handle_path(A2, B2, depth=2, tile_n=128, epilogue="swiglu", bias=bias)


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
