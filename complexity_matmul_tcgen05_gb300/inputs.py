"""Seeded synthetic inputs for fgemm.

This module draws random 16-bit matrices and nothing else: it holds none of
the GEMM arithmetic, so both the GPU path's tests and the CPU oracle can take
their inputs from it.  Values are drawn in fp32 with a seeded torch generator
and rounded once to the 16-bit type (torch's round-to-nearest-even cast).

Workloads (dense GEMMs shaped like LLM projection / FFN layers):

  square_256_f16        M=N=K=256, fp16, A,B ~ U[-1,1]
  proj_4096_bf16_bias   M=N=K=4096, bf16, A ~ N(0,1), B ~ N(0,1/K),
                        per-column bias ~ N(0, 0.02^2), alpha = 1
  ffn_up_swiglu_bf16    M=8192, N=28672 (gate | up, 2 x 14336), K=4096, bf16,
                        A ~ N(0,1), B ~ N(0,1/K), SwiGLU output M x 14336
  square_8192_bf16      M=N=K=8192, bf16, A,B ~ U[-1,1]
  square_16384_bf16     M=N=K=16384, bf16, A,B ~ U[-1,1]
  square_20480_bf16     M=N=K=20480, bf16, A,B ~ U[-1,1]
  square_24576_bf16     M=N=K=24576, bf16, A,B ~ U[-1,1]
  sweep                 bf16, M in {16,128,1024,8192} x N=K in
                        {2048,4096,8192,16384}, plus M=65536, N=K=1024;
                        A,B ~ N(0,1) / sqrt(K)
"""
from __future__ import annotations

import math

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}

WORKLOADS = {
    "square_256_f16": dict(M=256, N=256, K=256, dtype="f16", a="uniform", b="uniform",
                           epi="none", bias=None, algos=("classical", "strassen1")),
    "proj_4096_bf16_bias": dict(M=4096, N=4096, K=4096, dtype="bf16", a="normal",
                                b="normal_inv_k", epi="scale_bias", bias="normal_0.02",
                                algos=("classical", "auto")),
    "ffn_up_swiglu_bf16": dict(M=8192, N=28672, K=4096, dtype="bf16", a="normal",
                               b="normal_inv_k", epi="swiglu", bias=None,
                               algos=("classical", "strassen1", "auto")),
    "square_8192_bf16": dict(M=8192, N=8192, K=8192, dtype="bf16", a="uniform",
                             b="uniform", epi="none", bias=None,
                             algos=("classical", "strassen1", "winograd1", "auto")),
    "square_16384_bf16": dict(M=16384, N=16384, K=16384, dtype="bf16", a="uniform",
                              b="uniform", epi="none", bias=None,
                              algos=("classical", "strassen1", "strassen2", "winograd1", "auto")),
    "square_20480_bf16": dict(M=20480, N=20480, K=20480, dtype="bf16", a="uniform",
                              b="uniform", epi="none", bias=None,
                              algos=("classical", "strassen1", "winograd1", "auto")),
    "square_24576_bf16": dict(M=24576, N=24576, K=24576, dtype="bf16", a="uniform",
                              b="uniform", epi="none", bias=None,
                              algos=("classical", "strassen1", "winograd1", "auto")),
}

SWEEP_SHAPES = [(m, nk, nk) for m in (16, 128, 1024, 8192)
                for nk in (2048, 4096, 8192, 16384)] + [(65536, 1024, 1024)]

SEED_A, SEED_B, SEED_BIAS, SEED_SAMPLER = 0, 1, 2, 3


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def matrix(rows: int, cols: int, dist: str, dtype: str, seed: int, device="cpu",
           k: int | None = None) -> torch.Tensor:
    """A rows x cols 16-bit matrix drawn from ``dist`` with ``seed``.

    dist: "uniform" (U[-1,1]), "normal" (N(0,1)), "normal_inv_k" (N(0,1/k)),
    "normal_scaled" (N(0,1)/sqrt(k)), "normal_0.02" (N(0, 0.02^2)),
    "ternary" ({-1,0,1} uniformly), "ternary_bias" ({-2..2} uniformly).
    """
    g = _gen(seed, device)
    shape = (rows, cols)
    if dist == "uniform":
        x = torch.rand(shape, generator=g, device=device, dtype=torch.float32) * 2 - 1
    elif dist == "normal":
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    elif dist in ("normal_inv_k", "normal_scaled"):
        assert k is not None and k > 0
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) / math.sqrt(k)
    elif dist == "normal_0.02":
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 0.02
    elif dist == "ternary":
        x = torch.randint(-1, 2, shape, generator=g, device=device).to(torch.float32)
    elif dist == "ternary_bias":
        x = torch.randint(-2, 3, shape, generator=g, device=device).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(DTYPES[dtype])


def workload_inputs(name: str, device="cpu", M=None, N=None, K=None):
    """(A, B, bias or None) for a named workload (sizes may be overridden)."""
    w = WORKLOADS[name]
    M = w["M"] if M is None else M
    N = w["N"] if N is None else N
    K = w["K"] if K is None else K
    A = matrix(M, K, w["a"], w["dtype"], SEED_A, device, k=K)
    B = matrix(K, N, w["b"], w["dtype"], SEED_B, device, k=K)
    bias = None
    if w["bias"] is not None:
        bias = matrix(1, N, w["bias"], w["dtype"], SEED_BIAS, device, k=K)[0]
    return A, B, bias


def sweep_inputs(M: int, N: int, K: int, device="cpu"):
    A = matrix(M, K, "normal_scaled", "bf16", SEED_A, device, k=K)
    B = matrix(K, N, "normal_scaled", "bf16", SEED_B, device, k=K)
    return A, B


def sample_positions(M: int, Nout: int, n: int = 4096, seed: int = SEED_SAMPLER,
                     row_blocks: int = 1, col_blocks: int = 1, tile_m: int = 128,
                     tile_n: int = 256):
    """Stratified output positions: equal counts per (row block, col block)
    of the output (the quadrants of a Strassen split), plus the four corners
    and rows/cols on tile boundaries.  Returns (rows, cols) int64 tensors."""
    g = _gen(seed, "cpu")
    rows, cols = [], []
    nb = row_blocks * col_blocks
    per = max(1, n // nb)
    bm, bn = M // row_blocks, Nout // col_blocks
    for rb in range(row_blocks):
        for cb in range(col_blocks):
            r0, c0 = rb * bm, cb * bn
            rh = M - r0 if rb == row_blocks - 1 else bm
            ch = Nout - c0 if cb == col_blocks - 1 else bn
            rows.append(torch.randint(0, rh, (per,), generator=g) + r0)
            cols.append(torch.randint(0, ch, (per,), generator=g) + c0)
    fixed_r = [0, 0, M - 1, M - 1]
    fixed_c = [0, Nout - 1, 0, Nout - 1]
    for t in range(1, 5):  # tile-boundary rows and columns
        r = min(M - 1, t * tile_m - 1)
        c = min(Nout - 1, t * tile_n - 1)
        fixed_r += [r, min(M - 1, r + 1)]
        fixed_c += [c, min(Nout - 1, c + 1)]
    rows.append(torch.tensor(fixed_r, dtype=torch.int64))
    cols.append(torch.tensor(fixed_c, dtype=torch.int64))
    return torch.cat(rows), torch.cat(cols)


def bits(t: torch.Tensor):
    """The 16-bit patterns of a CPU fp16/bf16 tensor as a numpy uint16 array."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
