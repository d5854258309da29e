"""Randomised exact parity: seeded random legal shapes over every form, tile,
split and formation mode, bit for bit against the oracle.

Ternary inputs (entries in {-1, 0, 1}, bias in a small integer range) keep
every operand sum, product and fold exact in fp32 at these sizes, so each
form's C must equal RNE(exact C) in every entry whatever its schedule.  The
fixed cases elsewhere pin the known edges; this sweep looks for the
combinations nobody listed (short K with several tiles per pair, ragged
edges with splits, formation modes on small grids, ...).
"""
import random

import numpy as np
import pytest
import torch

import oracle
from complexity_matmul_tcgen05_gb300 import fgemm, inputs
from parity_util import gpu_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(rng):
    """One random legal (form, tile, shape, options) case."""
    kind = rng.choice(["pair", "pair", "cta", "small_m", "lcma_pair", "lcma_pair", "lcma_cta", "strassen2"])
    dtype = rng.choice(["bf16", "f16"])
    epi = rng.choice(["scale_bias", "scale_bias", "none"])
    split = rng.choice(["auto", "off", "force"])
    formation = rng.choice(["auto", "prepass", "in_kernel"])
    if kind == "pair":
        tm, tn, algo = 256, rng.choice([128, 256]), "classical"
        M = rng.choice([rng.randrange(1, 4097), 256 * rng.randrange(1, 17)])
        N = rng.choice([rng.randrange(8, 2049, 8), tn * rng.randrange(1, 9)])
        K = rng.choice([8 * rng.randrange(1, 25), 64 * rng.randrange(1, 9), 8 * rng.randrange(1, 129)])
    elif kind == "cta":
        tm, tn, algo = 128, rng.choice([64, 128, 256]), "classical"
        M = rng.randrange(1, 3000)
        N = rng.randrange(8, 3000, 8)
        K = 8 * rng.choice([rng.randrange(1, 25), rng.randrange(1, 129)])
    elif kind == "small_m":
        tm, tn, algo = rng.choice([16, 32, 64]), 128, "classical"
        M = rng.randrange(1, tm + 1)
        N = rng.randrange(8, 6000, 8)
        K = 8 * rng.choice([rng.randrange(1, 38), rng.randrange(1, 500)])
        epi = rng.choice(["scale_bias", "none"])
    elif kind == "lcma_pair":
        tm, tn, algo = 256, rng.choice([128, 256]), rng.choice(["strassen1", "winograd1"])
        M = 512 * rng.randrange(1, 5)
        N = 2 * tn * rng.randrange(1, 9)
        K = 128 * rng.randrange(1, 9)
    elif kind == "lcma_cta":
        tm, tn, algo = 128, rng.choice([128, 256]), rng.choice(["strassen1", "winograd1"])
        M = 256 * rng.randrange(1, 9)
        N = 2 * tn * rng.randrange(1, 5)
        K = 128 * rng.randrange(1, 9)
    else:  # two Strassen levels on one-CTA tiles
        tm, tn, algo = 128, rng.choice([128, 256]), "strassen2"
        M = 512 * rng.randrange(1, 4)
        N = 4 * tn * rng.randrange(1, 3)
        K = 256 * rng.randrange(1, 4)
    return dict(kind=kind, algo=algo, tile_m=tm, tile_n=tn, M=M, N=N, K=K, dtype=dtype, epi=epi,
                split=split, formation=formation)


def _many_case(rng):
    """Many tiles (or output positions) per pair with a short K: launches whose
    roles run far apart (the producer done long before the epilogue)."""
    dtype = rng.choice(["bf16", "f16"])
    split = rng.choice(["auto", "off", "force"])
    formation = rng.choice(["auto", "prepass", "in_kernel"])
    if rng.random() < 0.5:
        tn = rng.choice([128, 256])
        return dict(kind="pair_many", algo="classical", tile_m=256, tile_n=tn, M=rng.randrange(4096, 16385),
                    N=tn * rng.randrange(8, 33), K=8 * rng.randrange(1, 33), dtype=dtype,
                    epi=rng.choice(["scale_bias", "none"]), split=split, formation=formation)
    tn = rng.choice([128, 256])
    return dict(kind="lcma_many", algo=rng.choice(["strassen1", "winograd1"]), tile_m=256, tile_n=tn,
                M=512 * rng.randrange(8, 17), N=2 * tn * rng.randrange(8, 17), K=128 * rng.randrange(1, 5),
                dtype=dtype, epi=rng.choice(["scale_bias", "none"]), split=split, formation=formation)


def _strassen2_pair_case(rng):
    """Two Strassen levels on CTA pairs (the operands from the pre-pass)."""
    tn = rng.choice([128, 256])
    return dict(kind="strassen2_pair", algo="strassen2", tile_m=256, tile_n=tn, M=1024 * rng.randrange(1, 4),
                N=4 * tn * rng.randrange(1, 4), K=256 * rng.randrange(1, 4), dtype=rng.choice(["bf16", "f16"]),
                epi=rng.choice(["scale_bias", "none"]), split=rng.choice(["auto", "off", "force"]),
                formation=rng.choice(["auto", "prepass", "in_kernel"]))


_RNG = random.Random(20260603)
_RNG2 = random.Random(20261203)
CASES = [_case(_RNG) for _ in range(192)] + [_many_case(_RNG) for _ in range(32)] + \
    [_strassen2_pair_case(_RNG2) for _ in range(24)]


def _id(c):
    return f"{c['algo']}-{c['tile_m']}x{c['tile_n']}-{c['M']}x{c['N']}x{c['K']}-{c['dtype']}-{c['epi']}-" \
           f"split_{c['split']}-form_{c['formation']}"


@pytest.fixture
def handle_modes():
    h = fgemm.default_handle()
    yield h
    h.set_split_mode("auto")
    h.set_lcma_formation("auto")


@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_random_exact_ternary(case, handle_modes):
    c = case
    h = handle_modes
    h.set_split_mode(c["split"])
    h.set_lcma_formation(c["formation"])
    M, N, K, dtype = c["M"], c["N"], c["K"], c["dtype"]
    seed = (M * 131 + N * 17 + K) % 100000
    A = inputs.matrix(M, K, "ternary", dtype, seed, DEV)
    B = inputs.matrix(K, N, "ternary", dtype, seed + 1, DEV)
    bias = inputs.matrix(1, N, "ternary_bias", dtype, seed + 2, DEV)[0] if c["epi"] == "scale_bias" else None
    assert fgemm.validate(M, N, K, 16, K, 16, N, 16, N, fgemm.BF16 if dtype == "bf16" else fgemm.F16,
                          None, c["algo"], c["tile_n"], c["tile_m"]) == fgemm.OK, _id(c)
    ref = oracle.encode(oracle.reference(gpu_bits(A), gpu_bits(B), dtype,
                                         "scale_bias" if bias is not None else "none", 1.0,
                                         gpu_bits(bias) if bias is not None else None), dtype)
    for _ in range(2):  # two launches: also the same bits twice
        C = fgemm.matmul(A, B, epilogue=c["epi"], bias=bias, algo=c["algo"], tile_n=c["tile_n"],
                         tile_m=c["tile_m"])
        torch.cuda.synchronize()
        assert h.get_error() == fgemm.OK, h.last_message()
        bad = gpu_bits(C) != ref
        assert not bad.any(), f"{_id(c)}: {int(bad.sum())} entries differ, first at {np.argwhere(bad)[0]}"


def _host_case(rng):
    M = rng.choice([rng.randrange(1, 3000), 512 * rng.randrange(1, 17)])
    N = rng.choice([rng.randrange(1, 3000), 2048 * rng.randrange(1, 9)])
    K = rng.randrange(1, 700)
    return dict(M=M, N=N, K=K, dtype=rng.choice(["bf16", "f16"]), bias=rng.random() < 0.6,
                pinned=rng.random() < 0.8, blocking=rng.random() < 0.5,
                lda_pad=rng.choice([0, 0, 8, 13]), ldc_pad=rng.choice([0, 0, 5]))


_HRNG = random.Random(20260604)
HOST_CASES = [_host_case(_HRNG) for _ in range(24)]


@pytest.mark.parametrize("case", HOST_CASES,
                         ids=[f"{c['M']}x{c['N']}x{c['K']}-{c['dtype']}-bias{int(c['bias'])}-pin{int(c['pinned'])}-"
                              f"blk{int(c['blocking'])}-pad{c['lda_pad']}_{c['ldc_pad']}" for c in HOST_CASES])
def test_random_host_calls_exact_ternary(case):
    """Host buffers (any leading dimensions, pinned or not, blocking or not):
    RNE(exact C) bit for bit, two calls in a row into the same output."""
    c = case
    M, N, K, dtype = c["M"], c["N"], c["K"], c["dtype"]
    seed = (M * 7 + N * 3 + K) % 100000 + 500
    A = inputs.matrix(M, K, "ternary", dtype, seed, DEV)
    B = inputs.matrix(K, N, "ternary", dtype, seed + 1, DEV)
    bias = inputs.matrix(1, N, "ternary_bias", dtype, seed + 2, DEV)[0] if c["bias"] else None
    ref = oracle.encode(oracle.reference(gpu_bits(A), gpu_bits(B), dtype,
                                         "scale_bias" if bias is not None else "none", 1.0,
                                         gpu_bits(bias) if bias is not None else None), dtype)
    td = A.dtype
    hA = torch.zeros(M, K + c["lda_pad"], dtype=td)
    hA[:, :K] = A.cpu()
    hB = B.cpu().contiguous()
    hC = torch.full((M, N + c["ldc_pad"]), 3.0, dtype=td)
    if c["pinned"]:
        hA, hB, hC = hA.pin_memory(), hB.pin_memory(), hC.pin_memory()
    hbias = None if bias is None else bias.cpu().contiguous()
    out = hC[:, :N]
    for _ in range(2):
        fgemm.matmul(hA[:, :K], hB, out=out, epilogue="scale_bias" if bias is not None else "none",
                     bias=hbias, blocking=c["blocking"])
    torch.cuda.current_stream().synchronize()
    assert fgemm.default_handle().get_error() == fgemm.OK
    bad = gpu_bits(out) != ref
    assert not bad.any(), f"{int(bad.sum())} entries differ, first at {np.argwhere(bad)[0]}"
    if c["ldc_pad"]:
        assert torch.all(hC[:, N:] == 3.0)
