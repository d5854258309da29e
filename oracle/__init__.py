"""fp64 CPU oracle for fgemm -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product (the CUDA library
and its Python binding) never does.  The oracle shares no code with the GPU
path: its arithmetic lives in ``oracle.c`` (plain C, fp64), built here with
gcc into ``oracle/_build/liboracle.so``.

Every function follows the definition stated in ``oracle.c``'s header:
classical product (CS336 Lecture 05 notes, "Page 40. Trick 5: tiling"),
epilogue (PingPong GEMM / CODA note), Strassen and Winograd recursions
(FalconGEMM summary, "Methodology" items 1 and 4; textbook identities, since
the pages print none).  Arrays are numpy, row-major.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16, F64 = 0, 1, 2
EPI = {"none": 0, "scale_bias": 1, "silu": 2, "swiglu": 3}
DTYPES = {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no -ffast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_SO)
        i64, dp, u16p = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint16)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [ctypes.c_int, i64, u16p, dp]
        lib.oracle_encode.argtypes = [ctypes.c_int, i64, dp, u16p]
        lib.oracle_gemm_f64.argtypes = [i64, i64, i64, dp, i64, dp, i64, dp, i64]
        lib.oracle_gemm_sampled.argtypes = [ctypes.c_int, i64, u16p, i64, u16p, i64,
                                            i64, i64p, i64p, dp]
        lib.oracle_epilogue.argtypes = [ctypes.c_int, i64, i64, dp, i64, ctypes.c_double,
                                        dp, dp, i64]
        lib.oracle_strassen_f64.argtypes = [ctypes.c_int, i64, i64, i64, dp, i64, dp, i64, dp, i64]
        lib.oracle_strassen_f64.restype = ctypes.c_int
        lib.oracle_strassen_emulated.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, i64, dp,
                                                 i64, dp, i64, dp, i64]
        lib.oracle_strassen_emulated.restype = ctypes.c_int
        lib.oracle_winograd_f64.argtypes = [ctypes.c_int, i64, i64, i64, dp, i64, dp, i64, dp, i64]
        lib.oracle_winograd_f64.restype = ctypes.c_int
        lib.oracle_winograd_emulated.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, i64, dp,
                                                 i64, dp, i64, dp, i64]
        lib.oracle_winograd_emulated.restype = ctypes.c_int
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_fp8_decode.argtypes = [ctypes.c_int, i64, u8p, dp]
        lib.oracle_e8m0_decode.argtypes = [i64, u8p, dp]
        lib.oracle_mx_values.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, u8p, i64, u8p, i64, dp]
        lib.oracle_rmsnorm.argtypes = [i64, i64, dp, i64, dp, ctypes.c_double, dp, i64]
        lib.oracle_block_sumsq.argtypes = [i64, i64, dp, i64, dp]
        lib.oracle_row_scale.argtypes = [i64, i64, dp, ctypes.c_double, ctypes.c_double, dp]
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_silu.restype = ctypes.c_double
        _lib = lib
        return lib


def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return DTYPES[str(dtype).replace("torch.", "")]


def _f64(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def decode(bits: np.ndarray, dtype) -> np.ndarray:
    """Exact value of every 16-bit pattern (uint16 array) as float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode(_dtype_code(dtype), b.size, _ptr(b, ctypes.c_uint16),
                          _ptr(out, ctypes.c_double))
    return out


def encode(x: np.ndarray, dtype) -> np.ndarray:
    """Round float64 values to the 16-bit type (RNE); returns uint16 bits."""
    v = _f64(x)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_encode(_dtype_code(dtype), v.size, _ptr(v, ctypes.c_double),
                          _ptr(out, ctypes.c_uint16))
    return out


def round_to(x: np.ndarray, dtype) -> np.ndarray:
    """RNE to the 16-bit type, returned as float64 values."""
    return decode(encode(x, dtype), dtype)


def gemm(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """Classical fp64 product A @ B by a plain triple loop."""
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    C = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_f64(M, N, K, _ptr(A, ctypes.c_double), K,
                            _ptr(B, ctypes.c_double), N, _ptr(C, ctypes.c_double), N)
    return C


def gemm_sampled(A_bits: np.ndarray, B_bits: np.ndarray, dtype, rows, cols) -> np.ndarray:
    """Raw products sum_k A[r,k] B[k,c] (fp64) at the given (row, col) pairs.

    A_bits (M x K) and B_bits (K x N) are uint16 arrays holding the inputs'
    16-bit patterns; they are decoded on the fly.
    """
    A = np.ascontiguousarray(A_bits, dtype=np.uint16)
    B = np.ascontiguousarray(B_bits, dtype=np.uint16)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    assert r.shape == c.shape
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    assert r.size == 0 or (r.min() >= 0 and r.max() < M and c.min() >= 0 and c.max() < N)
    out = np.empty(r.shape, dtype=np.float64)
    _load().oracle_gemm_sampled(_dtype_code(dtype), K, _ptr(A, ctypes.c_uint16), K,
                                _ptr(B, ctypes.c_uint16), N, r.size,
                                _ptr(r, ctypes.c_int64), _ptr(c, ctypes.c_int64),
                                _ptr(out, ctypes.c_double))
    return out


def epilogue(acc: np.ndarray, kind: str = "none", alpha: float = 1.0,
             bias: np.ndarray | None = None) -> np.ndarray:
    """alpha * acc + bias, then the activation (SwiGLU halves the width)."""
    acc = _f64(acc)
    M, N = acc.shape
    k = EPI[kind]
    Nout = N // 2 if k == EPI["swiglu"] else N
    out = np.empty((M, Nout), dtype=np.float64)
    b = None if bias is None else _f64(bias)
    if b is not None:
        assert b.shape == (N,)
    _load().oracle_epilogue(k, M, N, _ptr(acc, ctypes.c_double), N, float(alpha),
                            None if b is None else _ptr(b, ctypes.c_double),
                            _ptr(out, ctypes.c_double), Nout)
    return out


FP8 = {"e4m3": 0, "e5m2": 1}


def fp8_decode(bits: np.ndarray, fmt: str) -> np.ndarray:
    """Exact value of every 8-bit float pattern (uint8 array) as float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_fp8_decode(FP8[fmt], b.size, _ptr(b, ctypes.c_uint8), _ptr(out, ctypes.c_double))
    return out


def e8m0_decode(bits: np.ndarray) -> np.ndarray:
    """2^(e - 127) for every E8M0 pattern (255: NaN)."""
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_e8m0_decode(b.size, _ptr(b, ctypes.c_uint8), _ptr(out, ctypes.c_double))
    return out


def mx_values(X: np.ndarray, S: np.ndarray, fmt: str, along: str) -> np.ndarray:
    """Values of a block-scaled matrix: X (rows x cols, uint8 8-bit floats)
    times the E8M0 scale of its block of 32.  along="row": S is rows x
    ceil(cols/32); along="col": S is ceil(rows/32) x cols."""
    X = np.ascontiguousarray(X, dtype=np.uint8)
    S = np.ascontiguousarray(S, dtype=np.uint8)
    rows, cols = X.shape
    out = np.empty((rows, cols), dtype=np.float64)
    _load().oracle_mx_values(FP8[fmt], 0 if along == "row" else 1, rows, cols,
                             _ptr(X, ctypes.c_uint8), cols, _ptr(S, ctypes.c_uint8), S.shape[1],
                             _ptr(out, ctypes.c_double))
    return out


def rmsnorm(x: np.ndarray, g: np.ndarray | None = None, eps: float = 1e-6) -> np.ndarray:
    """RMSNorm of every row: x_ij * g_j / sqrt(mean_j x_ij^2 + eps)."""
    x = _f64(x)
    M, N = x.shape
    y = np.empty((M, N), dtype=np.float64)
    gg = None if g is None else _f64(g)
    if gg is not None:
        assert gg.shape == (N,)
    _load().oracle_rmsnorm(M, N, _ptr(x, ctypes.c_double), N,
                           None if gg is None else _ptr(gg, ctypes.c_double), float(eps),
                           _ptr(y, ctypes.c_double), N)
    return y


def block_sumsq(x: np.ndarray) -> np.ndarray:
    """[ceil(N/64), M]: per row, the sum of squares of each block of 64 columns."""
    x = _f64(x)
    M, N = x.shape
    out = np.empty(((N + 63) // 64, M), dtype=np.float64)
    _load().oracle_block_sumsq(M, N, _ptr(x, ctypes.c_double), N, _ptr(out, ctypes.c_double))
    return out


def row_scale(sumsq: np.ndarray, n: int, eps: float) -> np.ndarray:
    """r_i = 1 / sqrt(sum_p sumsq[p, i] / n + eps) for a [parts, M] array."""
    s = _f64(sumsq)
    parts, M = s.shape
    r = np.empty(M, dtype=np.float64)
    _load().oracle_row_scale(M, parts, _ptr(s, ctypes.c_double), float(n), float(eps),
                             _ptr(r, ctypes.c_double))
    return r


def silu(v: float) -> float:
    return float(_load().oracle_silu(float(v)))


def strassen(A: np.ndarray, B: np.ndarray, depth: int) -> np.ndarray:
    """Recursive Strassen in fp64 (depth levels, classical leaves)."""
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    _, N = B.shape
    C = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_strassen_f64(depth, M, N, K, _ptr(A, ctypes.c_double), K,
                                     _ptr(B, ctypes.c_double), N,
                                     _ptr(C, ctypes.c_double), N)
    if rc != 0:
        raise ValueError("Strassen needs M, N, K divisible by 2**depth")
    return C


def strassen_emulated(A: np.ndarray, B: np.ndarray, depth: int, dtype) -> np.ndarray:
    """Strassen with every leaf operand rounded to fp32 then to ``dtype``.

    ``dtype`` may be "f16", "bf16" or "f64" (no rounding at all).
    """
    code = F64 if str(dtype) in ("f64", "float64") else _dtype_code(dtype)
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    _, N = B.shape
    C = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_strassen_emulated(depth, code, M, N, K, _ptr(A, ctypes.c_double), K,
                                          _ptr(B, ctypes.c_double), N,
                                          _ptr(C, ctypes.c_double), N)
    if rc != 0:
        raise ValueError("Strassen needs M, N, K divisible by 2**depth")
    return C


def winograd(A: np.ndarray, B: np.ndarray, depth: int) -> np.ndarray:
    """Recursive Winograd variant of Strassen in fp64 (depth levels)."""
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    _, N = B.shape
    C = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_winograd_f64(depth, M, N, K, _ptr(A, ctypes.c_double), K,
                                     _ptr(B, ctypes.c_double), N,
                                     _ptr(C, ctypes.c_double), N)
    if rc != 0:
        raise ValueError("Winograd needs M, N, K divisible by 2**depth")
    return C


def winograd_emulated(A: np.ndarray, B: np.ndarray, depth: int, dtype) -> np.ndarray:
    """Winograd variant with every leaf operand rounded (fp32, then ``dtype``)
    once from the exact signed sum of source blocks it stands for."""
    code = F64 if str(dtype) in ("f64", "float64") else _dtype_code(dtype)
    A, B = _f64(A), _f64(B)
    M, K = A.shape
    _, N = B.shape
    C = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_winograd_emulated(depth, code, M, N, K, _ptr(A, ctypes.c_double), K,
                                          _ptr(B, ctypes.c_double), N,
                                          _ptr(C, ctypes.c_double), N)
    if rc != 0:
        raise ValueError("Winograd needs M, N, K divisible by 2**depth")
    return C


def reference(A_bits: np.ndarray, B_bits: np.ndarray, dtype, kind: str = "none",
              alpha: float = 1.0, bias_bits: np.ndarray | None = None) -> np.ndarray:
    """Full fp64 reference epi(alpha * A @ B + bias) for 16-bit inputs."""
    A = decode(A_bits, dtype)
    B = decode(B_bits, dtype)
    bias = None if bias_bits is None else decode(bias_bits, dtype)
    return epilogue(gemm(A, B), kind, alpha, bias)


def reference_sampled(A_bits: np.ndarray, B_bits: np.ndarray, dtype, rows, cols,
                      kind: str = "none", alpha: float = 1.0,
                      bias_bits: np.ndarray | None = None) -> np.ndarray:
    """epi(alpha * A @ B + bias) at sampled output positions (row, col).

    For SwiGLU, col indexes the M x N/2 output and two dot products are
    taken per entry (gate column col, up column col + N/2).  The samples are
    laid out as the columns of a one-row accumulator, so that the epilogue
    sees each sample's own bias entry.
    """
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    N = B_bits.shape[1]
    bias = None if bias_bits is None else decode(bias_bits, dtype)
    if kind == "swiglu":
        half = N // 2
        g = gemm_sampled(A_bits, B_bits, dtype, rows, cols)
        u = gemm_sampled(A_bits, B_bits, dtype, rows, cols + half)
        acc = np.concatenate([g, u]).reshape(1, -1)
        b = None if bias is None else np.concatenate([bias[cols], bias[cols + half]])
        return epilogue(acc, "swiglu", alpha, b)[0]
    raw = gemm_sampled(A_bits, B_bits, dtype, rows, cols)
    b = None if bias is None else bias[cols]
    return epilogue(raw.reshape(1, -1), kind, alpha, b)[0]
