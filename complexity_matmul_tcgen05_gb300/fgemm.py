"""Python binding of the fgemm C ABI (include/fgemm.h).

Argument marshalling only: every step of the product runs in the CUDA
library ``_build/libfgemm.so``.  If that library is missing, every call
raises -- there is no fallback of any kind.

``matmul`` takes torch CUDA tensors (fp16 or bf16, row-major, unit column
stride) and enqueues on torch's current stream.  Given CPU tensors it copies
them to the current device first and returns a CPU result (the end-to-end
path: host -> device -> kernel -> host).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfgemm.so")

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_NO_DEVICE, \
    ERR_CALIBRATION = range(8)
F16, BF16 = 0, 1
ALGOS = {"auto": 0, "classical": 1, "strassen1": 2, "strassen2": 3, "winograd1": 4}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
EPILOGUES = {"none": 0, "scale_bias": 1, "silu": 2, "swiglu": 3}


class Rms(ctypes.Structure):
    _fields_ = [("sumsq_out", ctypes.c_void_p), ("sumsq_in", ctypes.c_void_p),
                ("sumsq_parts", ctypes.c_int32), ("norm_width", ctypes.c_int64),
                ("eps", ctypes.c_float)]


class FgemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(message)


class Epilogue(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("alpha", ctypes.c_float), ("bias", ctypes.c_void_p)]


class DeviceModel(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("peak_tflops", ctypes.c_double), ("hbm_gbs", ctypes.c_double),
                ("eff_classical", ctypes.c_double * 3),
                ("eff_pair", ctypes.c_double * 2),
                ("eff_strassen", (ctypes.c_double * 2) * 2),
                ("eff_strassen_pair", ctypes.c_double * 2),
                ("launch_us", ctypes.c_double), ("tile_fill_us", ctypes.c_double),
                ("l2_bytes", ctypes.c_double), ("l2_gbs", ctypes.c_double),
                ("split_fix_us", ctypes.c_double),
                ("eff_winograd", ctypes.c_double * 2),
                ("eff_small_m", ctypes.c_double * 3), ("hbm_stream_eff", ctypes.c_double),
                ("small_m_stream_eff", ctypes.c_double), ("small_m_fix_us", ctypes.c_double),
                ("small_m_aligned_eff", ctypes.c_double),
                ("form_in_kernel_eff", ctypes.c_double),
                ("form_in_kernel_drag", ctypes.c_double),
                ("lcma_margin", ctypes.c_double),
                ("dram_miss_slope", ctypes.c_double),
                ("dram_exposed", ctypes.c_double),
                ("eff_strassen2_pair", ctypes.c_double * 2),
                ("fold2_unit_us", ctypes.c_double)]


_lib = None
_lib_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise FgemmError(ERR_CUDA, f"fgemm CUDA library not built: {LIB_PATH} is missing "
                                       "(run python -m complexity_matmul_tcgen05_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, vp, st = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int
        epi_p = ctypes.POINTER(Epilogue)
        model_p = ctypes.POINTER(DeviceModel)
        L.fgemm_create.argtypes = [ctypes.POINTER(vp)]
        L.fgemm_destroy.argtypes = [vp]
        L.fgemm_set_stream.argtypes = [vp, vp]
        mm = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, st, epi_p, st]
        L.fgemm_matmul.argtypes = mm
        L.fgemm_matmul_ex.argtypes = mm + [i32, i32]
        L.fgemm_matmul_rms.argtypes = mm + [i32, i32, ctypes.POINTER(Rms)]
        L.fgemm_matmul_mx.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, i32, vp, i64, vp, i64,
                                      i32, vp, i64, epi_p, st, i32, i32]
        L.fgemm_mx_to_bf16.argtypes = [vp, i64, i64, vp, i64, vp, i64, i32, i32, vp, i64]
        L.fgemm_plan.argtypes = [vp, i64, i64, i64, st, epi_p, ctypes.POINTER(st),
                                 ctypes.POINTER(i32), ctypes.POINTER(i32),
                                 ctypes.POINTER(ctypes.c_double)]
        L.fgemm_plan_ex.argtypes = [vp, i64, i64, i64, st, epi_p, st, i32, i32, ctypes.POINTER(st),
                                    ctypes.POINTER(i32), ctypes.POINTER(i32),
                                    ctypes.POINTER(ctypes.c_double)]
        L.fgemm_get_error.argtypes = [vp]
        L.fgemm_matmul_host.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, st, epi_p, st, i32, i32]
        L.fgemm_matmul_host_ex.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, st, epi_p, st, i32,
                                           i32, i32]
        L.fgemm_call_launches.argtypes = [vp, i64, i64, i64, epi_p, st, i32, i32, ctypes.POINTER(i32)]
        L.fgemm_selftest_wait_timeout.argtypes = [vp, i32]
        L.fgemm_calibrate.argtypes = [vp, ctypes.c_char_p]
        L.fgemm_calibrate_ex.argtypes = [vp, i64, ctypes.c_char_p]
        L.fgemm_model_load_json.argtypes = [ctypes.c_char_p, model_p]
        L.fgemm_model_save_json.argtypes = [model_p, ctypes.c_char_p]
        L.fgemm_status_string.argtypes = [st]
        L.fgemm_status_string.restype = ctypes.c_char_p
        L.fgemm_last_message.argtypes = [vp]
        L.fgemm_last_message.restype = ctypes.c_char_p
        L.fgemm_validate.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, st, epi_p, st, i32,
                                     i32]
        L.fgemm_model_default.argtypes = [model_p, i32, ctypes.c_double, ctypes.c_double]
        L.fgemm_model_default.restype = None
        L.fgemm_model_tiles.argtypes = [i64, i64, i32, i32]
        L.fgemm_model_tiles.restype = i64
        L.fgemm_model_waves.argtypes = [i64, i32, ctypes.POINTER(ctypes.c_double)]
        L.fgemm_model_waves.restype = i64
        L.fgemm_model_tiled_reads.argtypes = [i64, i64, i64, i32, i32]
        L.fgemm_model_tiled_reads.restype = ctypes.c_double
        L.fgemm_model_roofline.argtypes = [ctypes.c_double] * 4
        L.fgemm_model_roofline.restype = ctypes.c_double
        L.fgemm_model_predict.argtypes = [model_p, i64, i64, i64, i32, st, i32, i32,
                                          ctypes.POINTER(ctypes.c_double)]
        L.fgemm_model_plan.argtypes = [model_p, i64, i64, i64, i32, ctypes.POINTER(st),
                                       ctypes.POINTER(i32), ctypes.POINTER(i32),
                                       ctypes.POINTER(ctypes.c_double)]
        L.fgemm_strassen_matmul_static.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, st,
                                                   epi_p, i32, i32, vp]
        L.fgemm_strassen_static_get_error.argtypes = [vp]
        L.fgemm_strassen_static_selftest_timeout.argtypes = [i32, vp]
        L.fgemm_model_split_tail.argtypes = [model_p, i64, i32, i32, i32, i32, ctypes.POINTER(i32)]
        L.fgemm_model_split_tail.restype = i32
        L.fgemm_split_work_item.argtypes = [i64, i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32)]
        L.fgemm_split_work_item.restype = i32
        L.fgemm_set_split_mode.argtypes = [vp, i32]
        L.fgemm_set_lcma_formation.argtypes = [vp, i32]
        L.fgemm_stream_k_work_item.argtypes = [i64, i32, i32, i32, i32, ctypes.POINTER(i64)]
        L.fgemm_stream_k_work_item.restype = i32
        L.fgemm_small_m_grid.argtypes = [i64, i32, i32, ctypes.POINTER(i32)]
        L.fgemm_small_m_grid.restype = i32
        L.fgemm_lcma_pair_clusters.argtypes = [i64, i32, i32]
        L.fgemm_lcma_pair_clusters.restype = i64
        L.fgemm_get_device_model.argtypes = [vp, model_p]
        L.fgemm_set_device_model.argtypes = [vp, model_p]
        for name in ("fgemm_create", "fgemm_destroy", "fgemm_set_stream", "fgemm_matmul",
                     "fgemm_matmul_ex", "fgemm_plan", "fgemm_plan_ex", "fgemm_get_error", "fgemm_calibrate",
                     "fgemm_calibrate_ex", "fgemm_model_load_json", "fgemm_model_save_json",
                     "fgemm_validate", "fgemm_model_predict", "fgemm_model_plan",
                     "fgemm_get_device_model", "fgemm_set_device_model",
                     "fgemm_strassen_matmul_static", "fgemm_selftest_wait_timeout",
                     "fgemm_set_split_mode", "fgemm_set_lcma_formation", "fgemm_call_launches", "fgemm_matmul_host", "fgemm_matmul_host_ex", "fgemm_matmul_rms", "fgemm_matmul_mx",
                     "fgemm_mx_to_bf16", "fgemm_strassen_static_get_error",
                     "fgemm_strassen_static_selftest_timeout"):
            getattr(L, name).restype = st
        _lib = L
        return L


SPLIT_MODES = {"off": 0, "auto": 1, "force": 2}
FORMATION_MODES = {"auto": 0, "prepass": 1, "in_kernel": 2}


def split_work_items(tiles: int, split_tiles: int, split_pieces: int, clusters: int,
                     k_blocks: int, cluster: int):
    """The work list of one pair in the K-split schedule, as (unit, k0, k1,
    piece, npieces) tuples (host-side copy of what the kernel runs)."""
    out = (ctypes.c_int32 * 5)()
    items = []
    n = 0
    while lib().fgemm_split_work_item(tiles, split_tiles, split_pieces, clusters, k_blocks,
                                      cluster, n, out):
        items.append(tuple(out))
        n += 1
    return items


def stream_k_work_items(tiles: int, k_blocks: int, ctas: int, cta: int):
    """The work list of one CTA of the small-M kernel, as (unit, k0, k1,
    piece, npieces, slot) tuples (host-side copy of what the kernel runs)."""
    out = (ctypes.c_int64 * 6)()
    items = []
    n = 0
    while lib().fgemm_stream_k_work_item(tiles, k_blocks, ctas, cta, n, out):
        items.append(tuple(out))
        n += 1
    return items


def small_m_grid(tiles: int, k_blocks: int, num_sms: int):
    """(CTA count, phases) of the small-M kernel's grid (fgemm_small_m_grid)."""
    ph = ctypes.c_int32()
    return lib().fgemm_small_m_grid(tiles, k_blocks, num_sms, ctypes.byref(ph)), ph.value


def status_string(status: int) -> str:
    return lib().fgemm_status_string(status).decode()


def _check(status: int, handle_ptr=None):
    if status != OK:
        msg = lib().fgemm_last_message(handle_ptr).decode()
        raise FgemmError(status, f"{status_string(status)}: {msg}")


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float16:
        return F16
    if t == torch.bfloat16:
        return BF16
    raise FgemmError(ERR_INVALID_ARG, f"fgemm supports float16 and bfloat16, not {t}")


def make_epilogue(kind: str = "none", alpha: float = 1.0, bias_ptr: int | None = None) -> Epilogue:
    return Epilogue(EPILOGUES[kind], float(alpha), bias_ptr)


def validate(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, dtype: int, epilogue: Epilogue | None,
             algo: str = "auto", tile_n: int = 0, tile_m: int = 0) -> int:
    """Host-only argument check (no device): the status fgemm_matmul_ex would return."""
    return lib().fgemm_validate(M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, dtype,
                                ctypes.byref(epilogue) if epilogue is not None else None,
                                ALGOS[algo], tile_m, tile_n)


class Handle:
    """An fgemm handle on the current CUDA device."""

    def __init__(self):
        h = ctypes.c_void_p()
        _check(lib().fgemm_create(ctypes.byref(h)))
        self._h = h
        self.device = torch.cuda.current_device()

    @property
    def ptr(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().fgemm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):  # pragma: no cover - interpreter teardown order
        try:
            self.close()
        except Exception:
            pass

    def set_stream(self, stream_ptr: int):
        _check(lib().fgemm_set_stream(self._h, ctypes.c_void_p(stream_ptr)), self._h)

    def set_split_mode(self, mode):
        """K split of the last wave of CTA-pair tiles: "off" (0), "auto" (1,
        the default) or "force" (2, whenever possible)."""
        code = SPLIT_MODES[mode] if isinstance(mode, str) else int(mode)
        _check(lib().fgemm_set_split_mode(self._h, code), self._h)

    def set_lcma_formation(self, mode):
        """Where one-level Strassen-like launches on CTA pairs form their
        summed operands: "auto" (0, the default), "prepass" (1, a separate
        launch) or "in_kernel" (2, inside the product kernel while the
        scheme's leading products that read only blocks of A and B run)."""
        code = FORMATION_MODES[mode] if isinstance(mode, str) else int(mode)
        _check(lib().fgemm_set_lcma_formation(self._h, code), self._h)

    def matmul_raw(self, M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, dtype: int,
                   epilogue: Epilogue | None = None, algo: str = "auto", tile_n: int = 0,
                   tile_m: int = 0) -> int:
        """Direct C-ABI call on raw device pointers; returns the status."""
        return lib().fgemm_matmul_ex(self._h, M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, dtype,
                                     ctypes.byref(epilogue) if epilogue is not None else None,
                                     ALGOS[algo], tile_m, tile_n)

    def matmul_rms_raw(self, M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, dtype: int,
                       epilogue: Epilogue | None, algo: str, tile_n: int, tile_m: int,
                       rms: Rms) -> int:
        """fgemm_matmul_rms on raw device pointers; returns the status."""
        return lib().fgemm_matmul_rms(self._h, M, N, K, A_ptr, lda, B_ptr, ldb, C_ptr, ldc, dtype,
                                      ctypes.byref(epilogue) if epilogue is not None else None,
                                      ALGOS[algo], tile_m, tile_n, ctypes.byref(rms))

    def plan(self, M, N, K, dtype: int = BF16, epilogue: Epilogue | None = None,
             algo: str = "auto", tile_m: int = 0, tile_n: int = 0):
        """(algorithm, tile_m, tile_n, predicted us) of the model's choice,
        restricted to a form / tile when those are given."""
        a = ctypes.c_int()
        tm = ctypes.c_int32()
        tn = ctypes.c_int32()
        us = ctypes.c_double()
        _check(lib().fgemm_plan_ex(self._h, M, N, K, dtype,
                                   ctypes.byref(epilogue) if epilogue is not None else None,
                                   ALGOS[algo], tile_m, tile_n, ctypes.byref(a), ctypes.byref(tm),
                                   ctypes.byref(tn), ctypes.byref(us)), self._h)
        return ALGO_NAMES[a.value], tm.value, tn.value, us.value

    def call_launches(self, M, N, K, epilogue: Epilogue | None = None, algo: str = "auto",
                      tile_m: int = 0, tile_n: int = 0) -> int:
        """Kernels of this library one matmul call with these arguments
        launches on this handle (host only)."""
        n = ctypes.c_int32()
        _check(lib().fgemm_call_launches(self._h, M, N, K,
                                         ctypes.byref(epilogue) if epilogue is not None else None,
                                         ALGOS[algo], tile_m, tile_n, ctypes.byref(n)), self._h)
        return n.value

    def get_error(self) -> int:
        return lib().fgemm_get_error(self._h)

    def last_message(self) -> str:
        return lib().fgemm_last_message(self._h).decode()

    def calibrate(self, json_path: str | None = None, n: int = 8192):
        _check(lib().fgemm_calibrate_ex(self._h, n, json_path.encode() if json_path else None),
               self._h)

    def device_model(self) -> DeviceModel:
        m = DeviceModel()
        _check(lib().fgemm_get_device_model(self._h, ctypes.byref(m)), self._h)
        return m

    def set_device_model(self, m: DeviceModel):
        _check(lib().fgemm_set_device_model(self._h, ctypes.byref(m)), self._h)


_handles: dict[int, Handle] = {}


def default_handle() -> Handle:
    dev = torch.cuda.current_device()
    h = _handles.get(dev)
    if h is None:
        h = Handle()
        _handles[dev] = h
    return h


def _check_matrix(t: torch.Tensor, name: str):
    if t.dim() != 2:
        raise FgemmError(ERR_INVALID_ARG, f"{name} must be 2-D")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise FgemmError(ERR_INVALID_ARG, f"{name} must be row-major with unit column stride")


def matmul(A: torch.Tensor, B: torch.Tensor, *, out: torch.Tensor | None = None,
           epilogue: str = "none", alpha: float = 1.0, bias: torch.Tensor | None = None,
           algo: str = "auto", tile_n: int = 0, tile_m: int = 0,
           handle: Handle | None = None, sumsq_out: torch.Tensor | None = None,
           sumsq_in: torch.Tensor | None = None, norm_width: int = 0,
           rms_eps: float = 1e-6, blocking: bool = True) -> torch.Tensor:
    """C = epi(alpha * A @ B + bias) through fgemm_matmul_ex.

    A is M x K, B is K x N (row-major), bias has N entries; for
    epilogue="swiglu" the output is M x N/2 (gate | up halves of B's columns).

    RMSNorm statistics (fgemm_matmul_rms): ``sumsq_out`` (fp32, shape
    [ceil(N_out/64), M]) receives each row's sums of squares of the stored
    outputs per 64-column block; ``sumsq_in`` (fp32 [parts, M], from an earlier
    call) scales accumulator row i by 1/sqrt(sum / norm_width + rms_eps).

    A and B on the host (CPU tensors, pinned for overlapped copies): the
    product goes through fgemm_matmul_host and ``out`` (or the returned
    tensor) is on the host.  With ``blocking=False`` the call returns once it
    is enqueued (fgemm_matmul_host_ex with FGEMM_HOST_OVERLAP: its uploads may
    run under the previous host call's products); C is written once the
    current CUDA stream has reached the call, and the inputs must not be
    written by other work still pending on that stream.
    """
    if A.device.type == "cpu" and B.device.type == "cpu":
        return _matmul_host(A, B, out, epilogue, alpha, bias, algo, tile_n, tile_m, handle, blocking)
    _check_matrix(A, "A")
    _check_matrix(B, "B")
    if not (A.is_cuda and B.is_cuda):
        raise FgemmError(ERR_INVALID_ARG, "A and B must both be CUDA tensors (or both CPU)")
    if A.dtype != B.dtype:
        raise FgemmError(ERR_INVALID_ARG, "A and B must have the same dtype")
    dt = _dtype_code(A.dtype)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise FgemmError(ERR_INVALID_ARG, f"inner dimensions differ: {K} vs {K2}")
    n_out = N // 2 if epilogue == "swiglu" else N
    if out is None:
        out = torch.empty((M, n_out), dtype=A.dtype, device=A.device)
    else:
        _check_matrix(out, "out")
        if out.dtype != A.dtype or tuple(out.shape) != (M, n_out):
            raise FgemmError(ERR_INVALID_ARG, "out has the wrong dtype or shape")
    bias_ptr = None
    if bias is not None:
        if bias.dtype != A.dtype or bias.numel() != N or not bias.is_cuda:
            raise FgemmError(ERR_INVALID_ARG, "bias must be a CUDA vector of N entries, same dtype")
        bias = bias.contiguous()
        bias_ptr = bias.data_ptr()
    h = handle if handle is not None else default_handle()
    h.set_stream(torch.cuda.current_stream(A.device).cuda_stream)
    epi = make_epilogue(epilogue, alpha, bias_ptr)
    lda = A.stride(0) if M > 1 else max(K, 1)
    ldb = B.stride(0) if K > 1 else max(N, 1)
    ldc = out.stride(0) if M > 1 else max(n_out, 1)
    if sumsq_out is None and sumsq_in is None:
        s = h.matmul_raw(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, dt,
                         epi, algo, tile_n, tile_m)
    else:
        parts = 0
        for t, name in ((sumsq_out, "sumsq_out"), (sumsq_in, "sumsq_in")):
            if t is not None and (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()):
                raise FgemmError(ERR_INVALID_ARG, f"{name} must be a contiguous CUDA float32 tensor")
        if sumsq_out is not None and tuple(sumsq_out.shape) != ((n_out + 63) // 64, M):
            raise FgemmError(ERR_INVALID_ARG, "sumsq_out must have shape [ceil(N_out / 64), M]")
        if sumsq_in is not None:
            if sumsq_in.dim() != 2 or sumsq_in.shape[1] != M:
                raise FgemmError(ERR_INVALID_ARG, "sumsq_in must have shape [parts, M]")
            parts = sumsq_in.shape[0]
        rms = Rms(None if sumsq_out is None else sumsq_out.data_ptr(),
                  None if sumsq_in is None else sumsq_in.data_ptr(), parts, int(norm_width),
                  float(rms_eps))
        s = h.matmul_rms_raw(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, dt,
                             epi, algo, tile_n, tile_m, rms)
    _check(s, h.ptr)
    return out


HOST_OVERLAP = 1


def _matmul_host(A, B, out, epilogue, alpha, bias, algo, tile_n, tile_m, handle, blocking=True):
    """Host tensors through fgemm_matmul_host_ex (pipelined copies; they
    overlap when the tensors are pinned); returns once C is written, or
    (blocking=False) once the call is enqueued."""
    for t, name in ((A, "A"), (B, "B")):
        if t.dim() != 2 or t.stride(1) != 1:
            raise FgemmError(ERR_INVALID_ARG, f"{name} must be a 2-D tensor with unit column stride")
    if A.dtype != B.dtype:
        raise FgemmError(ERR_INVALID_ARG, "A and B must have the same dtype")
    dt = _dtype_code(A.dtype)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise FgemmError(ERR_INVALID_ARG, f"inner dimensions differ: {K} vs {K2}")
    n_out = N // 2 if epilogue == "swiglu" else N
    if out is None:
        out = torch.empty((M, n_out), dtype=A.dtype, pin_memory=A.is_pinned())
    elif (out.device.type != "cpu" or out.dtype != A.dtype or tuple(out.shape) != (M, n_out)
          or out.stride(1) != 1):
        raise FgemmError(ERR_INVALID_ARG, "out must be a host tensor of the right dtype and shape")
    bias_ptr = None
    if bias is not None:
        if bias.device.type != "cpu" or bias.dtype != A.dtype or bias.numel() != N:
            raise FgemmError(ERR_INVALID_ARG, "bias must be a host vector of N entries, same dtype")
        if not blocking and not bias.is_contiguous():
            raise FgemmError(ERR_INVALID_ARG, "a non-blocking call needs a contiguous bias")
        bias = bias.contiguous()
        bias_ptr = bias.data_ptr()
    h = handle if handle is not None else default_handle()
    h.set_stream(torch.cuda.current_stream().cuda_stream)
    epi = make_epilogue(epilogue, alpha, bias_ptr)
    s = lib().fgemm_matmul_host_ex(h.ptr, M, N, K, A.data_ptr(), A.stride(0) if M > 1 else max(K, 1),
                                   B.data_ptr(), B.stride(0) if K > 1 else max(N, 1), out.data_ptr(),
                                   out.stride(0) if M > 1 else max(n_out, 1), dt, ctypes.byref(epi),
                                   ALGOS[algo], tile_m, tile_n, 0 if blocking else HOST_OVERLAP)
    _check(s, h.ptr)
    if blocking:
        torch.cuda.current_stream().synchronize()
        _check(h.get_error(), h.ptr)
    return out


FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def matmul_mx(A: torch.Tensor, scale_a: torch.Tensor, B: torch.Tensor, scale_b: torch.Tensor, *,
              a_format: str = "e4m3", b_format: str = "e4m3", out: torch.Tensor | None = None,
              epilogue: str = "none", alpha: float = 1.0, bias: torch.Tensor | None = None,
              algo: str = "auto", tile_n: int = 0, tile_m: int = 0,
              handle: Handle | None = None) -> torch.Tensor:
    """C = epi(alpha * A @ B + bias) for block-scaled 8-bit A (M x K) and B
    (K x N), given as uint8 (or float8) CUDA tensors, with E8M0 scales
    scale_a (M x ceil(K/32)) and scale_b (ceil(K/32) x N) as uint8; C is bf16."""
    for t, name in ((A, "A"), (B, "B"), (scale_a, "scale_a"), (scale_b, "scale_b")):
        if not t.is_cuda or t.dim() != 2 or t.element_size() != 1 or t.stride(1) != 1:
            raise FgemmError(ERR_INVALID_ARG, f"{name} must be a 2-D CUDA byte tensor with unit column stride")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise FgemmError(ERR_INVALID_ARG, f"inner dimensions differ: {K} vs {K2}")
    kb = (K + 31) // 32
    if tuple(scale_a.shape) != (M, kb) or tuple(scale_b.shape) != (kb, N):
        raise FgemmError(ERR_INVALID_ARG, "scales must be M x ceil(K/32) and ceil(K/32) x N")
    n_out = N // 2 if epilogue == "swiglu" else N
    if out is None:
        out = torch.empty((M, n_out), dtype=torch.bfloat16, device=A.device)
    bias_ptr = None
    if bias is not None:
        if bias.dtype != torch.bfloat16 or bias.numel() != N or not bias.is_cuda:
            raise FgemmError(ERR_INVALID_ARG, "bias must be a CUDA bf16 vector of N entries")
        bias = bias.contiguous()
        bias_ptr = bias.data_ptr()
    h = handle if handle is not None else default_handle()
    h.set_stream(torch.cuda.current_stream(A.device).cuda_stream)
    epi = make_epilogue(epilogue, alpha, bias_ptr)
    s = lib().fgemm_matmul_mx(h.ptr, M, N, K, A.data_ptr(), A.stride(0) if M > 1 else max(K, 1),
                              scale_a.data_ptr(), scale_a.stride(0) if M > 1 else max(kb, 1),
                              FP8_FORMATS[a_format], B.data_ptr(), B.stride(0) if K > 1 else max(N, 1),
                              scale_b.data_ptr(), scale_b.stride(0) if kb > 1 else max(N, 1),
                              FP8_FORMATS[b_format], out.data_ptr(),
                              out.stride(0) if M > 1 else max(n_out, 1), ctypes.byref(epi),
                              ALGOS[algo], tile_m, tile_n)
    _check(s, h.ptr)
    return out


def mx_to_bf16(X: torch.Tensor, S: torch.Tensor, fmt: str = "e4m3", along: str = "row",
               handle: Handle | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 values of a block-scaled 8-bit matrix X (uint8, rows x cols) with
    E8M0 scales S: blocks of 32 along each row (S rows x ceil(cols/32)) or
    down each column (S ceil(rows/32) x cols).  `out`, if given, is a bf16
    rows x cols tensor on X's device with unit column stride."""
    rows, cols = X.shape
    if out is not None and (out.dtype != torch.bfloat16 or tuple(out.shape) != (rows, cols)
                            or out.device != X.device or (cols > 1 and out.stride(1) != 1)):
        raise ValueError("out must be a bf16 tensor of X's shape and device with unit column stride")
    Y = out if out is not None else torch.empty((rows, cols), dtype=torch.bfloat16, device=X.device)
    h = handle if handle is not None else default_handle()
    h.set_stream(torch.cuda.current_stream(X.device).cuda_stream)
    s = lib().fgemm_mx_to_bf16(h.ptr, rows, cols, X.data_ptr(), X.stride(0) if rows > 1 else max(cols, 1),
                               S.data_ptr(), S.stride(0) if S.shape[0] > 1 else max(S.shape[1], 1),
                               FP8_FORMATS[fmt], 0 if along == "row" else 1, Y.data_ptr(),
                               Y.stride(0) if rows > 1 else max(cols, 1))
    _check(s, h.ptr)
    return Y


def plan(M: int, N: int, K: int, dtype: torch.dtype = torch.bfloat16, epilogue: str = "none"):
    """(algorithm, tile_m, tile_n, predicted microseconds) the decision model picks."""
    h = default_handle()
    return h.plan(M, N, K, _dtype_code(dtype), make_epilogue(epilogue))
