"""Python binding of libqgemv (ctypes, argument marshalling only).

Every entry point has the C name without the ``qgemv_`` prefix.  Tensors are passed as
raw device pointers (``tensor.data_ptr()``); PyTorch is used for device memory and
streams only.  All work runs in the CUDA library; if it is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

Q4_K, NVFP4, TQ1_0, Q5_K, Q6_K, Q8_0 = 0, 1, 2, 3, 4, 5
OPT_FORCE_PATH, OPT_RING_DEPTH, OPT_ROWS_PER_STAGE, OPT_SPIN_LIMIT_NS, OPT_PDL, OPT_TEST_STALL, OPT_CTAS_PER_SM, \
    OPT_KSPLIT, OPT_GRID_PER_SM = 0, 2, 3, 4, 5, 6, 7, 8, 9
STATUS = {0: "QGEMV_OK", 1: "QGEMV_ERR_INVALID_ARG", 2: "QGEMV_ERR_UNSUPPORTED_FORMAT", 3: "QGEMV_ERR_BAD_SHAPE",
          4: "QGEMV_ERR_MISALIGNED", 5: "QGEMV_ERR_CUDA", 6: "QGEMV_ERR_TIMEOUT", 7: "QGEMV_ERR_OOM",
          8: "QGEMV_ERR_NO_DEVICE", 9: "QGEMV_ERR_TOO_LARGE"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_FORMAT, ERR_BAD_SHAPE, ERR_MISALIGNED, ERR_CUDA, ERR_TIMEOUT, ERR_OOM, \
    ERR_NO_DEVICE, ERR_TOO_LARGE = range(10)
NOALLOC_MAX_COLUMN_SUMS = 262144  # QGEMV_NOALLOC_MAX_COLUMN_SUMS
OUT_F32, OUT_F16, OUT_BF16 = 0, 1, 2
MAX_GROUP = 8  # QGEMV_MAX_GROUP
MAX_BATCH = 8  # QGEMV_MAX_BATCH


class Problem(ctypes.Structure):
    """qgemv_problem_t: one matrix of run_group."""
    _fields_ = [("fmt", ctypes.c_int), ("packed_W", ctypes.c_void_p), ("packed_W_up", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("y", ctypes.c_void_p), ("alpha", ctypes.c_float),
                ("beta", ctypes.c_float), ("out", ctypes.c_int), ("swiglu", ctypes.c_int)]

EXPORTS = ["qgemv_create", "qgemv_destroy", "qgemv_run", "qgemv_unpack", "qgemv_check_error",
           "qgemv_status_string", "qgemv_packed_bytes", "qgemv_group_size", "qgemv_set_option",
           "qgemv_describe", "qgemv_build_marker", "qgemv_run_noalloc", "qgemv_run_group", "qgemv_run_ex", "qgemv_run_batch",
           "qgemv_run_gemm"]

_lib = None


class QgemvError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load the in-tree libqgemv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"libqgemv.so is not built ({LIB}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB)
        vp, i64, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.qgemv_create.argtypes = [ctypes.POINTER(vp), ctypes.c_int]
        L.qgemv_destroy.argtypes = [vp]
        L.qgemv_run.argtypes = [vp, ctypes.c_int, vp, vp, i64, i64, vp, vp]
        L.qgemv_unpack.argtypes = [vp, ctypes.c_int, vp, i64, i64, vp, vp, vp, vp]
        L.qgemv_check_error.argtypes = [vp, vp]
        L.qgemv_status_string.argtypes = [ctypes.c_int]
        L.qgemv_status_string.restype = ctypes.c_char_p
        L.qgemv_packed_bytes.argtypes = [ctypes.c_int, i64, i64]
        L.qgemv_packed_bytes.restype = ctypes.c_size_t
        L.qgemv_group_size.argtypes = [ctypes.c_int]
        L.qgemv_set_option.argtypes = [vp, ctypes.c_int, i64]
        L.qgemv_describe.argtypes = [vp, ctypes.c_int, i64, i64, ctypes.c_char_p, ctypes.c_size_t]
        L.qgemv_build_marker.restype = ctypes.c_char_p
        L.qgemv_run_noalloc.argtypes = [ctypes.c_int, vp, vp, i64, i64, vp, vp]
        L.qgemv_run_group.argtypes = [vp, vp, i64, ctypes.c_int, ctypes.POINTER(Problem), vp]
        L.qgemv_run_ex.argtypes = [vp, ctypes.c_int, vp, vp, i64, i64, ctypes.c_float, ctypes.c_float, vp,
                                   ctypes.c_int, vp]
        L.qgemv_run_batch.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, vp, i64, i64, vp, vp]
        L.qgemv_run_gemm.argtypes = [vp, ctypes.c_int, vp, i64, vp, i64, i64, vp, vp]
        for name in ("qgemv_create", "qgemv_destroy", "qgemv_run", "qgemv_unpack", "qgemv_check_error",
                     "qgemv_set_option", "qgemv_describe", "qgemv_run_noalloc", "qgemv_run_group",
                     "qgemv_run_ex", "qgemv_run_batch", "qgemv_run_gemm"):
            getattr(L, name).restype = st
        _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != OK:
        raise QgemvError(status, where)


def status_string(status: int) -> str:
    return lib().qgemv_status_string(status).decode()


def build_marker() -> str:
    return lib().qgemv_build_marker().decode()


def packed_bytes(fmt: int, N: int, K: int) -> int:
    return lib().qgemv_packed_bytes(fmt, N, K)


def group_size(fmt: int) -> int:
    return lib().qgemv_group_size(fmt)


class Handle:
    """Owns a qgemv_handle_t (split-K workspace and error word on one device)."""

    def __init__(self, device: int = 0):
        h = ctypes.c_void_p()
        _check(lib().qgemv_create(ctypes.byref(h), device), "qgemv_create")
        self._h = h
        self.device = device

    @property
    def ptr(self):
        return self._h

    def close(self) -> None:
        if self._h is not None and self._h.value:
            lib().qgemv_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def create(device: int = 0) -> Handle:
    return Handle(device)


def destroy(h: Handle) -> None:
    h.close()


def run(h: Handle, fmt: int, x, packed_W, N: int, K: int, y, stream=None, check: bool = True) -> int:
    """y = x . dequant(W)^T, asynchronous on `stream` (default: torch's current stream)."""
    st = lib().qgemv_run(h.ptr, fmt, _ptr(x), _ptr(packed_W), N, K, _ptr(y), _stream(stream))
    if check:
        _check(st, "qgemv_run")
    return st


def run_noalloc(fmt: int, x, packed_W, N: int, K: int, y, stream=None, check: bool = True) -> int:
    """qgemv_run_noalloc: the same GEMV without a handle, using the library's fixed scratch
    (for callers that may not allocate device memory).  Calls must not overlap on the GPU."""
    st = lib().qgemv_run_noalloc(fmt, _ptr(x), _ptr(packed_W), N, K, _ptr(y), _stream(stream))
    if check:
        _check(st, "qgemv_run_noalloc")
    return st


def run_ex(h: Handle, fmt: int, x, packed_W, N: int, K: int, y, alpha: float = 1.0, beta: float = 0.0,
           out: int = OUT_F32, stream=None, check: bool = True) -> int:
    """y = alpha * x . dequant(W)^T + beta * y, y of type `out` (OUT_F32 / OUT_F16 / OUT_BF16)."""
    st = lib().qgemv_run_ex(h.ptr, fmt, _ptr(x), _ptr(packed_W), N, K, alpha, beta, _ptr(y), out,
                            _stream(stream))
    if check:
        _check(st, "qgemv_run_ex")
    return st


def run_batch(h: Handle, fmt: int, x, M: int, packed_W, N: int, K: int, y, stream=None, check: bool = True) -> int:
    """Y[m] = X[m] . dequant(W)^T for M (<= MAX_BATCH) row-major activation vectors x [M, K]."""
    st = lib().qgemv_run_batch(h.ptr, fmt, _ptr(x), M, _ptr(packed_W), N, K, _ptr(y), _stream(stream))
    if check:
        _check(st, "qgemv_run_batch")
    return st


def run_gemm(h: Handle, fmt: int, x, M: int, packed_W, N: int, K: int, y, stream=None, check: bool = True) -> int:
    """Y = X . dequant(W)^T for any number M of row-major activation rows x [M, K] (NVFP4 with
    M > MAX_BATCH on the tcgen05 tensor-core kernel)."""
    st = lib().qgemv_run_gemm(h.ptr, fmt, _ptr(x), M, _ptr(packed_W), N, K, _ptr(y), _stream(stream))
    if check:
        _check(st, "qgemv_run_gemm")
    return st


def problem(fmt: int, packed_W, N: int, y, packed_W_up=None, alpha: float = 1.0, beta: float = 0.0,
            out: int = OUT_F32, swiglu: bool = False) -> Problem:
    return Problem(fmt, _ptr(packed_W), _ptr(packed_W_up), N, _ptr(y), alpha, beta, out, int(swiglu))


def run_group(h: Handle, x, K: int, problems, stream=None, check: bool = True) -> int:
    """GEMVs sharing x (a list of `problem(...)` entries, at most MAX_GROUP), one launch."""
    arr = (Problem * max(1, len(problems)))(*problems)
    st = lib().qgemv_run_group(h.ptr, _ptr(x), K, len(problems), arr, _stream(stream))
    if check:
        _check(st, "qgemv_run_group")
    return st


def unpack(h: Handle, fmt: int, packed_W, N: int, K: int, codes, scales, mins=None, stream=None,
           check: bool = True) -> int:
    st = lib().qgemv_unpack(h.ptr, fmt, _ptr(packed_W), N, K, _ptr(codes), _ptr(scales), _ptr(mins),
                            _stream(stream))
    if check:
        _check(st, "qgemv_unpack")
    return st


def check_error(h: Handle, stream=None) -> int:
    return lib().qgemv_check_error(h.ptr, _stream(stream))


def set_option(h: Handle, opt: int, value: int, check: bool = True) -> int:
    st = lib().qgemv_set_option(h.ptr, opt, value)
    if check:
        _check(st, "qgemv_set_option")
    return st


def describe(h: Handle, fmt: int, N: int, K: int) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(lib().qgemv_describe(h.ptr, fmt, N, K, buf, 512), "qgemv_describe")
    return buf.value.decode()
