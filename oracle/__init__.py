"""CPU fp64 oracle for the batch-1 dequant GEMV (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never loads it; the two share no code.

The arithmetic lives in ``qgemv_oracle.c`` (plain C, fp64, one weight at a time); this
module only builds that file with the host C compiler and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qgemv_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

Q4_K, NVFP4, TQ1_0, Q5_K, Q6_K, Q8_0 = 0, 1, 2, 3, 4, 5


def build(force: bool = False) -> str:
    """Compile qgemv_oracle.c into _build/liboracle.so (plain -O2, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        d, u8p, u16p, i64, i64p = (ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int64, ctypes.c_void_p)
        L.oracle_minifloat.restype = d
        L.oracle_minifloat.argtypes = [ctypes.c_uint32, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        for name, argt in (("oracle_fp16", ctypes.c_uint16), ("oracle_bf16", ctypes.c_uint16),
                           ("oracle_e4m3", ctypes.c_uint8), ("oracle_e5m2", ctypes.c_uint8),
                           ("oracle_e2m1", ctypes.c_uint8)):
            getattr(L, name).restype = d
            getattr(L, name).argtypes = [argt]
        L.oracle_tq1_digit.restype = ctypes.c_int
        L.oracle_tq1_digit.argtypes = [ctypes.c_uint8, ctypes.c_int]
        L.oracle_group_size.restype = ctypes.c_int
        L.oracle_group_size.argtypes = [ctypes.c_int]
        L.oracle_dequant_rows.restype = ctypes.c_int
        L.oracle_dequant_rows.argtypes = [ctypes.c_int, u8p, i64, i64, i64p, i64, ctypes.c_void_p]
        L.oracle_unpack.restype = ctypes.c_int
        L.oracle_unpack.argtypes = [ctypes.c_int, u8p, i64, i64, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p]
        L.oracle_gemv_rows.restype = ctypes.c_int
        L.oracle_gemv_rows.argtypes = [ctypes.c_int, u16p, u8p, i64, i64, i64p, i64, ctypes.c_void_p,
                                       ctypes.c_void_p]
        L.oracle_gemv_range.restype = ctypes.c_int
        L.oracle_gemv_range.argtypes = [ctypes.c_int, u16p, u8p, i64, i64, i64, i64, ctypes.c_void_p,
                                        ctypes.c_void_p]
        L.oracle_silu.restype = d
        L.oracle_silu.argtypes = [d]
        L.oracle_gemv_general.restype = ctypes.c_int
        L.oracle_gemv_general.argtypes = [ctypes.c_int, u16p, u8p, i64, i64, d, d, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_swiglu.restype = ctypes.c_int
        L.oracle_swiglu.argtypes = [ctypes.c_int, u16p, u8p, u8p, i64, i64] + [ctypes.c_void_p] * 5
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def fp16(bits: int) -> float:
    return lib().oracle_fp16(bits)


def bf16(bits: int) -> float:
    return lib().oracle_bf16(bits)


def e4m3(bits: int) -> float:
    return lib().oracle_e4m3(bits)


def e5m2(bits: int) -> float:
    return lib().oracle_e5m2(bits)


def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def minifloat(bits: int, ebits: int, mbits: int, bias: int, special: int) -> float:
    return lib().oracle_minifloat(bits, ebits, mbits, bias, special)


def tq1_digit(b: int, n: int) -> int:
    return lib().oracle_tq1_digit(b, n)


def group_size(fmt: int) -> int:
    return lib().oracle_group_size(fmt)


def dequant_rows(fmt: int, W: np.ndarray, N: int, K: int, rows) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((len(rows), K), dtype=np.float64)
    rc = lib().oracle_dequant_rows(fmt, _ptr(W), N, K, _ptr(rows), len(rows), _ptr(out))
    if rc:
        raise ValueError(f"oracle_dequant_rows failed ({rc})")
    return out


def unpack(fmt: int, W: np.ndarray, N: int, K: int):
    """(codes int8 [N,K], scales f64 [N,K/G], mins f64 [N,K/G]) with w = scales*codes - mins."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    G = group_size(fmt)
    codes = np.empty((N, K), dtype=np.int8)
    scales = np.empty((N, K // G), dtype=np.float64)
    mins = np.empty((N, K // G), dtype=np.float64)
    rc = lib().oracle_unpack(fmt, _ptr(W), N, K, _ptr(codes), _ptr(scales), _ptr(mins))
    if rc:
        raise ValueError(f"oracle_unpack failed ({rc})")
    return codes, scales, mins


def gemv_rows(fmt: int, x_bits: np.ndarray, W: np.ndarray, N: int, K: int, rows):
    """(y, S) in fp64 for the given rows: y = sum x w, S = sum |x w|."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    y = np.empty(len(rows), dtype=np.float64)
    S = np.empty(len(rows), dtype=np.float64)
    rc = lib().oracle_gemv_rows(fmt, _ptr(x_bits), _ptr(W), N, K, _ptr(rows), len(rows), _ptr(y), _ptr(S))
    if rc:
        raise ValueError(f"oracle_gemv_rows failed ({rc})")
    return y, S


def gemv(fmt: int, x_bits: np.ndarray, W: np.ndarray, N: int, K: int, r0: int = 0, r1: int | None = None):
    """(y, S) in fp64 for rows [r0, r1)."""
    r1 = N if r1 is None else r1
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    y = np.empty(r1 - r0, dtype=np.float64)
    S = np.empty(r1 - r0, dtype=np.float64)
    rc = lib().oracle_gemv_range(fmt, _ptr(x_bits), _ptr(W), N, K, r0, r1, _ptr(y), _ptr(S))
    if rc:
        raise ValueError(f"oracle_gemv_range failed ({rc})")
    return y, S


def silu(g: float) -> float:
    return lib().oracle_silu(float(g))


def gemv_general(fmt: int, x_bits: np.ndarray, W: np.ndarray, N: int, K: int, alpha: float, beta: float,
                 c=None):
    """(y, S) in fp64: y = alpha * x.W^T + beta * c (c unused when beta == 0), S = |alpha| sum|x w|."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    cc = np.ascontiguousarray(np.zeros(N) if c is None else c, dtype=np.float64)
    y = np.empty(N, dtype=np.float64)
    S = np.empty(N, dtype=np.float64)
    rc = lib().oracle_gemv_general(fmt, _ptr(x_bits), _ptr(W), N, K, float(alpha), float(beta), _ptr(cc),
                                   _ptr(y), _ptr(S))
    if rc:
        raise ValueError(f"oracle_gemv_general failed ({rc})")
    return y, S


def swiglu(fmt: int, x_bits: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, N: int, K: int):
    """dict of fp64 arrays h = silu(g) * u, g, u, Sg, Su for gate / up matrices Wg, Wu."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    Wg = np.ascontiguousarray(Wg, dtype=np.uint8)
    Wu = np.ascontiguousarray(Wu, dtype=np.uint8)
    out = {k: np.empty(N, dtype=np.float64) for k in ("h", "g", "u", "Sg", "Su")}
    rc = lib().oracle_swiglu(fmt, _ptr(x_bits), _ptr(Wg), _ptr(Wu), N, K, *(_ptr(out[k]) for k in
                                                                           ("h", "g", "u", "Sg", "Su")))
    if rc:
        raise ValueError(f"oracle_swiglu failed ({rc})")
    return out
