"""CPU oracle for C[M,N] = A[M,K] . B[K,N] with fp16/bf16 inputs (fp64 inside).

TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU-baseline
leg of the benchmark may import this package; the product library never does,
and it shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, compiled with gcc).  This module
only builds it when needed and marshals numpy arrays through ctypes.  Inputs
and outputs are the raw 16-bit patterns (numpy ``uint16``), so the oracle sees
exactly the bytes the device sees.

Reading of the pages implemented here (the plain definition of the product,
"tcgen05 for dummies: a B200 GEMM from scratch", section "Recap: how to write
a fast matmul kernel"): exact decode to double, exact products, double sum in k
order, one IEEE round-to-nearest-even to the output format.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16 = 0, 1
TN, NN = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    """The library at `path` with its entry points' argument types declared."""
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_decode.restype = ctypes.c_double
    lib.oracle_decode.argtypes = [ctypes.c_uint16, ctypes.c_int]
    lib.oracle_encode.restype = ctypes.c_uint16
    lib.oracle_encode.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.oracle_decode_array.argtypes = [u16p, f64p, i64, ctypes.c_int]
    lib.oracle_encode_array.argtypes = [f64p, u16p, i64, ctypes.c_int]
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [u16p, u16p, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, u16p, f64p, f64p, ctypes.c_int]
    lib.oracle_gemm_entries.restype = ctypes.c_int
    lib.oracle_gemm_entries.argtypes = [u16p, u16p, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                        i64p, i64p, i64, f64p, f64p, ctypes.c_int]
    lib.oracle_gemm_tiled.restype = ctypes.c_int
    lib.oracle_gemm_tiled.argtypes = [u16p, u16p, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                      i64, i64, i64, f64p]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _dt(dtype) -> int:
    if dtype in (F16, "f16", "fp16", "float16"):
        return F16
    if dtype in (BF16, "bf16", "bfloat16"):
        return BF16
    raise ValueError("dtype must be f16 or bf16, got %r" % (dtype,))


def _lay(layout) -> int:
    if layout in (TN, "TN"):
        return TN
    if layout in (NN, "NN"):
        return NN
    raise ValueError("layout must be TN or NN, got %r" % (layout,))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("expected raw uint16 bit patterns, got %s" % a.dtype)
    return a


def _p(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def decode(bits, dtype) -> np.ndarray:
    """Exact decode of 16-bit patterns to float64."""
    bits = _u16(bits)
    out = np.empty(bits.shape, np.float64)
    _load().oracle_decode_array(_p(bits, ctypes.c_uint16), _p(out, ctypes.c_double), bits.size, _dt(dtype))
    return out


def encode(values, dtype) -> np.ndarray:
    """float64 -> 16-bit patterns, round-to-nearest-even, overflow to Inf."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_encode_array(_p(v, ctypes.c_double), _p(out, ctypes.c_uint16), v.size, _dt(dtype))
    return out


def gemm(A_bits, B_bits, M, N, K, layout, in_dtype, out_dtype, nthreads=0, want_exact=False, want_abs=False):
    """Full product.  Returns (C_bits, C_exact or None, C_abs or None).

    A_bits is [M,K] row-major; B_bits is [N,K] (TN) or [K,N] (NN).  C_abs holds
    sum_k |a_mk * b_kn|, the scale the tolerances are written against."""
    A = _u16(A_bits)
    B = _u16(B_bits)
    if A.size != M * K or B.size != K * N:
        raise ValueError("operand sizes do not match M, N, K")
    C = np.empty((M, N), np.uint16)
    ex = np.empty((M, N), np.float64) if want_exact else None
    ab = np.empty((M, N), np.float64) if want_abs else None
    rc = _load().oracle_gemm(
        _p(A, ctypes.c_uint16), _p(B, ctypes.c_uint16), M, N, K, _lay(layout), _dt(in_dtype), _dt(out_dtype),
        _p(C, ctypes.c_uint16),
        _p(ex, ctypes.c_double) if ex is not None else None,
        _p(ab, ctypes.c_double) if ab is not None else None,
        int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_gemm failed")
    return C, ex, ab


def gemm_entries(A_bits, B_bits, M, N, K, layout, in_dtype, rows, cols, nthreads=0):
    """Exact (double) dot products and sum|ab| for selected entries."""
    A = _u16(A_bits)
    B = _u16(B_bits)
    if A.size != M * K or B.size != K * N:
        raise ValueError("operand sizes do not match M, N, K")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in shape")
    ex = np.empty(r.shape, np.float64)
    ab = np.empty(r.shape, np.float64)
    rc = _load().oracle_gemm_entries(
        _p(A, ctypes.c_uint16), _p(B, ctypes.c_uint16), M, N, K, _lay(layout), _dt(in_dtype),
        _p(r, ctypes.c_int64), _p(c, ctypes.c_int64), r.size,
        _p(ex, ctypes.c_double), _p(ab, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_entries failed (index out of range?)")
    return ex, ab


def gemm_tiled(A_bits, B_bits, M, N, K, layout, in_dtype, BM=128, BN=128, BK=64):
    """The tiled loop nest of the same section, in double (self-check only)."""
    A = _u16(A_bits)
    B = _u16(B_bits)
    ex = np.empty((M, N), np.float64)
    rc = _load().oracle_gemm_tiled(
        _p(A, ctypes.c_uint16), _p(B, ctypes.c_uint16), M, N, K, _lay(layout), _dt(in_dtype),
        BM, BN, BK, _p(ex, ctypes.c_double))
    if rc != 0:
        raise RuntimeError("oracle_gemm_tiled failed")
    return ex
