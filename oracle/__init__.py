"""CPU oracle for the tiled GEMM: FP64 reference arithmetic and schedule enumeration.

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
library (`tile_scheduled_tensor_gb300`) never imports, links or runs it, and
this package never imports the product: the two share no code.  The seeded
input generator (`synthetic`) is the only module both sides use.

Parts:
  * gemm_ref.c  - exact BF16 / e4m3 / e5m2 decode, FP64 GEMM with the fused epilogue,
                  FP64 -> BF16 round-to-nearest-even (built into liboracle.so
                  by build_oracle(); plain C, OpenMP over rows).
  * epilogue.py - the extended fused epilogue in the pages' order (alpha, beta*C,
                  vector scales, row/column bias, ReLU/GELU/SiLU, amax, output
                  scale, FP8 e4m3 output encoding), FP64 on the raw accumulator.
  * schedule.py - mappings F(i) -> (m, n), static / persistent / Stream-K work
                  lists, wave efficiency, operand band counts.
  * grouped.py  - the grouped (many-GEMM) persistent schedule: concatenated
                  tile sequence, the warp-level speculative group search.
  * blockscale.py - block-scaled operands (one scale per tile of A and of B).
Every function cites the passage it follows in its own source file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import blockscale, epilogue, grouped, schedule  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

BF16, E4M3, E5M2 = 0, 1, 2


def build_oracle(force: bool = False) -> str:
    """Compile gemm_ref.c with gcc (FP contraction off, so the FP64 sums are
    performed exactly as written)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_e4m3.restype = ctypes.c_double
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e5m2.restype = ctypes.c_double
        lib.oracle_decode_e5m2.argtypes = [ctypes.c_uint8]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_decode_array.restype = None
        lib.oracle_decode_array.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        lib.oracle_gemm_rows_bdec.restype = None
        lib.oracle_gemm_rows_bdec.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                              ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_gemm_rows.restype = None
        lib.oracle_gemm_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                         ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        _lib = lib
    return _lib


def _dtype_code(dtype) -> int:
    if dtype in (BF16, "bf16"):
        return BF16
    if dtype in (E4M3, "e4m3"):
        return E4M3
    if dtype in (E5M2, "e5m2"):
        return E5M2
    raise ValueError(dtype)


def decode(codes: np.ndarray, dtype) -> np.ndarray:
    """Exact FP64 values of BF16 (uint16), e4m3 or e5m2 (uint8) codes."""
    d = _dtype_code(dtype)
    want = np.uint16 if d == BF16 else np.uint8
    c = np.ascontiguousarray(codes, dtype=want)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_decode_array(d, c.ctypes.data, c.size, out.ctypes.data)
    return out


def round_bf16(z: np.ndarray) -> np.ndarray:
    """FP64 -> BF16 bit patterns (uint16), round to nearest even."""
    lib = _load()
    flat = np.ascontiguousarray(z, dtype=np.float64).ravel()
    return np.array([lib.oracle_round_bf16(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(z))


def gemm(A: np.ndarray, B: np.ndarray, dtype, alpha: float = 1.0, scales=None, bias=None,
         relu: bool = False, rows=None, dtype_b=None, b_decoded=None):
    """z (FP64, unrounded, after the epilogue) and absdot = |alpha sA sB| * sum_k |a||b|.

    A: (M, K) codes of `dtype`, B: (N, K) codes of `dtype_b` (default: the same;
    the FP8 formats may be mixed).  rows: optional row indices to compute.
    b_decoded: optional (N, K) FP64 array holding decode(B, dtype_b), for a caller
    that computes many row samples of one B; the arithmetic is the same loop.
    Returns arrays of shape (len(rows) or M, N).
    """
    d = _dtype_code(dtype)
    db = d if dtype_b is None else _dtype_code(dtype_b)
    if (d == BF16) != (db == BF16):
        raise ValueError("BF16 pairs only with BF16")
    want = np.uint16 if d == BF16 else np.uint8
    A = np.ascontiguousarray(A, dtype=want)
    M, K = A.shape
    if b_decoded is None:
        B = np.ascontiguousarray(B, dtype=want)
        N, K2 = B.shape
    else:
        b_decoded = np.ascontiguousarray(b_decoded, dtype=np.float64)
        N, K2 = b_decoded.shape
    assert K == K2
    sA, sB = (1.0, 1.0) if scales is None else (float(scales[0]), float(scales[1]))
    if rows is None:
        rows_arr, nrows, rows_ptr = None, M, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rows_ptr = rows_arr.size, rows_arr.ctypes.data
    bias_arr = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    bias_ptr = None if bias_arr is None else bias_arr.ctypes.data
    z = np.empty((nrows, N), dtype=np.float64)
    ad = np.empty((nrows, N), dtype=np.float64)
    if b_decoded is None:
        _load().oracle_gemm_rows(M, N, K, d, db, A.ctypes.data, B.ctypes.data, rows_ptr, nrows,
                                 float(alpha), sA, sB, bias_ptr, int(bool(relu)), z.ctypes.data, ad.ctypes.data)
    else:
        _load().oracle_gemm_rows_bdec(N, K, d, A.ctypes.data, b_decoded.ctypes.data, rows_ptr, nrows,
                                      float(alpha), sA, sB, bias_ptr, int(bool(relu)), z.ctypes.data,
                                      ad.ctypes.data)
    return z, ad
