"""Oracle for D = alpha*A*B + beta*C (TEST INFRASTRUCTURE ONLY).

Thin ctypes wrapper over ``gemm_ref.c`` plus the acceptance bound.  Only tests/, the
smoke check and the bench's CPU-baseline leg may import this module; the product path
never does.

Definitions followed:
  * "CUTLASS, in depth", section "The problem CUTLASS solves": D = alpha*A*B + beta*C.
  * "Day 84: CUTLASS and CuTe layouts", section "Two programs": the reference sums the
    same half values in double precision.
  * The acceptance rule for a GPU result d against the fp64 reference r (stated with the
    workload definition): |d - r| <= 2^-9 * (|alpha| * sum_k |a_ik b_kj| + |beta c_ij|)
    + one output ulp at |r|; integer-valued workloads must match exactly.
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

F16, BF16, E4M3, E5M2 = 0, 1, 2, 3
K_MAJOR, MN_MAJOR = 0, 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm.argtypes = [i64, i64, i64, dbl, vp, i64, ctypes.c_int, vp, i64,
                                    ctypes.c_int, dbl, vp, i64, ctypes.c_int, vp, vp, i64,
                                    vp, vp, ctypes.c_int]
        ci = ctypes.c_int
        lib.oracle_gemm_typed.restype = ci
        lib.oracle_gemm_typed.argtypes = [i64, i64, i64, dbl, vp, i64, ci, ci, vp, i64, ci, ci,
                                          dbl, vp, i64, ci, vp, vp, i64, vp, vp, ci]
        lib.oracle_gemm_mx.restype = ci
        lib.oracle_gemm_mx.argtypes = [i64, i64, i64, dbl, vp, i64, ci, vp, i64, vp, i64, ci, vp,
                                       i64, dbl, vp, i64, ci, vp, vp, i64, vp, vp, ci]
        lib.oracle_decode.restype = None
        lib.oracle_decode.argtypes = [ctypes.c_int, vp, i64, vp]
        lib.oracle_round.restype = None
        lib.oracle_round.argtypes = [ctypes.c_int, vp, i64, vp]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def dtype_code(name):
    return {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16,
            "e4m3": E4M3, "e5m2": E5M2}[name]


def _bits(arr):
    a = np.ascontiguousarray(arr)
    if a.dtype != np.uint16:
        raise TypeError("oracle operands are raw 16-bit patterns (uint16)")
    return a


def decode(dtype, bits):
    """16-bit patterns -> exact float64 values."""
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode(dtype, b.ctypes.data, b.size, out.ctypes.data)
    return out


def round_to(dtype, values):
    """float64 -> 16-bit patterns, round to nearest, ties to even."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round(dtype, v.ctypes.data, v.size, out.ctypes.data)
    return out


def max_threads():
    return _load().oracle_max_threads()


def gemm(M, N, K, alpha, A, lda, majorA, B, ldb, majorB, beta, C, ldc, dtype,
         rows=None, cols=None, threads=0, a_dtype=None, b_dtype=None):
    """fp64 reference outputs and sum_k |a b| for the requested entries.

    A, B, C are flat uint16 arrays holding the stored operands (C may be None when
    beta == 0); FP8 operands are their one-byte codes widened to uint16.  dtype is the
    format of C (and of A and B unless a_dtype / b_dtype name theirs).  With rows/cols None
    every output is returned as an (M, N) array; otherwise 1-D arrays for the entries
    (rows[e], cols[e]).
    """
    dtA = dtype if a_dtype is None else a_dtype
    dtB = dtype if b_dtype is None else b_dtype
    A = _bits(A)
    B = _bits(B)
    Cp = None
    if C is not None:
        C = _bits(C)
        Cp = C.ctypes.data
    if rows is None:
        n = M * N
        r_p = c_p = None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        n = rows.size
        r_p, c_p = rows.ctypes.data, cols.ctypes.data
    ref = np.empty(n, dtype=np.float64)
    sab = np.empty(n, dtype=np.float64)
    rc = _load().oracle_gemm_typed(M, N, K, float(alpha), A.ctypes.data, lda, majorA, dtA,
                                   B.ctypes.data, ldb, majorB, dtB, float(beta), Cp, ldc,
                                   dtype, r_p, c_p, n, ref.ctypes.data, sab.ctypes.data,
                                   threads)
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    if rows is None:
        return ref.reshape(M, N), sab.reshape(M, N)
    return ref, sab


def gemm_mx(M, N, K, alpha, A, lda, a_dtype, SFA, ld_sfa, B, ldb, b_dtype, SFB, ld_sfb, beta, C,
            ldc, dtype, rows=None, cols=None, threads=0):
    """Block-scaled FP8 GEMM reference (see oracle_gemm_mx): K-major FP8 codes A (M x K) and
    B (N rows of K) as uint16-widened codes, E8M0 scales SFA (M x ceil(K/32), row pitch
    ld_sfa) and SFB (N x ceil(K/32), ld_sfb) as uint8, C in `dtype`.  Returns (ref, sumabs)
    like ``gemm``."""
    A = _bits(A)
    B = _bits(B)
    SFA = np.ascontiguousarray(SFA, dtype=np.uint8)
    SFB = np.ascontiguousarray(SFB, dtype=np.uint8)
    Cp = None
    if C is not None:
        C = _bits(C)
        Cp = C.ctypes.data
    if rows is None:
        n = M * N
        r_p = c_p = None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        n = rows.size
        r_p, c_p = rows.ctypes.data, cols.ctypes.data
    ref = np.empty(n, dtype=np.float64)
    sab = np.empty(n, dtype=np.float64)
    rc = _load().oracle_gemm_mx(M, N, K, float(alpha), A.ctypes.data, lda, a_dtype, SFA.ctypes.data,
                                ld_sfa, B.ctypes.data, ldb, b_dtype, SFB.ctypes.data, ld_sfb,
                                float(beta), Cp, ldc, dtype, r_p, c_p, n, ref.ctypes.data,
                                sab.ctypes.data, threads)
    if rc != 0:
        raise ValueError("oracle_gemm_mx rejected its arguments")
    if rows is None:
        return ref.reshape(M, N), sab.reshape(M, N)
    return ref, sab


def gelu(v):
    """GELU in its erf form, 0.5 v (1 + erf(v / sqrt 2)), in float64."""
    from scipy.special import erf
    v = np.asarray(v, dtype=np.float64)
    return 0.5 * v * (1.0 + erf(v / math.sqrt(2.0)))


def fused(ref, bias_cols=None, activation="none"):
    """The fused epilogue after alpha*acc + beta*c ("CUTLASS, in depth", "Epilogue fusion"):
    add the column's bias, then activate.  ref is (M, N) or per-entry with bias_cols given per
    entry."""
    v = np.asarray(ref, dtype=np.float64)
    if bias_cols is not None:
        v = v + bias_cols
    if activation == "relu":
        v = np.maximum(v, 0.0)
    elif activation == "gelu":
        v = gelu(v)
    return v


# Largest Lipschitz constant of the activations (bounds how accumulated error propagates):
# ReLU 1; GELU max |d/dv| = 1.1289 (at v = +-sqrt(2)).
LIPSCHITZ = {"none": 1.0, "relu": 1.0, "gelu": 1.13}


def ulp_fp8(dtype, r):
    """Spacing of an FP8 format at |r| (subnormal spacing near zero)."""
    r = np.abs(np.asarray(r, dtype=np.float64))
    emin, frac = (-6, 3) if dtype == E4M3 else (-14, 2)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    e = np.where(r > 0, np.maximum(e, emin), emin)
    return np.ldexp(1.0, (e - frac).astype(np.int64))


def ulp_out(dtype, r):
    """Spacing of the output format at |r| (the smallest subnormal spacing near zero)."""
    r = np.abs(np.asarray(r, dtype=np.float64))
    if dtype == F16:
        emin, frac = -14, 10
    else:
        emin, frac = -126, 7
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    e = np.where(r > 0, np.maximum(e, emin), emin)
    return np.ldexp(1.0, (e - frac).astype(np.int64))


def bound(dtype, alpha, beta, ref, sumabs, c_values=None):
    """Acceptance bound 2^-9 (|alpha| S + |beta c|) + ulp_out(ref)."""
    t = abs(alpha) * np.asarray(sumabs, dtype=np.float64)
    if c_values is not None and beta != 0:
        t = t + np.abs(beta * np.asarray(c_values, dtype=np.float64))
    return math.ldexp(1.0, -9) * t + ulp_out(dtype, ref)
