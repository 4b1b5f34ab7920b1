"""CPU oracle for C := alpha*A*B + beta*C (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the bench are the only callers.  Nothing in the CUDA library imports,
links or runs this package, and this package imports nothing from it.

The arithmetic lives in ``gemm_oracle.c`` (plain triple loop, double, k
ascending).  This module builds and loads it, widens half operands to float32
(exact), holds the parity tolerances, and gives the float-to-half rounding
that the conversion entry point must reproduce bit for bit:

* fp16 path: |gpu - ref| <= 2e-3 * sum_k |a_ik||b_kj| + ulp16(ref), per element;
* fp16 operands with an fp32 C: the same bound with the output rounding term
  of binary32, 2e-3 * sum_k |a_ik||b_kj| + ulp32(ref);
* fp32 path: |gpu - ref| <= 1e-6 * K * max|A| * max|B|, per element, with the
  maxima over the whole matrices (the bound exactly as stated, no extra term).

ulp16/ulp32 are the spacings of binary16/binary32 at |ref| (the subnormal
spacing below the smallest normal).

Pins (tests/test_oracle_pins.py) tie every function here to something other
than itself: exact rational brute force, identity/permutation/single-entry
matrices, the alpha=0 / beta=0 / K=0 closed forms, numpy.matmul, and the
algebraic checksum and Freivalds identities.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_gemm.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                _fp, ctypes.c_long, _fp, ctypes.c_long,
                ctypes.c_double, _fp, ctypes.c_long,
                _dp, _dp, ctypes.c_long, _ip, ctypes.c_int]
            lib.oracle_sum_f64.restype = ctypes.c_double
            lib.oracle_sum_f64.argtypes = [ctypes.c_int, ctypes.c_int, _dp, ctypes.c_long]
            lib.oracle_sum_f32.restype = ctypes.c_double
            lib.oracle_sum_f32.argtypes = [ctypes.c_int, ctypes.c_int, _fp, ctypes.c_long]
            lib.oracle_checksum_closed_form.restype = ctypes.c_double
            lib.oracle_checksum_closed_form.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                _fp, ctypes.c_long, _fp, ctypes.c_long,
                ctypes.c_double, _fp, ctypes.c_long, _dp]
            lib.oracle_freivalds_rhs.restype = None
            lib.oracle_freivalds_rhs.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                _fp, ctypes.c_long, _fp, ctypes.c_long,
                ctypes.c_double, _fp, ctypes.c_long, _dp, _dp, _dp]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def max_threads() -> int:
    return _load().oracle_max_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def _as_f32(x, rows: int, ld: int) -> np.ndarray:
    """Widen to a float32 row-major buffer with at least rows*ld... elements."""
    if x is None:
        return None
    a = np.asarray(x)
    if a.dtype == np.float16:
        a = a.astype(np.float32)          # exact: every binary16 is a binary32
    elif a.dtype != np.float32:
        raise TypeError("oracle inputs are float16 or float32, got %s" % a.dtype)
    return np.ascontiguousarray(a).reshape(-1)


def _ptr(a, t):
    return None if a is None else a.ctypes.data_as(t)


def _check_extent(name, buf, rows, cols, ld):
    if rows == 0 or cols == 0:
        return
    need = (rows - 1) * ld + cols
    if buf is None or buf.size < need:
        raise ValueError("%s: buffer of %s elements, need %d" % (name, None if buf is None else buf.size, need))


def gemm(A, B, C0, alpha: float, beta: float, M: int = None, N: int = None, K: int = None,
         lda: int = None, ldb: int = None, ldc: int = None, rows=None, with_absdot: bool = False):
    """Unrounded double result of alpha*A*B + beta*C0.

    ``A``, ``B``, ``C0`` are row-major arrays (float16 or float32); either 2-D
    with the natural leading dimension or flat buffers with explicit ld.  With
    ``rows`` (a list of row indices) only those rows are computed.
    Returns ``out`` (and ``absdot`` = sum_k |a||b| when asked), each
    ``len(rows) x N`` (or ``M x N``).
    """
    A_ = np.asarray(A) if A is not None else None
    B_ = np.asarray(B) if B is not None else None
    if M is None:
        M = A_.shape[0]
    if K is None:
        K = A_.shape[1] if A_ is not None and A_.ndim == 2 else 0
    if N is None:
        N = B_.shape[1]
    lda = lda if lda is not None else (A_.shape[1] if A_ is not None and A_.ndim == 2 else K)
    ldb = ldb if ldb is not None else (B_.shape[1] if B_ is not None and B_.ndim == 2 else N)
    ldc = ldc if ldc is not None else (np.asarray(C0).shape[1] if C0 is not None and np.asarray(C0).ndim == 2 else N)
    a = _as_f32(A, M, lda)
    b = _as_f32(B, K, ldb)
    c = _as_f32(C0, M, ldc)
    read_ab = alpha != 0.0 and K > 0
    if read_ab:
        _check_extent("A", a, M, K, lda)
        _check_extent("B", b, K, N, ldb)
    if beta != 0.0:
        _check_extent("C0", c, M, N, ldc)
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        if rows_arr.size and (rows_arr.min() < 0 or rows_arr.max() >= M):
            raise ValueError("row index out of range")
        R = rows_arr.size
    else:
        rows_arr = None
        R = M
    out = np.zeros((R, N), dtype=np.float64)
    absd = np.zeros((R, N), dtype=np.float64) if with_absdot else None
    dummy = np.zeros(1, dtype=np.float32)
    rc = _load().oracle_gemm(
        int(M), int(N), int(K), float(alpha),
        _ptr(a if a is not None else dummy, _fp), int(lda),
        _ptr(b if b is not None else dummy, _fp), int(ldb),
        float(beta), _ptr(c if c is not None else dummy, _fp), int(ldc),
        _ptr(out, _dp), _ptr(absd, _dp) if absd is not None else None, int(N),
        _ptr(rows_arr, _ip) if rows_arr is not None else None, int(R))
    if rc != 0:
        raise MemoryError("oracle_gemm could not allocate its row buffers")
    return (out, absd) if with_absdot else out


def gemm_cols(A, B, C0, alpha, beta, cols, M=None, N=None, K=None, lda=None, ldb=None, ldc=None,
              with_absdot: bool = False):
    """Columns ``cols`` of the result (an M x len(cols) array), computed by the
    same definition on B and C0 restricted to those columns."""
    A_ = np.asarray(A)
    if M is None:
        M = A_.shape[0]
    if K is None:
        K = A_.shape[1]
    Bm = np.asarray(B).reshape(-1)
    ldb = ldb if ldb is not None else (np.asarray(B).shape[1] if np.asarray(B).ndim == 2 else N)
    cols = np.asarray(cols, dtype=np.int64)
    Bsub = np.stack([Bm[k * ldb + cols] for k in range(K)]) if K > 0 else np.zeros((0, cols.size), Bm.dtype)
    Csub = None
    if C0 is not None and beta != 0.0:
        Cm = np.asarray(C0).reshape(-1)
        ldc = ldc if ldc is not None else (np.asarray(C0).shape[1] if np.asarray(C0).ndim == 2 else N)
        Csub = np.stack([Cm[i * ldc + cols] for i in range(M)])
    return gemm(A, Bsub, Csub, alpha, beta, M=M, N=cols.size, K=K, lda=lda,
                ldb=cols.size, ldc=cols.size, with_absdot=with_absdot)


# ----------------------------------------------------------------------------
# Tolerances
# ----------------------------------------------------------------------------

def ulp16(x) -> np.ndarray:
    """Spacing of binary16 numbers at |x|: 2^(floor(log2|x|) - 10) for normal
    magnitudes (|x| >= 2^-14), the subnormal spacing 2^-24 below."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax >= 2.0 ** -14, ax, 1.0)))
    return np.where(ax >= 2.0 ** -14, np.exp2(e - 10.0), 2.0 ** -24)


def ulp32(x) -> np.ndarray:
    """Spacing of binary32 numbers at |x| (2^-149 below the smallest normal)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax >= 2.0 ** -126, ax, 1.0)))
    return np.where(ax >= 2.0 ** -126, np.exp2(e - 23.0), 2.0 ** -149)


def tol_f16(ref, absdot) -> np.ndarray:
    return 2e-3 * np.asarray(absdot, dtype=np.float64) + ulp16(ref)


def tol_f32(ref, K: int, max_a: float, max_b: float) -> np.ndarray:
    """1e-6 * K * max|A| * max|B| for every element of ``ref`` (broadcast to
    its shape)."""
    return np.broadcast_to(np.float64(1e-6 * float(K) * float(max_a) * float(max_b)),
                           np.shape(ref))


def tol_f16_f32out(ref, absdot) -> np.ndarray:
    return 2e-3 * np.asarray(absdot, dtype=np.float64) + ulp32(ref)


def f32_to_f16(x) -> np.ndarray:
    """binary32 -> binary16, round to nearest with ties to even, overflow to
    +-Inf, NaN to NaN (IEEE 754 conversion; numpy's cast implements it).
    The float-to-half kernel of the "Tensorcore_wmma_vs_fp32 test code" page
    (section on the float - half conversion kernel) applies __float2half,
    which rounds the same way."""
    with np.errstate(over="ignore", invalid="ignore"):   # overflow to Inf is the rule
        return np.asarray(x, dtype=np.float32).astype(np.float16)


def compare(got, ref, tol):
    """Elementwise |got - ref| <= tol.  Returns a dict with ``ok``, the worst
    ratio err/tol, its index, and diagnostics."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    t = np.broadcast_to(np.asarray(tol, dtype=np.float64), r.shape)
    if g.shape != r.shape:
        raise ValueError("shape mismatch %s vs %s" % (g.shape, r.shape))
    err = np.abs(g - r)
    bad = ~(err <= t)                      # NaN in got -> bad
    ratio = np.where(t > 0, err / np.where(t > 0, t, 1.0), np.where(err > 0, np.inf, 0.0))
    ratio = np.where(np.isnan(ratio), np.inf, ratio)
    worst = int(np.argmax(ratio)) if ratio.size else 0
    return {
        "ok": not bool(bad.any()),
        "n_bad": int(bad.sum()),
        "max_ratio": float(ratio.reshape(-1)[worst]) if ratio.size else 0.0,
        "worst_index": np.unravel_index(worst, r.shape) if ratio.size else None,
        "max_abs_err": float(err.max()) if err.size else 0.0,
    }


def f16_diagnostics(got, ref) -> dict:
    """Non-gating: error in units of the fp16 spacing, and the share of
    outputs equal to ref rounded once to fp16."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    rn = r.astype(np.float16).astype(np.float64)
    ulps = np.abs(g - r) / ulp16(r)
    return {"max_ulp16": float(ulps.max()) if ulps.size else 0.0,
            "frac_equal_rn16": float((g == rn).mean()) if g.size else 1.0}


# ----------------------------------------------------------------------------
# Whole-matrix properties for sizes too large to recompute in full
# ----------------------------------------------------------------------------

def checksum(X) -> float:
    """Double-precision sum of all elements (rows, then columns, ascending)."""
    x = np.asarray(X)
    if x.dtype == np.float16:
        x = x.astype(np.float32)
    x = np.ascontiguousarray(x)
    M, N = x.shape
    if x.dtype == np.float32:
        return float(_load().oracle_sum_f32(M, N, x.ctypes.data_as(_fp), N))
    x = x.astype(np.float64, copy=False)
    return float(_load().oracle_sum_f64(M, N, x.ctypes.data_as(_dp), N))


def checksum_closed_form(A, B, C0, alpha, beta, M, N, K, lda=None, ldb=None, ldc=None):
    """(sum, scale): alpha*sum_k colsum(A)_k*rowsum(B)_k + beta*sum(C0), and the
    same with absolute values (scale for an error bound)."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    a = _as_f32(A, M, lda)
    b = _as_f32(B, K, ldb)
    c = _as_f32(C0, M, ldc) if C0 is not None else np.zeros(1, np.float32)
    bound = ctypes.c_double(0.0)
    s = _load().oracle_checksum_closed_form(
        int(M), int(N), int(K), float(alpha), a.ctypes.data_as(_fp), int(lda),
        b.ctypes.data_as(_fp), int(ldb), float(beta), c.ctypes.data_as(_fp), int(ldc),
        ctypes.byref(bound))
    return float(s), float(bound.value)


def freivalds_rhs(A, B, C0, alpha, beta, x, M, N, K, lda=None, ldb=None, ldc=None):
    """(y, yabs) with y = alpha*A(Bx) + beta*C0 x for a length-N vector x."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    a = _as_f32(A, M, lda) if K > 0 else np.zeros(1, np.float32)
    b = _as_f32(B, K, ldb) if K > 0 else np.zeros(1, np.float32)
    c = _as_f32(C0, M, ldc) if C0 is not None else np.zeros(1, np.float32)
    xv = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.zeros(M, np.float64)
    ya = np.zeros(M, np.float64)
    _load().oracle_freivalds_rhs(
        int(M), int(N), int(K), float(alpha), a.ctypes.data_as(_fp), int(lda),
        b.ctypes.data_as(_fp), int(ldb), float(beta), c.ctypes.data_as(_fp), int(ldc),
        xv.ctypes.data_as(_dp), y.ctypes.data_as(_dp), ya.ctypes.data_as(_dp))
    return y, ya


def sample_rows(M: int, block: int = 128, extra: int = 8, seed: int = 7):
    """Row indices to check at sizes too large for the full oracle: one seeded
    row inside every block of ``block`` rows (so every output tile row-band is
    visited), the first and last rows, and ``extra`` more seeded rows."""
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    for start in range(0, M, block):
        rows.add(int(rng.integers(start, min(M, start + block))))
    for r in rng.integers(0, M, size=extra):
        rows.add(int(r))
    return sorted(rows)


def sample_cols(N: int, block: int = 64, extra: int = 8, seed: int = 11):
    """Column indices: one seeded column per ``block`` columns, the first and
    last columns, and ``extra`` more."""
    return sample_rows(N, block=block, extra=extra, seed=seed)
