"""Shared helpers for the GPU parity tests: move seeded host operands to the
device, call the library through its C ABI, bring C back, and compare with
the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np

import oracle
import synthetic

F16_SENTINEL = np.uint16(0x7E55)   # a quiet NaN pattern for padding that must stay untouched
F32_SENTINEL = np.uint32(0x7FC0DEAD)


def torch():
    import torch as t
    return t


def to_dev(x: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(x)).cuda()


def operands(seed, M, N, K, lda, ldb, ldc, dtype, dist="uniform", c_fill="uniform"):
    """Seeded A, B, C0 as flat row-major buffers with their leading dimensions.
    Padding columns hold a NaN sentinel."""
    rows_a, rows_b = M, K
    A = synthetic.padded(seed, synthetic.STREAM_A, rows_a, K, lda, dtype, dist=dist)
    B = synthetic.padded(seed, synthetic.STREAM_B, rows_b, N, ldb, dtype, dist=dist)
    if c_fill == "nan":
        C0 = np.full((M, ldc), np.nan, dtype=dtype)
    elif c_fill == "zero":
        C0 = np.zeros((M, ldc), dtype=dtype)
        if ldc > N:
            C0[:, N:] = np.nan
    else:
        C0 = synthetic.padded(seed, synthetic.STREAM_C, M, N, ldc, dtype, dist=dist)
    if ldc > N:
        if dtype == np.float16:
            C0.view(np.uint16)[:, N:] = F16_SENTINEL
        else:
            C0.view(np.uint32)[:, N:] = F32_SENTINEL
    return A, B, C0


def run(kind, A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, path=0, splits=0, stream=None):
    """One call through the C ABI on device copies; returns C as a host array
    shaped like C0 and the path the library reports."""
    import dense_gemm_03_gb300 as g
    t = torch()
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C0)
    prev_p = g.force_path(path)
    prev_s = g.force_splits(splits)
    try:
        fn = g.gemm_f16 if kind == "f16" else g.sgemm_f32
        fn(dA, dB, dC, alpha, beta, M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc, stream=stream)
        taken = g.last_path()
    finally:
        g.force_path(prev_p)
        g.force_splits(prev_s)
    t.cuda.synchronize()
    assert g.debug_status() == 0, "a kernel reported a timeout"
    return dC.cpu().numpy().reshape(C0.shape), taken


def check(kind, got, A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, rows=None, cols=None):
    """Elementwise comparison with the oracle (all of C, or the given rows and
    columns).  Returns the comparison record; asserts on failure."""
    view = got[:, :N].astype(np.float64)
    kw = dict(M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc)
    recs = []
    if kind == "f16":
        if rows is None and cols is None:
            ref, absd = oracle.gemm(A, B, C0, alpha, beta, with_absdot=True, **kw)
            recs.append(("all", oracle.compare(view, ref, oracle.tol_f16(ref, absd))))
        else:
            if rows is not None:
                ref, absd = oracle.gemm(A, B, C0, alpha, beta, rows=rows, with_absdot=True, **kw)
                recs.append(("rows", oracle.compare(view[rows], ref, oracle.tol_f16(ref, absd))))
            if cols is not None:
                ref, absd = oracle.gemm_cols(A, B, C0, alpha, beta, cols, with_absdot=True, **kw)
                recs.append(("cols", oracle.compare(view[:, cols], ref, oracle.tol_f16(ref, absd))))
    else:
        amax = float(np.nanmax(np.abs(_valid(A, M, K, lda)))) if M and K else 0.0
        bmax = float(np.nanmax(np.abs(_valid(B, K, N, ldb)))) if K and N else 0.0
        if rows is None and cols is None:
            ref = oracle.gemm(A, B, C0, alpha, beta, **kw)
            recs.append(("all", oracle.compare(view, ref, oracle.tol_f32(ref, K, amax, bmax))))
        else:
            if rows is not None:
                ref = oracle.gemm(A, B, C0, alpha, beta, rows=rows, **kw)
                recs.append(("rows", oracle.compare(view[rows], ref, oracle.tol_f32(ref, K, amax, bmax))))
            if cols is not None:
                ref = oracle.gemm_cols(A, B, C0, alpha, beta, cols, **kw)
                recs.append(("cols", oracle.compare(view[:, cols], ref, oracle.tol_f32(ref, K, amax, bmax))))
    for name, r in recs:
        assert r["ok"], "%s: %d elements out of tolerance, worst %s at %s (abs err %g)" % (
            name, r["n_bad"], r["max_ratio"], r["worst_index"], r["max_abs_err"])
    return recs


def _valid(X, rows, cols, ld):
    return np.asarray(X).reshape(-1)[: rows * ld].reshape(rows, ld)[:, :cols]


def padding_untouched(got, C0, N):
    """Columns beyond N of a padded C must keep their sentinel bits."""
    if got.shape[1] == N:
        return True
    bits = np.uint16 if got.dtype == np.float16 else np.uint32
    return np.array_equal(got.view(bits)[:, N:], C0.view(bits)[:, N:])
