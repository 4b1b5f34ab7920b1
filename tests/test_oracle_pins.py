"""Pins for the CPU oracle and the seeded generator (no GPU).

Every check here ties the oracle to something other than itself: exact
rational arithmetic by brute force, matrices whose product is known by
construction (identity, permutation, single entry, small integers), the
alpha=0 / beta=0 / K=0 closed forms, numpy.matmul, and the algebraic
checksum and Freivalds identities.  The last group plants mistakes in the
oracle's output or inputs and checks that the pins notice.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, dtype=np.float32):
    return synthetic.uniform(seed, 1, shape, dtype=dtype)


def _exact(A, B, C0, alpha, beta):
    """Exact rational alpha*A*B + beta*C0 (pure Python, tiny sizes only)."""
    M, K = A.shape
    N = B.shape[1]
    fa = [[Fraction(float(A[i, k])) for k in range(K)] for i in range(M)]
    fb = [[Fraction(float(B[k, j])) for j in range(N)] for k in range(K)]
    al, be = Fraction(alpha), Fraction(beta)
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = sum((fa[i][k] * fb[k][j] for k in range(K)), Fraction(0))
            v = al * s
            if beta != 0:
                v += be * Fraction(float(C0[i, j]))
            row.append(v)
        out.append(row)
    return out


# ---------------------------------------------------------------- generator

def test_splitmix64_published_vector():
    want = [int(l) for l in open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt"))
            if l.strip() and not l.startswith("#")]
    got = synthetic.splitmix64(1234567, 5)
    assert [int(x) for x in got] == want


def test_splitmix64_counter_based():
    full = synthetic.splitmix64(99, 1000)
    part = synthetic.splitmix64(99, 100, offset=450)
    assert np.array_equal(full[450:550], part)


def test_uniform_range_and_rounding_chain():
    u32 = synthetic.uniform(5, 1, (257, 129))
    assert u32.dtype == np.float32 and u32.min() >= -1.0 and u32.max() < 1.0
    u16 = synthetic.uniform(5, 1, (257, 129), dtype=np.float16)
    assert np.array_equal(u16, u32.astype(np.float16))
    # different streams differ, same stream repeats
    assert not np.array_equal(u32, synthetic.uniform(5, 2, (257, 129)))
    assert np.array_equal(u32, synthetic.uniform(5, 1, (257, 129)))
    # mean and variance of U(-1,1): 0 and 1/3
    assert abs(float(u32.mean())) < 0.02 and abs(float(u32.var()) - 1 / 3) < 0.02


def test_normal_moments():
    z = synthetic.normal(3, 1, (200000,))
    assert abs(float(z.mean())) < 0.01 and abs(float(z.std()) - 1.0) < 0.01


def test_padded_sentinel():
    buf = synthetic.padded(1, 1, 5, 7, 10, np.float16)
    assert buf.shape == (5, 10) and np.isnan(buf[:, 7:]).all() and np.isfinite(buf[:, :7]).all()


# ---------------------------------------------------------------- oracle core

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (7, 3, 5), (4, 9, 2), (6, 6, 11)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, 0.5), (-0.75, -0.25), (2.0, 1.0)])
def test_exact_rational_brute_force(M, N, K, alpha, beta):
    A = _rand((M, K), 10 + M)
    B = synthetic.uniform(20 + N, 2, (K, N))
    C0 = synthetic.uniform(30 + K, 3, (M, N))
    ref = oracle.gemm(A, B, C0, alpha, beta)
    exact = _exact(A, B, C0, alpha, beta)
    for i in range(M):
        for j in range(N):
            scale = abs(alpha) * sum(abs(float(A[i, k]) * float(B[k, j])) for k in range(K)) + abs(beta) * abs(float(C0[i, j]))
            assert abs(ref[i, j] - float(exact[i][j])) <= 1e-14 * max(scale, 1e-300)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (2.0, -1.0)])
def test_small_integer_exact(alpha, beta):
    rng = np.random.default_rng(0)
    M, N, K = 17, 23, 64
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float16)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float16)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float16)
    ref = oracle.gemm(A, B, C0, alpha, beta)
    Ai = A.astype(np.int64)
    Bi = B.astype(np.int64)
    want = [[int(alpha) * sum(int(Ai[i, k]) * int(Bi[k, j]) for k in range(K)) + int(beta) * int(C0[i, j])
             for j in range(N)] for i in range(M)]
    assert np.array_equal(ref, np.array(want, dtype=np.float64))


def test_identity_gives_alpha_B():
    K = N = 40
    A = np.eye(K, dtype=np.float16)
    B = synthetic.uniform(1, 2, (K, N), dtype=np.float16)
    ref = oracle.gemm(A, B, None, 1.5, 0.0)
    assert np.array_equal(ref, 1.5 * B.astype(np.float64))


def test_permutation_permutes_rows():
    rng = np.random.default_rng(1)
    K, N = 33, 19
    p = rng.permutation(K)
    A = np.zeros((K, K), np.float32)
    A[np.arange(K), p] = 1.0
    B = synthetic.uniform(2, 2, (K, N))
    ref = oracle.gemm(A, B, None, 1.0, 0.0)
    assert np.array_equal(ref, B[p].astype(np.float64))


@pytest.mark.parametrize("i0,k0,j0", [(0, 0, 0), (4, 2, 6), (6, 8, 1)])
def test_single_entry(i0, k0, j0):
    M, N, K = 7, 9, 11
    A = np.zeros((M, K), np.float32)
    B = np.zeros((K, N), np.float32)
    A[i0, k0] = 3.0
    B[k0, j0] = -0.5
    ref = oracle.gemm(A, B, None, 2.0, 0.0)
    want = np.zeros((M, N))
    want[i0, j0] = -3.0
    assert np.array_equal(ref, want)


def test_alpha_zero_is_beta_C_and_ignores_AB():
    M, N, K = 9, 13, 5
    A = np.full((M, K), np.nan, np.float32)
    B = np.full((K, N), np.nan, np.float32)
    C0 = synthetic.uniform(4, 3, (M, N), dtype=np.float16)
    ref = oracle.gemm(A, B, C0, 0.0, -0.25)
    assert np.array_equal(ref, -0.25 * C0.astype(np.float64))


def test_beta_zero_ignores_C():
    M, N, K = 9, 13, 5
    A = synthetic.uniform(5, 1, (M, K))
    B = synthetic.uniform(5, 2, (K, N))
    C0 = np.full((M, N), np.nan, np.float32)
    ref = oracle.gemm(A, B, C0, 0.75, 0.0)
    assert np.isfinite(ref).all()
    assert np.array_equal(ref, oracle.gemm(A, B, None, 0.75, 0.0))


def test_K_zero_is_beta_C():
    M, N = 6, 4
    C0 = synthetic.uniform(6, 3, (M, N))
    ref = oracle.gemm(np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), C0, 1.5, 0.5, K=0)
    assert np.array_equal(ref, 0.5 * C0.astype(np.float64))


def test_leading_dimensions_with_sentinels():
    M, N, K = 11, 13, 9
    lda, ldb, ldc = K + 3, N + 5, N + 1
    Ap = synthetic.padded(7, 1, M, K, lda, np.float16)
    Bp = synthetic.padded(7, 2, K, N, ldb, np.float16)
    Cp = synthetic.padded(7, 3, M, N, ldc, np.float16)
    got = oracle.gemm(Ap.reshape(-1), Bp.reshape(-1), Cp.reshape(-1), 0.75, -0.25,
                      M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc)
    want = oracle.gemm(Ap[:, :K].copy(), Bp[:, :N].copy(), Cp[:, :N].copy(), 0.75, -0.25)
    assert np.isfinite(got).all() and np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(64, 64, 64), (33, 17, 50), (1, 64, 7)])
def test_against_numpy_matmul(M, N, K):
    A = synthetic.uniform(8, 1, (M, K), dtype=np.float16)
    B = synthetic.uniform(8, 2, (K, N), dtype=np.float16)
    C0 = synthetic.uniform(8, 3, (M, N), dtype=np.float16)
    ref, absd = oracle.gemm(A, B, C0, 1.5, 0.5, with_absdot=True)
    a = A.astype(np.float64)
    b = B.astype(np.float64)
    lib = 1.5 * (a @ b) + 0.5 * C0.astype(np.float64)
    scale = 1.5 * (np.abs(a) @ np.abs(b)) + 0.5 * np.abs(C0.astype(np.float64))
    assert np.all(np.abs(ref - lib) <= 1e-12 * scale + 1e-300)
    assert np.allclose(absd, np.abs(a) @ np.abs(b), rtol=1e-12, atol=0)


def test_row_subset_matches_full():
    M, N, K = 50, 21, 30
    A = synthetic.uniform(9, 1, (M, K))
    B = synthetic.uniform(9, 2, (K, N))
    C0 = synthetic.uniform(9, 3, (M, N))
    full = oracle.gemm(A, B, C0, 1.5, 0.5)
    rows = [0, 7, 49, 13]
    assert np.array_equal(oracle.gemm(A, B, C0, 1.5, 0.5, rows=rows), full[rows])


def test_column_subset_matches_full():
    M, N, K = 20, 37, 15
    A = synthetic.uniform(10, 1, (M, K))
    B = synthetic.uniform(10, 2, (K, N))
    C0 = synthetic.uniform(10, 3, (M, N))
    full = oracle.gemm(A, B, C0, 0.75, -0.25)
    cols = [0, 5, 36, 11]
    assert np.array_equal(oracle.gemm_cols(A, B, C0, 0.75, -0.25, cols), full[:, cols])


def test_thread_count_does_not_change_result():
    M, N, K = 64, 48, 80
    A = synthetic.uniform(11, 1, (M, K))
    B = synthetic.uniform(11, 2, (K, N))
    n0 = oracle.max_threads()
    try:
        oracle.set_threads(1)
        one = oracle.gemm(A, B, None, 1.0, 0.0)
        oracle.set_threads(max(2, n0))
        many = oracle.gemm(A, B, None, 1.0, 0.0)
    finally:
        oracle.set_threads(n0)
    assert np.array_equal(one, many)


# ---------------------------------------------------------------- whole-matrix identities

def test_checksum_identity():
    M, N, K = 70, 45, 33
    A = synthetic.uniform(12, 1, (M, K), dtype=np.float16)
    B = synthetic.uniform(12, 2, (K, N), dtype=np.float16)
    C0 = synthetic.uniform(12, 3, (M, N), dtype=np.float16)
    ref = oracle.gemm(A, B, C0, 1.5, 0.5)
    s, scale = oracle.checksum_closed_form(A, B, C0, 1.5, 0.5, M, N, K)
    assert abs(oracle.checksum(ref) - s) <= 1e-12 * scale
    assert abs(float(np.sum(ref, dtype=np.float64)) - s) <= 1e-12 * scale


def test_freivalds_identity():
    M, N, K = 40, 31, 27
    A = synthetic.uniform(13, 1, (M, K))
    B = synthetic.uniform(13, 2, (K, N))
    C0 = synthetic.uniform(13, 3, (M, N))
    x = np.where(synthetic.uniform(13, 4, (N,)) > 0, 1.0, -1.0)
    ref = oracle.gemm(A, B, C0, 0.75, -0.25)
    y, ya = oracle.freivalds_rhs(A, B, C0, 0.75, -0.25, x, M, N, K)
    assert np.all(np.abs(ref @ x - y) <= 1e-12 * ya)


# ---------------------------------------------------------------- tolerances

def test_ulp16_matches_numpy_spacing():
    vals = np.array([1.0, 1.5, 2.0, 3.0, 32768.0, 2.0 ** -14, 0.1, 1000.0], dtype=np.float16)
    assert np.array_equal(oracle.ulp16(vals.astype(np.float64)), np.spacing(vals).astype(np.float64))
    # the largest finite half (numpy's spacing there overflows to inf): binade [2^15, 2^16) -> 32
    assert oracle.ulp16(65504.0) == 32.0
    assert oracle.ulp16(0.0) == 2.0 ** -24 and oracle.ulp16(2.0 ** -20) == 2.0 ** -24


def test_ulp32_matches_numpy_spacing():
    vals = np.array([1.0, 3.0, 1e-3, 12345.678, 2.0 ** -126], dtype=np.float32)
    assert np.array_equal(oracle.ulp32(vals.astype(np.float64)), np.spacing(vals).astype(np.float64))


def test_half_rounding_is_nearest_even():
    # ties go to the even neighbour: 1 + 2^-11 -> 1, 1 + 3*2^-11 -> 1 + 2^-9
    x = np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, -(1 + 2.0 ** -11)], dtype=np.float32)
    assert list(x.astype(np.float16).astype(np.float64)) == [1.0, 1 + 2.0 ** -9, -1.0]


def test_tol_f16_accepts_rounded_reference():
    M, N, K = 32, 32, 64
    A = synthetic.uniform(14, 1, (M, K), dtype=np.float16)
    B = synthetic.uniform(14, 2, (K, N), dtype=np.float16)
    C0 = synthetic.uniform(14, 3, (M, N), dtype=np.float16)
    ref, absd = oracle.gemm(A, B, C0, 1.5, 0.5, with_absdot=True)
    rounded = ref.astype(np.float16).astype(np.float64)
    assert oracle.compare(rounded, ref, oracle.tol_f16(ref, absd))["ok"]


def test_tol_f16_f32out_is_the_fp16_bound_with_binary32_rounding():
    ref = np.array([1.0, -3.0, 1000.0, 0.0])
    absd = np.array([10.0, 0.0, 5.0, 0.0])
    want = 2e-3 * absd + np.array([2.0 ** -23, 2.0 ** -22, 2.0 ** -14, 2.0 ** -149])
    assert np.array_equal(oracle.tol_f16_f32out(ref, absd), want)


# ---------------------------------------------------------------- float -> half rounding

def test_f32_to_f16_worked_values():
    """IEEE binary16 facts: the largest finite half is 65504 (0x7BFF); values
    at or beyond 65520 (halfway to the next binade step) overflow to Inf; the
    smallest subnormal is 2^-24 (0x0001); ties round to the even neighbour
    (2049 -> 2048, 2051 -> 2052 = 0x6802 since the spacing above 2048 is 2,
    2^-25 -> 0, 3*2^-25 -> 2*2^-24)."""
    cases = [
        (1.0 / 3.0, 0x3555), (1.0, 0x3C00), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
        (65504.0, 0x7BFF), (65519.0, 0x7BFF), (65520.0, 0x7C00), (-1e6, 0xFC00),
        (2049.0, 0x6800), (2051.0, 0x6802), (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000),
        (3 * 2.0 ** -25, 0x0002), (2.0 ** -14, 0x0400), (float("inf"), 0x7C00),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    got = oracle.f32_to_f16(x).view(np.uint16)
    assert [int(v) for v in got] == [c[1] for c in cases]
    assert np.isnan(oracle.f32_to_f16(np.array([np.nan], np.float32))).all()


# ---------------------------------------------------------------- planted mistakes

def test_compare_flags_planted_error_and_nan():
    ref = np.linspace(-1, 1, 64).reshape(8, 8)
    tol = np.full_like(ref, 1e-3)
    bad = ref.copy()
    bad[3, 5] += 2.5e-3
    r = oracle.compare(bad, ref, tol)
    assert not r["ok"] and r["n_bad"] == 1 and tuple(r["worst_index"]) == (3, 5)
    bad = ref.copy()
    bad[0, 0] = np.nan
    assert not oracle.compare(bad, ref, tol)["ok"]


@pytest.mark.parametrize("mistake", ["transpose_B", "drop_beta", "flip_alpha", "shift_k"])
def test_pins_catch_planted_oracle_mistakes(mistake):
    """Run the oracle with one plausible mistake planted in how it is called
    and check that the exact brute force disagrees."""
    M, N, K = 5, 5, 5
    A = _rand((M, K), 40)
    B = synthetic.uniform(41, 2, (K, N))
    C0 = synthetic.uniform(42, 3, (M, N))
    alpha, beta = 1.5, 0.5
    if mistake == "transpose_B":
        got = oracle.gemm(A, np.ascontiguousarray(B.T), C0, alpha, beta)
    elif mistake == "drop_beta":
        got = oracle.gemm(A, B, C0, alpha, 0.0)
    elif mistake == "flip_alpha":
        got = oracle.gemm(A, B, C0, -alpha, beta)
    else:  # A read one column off (index slip in k)
        got = oracle.gemm(np.roll(A, 1, axis=1), B, C0, alpha, beta)
    exact = np.array([[float(v) for v in row] for row in _exact(A, B, C0, alpha, beta)])
    assert np.max(np.abs(got - exact)) > 1e-6
