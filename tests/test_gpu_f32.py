"""Parity of the fp32 SGEMM path (sgemm_f32 / sgemm_f32_ld) with the CPU
oracle, through the C ABI: vectorised and predicated-scalar kernels."""
import numpy as np
import pytest

import oracle
from helpers import check, operands, padding_untouched, run

pytestmark = pytest.mark.gpu

AUTO, SCALAR = 0, 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_03_gb300 import build
    build.build()


@pytest.mark.parametrize("path", [AUTO, SCALAR])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (129, 257, 65), (1, 1, 1), (300, 700, 1000),
                                   (128, 128, 8), (5, 300, 9)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (2.0, -1.0)])
def test_small_integers_bit_exact(path, M, N, K, alpha, beta):
    rng = np.random.default_rng(M + 11 * N + 101 * K)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    got, taken = run("f32", A, B, C0, alpha, beta, M, N, K, K, N, N, path=path)
    if path == SCALAR:
        assert taken == "f32.ffma.scalar"
    ref = oracle.gemm(A, B, C0, alpha, beta)
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("path", [AUTO, SCALAR])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (129, 257, 65), (7, 9, 13), (300, 500, 1000),
                                   (1000, 1000, 1000), (64, 2000, 33)])
@pytest.mark.parametrize("alpha,beta,c_fill", [(1.0, 0.0, "nan"), (1.5, 0.5, "uniform"),
                                               (0.75, -0.25, "uniform")])
def test_random_parity(path, M, N, K, alpha, beta, c_fill):
    A, B, C0 = operands(500 + M + N + K, M, N, K, K, N, N, np.float32, c_fill=c_fill)
    got, _ = run("f32", A, B, C0, alpha, beta, M, N, K, K, N, N, path=path)
    check("f32", got, A, B, C0, alpha, beta, M, N, K, K, N, N)


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc", [
    (257, 255, 77, 78, 255, 255),     # odd strides: scalar path
    (200, 300, 150, 152, 304, 308),   # 16-byte strides with padding: vector path
    (130, 190, 100, 101, 193, 191),
])
def test_leading_dimensions(M, N, K, lda, ldb, ldc):
    """Leading dimensions on the FFMA kernel (vector or scalar accesses) and on
    the automatic tensor-core path, whose split pre-pass reads any stride."""
    A, B, C0 = operands(17 + lda, M, N, K, lda, ldb, ldc, np.float32)
    got, taken = run("f32", A, B, C0, 0.75, -0.25, M, N, K, lda, ldb, ldc, path=FFMA_ONLY)
    vec = lda % 4 == 0 and ldb % 4 == 0 and ldc % 4 == 0
    assert taken == ("f32.ffma.vec" if vec else "f32.ffma.scalar")
    check("f32", got, A, B, C0, 0.75, -0.25, M, N, K, lda, ldb, ldc)
    assert padding_untouched(got, C0, N)
    for path, prefix in ((0, "f32.3xtf32.pair"), (16, "f32.3xf16.pair")):   # tiny: 3xTF32
        got, taken = run("f32", A, B, C0, 0.75, -0.25, M, N, K, lda, ldb, ldc, path=path)
        assert taken.startswith(prefix), taken
        check("f32", got, A, B, C0, 0.75, -0.25, M, N, K, lda, ldb, ldc)
        assert padding_untouched(got, C0, N)


def test_alpha_zero_and_K_zero():
    M, N, K = 70, 90, 30
    A, B, C0 = operands(2, M, N, K, K, N, N, np.float32)
    A[:] = np.nan
    got, path = run("f32", A, B, C0, 0.0, 0.5, M, N, K, K, N, N)
    assert path == "f32.scale"
    assert np.array_equal(got, C0 * np.float32(0.5))
    got, _ = run("f32", A[:, :0], B[:0], C0, 1.0, -0.25, M, N, 0, 1, N, N)
    assert np.array_equal(got, C0 * np.float32(-0.25))


def test_deterministic():
    M = N = K = 777
    A, B, C0 = operands(8, M, N, K, K, N, N, np.float32)
    r1, _ = run("f32", A, B, C0, 1.0, 1.0, M, N, K, K, N, N)
    r2, _ = run("f32", A, B, C0, 1.0, 1.0, M, N, K, K, N, N)
    assert np.array_equal(r1, r2)


# ---------------------------------------------------------------- tensor-core paths (split operands)
FFMA_ONLY, TF32_FORCED, F16X3_FORCED = 7, 8, 16
# (forced path, path prefix): path 16 forces 3xFP16 (scaled half parts,
# kind::f16), path 8 3xTF32 (tf32 parts, kind::tf32); the automatic choice
# between them is tested on its own below
KINDS = [(F16X3_FORCED, "f32.3xf16.pair"), (TF32_FORCED, "f32.3xtf32.pair")]


@pytest.mark.parametrize("kind,prefix", KINDS)
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 520, 200), (129, 257, 65), (7, 9, 13),
                                   (1000, 1000, 1000), (513, 1025, 4100), (64, 2000, 33)])
@pytest.mark.parametrize("alpha,beta,c_fill", [(1.0, 0.0, "nan"), (1.5, 0.5, "uniform"),
                                               (0.75, -0.25, "uniform")])
def test_split_parity(kind, prefix, M, N, K, alpha, beta, c_fill):
    A, B, C0 = operands(900 + M + N + K, M, N, K, K, N, N, np.float32, c_fill=c_fill)
    got, taken = run("f32", A, B, C0, alpha, beta, M, N, K, K, N, N, path=kind)
    assert taken.startswith(prefix), taken
    check("f32", got, A, B, C0, alpha, beta, M, N, K, K, N, N)


@pytest.mark.parametrize("kind,prefix", KINDS)
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 700, 1000)])
def test_split_small_integers_bit_exact(kind, prefix, M, N, K):
    """Integers in {-3..3}: tf32 values, and halves after any power-of-two
    scaling, so the small parts are zero and every partial sum is exact."""
    rng = np.random.default_rng(M + N + K)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    got, taken = run("f32", A, B, C0, 2.0, -1.0, M, N, K, K, N, N, path=kind)
    assert taken.startswith(prefix), taken
    assert np.array_equal(got.astype(np.float64), oracle.gemm(A, B, C0, 2.0, -1.0))


@pytest.mark.parametrize("kind,prefix", KINDS)
def test_split_close_to_ffma(kind, prefix):
    """The split keeps enough bits: at K = 1024 both the tensor-core and the
    FFMA product stay below an eighth of the fp32 bound (a single tf32 or half
    product, with its 2^-11 relative rounding per term, lands near or above
    the whole bound)."""
    M = N = K = 1024
    A, B, C0 = operands(77, M, N, K, K, N, N, np.float32)
    tc, t1 = run("f32", A, B, C0, 1.0, 0.0, M, N, K, K, N, N, path=kind)
    ff, t2 = run("f32", A, B, C0, 1.0, 0.0, M, N, K, K, N, N, path=FFMA_ONLY)
    assert t1.startswith(prefix) and t2.startswith("f32.ffma")
    ref = oracle.gemm(A, B, None, 1.0, 0.0)
    err_tc = np.abs(tc - ref).max()
    err_ff = np.abs(ff - ref).max()
    bound = 1e-6 * K * np.abs(A).max() * np.abs(B).max()
    assert err_tc < bound / 8 and err_ff < bound / 8, (err_tc, err_ff, bound)


@pytest.mark.parametrize("kind,prefix", KINDS)
def test_split_long_k_no_drift(kind, prefix):
    """Long K: the tensor core's own fp32 accumulation drifts toward zero by a
    bias growing like K*|C| (past the bound by K = 16384); the kernel folds
    128-deep chunks into round-to-nearest register sums, so the error stays a
    small fraction of the bound and shows no systematic sign."""
    M, N, K = 256, 256, 16384
    A, B, C0 = operands(4242, M, N, K, K, N, N, np.float32)
    got, taken = run("f32", A, B, C0, 1.0, 0.0, M, N, K, K, N, N, path=kind)
    assert taken.startswith(prefix), taken
    ref = oracle.gemm(A, B, None, 1.0, 0.0)
    err = got.astype(np.float64) - ref
    bound = 1e-6 * K * np.abs(A).max() * np.abs(B).max()
    assert np.abs(err).max() < bound / 10, (np.abs(err).max(), bound)
    # drift toward zero would make err * sign(ref) consistently negative
    bias = np.mean(err * np.sign(ref))
    assert abs(bias) < bound / 100, (bias, bound)


def test_f16x3_scaled_rows_and_columns():
    """3xFP16 scales each row of A and each column of B by its own power of
    two before the split: rows and columns whose magnitudes differ by 2^+-60
    (far outside the half range, and far apart) keep fp32 accuracy, each
    output within the fp32 bound taken over its own row and column."""
    rng = np.random.default_rng(61)
    M, N, K = 300, 260, 700
    A = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-60, 61, (M, 1)))).astype(np.float32)
    B = (rng.standard_normal((K, N)) * np.exp2(rng.integers(-60, 61, (1, N)))).astype(np.float32)
    C0 = np.zeros((M, N), np.float32)
    got, taken = run("f32", A, B, C0, 1.0, 0.0, M, N, K, K, N, N, path=F16X3_FORCED)
    assert taken.startswith("f32.3xf16.pair"), taken
    ref = oracle.gemm(A, B, None, 1.0, 0.0)
    per = 1e-6 * K * np.abs(A).max(axis=1)[:, None] * np.abs(B).max(axis=0)[None, :]
    assert (np.abs(got.astype(np.float64) - ref) <= per).all()
    check("f32", got, A, B, C0, 1.0, 0.0, M, N, K, K, N, N)


@pytest.mark.parametrize("kind,prefix", KINDS)
@pytest.mark.parametrize("M,N,K", [(2560, 2560, 512), (2500, 2000, 300)])
def test_split_half_width_tail(kind, prefix, M, N, K):
    """The last, partial wave of pair tiles runs as half-width units: exact on
    integers, and within the fp32 bound of the oracle (and, for the automatic
    path, of whole tiles)."""
    rng = np.random.default_rng(M + K)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    got, taken = run("f32", A, B, C0, 2.0, -1.0, M, N, K, K, N, N, path=kind)
    assert taken == prefix + ".halves", taken
    rows = oracle.sample_rows(M, block=64)
    assert np.array_equal(got[rows].astype(np.float64), oracle.gemm(A, B, C0, 2.0, -1.0, rows=rows))
    A, B, C0 = operands(55 + M, M, N, K, K, N, N, np.float32)
    got, _ = run("f32", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=kind)
    check("f32", got, A, B, C0, 1.5, 0.5, M, N, K, K, N, N, rows=rows)
    if kind == F16X3_FORCED:   # these shapes have more tiles than pairs: automatic 3xFP16
        whole, t2 = run("f32", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=5)
        assert t2 == "f32.3xf16.pair"
        bound = 1e-6 * K * np.abs(A).max() * np.abs(B).max()
        assert np.abs(got.astype(np.float64) - whole).max() <= 2 * bound


@pytest.mark.parametrize("kind,prefix", KINDS)
def test_split_two_slice_tail(kind, prefix):
    """The tiles of the last, partial wave cut into two K slices each, the
    first a worker's first unit and the second a worker's last (90 pair
    tiles on at most 76 pairs, 2048-deep K): exact on integers, within the fp32
    bound of the oracle, bit-identical run to run, and within twice the bound
    of the half-width form of the same wave (path 15, 3xFP16)."""
    M, N, K = 2560, 2304, 2048
    rng = np.random.default_rng(2304)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    got, taken = run("f32", A, B, C0, 2.0, -1.0, M, N, K, K, N, N, path=kind)
    assert taken == prefix + ".ktail", taken
    rows = oracle.sample_rows(M, block=64)
    assert np.array_equal(got[rows].astype(np.float64), oracle.gemm(A, B, C0, 2.0, -1.0, rows=rows))
    A, B, C0 = operands(2305, M, N, K, K, N, N, np.float32)
    got, _ = run("f32", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=kind)
    again, _ = run("f32", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=kind)
    assert np.array_equal(got, again)
    check("f32", got, A, B, C0, 1.5, 0.5, M, N, K, K, N, N, rows=rows)
    halves, t2 = run("f32", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=15)   # 3xFP16 halves
    assert t2.endswith(".halves"), t2
    bound = 1e-6 * K * np.abs(A).max() * np.abs(B).max()
    assert np.abs(got.astype(np.float64) - halves).max() <= 2 * bound
    # beta = 0: C (NaN-filled here) is never read, by whole tiles or by the slices
    Cn = np.full_like(C0, np.nan)
    got0, _ = run("f32", A, B, Cn, 1.5, 0.0, M, N, K, K, N, N, path=kind)
    check("f32", got0, A, B, Cn, 1.5, 0.0, M, N, K, K, N, N, rows=rows)


@pytest.mark.parametrize("kind,prefix", KINDS)
@pytest.mark.parametrize("M,N,K,lda,ldb,ldc", [
    (2560, 2303, 2100, 2103, 2305, 2307),   # ragged last K chunk, odd N, unaligned rows
    (2304, 2560, 1800, 1800, 2560, 2561),
])
def test_split_two_slice_tail_ragged(kind, prefix, M, N, K, lda, ldb, ldc):
    """The two-slice tail with a K that ends inside an accumulation chunk, a
    column count that is not a multiple of 4 and leading dimensions off the
    16-byte grid (the pre-pass reads them with element loads, C is written row
    by row): parity with the oracle on sampled rows and C's padding intact."""
    A, B, C0 = operands(7000 + K, M, N, K, lda, ldb, ldc, np.float32)
    got, taken = run("f32", A, B, C0, 0.75, -0.25, M, N, K, lda, ldb, ldc, path=kind)
    assert taken == prefix + ".ktail", taken
    check("f32", got, A, B, C0, 0.75, -0.25, M, N, K, lda, ldb, ldc,
          rows=oracle.sample_rows(M, block=64))
    assert padding_untouched(got, C0, N)


@pytest.mark.parametrize("M,N,K", [(1, 1, 65536), (300, 260, 1), (257, 1000, 64), (3000, 1, 4)])
def test_fp32_extreme_dimensions(M, N, K):
    A, B, C0 = operands(4242 + M + K, M, N, K, K, N, N, np.float32)
    got, _ = run("f32", A, B, C0, 0.75, -0.25, M, N, K, K, N, N)
    check("f32", got, A, B, C0, 0.75, -0.25, M, N, K, K, N, N)


# ---------------------------------------------------------------- K slices (few tiles)
@pytest.mark.parametrize("kind,prefix", KINDS)
@pytest.mark.parametrize("M,N,K", [(1000, 1100, 4000), (256, 256, 4096), (513, 1025, 4100),
                                   (300, 300, 8200)])
def test_split_k_slices(kind, prefix, M, N, K):
    """Few pair tiles and a long K: every tile is cut into K slices whose fp32
    partial sums the last slice to finish adds up.  Exact on integers; within
    the fp32 bound of the oracle and of whole-K units; bit-identical run to
    run."""
    rng = np.random.default_rng(M + 3 * K)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    got, taken = run("f32", A, B, C0, 2.0, -1.0, M, N, K, K, N, N, path=kind)
    assert taken == prefix + ".ksplit", taken
    assert np.array_equal(got.astype(np.float64), oracle.gemm(A, B, C0, 2.0, -1.0))
    A, B, C0 = operands(606 + M + K, M, N, K, K, N, N, np.float32)
    got, _ = run("f32", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=kind)
    again, _ = run("f32", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=kind)
    assert np.array_equal(got, again)
    check("f32", got, A, B, C0, 1.5, 0.5, M, N, K, K, N, N)
    whole, t2 = run("f32", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=kind, splits=1)
    assert not t2.endswith(".ksplit"), t2
    bound = 1e-6 * K * np.abs(A).max() * np.abs(B).max()
    assert np.abs(got.astype(np.float64) - whole).max() <= 2 * bound


@pytest.mark.parametrize("kind,prefix", KINDS)
@pytest.mark.parametrize("splits", [2, 3, 7, 16])
def test_split_forced_slice_counts(kind, prefix, splits):
    """Any slice count (slices are whole 4-k-block chunks; a count that would
    leave a slice empty is reduced): parity with the oracle, NaN-filled C with
    beta = 0 never read."""
    M, N, K = 700, 900, 3000
    A, B, C0 = operands(707 + splits, M, N, K, K, N, N, np.float32, c_fill="nan")
    got, taken = run("f32", A, B, C0, 1.0, 0.0, M, N, K, K, N, N, path=kind, splits=splits)
    assert taken == prefix + ".ksplit", taken
    check("f32", got, A, B, C0, 1.0, 0.0, M, N, K, K, N, N)


@pytest.mark.parametrize("kind,prefix", KINDS)
def test_split_k_slices_padded_ldc(kind, prefix):
    """Sliced tiles with ldc > N: the padding of C stays untouched."""
    M, N, K, ldc = 600, 700, 4000, 712
    A, B, C0 = operands(808, M, N, K, K, N, ldc, np.float32)
    got, taken = run("f32", A, B, C0, 0.75, -0.25, M, N, K, K, N, ldc, path=kind)
    assert taken == prefix + ".ksplit", taken
    check("f32", got, A, B, C0, 0.75, -0.25, M, N, K, K, N, ldc)
    assert padding_untouched(got, C0, N)


@pytest.mark.parametrize("kind,prefix", KINDS)
@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (256, 256, 256), (1000, 1100, 900)])
def test_split_short_k_keeps_whole_units(kind, prefix, M, N, K):
    """Few tiles with a short K: slicing would cost more in its fix-up than it
    saves, so the tiles run as whole-K half-width units."""
    A, B, C0 = operands(909 + K, M, N, K, K, N, N, np.float32)
    got, taken = run("f32", A, B, C0, 1.0, 0.0, M, N, K, K, N, N, path=kind)
    assert taken == prefix + ".halves", taken
    check("f32", got, A, B, C0, 1.0, 0.0, M, N, K, K, N, N)


@pytest.mark.parametrize("M,N,K,expect", [
    (16, 8192, 1024, "f32.3xf16"), (1, 4096, 512, "f32.3xtf32"), (200, 200, 200, "f32.3xtf32"),
    (16, 16, 4096, "f32.3xtf32"), (1024, 1024, 16, "f32.ffma"), (300, 260, 1, "f32.ffma"),
    (2560, 2048, 64, "f32.3xf16"), (2048, 2048, 2048, "f32.3xf16"), (256, 256, 256, "f32.3xtf32"),
    (256, 256, 257, "f32.3xf16"),
])
def test_fp32_path_choice_small_and_skinny(M, N, K, expect):
    """K >= 64 takes the tensor cores whatever M and N (skinny and tiny shapes
    included): 3xFP16 when M*N*K exceeds 256^3, 3xTF32 up to that; a shorter
    K takes the FFMA kernel.  Parity either way."""
    A, B, C0 = operands(3030 + M + K, M, N, K, K, N, N, np.float32)
    got, taken = run("f32", A, B, C0, 1.25, -0.5, M, N, K, K, N, N)
    assert taken.startswith(expect), taken
    rows = oracle.sample_rows(M, block=64) if M * N * K > 2e9 else None
    check("f32", got, A, B, C0, 1.25, -0.5, M, N, K, K, N, N, rows=rows)


@pytest.mark.parametrize("M,N,K,ldc", [(700, 900, 500, 900), (2600, 1000, 700, 1004)])
def test_fp32_host_form(M, N, K, ldc):
    """sgemm_f32_host: pinned host operands copied in, computed (in four row
    blocks when M >= 2048, each block with its own split pre-pass) and copied
    back; parity with the oracle and C's padding unchanged."""
    import dense_gemm_03_gb300 as g
    from helpers import torch
    t = torch()
    A, B, C0 = operands(4400 + M, M, N, K, K, N, ldc, np.float32)
    hA = t.from_numpy(A).pin_memory()
    hB = t.from_numpy(B).pin_memory()
    hC = t.from_numpy(C0.copy()).pin_memory()
    g.sgemm_f32_host(hA, hB, hC, 0.75, -0.25, M=M, N=N, K=K, ldc=ldc)
    got = hC.numpy()
    check("f32", got, A, B, C0, 0.75, -0.25, M, N, K, K, N, ldc,
          rows=oracle.sample_rows(M, block=64) if M >= 2048 else None)
    assert padding_untouched(got, C0, N)
    assert g.debug_status() == 0
