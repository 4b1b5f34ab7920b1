"""Overflow and non-finite values on every half-precision path, against the
oracle, through the C ABI.

The epilogue of the "LeetGPU GEMM T4" page (baseline section) evaluates
acc*alpha + C*beta in fp32 and converts it with __float2half: round to nearest,
ties to even, and a result beyond the half range becomes +-Inf.  The operands
here are small integers (sparse A, so that every dot product stays small) and
C sits at the edge of the half range (+-65504, +-65472, 32768, 2048, ...), so
every fp32 value on the way is exact whatever the order of accumulation:
each output must equal the oracle's exact value rounded once to half -- an
overflow to +-Inf, a tie at the top of the range (65488 -> 65472), or a tie
between two halves (2049 -> 2048) -- bit for bit, on every schedule (CTA
pairs, single CTAs, predicated loads and epilogue, realigned operands,
split-K, stream-K, two-slice tails, half-width units, skinny and tall
shapes, 64-row tiles).

Operands holding +-Inf follow IEEE arithmetic: a product with Inf is +-Inf
(NaN for Inf * 0) and a sum that meets both +Inf and -Inf is NaN, whatever
the order; those outputs must be NaN or the same infinity as the oracle's.
"""
import numpy as np
import pytest

import oracle
from helpers import run, to_dev, torch

pytestmark = pytest.mark.gpu

AUTO, MANUAL, SPLITK = 0, 2, 3
NO_TAIL, NO_PAIR, TAIL2, SK, SK_ALL = 5, 6, 9, 10, 11
FFMA_ONLY, TF32, F16X3 = 7, 8, 16

# values of C at and near the top of the half range and at a spacing-2 binade
EDGE_C = np.array([65504, -65504, 65472, -65472, 65440, 32768, -32768, 2048, -2048, 1024, 0],
                  dtype=np.float16)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_03_gb300 import build
    build.build()


def _operands(seed, M, N, K, lda=None, ldb=None, ldc=None, dtype=np.float16):
    """Sparse small-integer A (about 32 nonzeros per row), dense small-integer
    B, C from EDGE_C; padded rows hold NaN (never read)."""
    lda, ldb, ldc = lda or K, ldb or N, ldc or N
    rng = np.random.default_rng(seed)
    dens = min(1.0, 32.0 / K)
    A = np.full((M, lda), np.nan, dtype=dtype)
    A[:, :K] = rng.integers(-3, 4, size=(M, K)) * (rng.random((M, K)) < dens)
    B = np.full((K, ldb), np.nan, dtype=dtype)
    B[:, :N] = rng.integers(-3, 4, size=(K, N))
    C0 = np.full((M, ldc), np.nan, dtype=dtype)
    C0[:, :N] = EDGE_C[rng.integers(0, EDGE_C.size, size=(M, N))]
    return A, B, C0


def _expected(A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, rows=None):
    ref = oracle.gemm(A, B, C0, alpha, beta, M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc, rows=rows)
    return oracle.f32_to_f16(ref), ref


def _same_bits_or_both_nan(got, want):
    g = np.asarray(got, dtype=np.float16)
    w = np.asarray(want, dtype=np.float16)
    nan_g, nan_w = np.isnan(g), np.isnan(w)
    if not np.array_equal(nan_g, nan_w):
        return False
    return np.array_equal(g.view(np.uint16)[~nan_g], w.view(np.uint16)[~nan_w])


# (M, N, K, lda, ldb, ldc, forced path, splits, mark in the reported path)
PATHS = [
    (512, 512, 64, 64, 512, 512, NO_TAIL, 0, ".pair.bn256.tma.epi_tma"),
    (512, 1001, 64, 64, 1001, 1001, NO_TAIL, 0, ".pair.bn256.tma.epi_tma.realigned.c"),
    (300, 384, 64, 64, 384, 384, NO_PAIR, 0, ".bn256.tma.epi_tma"),
    (300, 100, 200, 200, 100, 100, AUTO, 0, ".bn128.tma.epi_tma.halves.realigned.c"),
    (300, 1001, 200, 200, 1001, 1001, MANUAL, 0, ".manual.epi_manual"),
    (300, 400, 200, 200, 400, 400, MANUAL, 0, ".manual."),
    (300, 520, 200, 201, 520, 523, AUTO, 0, ".realigned"),
    (200, 300, 1024, 1024, 300, 300, SPLITK, 3, ".splitk"),
    (64, 128, 4096, 4096, 128, 128, SK_ALL, 0, ".sk"),
    (2000, 2600, 4096, 4096, 2600, 2600, SK, 0, ".pair.bn256.tma.epi_tma.sk"),
    (2000, 2600, 4096, 4096, 2600, 2600, TAIL2, 0, ".tail"),
    (2000, 2600, 4096, 4096, 2600, 2600, AUTO, 0, ".pair.bn256.tma.epi_tma.ktail"),
    (2560, 2560, 1024, 1024, 2560, 2560, 15, 0, ".pair.bn256.tma.epi_tma.halves"),
    (2000, 2600, 4096, 4096, 2600, 2600, 14, 0, ".pair.bn256.tma.epi_tma.sktail"),
    (600, 1000, 300, 300, 1000, 1000, 12, 0, ".pair.bn224.tma.epi_tma"),
    (600, 1001, 300, 300, 1001, 1001, 13, 0, ".pair.bn192.tma.epi_tma"),
    (16, 1000, 700, 700, 1000, 1000, AUTO, 0, ".a32"),
    (4096, 64, 8192, 8192, 64, 64, AUTO, 0, ".bn64.tma.epi_tma.sk"),
    (4096, 64, 2048, 2048, 64, 64, AUTO, 0, ".bn64.tma.epi_tma"),
    (4096, 64, 2048, 2048, 64, 64, 17, 0, ".bn64.tma.epi_tma.m64"),
]


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,path,splits,mark", PATHS)
@pytest.mark.parametrize("alpha,beta", [(1.0, 1.0), (2.0, 2.0), (2048.0, 0.0)])
def test_overflow_rounds_to_inf_on_every_path(M, N, K, lda, ldb, ldc, path, splits, mark, alpha,
                                              beta):
    A, B, C0 = _operands(M + 3 * N + 7 * K + int(alpha), M, N, K, lda, ldb, ldc)
    got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, path=path,
                     splits=splits)
    assert mark in taken, taken
    rows = list(range(M)) if M * N * K <= 2e9 else oracle.sample_rows(M, block=64)
    want, ref = _expected(A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, rows=rows)
    # the operands reach both sides of the range edge
    assert np.isinf(want).any() and np.isfinite(want).any()
    assert np.array_equal(got[rows, :N].view(np.uint16), want.view(np.uint16)), taken
    if ldc > N:   # padding of C untouched
        assert np.isnan(got[:, N:]).all()


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc,path,splits,mark", [PATHS[i] for i in (0, 1, 4, 5, 7, 8, 11, 12)])
def test_infinite_operands_follow_ieee(M, N, K, lda, ldb, ldc, path, splits, mark):
    A, B, C0 = _operands(11 + M + N + K, M, N, K, lda, ldb, ldc)
    rng = np.random.default_rng(M * N)
    # a few infinities of either sign in A and B, some C entries infinite
    for X, rows_, cols_ in ((A, M, K), (B, K, N)):
        idx = rng.integers(0, rows_ * cols_, size=max(4, rows_ * cols_ // 20000))
        r, c = np.divmod(idx, cols_)
        X[r, c] = np.where(rng.random(idx.size) < 0.5, np.inf, -np.inf)
    C0[rng.integers(0, M, 8), rng.integers(0, N, 8)] = np.inf
    got, taken = run("f16", A, B, C0, 0.75, -0.5, M, N, K, lda, ldb, ldc, path=path,
                     splits=splits)
    assert mark in taken, taken
    rows = list(range(M)) if M * N * K <= 2e9 else oracle.sample_rows(M, block=64)
    with np.errstate(invalid="ignore"):
        want, ref = _expected(A, B, C0, 0.75, -0.5, M, N, K, lda, ldb, ldc, rows=rows)
    assert np.isnan(want).any() and np.isposinf(want).any() and np.isneginf(want).any()
    assert _same_bits_or_both_nan(got[rows, :N], want), taken


def test_f32_output_then_conversion_overflows_like_gemm_f16():
    """gemm_f16_f32out keeps the fp32 value (no overflow at these magnitudes);
    converting it with gemm_f32_to_f16 rounds it once, to +-Inf beyond the
    half range, exactly as gemm_f16 does."""
    import dense_gemm_03_gb300 as g
    t = torch()
    M, N, K = 512, 512, 64
    A, B, C0 = _operands(5, M, N, K)
    C32 = C0.astype(np.float32)
    dA, dB, dC = to_dev(A), to_dev(B), to_dev(C32)
    g.gemm_f16_f32out(dA, dB, dC, 1.0, 1.0)
    h = t.empty((M, N), dtype=t.float16, device="cuda")
    g.f32_to_f16(dC, h)
    t.cuda.synchronize()
    assert g.debug_status() == 0
    ref = oracle.gemm(A, B, C32, 1.0, 1.0)
    assert np.array_equal(dC.cpu().numpy().astype(np.float64), ref)   # exact in fp32
    want = oracle.f32_to_f16(ref)
    assert np.isinf(want).any()
    assert np.array_equal(h.cpu().numpy().view(np.uint16), want.view(np.uint16))


def test_host_form_overflow():
    import dense_gemm_03_gb300 as g
    t = torch()
    M, N, K = 2304, 512, 128     # four row blocks of the pipelined host form
    A, B, C0 = _operands(6, M, N, K)
    pA, pB, pC = (t.from_numpy(x.copy()).pin_memory() for x in (A, B, C0))
    g.gemm_f16_host(pA, pB, pC, 1.0, 1.0)
    want, _ = _expected(A, B, C0, 1.0, 1.0, M, N, K, K, N, N)
    assert np.isinf(want).any()
    assert np.array_equal(pC.numpy().view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("path", [FFMA_ONLY, TF32, F16X3])
def test_fp32_non_finite_operands(path):
    """fp32: the FFMA kernel follows IEEE exactly.  The tensor-core paths split
    each operand into a part and a remainder (Inf - Inf = NaN for an infinite
    operand; 3xFP16 also leaves the row or column of an infinite operand
    unscaled), so an output that meets an infinite operand is NaN there: it is
    still non-finite, and every other output is exact."""
    M, N, K = 300, 400, 200
    A, B, C0 = _operands(9, M, N, K, dtype=np.float32)
    A[5, 7], A[100, 50], B[3, 9] = np.inf, -np.inf, np.inf
    got, taken = run("f32", A, B, C0, 1.0, 1.0, M, N, K, K, N, N, path=path)
    with np.errstate(invalid="ignore"):
        ref = oracle.gemm(A, B, C0, 1.0, 1.0)
    g = got.astype(np.float64)
    fin = np.isfinite(ref)
    assert not fin.all()
    assert np.array_equal(np.isfinite(g), fin), taken
    assert np.array_equal(g[fin], ref[fin])
    if path == FFMA_ONLY:
        assert taken.startswith("f32.ffma")
        assert np.array_equal(np.isnan(g), np.isnan(ref))
        assert np.array_equal(g[np.isinf(ref)], ref[np.isinf(ref)])
    else:
        assert taken.startswith("f32.3xtf32" if path == TF32 else "f32.3xf16"), taken
