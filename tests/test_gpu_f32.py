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
    A, B, C0 = operands(17 + lda, M, N, K, lda, ldb, ldc, np.float32)
    got, taken = run("f32", A, B, C0, 0.75, -0.25, M, N, K, lda, ldb, ldc)
    vec = lda % 4 == 0 and ldb % 4 == 0 and ldc % 4 == 0
    assert taken == ("f32.ffma.vec" if vec else "f32.ffma.scalar")
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
