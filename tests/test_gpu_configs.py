"""The benchmark workloads at full size, checked against the oracle: all of C
where the oracle finishes in seconds, sampled rows and columns (one in every
output tile band) plus whole-matrix identities elsewhere.

Workloads (seeded, synthetic):
  fp32 256^3, alpha=1 beta=0, C zeroed
  fp32 square N in {256..4096}, alpha=1 beta=0, checksum + elementwise
  fp16 4096^3, alpha=1.5 beta=0.5, C0 ~ U(-1,1)
  fp32 sweep sizes (a sample of 1024..12800 step 128), A, B ~ N(0,1)
  fp16 edge shapes, alpha=0.75 beta=-0.25: 4097x1023x777 (lda=780),
       16x8192x8192, 8192x64x4096
"""
import numpy as np
import pytest

import oracle
import synthetic
from helpers import check, operands, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_03_gb300 import build
    build.build()


def _checksum_ok(got, A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, kind):
    s_gpu = oracle.checksum(got[:, :N])
    s_ref, scale = oracle.checksum_closed_form(A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc)
    # each element is within its tolerance; the sum of the tolerances bounds the sum
    if kind == "f16":
        bound = 2e-3 * scale + 2.0 ** -10 * scale + M * N * 2.0 ** -24
    else:
        amax = float(np.abs(A).max())
        bmax = float(np.abs(B).max())
        bound = M * N * (1e-6 * K * amax * bmax) + 2.0 ** -23 * scale
    assert abs(s_gpu - s_ref) <= bound, (s_gpu, s_ref, bound)


def test_fp32_256_cube():
    M = N = K = 256
    A, B, C0 = operands(synthetic.config_seed(0), M, N, K, K, N, N, np.float32, c_fill="zero")
    got, path = run("f32", A, B, C0, 1.0, 0.0, M, N, K, K, N, N)
    check("f32", got, A, B, C0, 1.0, 0.0, M, N, K, K, N, N)


@pytest.mark.parametrize("n", [256, 512, 1024, 2048, 4096])
def test_fp32_square(n):
    A, B, C0 = operands(synthetic.config_seed(1), n, n, n, n, n, n, np.float32, c_fill="zero")
    got, path = run("f32", A, B, C0, 1.0, 0.0, n, n, n, n, n, n)
    _checksum_ok(got, A, B, C0, 1.0, 0.0, n, n, n, n, n, n, "f32")
    if n <= 2048:
        check("f32", got, A, B, C0, 1.0, 0.0, n, n, n, n, n, n)
    else:
        check("f32", got, A, B, C0, 1.0, 0.0, n, n, n, n, n, n,
              rows=oracle.sample_rows(n), cols=oracle.sample_cols(n))


def test_fp16_4096_cube():
    n = 4096
    A, B, C0 = operands(synthetic.config_seed(2), n, n, n, n, n, n, np.float16)
    got, path = run("f16", A, B, C0, 1.5, 0.5, n, n, n, n, n, n)
    assert path.startswith("f16.tc") and "tma" in path
    check("f16", got, A, B, C0, 1.5, 0.5, n, n, n, n, n, n,
          rows=oracle.sample_rows(n), cols=oracle.sample_cols(n))
    _checksum_ok(got, A, B, C0, 1.5, 0.5, n, n, n, n, n, n, "f16")


@pytest.mark.parametrize("size", [1024, 1152, 2560, 4096 + 128, 12800])
def test_fp32_sweep_sizes(size):
    n = size
    A, B, C0 = operands(synthetic.config_seed(3) + n, n, n, n, n, n, n, np.float32,
                        dist="normal", c_fill="zero")
    got, _ = run("f32", A, B, C0, 1.0, 0.0, n, n, n, n, n, n)
    rows = oracle.sample_rows(n, block=128 if n <= 4096 else 512, extra=4)
    check("f32", got, A, B, C0, 1.0, 0.0, n, n, n, n, n, n, rows=rows)


@pytest.mark.parametrize("M,N,K,lda", [(4097, 1023, 777, 780), (16, 8192, 8192, 8192),
                                       (8192, 64, 4096, 4096)])
def test_fp16_edge_shapes(M, N, K, lda):
    A, B, C0 = operands(synthetic.config_seed(4), M, N, K, lda, N, N, np.float16)
    got, path = run("f16", A, B, C0, 0.75, -0.25, M, N, K, lda, N, N)
    if lda == 780:
        assert path.endswith(".realigned.c"), path   # A, B and C through aligned copies
    check("f16", got, A, B, C0, 0.75, -0.25, M, N, K, lda, N, N)
