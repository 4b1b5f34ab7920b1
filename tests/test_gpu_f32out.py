"""Half operands with an fp32 C (gemm_f16_f32out) and the float-to-half
conversion (gemm_f32_to_f16), through the C ABI, against the CPU oracle."""
import numpy as np
import pytest

import oracle
import synthetic
from helpers import operands, torch

pytestmark = pytest.mark.gpu

AUTO, NO_TAIL, NO_PAIR, SK = 0, 5, 6, 10
F32_SENTINEL = np.float32(-12345.5)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_03_gb300 import build
    build.build()


def run32(A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, path=AUTO):
    """gemm_f16_f32out on device copies; returns (C as float32 host array, path)."""
    import dense_gemm_03_gb300 as g
    t = torch()
    dA = t.from_numpy(np.ascontiguousarray(A).reshape(-1)).cuda()
    dB = t.from_numpy(np.ascontiguousarray(B).reshape(-1)).cuda()
    dC = t.from_numpy(np.ascontiguousarray(C0).reshape(-1)).cuda()
    prev = g.force_path(path)
    try:
        g.gemm_f16_f32out(dA, dB, dC, alpha, beta, M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc)
        taken = g.last_path()
    finally:
        g.force_path(prev)
    t.cuda.synchronize()
    assert g.debug_status() == 0
    return dC.cpu().numpy().reshape(C0.shape), taken


def _c32(seed, M, ldc, fill="uniform"):
    if fill == "nan":
        C0 = np.full((M, ldc), np.nan, np.float32)
    else:
        C0 = synthetic.uniform(seed, synthetic.STREAM_C, (M, ldc), dtype=np.float32)
    return C0


@pytest.mark.parametrize("M,N,K,path,mark", [
    (256, 512, 128, AUTO, ".epi_f32"),
    (2000, 2600, 4096, AUTO, ".pair.bn256.tma.epi_f32_tma.ktail"),
    (2000, 2601, 1024, AUTO, ".pair.bn256.tma.epi_f32.halves"),    # N % 4 != 0: direct stores
    (2000, 2601, 4096, AUTO, ".pair.bn256.tma.epi_f32.ktail"),
    (2000, 2600, 2048, SK, ".pair.bn256.tma.epi_f32_tma.sk"),
    (16, 8192, 8192, AUTO, ".bn128.tma.epi_f32.a32.sk"),
    (48, 3000, 1500, AUTO, ".epi_f32.a64"),
    (700, 300, 500, NO_PAIR, ".bn256.tma.epi_f32"),
    (129, 65, 17, AUTO, ".epi_f32"),
    (1, 1, 1, AUTO, ".epi_f32"),
])
def test_small_integers_exact(M, N, K, path, mark):
    """Entries in {-1, 0, 1} and integer C: every sum is an integer below 2^24,
    so the fp32 C equals the oracle exactly on every schedule."""
    rng = np.random.default_rng(M + 5 * N + 11 * K)
    A = rng.integers(-1, 2, size=(M, K)).astype(np.float16)
    B = rng.integers(-1, 2, size=(K, N)).astype(np.float16)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    got, taken = run32(A, B, C0, 2.0, -1.0, M, N, K, K, N, N, path=path)
    assert mark in taken, taken
    rows = list(range(M)) if M * N * K <= 4e9 else oracle.sample_rows(M, block=32)
    ref = oracle.gemm(A, B, C0, 2.0, -1.0, rows=rows)
    assert np.array_equal(got[rows].astype(np.float64), ref)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 700, 1000), (1024, 1024, 1024),
                                   (2000, 2600, 4096), (7, 9, 13), (64, 128, 4096)])
@pytest.mark.parametrize("alpha,beta,fill", [(1.0, 0.0, "nan"), (1.5, 0.5, "uniform"),
                                             (0.75, -0.25, "uniform")])
def test_random_parity(M, N, K, alpha, beta, fill):
    A, B, _ = operands(300 + M + N + K, M, N, K, K, N, N, np.float16)
    C0 = _c32(300 + M, M, N, fill)
    got, _ = run32(A, B, C0, alpha, beta, M, N, K, K, N, N)
    rows = None if M * N * K <= 2e9 else oracle.sample_rows(M)
    ref, absd = oracle.gemm(A, B, C0, alpha, beta, rows=rows, with_absdot=True)
    view = (got if rows is None else got[rows]).astype(np.float64)
    r = oracle.compare(view, ref, oracle.tol_f16_f32out(ref, absd))
    assert r["ok"], r
    # and far inside it: the error is that of fp32 accumulation
    r2 = oracle.compare(view, ref, 1e-5 * absd + oracle.ulp32(ref))
    assert r2["ok"], r2


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc", [
    (257, 255, 77, 80, 255, 257),       # odd ldc: predicated fp32 stores
    (200, 300, 150, 153, 305, 304),     # unaligned A and B rows: realigned copies
    (130, 190, 100, 104, 192, 200),     # padding everywhere, 16-byte strides
])
def test_leading_dimensions(M, N, K, lda, ldb, ldc):
    A, B, _ = operands(71 + lda, M, N, K, lda, ldb, ldc, np.float16)
    C0 = _c32(71 + ldc, M, ldc)
    C0[:, N:] = F32_SENTINEL
    got, _ = run32(A, B, C0, 0.75, -0.25, M, N, K, lda, ldb, ldc)
    ref, absd = oracle.gemm(A, B, C0, 0.75, -0.25, M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc,
                            with_absdot=True)
    r = oracle.compare(got[:, :N].astype(np.float64), ref, oracle.tol_f16_f32out(ref, absd))
    assert r["ok"], r
    assert (got[:, N:] == F32_SENTINEL).all()


def test_alpha_zero_and_K_zero_scale_C_exactly():
    M, N, K = 100, 130, 40
    A, B, _ = operands(9, M, N, K, K, N, N, np.float16)
    A[:] = np.nan
    C0 = _c32(9, M, N)
    got, path = run32(A, B, C0, 0.0, -0.25, M, N, K, K, N, N)
    assert path == "f16f32.scale"
    assert np.array_equal(got, C0 * np.float32(-0.25))


def test_rounded_to_half_equals_gemm_f16():
    """alpha*acc + beta*c in fp32, then rounded once to half, is what gemm_f16
    stores: converting this entry's output with gemm_f32_to_f16 reproduces
    gemm_f16's bits on the same schedule."""
    import dense_gemm_03_gb300 as g
    from helpers import run
    t = torch()
    M, N, K = 2000, 2600, 1024
    A, B, C16 = operands(404, M, N, K, K, N, N, np.float16)
    want, p16 = run("f16", A, B, C16, 1.5, 0.5, M, N, K, K, N, N)
    got32, p32 = run32(A, B, C16.astype(np.float32), 1.5, 0.5, M, N, K, K, N, N)
    assert p16.replace("epi_tma", "epi_f32_tma") == p32, (p16, p32)
    src = t.from_numpy(got32.reshape(-1)).cuda()
    dst = t.empty(src.numel(), dtype=t.float16, device="cuda")
    g.f32_to_f16(src, dst)
    t.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy().view(np.uint16).reshape(M, N), want.view(np.uint16))


# ---------------------------------------------------------------- float -> half conversion

def _special_values():
    v = [0.0, -0.0, 1.0, -1.0, 1 / 3, 65504.0, 65519.0, 65520.0, -65520.0, 1e30, -1e30,
         2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -14, 2049.0, 2051.0, np.inf, -np.inf]
    return np.array(v, dtype=np.float32)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 1 << 20, (1 << 20) + 3])
@pytest.mark.parametrize("src_off,dst_off", [(0, 0), (1, 0), (0, 1), (3, 5)])
def test_f32_to_f16_bit_exact(n, src_off, dst_off):
    import dense_gemm_03_gb300 as g
    t = torch()
    rng = np.random.default_rng(n + 7 * src_off + dst_off)
    # every exponent from deep subnormal-half range to beyond the half range
    x = (rng.standard_normal(n) * np.exp2(rng.integers(-30, 20, n))).astype(np.float32)
    sp = _special_values()
    x[:min(n, sp.size)] = sp[:min(n, sp.size)]
    src = t.zeros(n + 8, dtype=t.float32, device="cuda")
    src[src_off:src_off + n] = t.from_numpy(x).cuda()
    dst = t.full((n + 8,), -7.0, dtype=t.float16, device="cuda")
    g.f32_to_f16(src.data_ptr() + 4 * src_off, dst.data_ptr() + 2 * dst_off, n)
    t.cuda.synchronize()
    out = dst.cpu().numpy()
    got = out[dst_off:dst_off + n]
    want = oracle.f32_to_f16(x)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    # nothing outside [dst, dst + n) is written
    assert (out[:dst_off] == -7.0).all() and (out[dst_off + n:] == -7.0).all()


def test_f32_to_f16_nan_and_errors():
    import dense_gemm_03_gb300 as g
    t = torch()
    src = t.tensor([np.nan, -np.nan, 1.0], dtype=t.float32, device="cuda")
    dst = t.zeros(3, dtype=t.float16, device="cuda")
    g.f32_to_f16(src, dst)
    t.cuda.synchronize()
    h = dst.cpu().numpy()
    assert np.isnan(h[0]) and np.isnan(h[1]) and h[2] == 1.0
    L = g.lib()
    assert L.gemm_f32_to_f16(src.data_ptr(), dst.data_ptr(), -1, None) == -2      # negative n
    assert L.gemm_f32_to_f16(src.data_ptr(), dst.data_ptr() + 1, 2, None) == -7   # odd dst
    assert L.gemm_f32_to_f16(src.data_ptr(), dst.data_ptr(), 0, None) == 0        # no-op
