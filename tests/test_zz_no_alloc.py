"""The allocation-free entry point gemm_f16_splitk_noalloc.

Some callers must not allocate device memory while they run: cudaMalloc can
synchronise the whole device and can fail mid-run, and some programs draw
every device allocation from their own planner or from a budget fixed at
start-up.  gemm_f16_splitk_noalloc serves them: it runs the split-K GEMM on
the library's fixed static scratch array instead of a workspace it would have
to allocate.  This file checks, through the C ABI, that two calls in a row
match the CPU oracle within the fp16 tolerance the other tests use (and agree
with the ordinary entry point gemm_f16_ld within the same bound), on aligned
operands (tensor-memory-accelerator loads) and on unaligned ones (predicated
element loads), that the calls do not change the device's free memory, and
that a problem too large for the array is refused.

It is named so that pytest collects it last; it sets up everything it needs,
so it also passes when run on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
from helpers import operands, padding_untouched, to_dev, torch

pytestmark = pytest.mark.gpu

# M, N, K, lda, ldb, ldc, alpha, beta, K slices (0 = automatic), load mode in the path
CASES = [(16, 8192, 8192, 8192, 8192, 8192, 0.75, -0.25, 0, "tma"),
         (300, 512, 3000, 3000, 512, 512, 1.5, 0.5, 4, "tma"),
         # rows of A and B off the 16-byte grid (K + 3, N): predicated element loads
         (300, 1023, 777, 780, 1023, 1023, 0.75, -0.25, 4, "manual")]


@pytest.fixture(scope="module")
def L():
    from dense_gemm_03_gb300 import build
    build.build()
    import dense_gemm_03_gb300 as g
    return g.lib()


def _noalloc(L, dA, dB, dC, M, N, K, lda, ldb, ldc, alpha, beta, splits, stream):
    return L.gemm_f16_splitk_noalloc(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, lda,
                                     ldb, ldc, ctypes.c_float(alpha), ctypes.c_float(beta), splits,
                                     stream)


def test_two_calls_match_the_oracle(L):
    t = torch()
    stream = t.cuda.current_stream().cuda_stream
    prepared = []
    for i, (M, N, K, lda, ldb, ldc, alpha, beta, splits, mode) in enumerate(CASES):
        A, B, C0 = operands(900 + i, M, N, K, lda, ldb, ldc, np.float16)
        prepared.append((A, B, C0, to_dev(A), to_dev(B), to_dev(C0), to_dev(C0)))
    # one call per case first: the per-device set-up, and the CUDA runtime
    # loading each kernel's code on its first launch, may take device memory
    for w, case in zip(prepared, CASES):
        warm = to_dev(w[2])
        assert _noalloc(L, w[3], w[4], warm, *case[:9], stream) == 0
    t.cuda.synchronize()
    free_before = t.cuda.mem_get_info()[0]

    # two calls in a row on the shared scratch array
    paths = []
    for (A, B, C0, dA, dB, dC_new, _), case in zip(prepared, CASES):
        assert _noalloc(L, dA, dB, dC_new, *case[:9], stream) == 0
        paths.append(L.gemm_last_path().decode())
    t.cuda.synchronize()
    assert t.cuda.mem_get_info()[0] == free_before

    import dense_gemm_03_gb300 as g
    assert g.debug_status() == 0
    for (A, B, C0, dA, dB, dC_new, dC_old), case, path in zip(prepared, CASES, paths):
        M, N, K, lda, ldb, ldc, alpha, beta, splits, mode = case
        assert path == "f16.splitk.noalloc." + mode, path
        new = dC_new.cpu().numpy().reshape(C0.shape)
        ref, absd = oracle.gemm(A, B, C0, alpha, beta, M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc,
                                with_absdot=True)
        tol = oracle.tol_f16(ref, absd)
        r = oracle.compare(new[:, :N].astype(np.float64), ref, tol)
        assert r["ok"], r
        if ldc > N:
            assert padding_untouched(new, C0, N)
        # and within the same bound of the ordinary entry point
        assert L.gemm_f16_ld(dA.data_ptr(), dB.data_ptr(), dC_old.data_ptr(), M, N, K, lda, ldb,
                             ldc, ctypes.c_float(alpha), ctypes.c_float(beta), stream) == 0
        t.cuda.synchronize()
        old = dC_old.cpu().numpy().reshape(C0.shape)[:, :N].astype(np.float64)
        r = oracle.compare(new[:, :N].astype(np.float64), old, tol)
        assert r["ok"], r


def test_too_large_is_refused(L):
    t = torch()
    M = N = 2048
    K = 4096
    dA = t.zeros((M, K), dtype=t.float16, device="cuda")
    dB = t.zeros((K, N), dtype=t.float16, device="cuda")
    dC = t.full((M, N), 7.0, dtype=t.float16, device="cuda")
    # 2 slices x 2048 x 2048 x 4 bytes = 32 MiB > the 8 MiB array
    assert _noalloc(L, dA, dB, dC, M, N, K, K, N, N, 1.0, 0.0, 2, None) == -7
    t.cuda.synchronize()
    assert bool((dC == 7.0).all())
