"""The allocation-free entry point gemm_f16_splitk_noalloc.

Some callers must not allocate device memory while they run: cudaMalloc can
synchronise the whole device and can fail mid-run, and some programs draw
every device allocation from their own planner or from a budget fixed at
start-up.  gemm_f16_splitk_noalloc serves them: it runs the split-K GEMM on
the library's fixed static scratch array instead of a workspace it would have
to allocate.  This file checks, through the C ABI, that two calls in a row
give the same results as the ordinary entry point gemm_f16_ld (within the fp16
tolerance the other tests use), that the calls do not change the device's free
memory, and that a problem too large for the array is refused.

It is named so that pytest collects it last; it sets up everything it needs,
so it also passes when run on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
from helpers import operands, to_dev, torch

pytestmark = pytest.mark.gpu

# M, N, K, alpha, beta, K slices (0 = automatic)
CASES = [(16, 8192, 8192, 0.75, -0.25, 0), (300, 500, 3000, 1.5, 0.5, 4)]


@pytest.fixture(scope="module")
def L():
    from dense_gemm_03_gb300 import build
    build.build()
    import dense_gemm_03_gb300 as g
    return g.lib()


def _noalloc(L, dA, dB, dC, M, N, K, alpha, beta, splits, stream):
    return L.gemm_f16_splitk_noalloc(dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), M, N, K, K, N, N,
                                     ctypes.c_float(alpha), ctypes.c_float(beta), splits, stream)


def test_two_calls_match_existing_entry_point(L):
    t = torch()
    stream = t.cuda.current_stream().cuda_stream
    prepared = []
    for i, (M, N, K, alpha, beta, splits) in enumerate(CASES):
        A, B, C0 = operands(900 + i, M, N, K, K, N, N, np.float16)
        dA, dB = to_dev(A), to_dev(B)
        prepared.append((A, B, C0, dA, dB, to_dev(C0), to_dev(C0)))
    # one call per case first: the per-device set-up, and the CUDA runtime
    # loading each kernel's code on its first launch, may take device memory
    for w, case in zip(prepared, CASES):
        warm = to_dev(w[2])
        assert _noalloc(L, w[3], w[4], warm, *case[:5], case[5], stream) == 0
    t.cuda.synchronize()
    free_before = t.cuda.mem_get_info()[0]

    # two calls in a row on the shared scratch array
    for (A, B, C0, dA, dB, dC_new, _), (M, N, K, alpha, beta, splits) in zip(prepared, CASES):
        assert _noalloc(L, dA, dB, dC_new, M, N, K, alpha, beta, splits, stream) == 0
    t.cuda.synchronize()
    assert t.cuda.mem_get_info()[0] == free_before

    import dense_gemm_03_gb300 as g
    assert g.debug_status() == 0
    for (A, B, C0, dA, dB, dC_new, dC_old), (M, N, K, alpha, beta, splits) in zip(prepared, CASES):
        assert L.gemm_f16_ld(dA.data_ptr(), dB.data_ptr(), dC_old.data_ptr(), M, N, K, K, N, N,
                             ctypes.c_float(alpha), ctypes.c_float(beta), stream) == 0
        t.cuda.synchronize()
        new = dC_new.cpu().numpy().astype(np.float64)
        old = dC_old.cpu().numpy().astype(np.float64)
        ref, absd = oracle.gemm(A, B, C0, alpha, beta, with_absdot=True)
        r = oracle.compare(new, old, oracle.tol_f16(ref, absd))
        assert r["ok"], r


def test_too_large_is_refused(L):
    t = torch()
    M = N = 2048
    K = 4096
    dA = t.zeros((M, K), dtype=t.float16, device="cuda")
    dB = t.zeros((K, N), dtype=t.float16, device="cuda")
    dC = t.full((M, N), 7.0, dtype=t.float16, device="cuda")
    # 2 slices x 2048 x 2048 x 4 bytes = 32 MiB > the 8 MiB array
    assert _noalloc(L, dA, dB, dC, M, N, K, 1.0, 0.0, 2, None) == -7
    t.cuda.synchronize()
    assert bool((dC == 7.0).all())
