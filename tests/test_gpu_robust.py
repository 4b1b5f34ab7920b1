"""Robustness through the C ABI: concurrent calls from several host threads on
their own streams (per-stream scratch and counters), and operands larger
than 2^31 elements (64-bit offsets everywhere)."""
import threading

import numpy as np
import pytest

import oracle
import synthetic
from helpers import check, operands, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_03_gb300 import build
    build.build()


def test_concurrent_threads_own_streams():
    """Five threads, each on its own stream, repeatedly run shapes whose tiles
    are shared out (stream-K, half-width units, 3xTF32 whole-K and K slices);
    every result checks against the oracle."""
    import dense_gemm_03_gb300 as g
    t = torch()
    cases = [
        ("f16", 16, 8192, 8192), ("f16", 2000, 2600, 1024), ("f32", 700, 900, 500),
        ("f16", 1000, 1001, 4096), ("f32", 600, 700, 2000),
    ]
    prepared = []
    for i, (kind, M, N, K) in enumerate(cases):
        dt = np.float16 if kind == "f16" else np.float32
        A, B, C0 = operands(7000 + i, M, N, K, K, N, N, dt)
        prepared.append((kind, M, N, K, A, B, C0))
    errors = []

    def worker(idx):
        try:
            kind, M, N, K, A, B, C0 = prepared[idx]
            s = t.cuda.Stream()
            dA, dB = t.from_numpy(A).cuda(), t.from_numpy(B).cuda()
            fn = g.gemm_f16 if kind == "f16" else g.sgemm_f32
            for _ in range(5):
                dC = t.from_numpy(C0).cuda()
                with t.cuda.stream(s):
                    fn(dA, dB, dC, 0.75, -0.25, stream=s)
                s.synchronize()
                got = dC.cpu().numpy()
                big = M * N * K > 2e9
                check(kind, got, A, B, C0, 0.75, -0.25, M, N, K, K, N, N,
                      rows=oracle.sample_rows(M) if big else None,
                      cols=oracle.sample_cols(N) if big else None)
        except Exception as e:   # reported on the main thread
            errors.append((idx, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(prepared))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert g.debug_status() == 0


def test_operand_beyond_2_pow_31_elements():
    """A has 40000 x 60000 = 2.4e9 halves (4.8 GB): rows past element 2^31 are
    only reached with 64-bit offsets.  A's rows repeat a seeded block of 1021
    rows (a prime, so a wrapped 32-bit offset would land on another row)."""
    import dense_gemm_03_gb300 as g
    t = torch()
    M, N, K = 40000, 256, 60000
    base = synthetic.uniform(8001, synthetic.STREAM_A, (1021, K), dtype=np.float16)
    B = synthetic.uniform(8001, synthetic.STREAM_B, (K, N), dtype=np.float16)
    C0 = synthetic.uniform(8001, synthetic.STREAM_C, (M, N), dtype=np.float16)
    dbase = t.from_numpy(base).cuda()
    reps = (M + 1020) // 1021
    dA = dbase.repeat(reps, 1)[:M].contiguous()
    del dbase
    dB = t.from_numpy(B).cuda()
    dC = t.from_numpy(C0).cuda()
    g.gemm_f16(dA, dB, dC, 1.5, 0.5)
    t.cuda.synchronize()
    assert g.debug_status() == 0
    got = dC.cpu().numpy()
    del dA
    # rows whose first element lies beyond 2^31 elements, and a few before
    rows = [0, 1, 17000, 35791, 35792, 39999] + list(range(39000, 40000, 97))
    A_rows = base[np.array(rows) % 1021]
    ref, absd = oracle.gemm(A_rows, B, C0[rows], 1.5, 0.5, with_absdot=True)
    r = oracle.compare(got[rows].astype(np.float64), ref, oracle.tol_f16(ref, absd))
    assert r["ok"], r
    assert 35792 * K > 2 ** 31
