"""Failure detection on the GPU without a fault: a bounded wait that nothing
releases gives up, the kernel reports GEMM_ERR_TIMEOUT through the device
status word and returns normally, and the context keeps working."""
import time

import numpy as np
import pytest

from helpers import check, operands, run

pytestmark = pytest.mark.gpu

GEMM_ERR_TIMEOUT = -6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_03_gb300 import build
    build.build()


def test_wait_that_nothing_releases_reports_timeout_and_context_survives():
    import dense_gemm_03_gb300 as g
    assert g.debug_status() == 0          # clean start (reading also clears)
    t0 = time.perf_counter()
    g.debug_wait_probe(1_000_000)         # gives up after about a millisecond
    assert g.debug_status() == GEMM_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    assert g.debug_status() == 0          # the status word was cleared by the read
    # the same context still computes correctly
    M, N, K = 300, 520, 200
    A, B, C0 = operands(123, M, N, K, K, N, N, np.float16)
    got, _ = run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N)
    check("f16", got, A, B, C0, 1.5, 0.5, M, N, K, K, N, N)


def test_wait_probe_rejects_nonpositive_limit():
    import dense_gemm_03_gb300 as g
    assert g.lib().gemm_debug_wait_probe(0, None) == -7
