"""The GEMM captured in a CUDA graph and replayed: schedules whose shared
tiles count their pieces in device counters (stream-K, K slices) must give
the right result on every replay, with new operands each time."""
import numpy as np
import pytest

import oracle
from helpers import check, operands, torch

pytestmark = pytest.mark.gpu

AUTO, SPLITK, TAIL2, SK_ALL = 0, 3, 9, 11


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_03_gb300 import build
    build.build()


@pytest.mark.parametrize("M,N,K,path,mark", [
    (16, 8192, 8192, AUTO, ".sk"),
    (300, 500, 3000, SPLITK, ".splitk"),
    (2000, 2600, 4096, TAIL2, ".tail"),
    (2000, 2600, 4096, AUTO, ".ktail"),
    (2000, 2600, 4096, 14, ".sktail"),
    (64, 128, 4096, SK_ALL, ".sk"),
    (4096, 64, 2048, AUTO, ".kb2"),      # whole 64-wide tiles, two k-blocks per ring stage
    (4096, 64, 2048, 17, ".m64"),        # 64-row tiles
])
def test_graph_replays(M, N, K, path, mark):
    import dense_gemm_03_gb300 as g
    t = torch()
    s = t.cuda.Stream()
    dA = t.empty((M, K), dtype=t.float16, device="cuda")
    dB = t.empty((K, N), dtype=t.float16, device="cuda")
    dC = t.empty((M, N), dtype=t.float16, device="cuda")
    prev = g.force_path(path)
    try:
        # a first call outside the capture sets up scratch buffers and counters
        A, B, C0 = operands(5000, M, N, K, K, N, N, np.float16)
        dA.copy_(t.from_numpy(A)); dB.copy_(t.from_numpy(B)); dC.copy_(t.from_numpy(C0))
        g.gemm_f16(dA, dB, dC, 0.75, -0.25, stream=s)
        s.synchronize()
        assert mark in g.last_path()
        graph = t.cuda.CUDAGraph()
        with t.cuda.graph(graph, stream=s):
            g.gemm_f16(dA, dB, dC, 0.75, -0.25, stream=s)
    finally:
        g.force_path(prev)
    for i in range(3):
        A, B, C0 = operands(5001 + i, M, N, K, K, N, N, np.float16)
        dA.copy_(t.from_numpy(A)); dB.copy_(t.from_numpy(B)); dC.copy_(t.from_numpy(C0))
        t.cuda.synchronize()
        graph.replay()
        t.cuda.synchronize()
        got = dC.cpu().numpy()
        big = M * N * K > 2e9
        check("f16", got, A, B, C0, 0.75, -0.25, M, N, K, K, N, N,
              rows=oracle.sample_rows(M) if big else None, cols=oracle.sample_cols(N) if big else None)
    assert g.debug_status() == 0


@pytest.mark.parametrize("M,N,K,mark", [(600, 700, 4000, ".ksplit"), (2560, 2304, 2048, ".ktail")])
def test_graph_replays_fp32_k_slices(M, N, K, mark):
    """The fp32 tensor-core path with K slices (few pair tiles) or with the
    last wave's tiles in two K slices inside a graph: the operand split, the
    sliced kernel and its counters replay correctly."""
    import dense_gemm_03_gb300 as g
    t = torch()
    s = t.cuda.Stream()
    dA = t.empty((M, K), dtype=t.float32, device="cuda")
    dB = t.empty((K, N), dtype=t.float32, device="cuda")
    dC = t.empty((M, N), dtype=t.float32, device="cuda")
    A, B, C0 = operands(6000, M, N, K, K, N, N, np.float32)
    dA.copy_(t.from_numpy(A)); dB.copy_(t.from_numpy(B)); dC.copy_(t.from_numpy(C0))
    g.sgemm_f32(dA, dB, dC, 0.75, -0.25, stream=s)
    s.synchronize()
    assert g.last_path().endswith(mark), g.last_path()
    graph = t.cuda.CUDAGraph()
    with t.cuda.graph(graph, stream=s):
        g.sgemm_f32(dA, dB, dC, 0.75, -0.25, stream=s)
    for i in range(3):
        A, B, C0 = operands(6001 + i, M, N, K, K, N, N, np.float32)
        dA.copy_(t.from_numpy(A)); dB.copy_(t.from_numpy(B)); dC.copy_(t.from_numpy(C0))
        t.cuda.synchronize()
        graph.replay()
        t.cuda.synchronize()
        check("f32", dC.cpu().numpy(), A, B, C0, 0.75, -0.25, M, N, K, K, N, N,
              rows=oracle.sample_rows(M, block=64) if M * N * K > 2e9 else None)
    assert g.debug_status() == 0
