"""Parity of the half-precision path (gemm_f16 / gemm_f16_ld) with the CPU
oracle, through the C ABI, on every kernel path: TMA loads, predicated loads
(unaligned operands), split-K, and the scale-only case."""
import numpy as np
import pytest

import oracle
import synthetic
from helpers import check, operands, padding_untouched, run, to_dev, torch

pytestmark = pytest.mark.gpu

AUTO, MANUAL, SPLITK = 0, 2, 3
NO_TAIL, NO_PAIR, TAIL2, SK, SK_ALL, SKTAIL, HALVES, M64 = 5, 6, 9, 10, 11, 14, 15, 17


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dense_gemm_03_gb300 import build
    build.build()


def _exact16(ref):
    return ref.astype(np.float16)


def test_identity_one_tile_is_exact():
    M = K = 128
    N = 256
    A = np.eye(M, dtype=np.float16)
    B = synthetic.uniform(1, 2, (K, N), dtype=np.float16)
    C0 = np.full((M, N), np.nan, dtype=np.float16)
    got, path = run("f16", A, B, C0, 1.0, 0.0, M, N, K, K, N, N)
    assert "tma" in path
    assert np.array_equal(got.view(np.uint16), B.view(np.uint16))


@pytest.mark.parametrize("path", [AUTO, MANUAL])
def test_permutation_is_exact(path):
    M = K = 384
    N = 320
    rng = np.random.default_rng(5)
    p = rng.permutation(K)
    A = np.zeros((M, K), np.float16)
    A[np.arange(M), p] = 1.0
    B = synthetic.uniform(2, 2, (K, N), dtype=np.float16)
    C0 = np.zeros((M, N), np.float16)
    got, _ = run("f16", A, B, C0, 1.0, 0.0, M, N, K, K, N, N, path=path)
    assert np.array_equal(got.view(np.uint16), B[p].view(np.uint16))


@pytest.mark.parametrize("path", [AUTO, MANUAL, SPLITK])
@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (300, 700, 1000), (129, 65, 17), (1, 1, 1),
                                   (8, 8, 8), (130, 1000, 640)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (2.0, -1.0)])
def test_small_integers_bit_exact(path, M, N, K, alpha, beta):
    """Entries in {-1, 0, 1}: every partial sum is an integer below 2048, so
    the fp32 accumulation and the fp16 output are exact whatever the order."""
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = rng.integers(-1, 2, size=(M, K)).astype(np.float16)
    B = rng.integers(-1, 2, size=(K, N)).astype(np.float16)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float16)
    got, _ = run("f16", A, B, C0, alpha, beta, M, N, K, K, N, N, path=path,
                 splits=3 if path == SPLITK else 0)
    ref = oracle.gemm(A, B, C0, alpha, beta)
    assert np.array_equal(got.view(np.uint16), _exact16(ref).view(np.uint16))


@pytest.mark.parametrize("path", [AUTO, MANUAL, SPLITK])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (384, 640, 320), (129, 257, 65), (7, 9, 13),
                                   (300, 500, 1000), (1024, 1024, 1024), (200, 64, 2000),
                                   (64, 128, 4096)])
@pytest.mark.parametrize("alpha,beta,c_fill", [(1.5, 0.5, "uniform"), (1.0, 0.0, "nan"),
                                               (0.75, -0.25, "uniform")])
def test_random_parity(path, M, N, K, alpha, beta, c_fill):
    A, B, C0 = operands(100 + M + N + K, M, N, K, K, N, N, np.float16, c_fill=c_fill)
    got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, K, N, N, path=path,
                     splits=4 if path == SPLITK else 0)
    if path == MANUAL:
        assert "manual" in taken
    if path == SPLITK and (K + 63) // 64 >= 2:
        assert "splitk" in taken
    check("f16", got, A, B, C0, alpha, beta, M, N, K, K, N, N)


@pytest.mark.parametrize("M,N,K,lda,ldb,ldc", [
    (257, 255, 77, 80, 255, 255),        # nothing 16-byte aligned: predicated path
    (200, 300, 150, 153, 305, 301),      # padding everywhere
    (130, 190, 100, 104, 192, 200),      # strides 16-byte aligned, ld > cols
    (64, 70, 64, 64, 71, 77),
])
@pytest.mark.parametrize("alpha,beta", [(0.75, -0.25), (1.0, 0.0)])
def test_leading_dimensions(M, N, K, lda, ldb, ldc, alpha, beta):
    A, B, C0 = operands(7 + lda + ldb, M, N, K, lda, ldb, ldc, np.float16)
    got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc)
    check("f16", got, A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc)
    assert padding_untouched(got, C0, N)


def test_misaligned_base_pointers():
    """Operands starting 2 bytes past a 16-byte boundary: A and B go through
    aligned copies, and C through an aligned copy that is copied back."""
    t = torch()
    M, N, K = 150, 200, 90
    A, B, C0 = operands(31, M, N, K, K, N, N, np.float16)
    import dense_gemm_03_gb300 as g
    bufs = [t.zeros(x.size + 8, dtype=t.float16, device="cuda") for x in (A, B, C0)]
    for buf, x in zip(bufs, (A, B, C0)):
        buf[1:1 + x.size].copy_(t.from_numpy(x.reshape(-1)).cuda())
    es = bufs[0].element_size()
    g.gemm_f16(bufs[0].data_ptr() + es, bufs[1].data_ptr() + es, bufs[2].data_ptr() + es,
               1.5, 0.5, M=M, N=N, K=K)
    assert g.last_path().endswith(".realigned.c"), g.last_path()
    t.cuda.synchronize()
    got = bufs[2][1:1 + C0.size].cpu().numpy().reshape(M, N)
    check("f16", got, A, B, C0, 1.5, 0.5, M, N, K, K, N, N)


def test_alpha_zero_and_K_zero_scale_C():
    M, N, K = 100, 130, 40
    A, B, C0 = operands(9, M, N, K, K, N, N, np.float16)
    A[:] = np.nan
    got, path = run("f16", A, B, C0, 0.0, -0.25, M, N, K, K, N, N)
    assert path == "f16.scale"
    assert np.array_equal(got.view(np.uint16), (C0.astype(np.float64) * -0.25).astype(np.float16).view(np.uint16))
    got, _ = run("f16", A[:, :0], B[:0], C0, 1.5, 0.5, M, N, 0, 1, N, N)
    assert np.array_equal(got.view(np.uint16), (C0.astype(np.float64) * 0.5).astype(np.float16).view(np.uint16))
    got, _ = run("f16", A, B, C0, 0.0, 0.0, M, N, K, K, N, N)
    assert not got.any()


def test_empty_is_noop():
    t = torch()
    import dense_gemm_03_gb300 as g
    C = t.full((4, 4), 3.0, dtype=t.float16, device="cuda")
    g.gemm_f16(C, C, C, 1.0, 1.0, M=0, N=4, K=4)
    g.gemm_f16(C, C, C, 1.0, 1.0, M=4, N=0, K=4)
    assert g.last_path() == "noop"
    assert bool((C == 3.0).all())


def test_deterministic():
    M, N, K = 512, 768, 2048
    A, B, C0 = operands(3, M, N, K, K, N, N, np.float16)
    r1, _ = run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N)
    r2, _ = run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N)
    assert np.array_equal(r1.view(np.uint16), r2.view(np.uint16))
    s1, _ = run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=SPLITK, splits=5)
    s2, _ = run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=SPLITK, splits=5)
    assert np.array_equal(s1.view(np.uint16), s2.view(np.uint16))


def test_host_form_matches_device_form():
    import dense_gemm_03_gb300 as g
    t = torch()
    M, N, K = 333, 444, 555
    A, B, C0 = operands(21, M, N, K, K, N, N, np.float16)
    dev, _ = run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N)
    hA = t.from_numpy(A).pin_memory()
    hB = t.from_numpy(B).pin_memory()
    hC = t.from_numpy(C0.copy()).pin_memory()
    g.gemm_f16_host(hA, hB, hC, 1.5, 0.5, M=M, N=N, K=K)
    assert np.array_equal(hC.numpy().view(np.uint16), dev.view(np.uint16))


@pytest.mark.parametrize("M,N,K,ldc", [(4096, 1024, 512, 1024), (2100, 777, 300, 800)])
def test_host_form_in_row_blocks(M, N, K, ldc):
    """M >= 2048: four row blocks copied in, computed and copied back in turn;
    the result matches the oracle, and C's padding comes back unchanged."""
    import dense_gemm_03_gb300 as g
    t = torch()
    A, B, C0 = operands(808 + M, M, N, K, K, N, ldc, np.float16)
    hA = t.from_numpy(A).pin_memory()
    hB = t.from_numpy(B).pin_memory()
    hC = t.from_numpy(C0.copy()).pin_memory()
    g.gemm_f16_host(hA, hB, hC, 0.75, -0.25, M=M, N=N, K=K, ldc=ldc)
    got = hC.numpy()
    check("f16", got, A, B, C0, 0.75, -0.25, M, N, K, K, N, ldc,
          rows=oracle.sample_rows(M, block=64), cols=oracle.sample_cols(N))
    assert padding_untouched(got, C0, N)
    assert g.debug_status() == 0


def test_streams_are_respected():
    """Work goes on the caller's stream: a GEMM enqueued on a side stream after
    an event sees the inputs the main stream wrote before it."""
    import dense_gemm_03_gb300 as g
    t = torch()
    M, N, K = 256, 256, 512
    A, B, C0 = operands(4, M, N, K, K, N, N, np.float16)
    dA, dB = to_dev(A), to_dev(B)
    dC = t.zeros((M, N), dtype=t.float16, device="cuda")
    s = t.cuda.Stream()
    dA2 = t.empty_like(dA)
    dA2.copy_(dA)
    ev = t.cuda.Event()
    ev.record()
    s.wait_event(ev)
    with t.cuda.stream(s):
        g.gemm_f16(dA2, dB, dC, 1.0, 0.0, M=M, N=N, K=K, stream=s)
    s.synchronize()
    check("f16", dC.cpu().numpy(), A, B, np.zeros((M, N), np.float16), 1.0, 0.0, M, N, K, K, N, N)


# ---------------------------------------------------------------- last-wave balancing
@pytest.mark.parametrize("path,mark", [(AUTO, ".ktail"), (TAIL2, ".tail"), (SK, ".sk"),
                                       (SKTAIL, ".sktail"), (HALVES, ".halves")])
@pytest.mark.parametrize("M,N,K,lda,ldb,ldc", [
    (2000, 2600, 4096, 4096, 2600, 2600),     # 176 tiles: the last 24 cut into 2 K slices
    (2000, 2600, 4100, 4104, 2600, 2600),     # ragged last k-block
    (2000, 2601, 4096, 4096, 2601, 2601),     # N % 8 != 0: predicated epilogue
    (2000, 2600, 4096, 4097, 2600, 2600),     # odd lda: predicated loads
    (1300, 4000, 4096, 4104, 4008, 4000),     # padded operands
])
@pytest.mark.parametrize("alpha,beta,c_fill", [(1.5, 0.5, "uniform"), (1.0, 0.0, "nan")])
def test_tail_parity(path, mark, M, N, K, lda, ldb, ldc, alpha, beta, c_fill):
    """The last wave balanced by two K slices per tile (the first one worker's
    first unit, the second another worker's last), by two K slices run at the
    end, by stream-K over the last two waves or over the last wave (each worker
    runs the piece that starts a tile first and the piece that ends one last),
    or by half-width units; against the oracle and against whole tiles."""
    A, B, C0 = operands(40 + M + N + lda, M, N, K, lda, ldb, ldc, np.float16, c_fill=c_fill)
    got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, path=path)
    assert mark in taken, taken
    check("f16", got, A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc,
          rows=oracle.sample_rows(M, block=64), cols=oracle.sample_cols(N, block=32))
    assert padding_untouched(got, C0, N)
    whole, taken2 = run("f16", A, B, C0, alpha, beta, M, N, K, lda, ldb, ldc, path=NO_TAIL)
    assert ".tail" not in taken2 and ".sk" not in taken2
    ref, absd = oracle.gemm(A, B, C0, alpha, beta, M=M, N=N, K=K, lda=lda, ldb=ldb, ldc=ldc,
                            rows=list(range(0, M, 97)), with_absdot=True)
    r = oracle.compare(got[::97, :N].astype(np.float64), whole[::97, :N].astype(np.float64),
                       oracle.tol_f16(ref, absd))
    assert r["ok"], r


@pytest.mark.parametrize("path,mark", [(AUTO, ".ktail"), (TAIL2, ".tail"), (SK, ".sk"),
                                       (SKTAIL, ".sktail"), (HALVES, ".halves")])
def test_tail_deterministic(path, mark):
    """Shared tiles are summed in k order whichever piece finishes last (and
    whether or not the finishing piece published its own partial sums), so
    repeated calls give the same bits."""
    M, N, K = 2000, 3000, 4096
    A, B, C0 = operands(77, M, N, K, K, N, N, np.float16)
    r1, taken = run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=path)
    assert mark in taken
    for _ in range(3):
        r2, _ = run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=path)
        assert np.array_equal(r1.view(np.uint16), r2.view(np.uint16))
    check("f16", r1, A, B, C0, 1.5, 0.5, M, N, K, K, N, N,
          rows=oracle.sample_rows(M), cols=oracle.sample_cols(N))


@pytest.mark.parametrize("M,N,K,path,mark", [
    (2000, 2600, 4096, SK, ".pair.bn256.tma.epi_tma.sk"),    # CTA pairs, last waves shared
    (2000, 2601, 2048, SK, ".epi_tma.sk.realigned.c"),      # N % 8 != 0: C through an aligned copy
    (2000, 2600, 4096, AUTO, ".pair.bn256.tma.epi_tma.ktail"),    # 88 pair tiles: 12 in two slices
    (2000, 2600, 4096, SKTAIL, ".pair.bn256.tma.epi_tma.sktail"), # 12 shared out as stream-K
    (4096, 4096, 4096, AUTO, ".pair.bn256.tma.epi_tma.ktail"),    # 256 pair tiles: 28 in two slices
    (20000, 128, 4096, AUTO, ".bn128.tma.epi_tma.ktail"),         # 157 CTA tiles: 5 in two slices
    (20000, 128, 2048, AUTO, ".bn128.tma.epi_tma.halves"),        # a shorter K: halved instead
    (2560, 2560, 1024, AUTO, ".pair.bn256.tma.epi_tma.halves"),   # 100 pair tiles: 24 halved
    (2000, 2600, 4096, HALVES, ".pair.bn256.tma.epi_tma.halves"), # 88 pair tiles: 12 halved
    (2560, 2560, 1024, NO_PAIR, ".bn256.tma.epi_tma.halves"),     # 200 CTA tiles
    (3300, 2001, 700, AUTO, ".halves.realigned.c"),               # every operand realigned, halved
    (3300, 2001, 700, MANUAL, ".manual.epi_manual"),              # predicated loads and epilogue
    (16, 8192, 8192, AUTO, ".bn128.tma.epi_tma.a32.sk"),   # skinny: every tile shared
    (4096, 64, 8192, AUTO, ".bn64.tma.epi_tma.sk"),      # tall, long K: every tile shared
    (4096, 64, 2048, AUTO, ".bn64.tma.epi_tma"),         # tall, shorter K: one wave of whole tiles
    (4096, 64, 2048, M64, ".bn64.tma.epi_tma.m64"),      # the same on 64-row tiles
    (64, 128, 4096, SK_ALL, ".sk"),                      # one tile cut into 16 pieces
    (100, 300, 1000, SK_ALL, ".sk"),                     # ragged, small
    (64, 128, 4096, AUTO, ".halves"),                    # the same, as two half-width units
    (1024, 1024, 1024, AUTO, ".pair.bn256.tma.epi_tma.halves"),   # few tiles, short K
])
def test_balanced_schedules_integers_exact(M, N, K, path, mark):
    """Entries in {-1, 0, 1}: partial sums are integers below 2^24, exact in
    fp32 however the k-blocks are shared out, so C is exactly the oracle's
    value rounded once to half."""
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A = rng.integers(-1, 2, size=(M, K)).astype(np.float16)
    B = rng.integers(-1, 2, size=(K, N)).astype(np.float16)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float16)
    got, taken = run("f16", A, B, C0, 2.0, -1.0, M, N, K, K, N, N, path=path)
    assert mark in taken, taken
    rows = list(range(M)) if M * N * K <= 4e9 else oracle.sample_rows(M, block=32)
    ref = oracle.gemm(A, B, C0, 2.0, -1.0, rows=rows)
    assert np.array_equal(got[rows].view(np.uint16), _exact16(ref).view(np.uint16))


# ---------------------------------------------------------------- CTA pairs (cta_group::2)


@pytest.mark.parametrize("M,N,K,ldc", [
    (512, 512, 128, 512),        # one pair tile per cluster
    (384, 768, 640, 768),        # 1.5 pair rows: the second CTA of the last pair is half empty
    (300, 1000, 1000, 1000),     # ragged everything
    (257, 512, 256, 512),        # the second CTA of the last pair has one row
    (1000, 1001, 700, 1001),     # N % 8 != 0: predicated epilogue on pairs
    (2048, 2048, 4096, 2048),    # 64 pair tiles, one partial wave
])
@pytest.mark.parametrize("alpha,beta,c_fill", [(1.5, 0.5, "uniform"), (1.0, 0.0, "nan")])
def test_pair_parity(M, N, K, ldc, alpha, beta, c_fill):
    """Whole tiles forced (no stream-K), so that even the shapes with few tiles
    run on CTA pairs."""
    A, B, C0 = operands(60 + M + N + K, M, N, K, K, N, ldc, np.float16, c_fill=c_fill)
    got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, K, N, ldc, path=NO_TAIL)
    if (M + 127) // 128 >= 2 and N > 128:
        assert ".pair." in taken, taken
    big = M * N * K > 2e9
    check("f16", got, A, B, C0, alpha, beta, M, N, K, K, N, ldc,
          rows=oracle.sample_rows(M) if big else None, cols=oracle.sample_cols(N) if big else None)
    assert padding_untouched(got, C0, N)


def test_pair_identity_exact():
    M = K = 768
    N = 512
    A = np.eye(M, dtype=np.float16)
    B = synthetic.uniform(9, 2, (K, N), dtype=np.float16)
    C0 = np.full((M, N), np.nan, dtype=np.float16)
    import dense_gemm_03_gb300 as g
    got, taken = run("f16", A, B, C0, 1.0, 0.0, M, N, K, K, N, N, path=NO_TAIL)
    assert ".pair." in taken
    assert np.array_equal(got.view(np.uint16), B.view(np.uint16))


def test_pair_matches_single_cta_and_is_deterministic():
    M, N, K = 1536, 2048, 1024
    A, B, C0 = operands(61, M, N, K, K, N, N, np.float16)
    p1, t1 = run("f16", A, B, C0, 0.75, -0.25, M, N, K, K, N, N)
    p2, _ = run("f16", A, B, C0, 0.75, -0.25, M, N, K, K, N, N)
    s1, t2 = run("f16", A, B, C0, 0.75, -0.25, M, N, K, K, N, N, path=NO_PAIR)
    assert ".pair." in t1 and ".pair." not in t2
    assert np.array_equal(p1.view(np.uint16), p2.view(np.uint16))
    # same products, possibly another summation order inside the tensor core
    ref, absd = oracle.gemm(A, B, C0, 0.75, -0.25, rows=list(range(0, M, 61)), with_absdot=True)
    r = oracle.compare(p1[::61].astype(np.float64), s1[::61].astype(np.float64), oracle.tol_f16(ref, absd))
    assert r["ok"], r


# ---------------------------------------------------------------- unaligned operands (realigned copies)
@pytest.mark.parametrize("offset_elems", [1, 2, 3, 7])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (7, 9, 13), (130, 1023, 777)])
def test_realigned_base_offsets(offset_elems, M, N, K):
    """A and B start 2, 4, 6 or 14 bytes past a 16-byte boundary (every
    misalignment the copy has to shift away); C stays aligned."""
    import dense_gemm_03_gb300 as g
    t = torch()
    A, B, C0 = operands(70 + offset_elems + M, M, N, K, K, N, N, np.float16)
    bufs = []
    for x in (A, B):
        buf = t.zeros(x.size + 16, dtype=t.float16, device="cuda")
        buf[offset_elems:offset_elems + x.size].copy_(t.from_numpy(x.reshape(-1)).cuda())
        bufs.append(buf)
    dC = to_dev(C0)
    es = 2
    g.gemm_f16(bufs[0].data_ptr() + es * offset_elems, bufs[1].data_ptr() + es * offset_elems, dC,
               0.75, -0.25, M=M, N=N, K=K)
    assert ".realigned" in g.last_path(), g.last_path()
    t.cuda.synchronize()
    check("f16", dC.cpu().numpy(), A, B, C0, 0.75, -0.25, M, N, K, K, N, N)


def test_odd_pointers_are_rejected():
    import dense_gemm_03_gb300 as g
    t = torch()
    buf = t.zeros(4096, dtype=t.float16, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16(buf.data_ptr() + 1, buf, buf[1024:], 1.0, 0.0, M=8, N=8, K=8)
    assert e.value.code == -7
    f = t.zeros(4096, dtype=t.float32, device="cuda")
    with pytest.raises(g.GemmError):
        g.sgemm_f32(f, f.data_ptr() + 2, f[1024:], 1.0, 0.0, M=8, N=8, K=8)


# ---------------------------------------------------------------- skinny shapes (A rows staged: 32 or 64)
@pytest.mark.parametrize("M,N,K,mark", [
    (1, 300, 2000, ".a32"),
    (16, 8192, 2048, ".a32"),
    (31, 1000, 700, ".a32"),
    (32, 1000, 700, ".a32"),
    (33, 1000, 700, ".a64"),
    (64, 4096, 1024, ".a64"),
    (17, 1001, 513, ".a32"),                # N % 8 != 0: C through an aligned copy
])
@pytest.mark.parametrize("alpha,beta,c_fill", [(1.5, 0.5, "uniform"), (1.0, 0.0, "nan")])
def test_skinny_parity(M, N, K, mark, alpha, beta, c_fill):
    """At most 64 rows: only the rows of A that exist are staged; the MMA's
    other rows read the stage's B region and must never reach C."""
    A, B, C0 = operands(900 + M + N, M, N, K, K, N, N, np.float16, c_fill=c_fill)
    got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, K, N, N)
    assert mark in taken, taken
    check("f16", got, A, B, C0, alpha, beta, M, N, K, K, N, N)


# ---------------------------------------------------------------- extreme dimensions
@pytest.mark.parametrize("M,N,K", [
    (4096, 1024, 1),       # K = 1: one ragged k-block, realigned operands
    (1, 1, 65536),         # one output, a very long K
    (1, 16384, 256),       # one row
    (3, 5, 100003),        # ragged everything, long K
    (16384, 1, 64),        # one column
])
def test_extreme_dimensions(M, N, K):
    A, B, C0 = operands(31337 + M + N, M, N, K, K, N, N, np.float16)
    got, taken = run("f16", A, B, C0, 0.75, -0.25, M, N, K, K, N, N)
    check("f16", got, A, B, C0, 0.75, -0.25, M, N, K, K, N, N)


# ---------------------------------------------------------------- narrower CTA-pair tiles (224, 192)
W224, W192 = 12, 13


@pytest.mark.parametrize("width,path", [(224, W224), (192, W192)])
@pytest.mark.parametrize("M,N,K,ldc", [
    (512, 448, 128, 448),        # exactly two 224-wide tiles
    (600, 1000, 300, 1000),      # ragged rows, columns and k-blocks
    (257, 300, 640, 304),        # the second CTA of the last pair has one row; padded C
    (1000, 1001, 700, 1001),     # N % 8 != 0: predicated epilogue
    (4096, 4096, 512, 4096),     # several waves; the last column tile 64 (224) or 64 (192) wide
])
@pytest.mark.parametrize("alpha,beta,c_fill", [(1.5, 0.5, "uniform"), (1.0, 0.0, "nan")])
def test_narrow_pair_tiles_parity(width, path, M, N, K, ldc, alpha, beta, c_fill):
    """Pair tiles of 256 x 224 and 256 x 192: each CTA stages two whole
    64-column boxes of B and the MMA reads the first 112 or 96 columns; the
    epilogue splits the unit's 7 or 6 column chunks between two warps per row
    quadrant."""
    A, B, C0 = operands(70 + M + N + K + width, M, N, K, K, N, ldc, np.float16, c_fill=c_fill)
    got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, K, N, ldc, path=path)
    assert ".pair.bn%d." % width in taken, taken
    big = M * N * K > 2e9
    check("f16", got, A, B, C0, alpha, beta, M, N, K, K, N, ldc,
          rows=oracle.sample_rows(M) if big else None, cols=oracle.sample_cols(N) if big else None)
    assert padding_untouched(got, C0, N)


@pytest.mark.parametrize("path", [W224, W192])
def test_narrow_pair_tiles_integers_exact(path):
    M, N, K = 700, 900, 1000
    rng = np.random.default_rng(path)
    A = rng.integers(-1, 2, size=(M, K)).astype(np.float16)
    B = rng.integers(-1, 2, size=(K, N)).astype(np.float16)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float16)
    got, taken = run("f16", A, B, C0, 2.0, -1.0, M, N, K, K, N, N, path=path)
    assert ".pair.bn" in taken and ".bn256" not in taken, taken
    ref = oracle.gemm(A, B, C0, 2.0, -1.0)
    assert np.array_equal(got.view(np.uint16), _exact16(ref).view(np.uint16))


def test_narrow_pair_tiles_match_256_wide_bitwise_on_integers():
    """The same integer problem through 256-, 224- and 192-wide pair tiles gives
    the same bits (every partial sum exact)."""
    M, N, K = 1024, 1344, 512
    rng = np.random.default_rng(3)
    A = rng.integers(-2, 3, size=(M, K)).astype(np.float16)
    B = rng.integers(-2, 3, size=(K, N)).astype(np.float16)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float16)
    outs = [run("f16", A, B, C0, 1.0, 1.0, M, N, K, K, N, N, path=p)[0] for p in (NO_TAIL, W224, W192)]
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    assert np.array_equal(outs[0].view(np.uint16), outs[2].view(np.uint16))


# ---------------------------------------------------------------- C off the 16-byte grid: copied back
@pytest.mark.parametrize("offset_elems", [1, 3, 7])
@pytest.mark.parametrize("M,N,ldc", [(300, 1000, 1003), (257, 9, 13), (64, 1, 1), (130, 520, 523),
                                     (600, 1024, 1025)])
@pytest.mark.parametrize("beta", [0.5, 0.0])
def test_unaligned_c_copied_back(offset_elems, M, N, ldc, beta):
    """C starts 2, 6 or 14 bytes past a 16-byte boundary with an odd leading
    dimension: the kernel writes an aligned copy by TMA and a last kernel
    copies it back.  Every element outside C's columns -- before its first
    row, between its rows and after its last row -- keeps its sentinel."""
    import dense_gemm_03_gb300 as g
    t = torch()
    K = 200
    A, B, C0 = operands(90 + offset_elems + M + N, M, N, K, K, N, ldc, np.float16)
    pad = 64
    buf = np.full(C0.size + 2 * pad, np.nan, dtype=np.float16)
    buf.view(np.uint16)[:] = 0x7E55
    buf[pad + offset_elems:pad + offset_elems + C0.size] = C0.reshape(-1)
    dbuf = to_dev(buf)
    dA, dB = to_dev(A), to_dev(B)
    g.gemm_f16(dA, dB, dbuf.data_ptr() + 2 * (pad + offset_elems), 0.75, beta, M=M, N=N, K=K,
               lda=K, ldb=N, ldc=ldc)
    assert g.last_path().endswith(".c"), g.last_path()
    t.cuda.synchronize()
    assert g.debug_status() == 0
    out = dbuf.cpu().numpy()
    got = out[pad + offset_elems:pad + offset_elems + C0.size].reshape(M, ldc)
    check("f16", got, A, B, C0, 0.75, beta, M, N, K, K, N, ldc)
    assert padding_untouched(got, C0, N)
    ref_bits = buf.view(np.uint16)
    out_bits = out.view(np.uint16)
    assert np.array_equal(out_bits[:pad + offset_elems], ref_bits[:pad + offset_elems])
    assert np.array_equal(out_bits[pad + offset_elems + C0.size:], ref_bits[pad + offset_elems + C0.size:])


# ---------------------------------------------------------------- 64-row tiles (tcgen05.mma with M = 64)

@pytest.mark.parametrize("M,N,K,ldc", [
    (8192, 64, 4096, 64),     # the tall shape: 128 tiles, one wave of whole-K units
    (1000, 64, 700, 64),      # a 40-row last tile and a ragged k-block
    (64, 64, 64, 64),         # one tile, one k-block
    (4000, 40, 1000, 48),     # N < 64 with a padded C
    (129, 56, 4100, 56),      # three tiles, the last with one row; a long ragged K
])
@pytest.mark.parametrize("alpha,beta,c_fill", [(0.75, -0.25, "uniform"), (1.0, 0.0, "nan")])
def test_m64_tiles_parity(M, N, K, ldc, alpha, beta, c_fill):
    """64-row tiles: the M = 64 accumulator holds row 16q + l of the tile in
    TMEM lane 32q + l (l < 16) and each epilogue warp stores 16 rows; rows past
    M and the padding of C stay untouched."""
    A, B, C0 = operands(640 + M + N + K, M, N, K, K, N, ldc, np.float16, c_fill=c_fill)
    got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, K, N, ldc, path=M64)
    assert ".m64" in taken, taken
    big = M * N * K > 1e9
    check("f16", got, A, B, C0, alpha, beta, M, N, K, K, N, ldc,
          rows=oracle.sample_rows(M, block=16) if big else None)   # every 16-row quadrant
    assert padding_untouched(got, C0, N)


def test_m64_tiles_integers_exact():
    """Small integers: every partial sum is exact, so the 64-row tiles give
    the oracle's bits."""
    M, N, K = 3000, 64, 2000
    rng = np.random.default_rng(64)
    A = rng.integers(-2, 3, size=(M, K)).astype(np.float16)
    B = rng.integers(-2, 3, size=(K, N)).astype(np.float16)
    C0 = rng.integers(-3, 4, size=(M, N)).astype(np.float16)
    got, taken = run("f16", A, B, C0, 1.0, -1.0, M, N, K, K, N, N, path=M64)
    assert ".m64" in taken, taken
    ref = oracle.gemm(A, B, C0, 1.0, -1.0)
    assert np.array_equal(got.view(np.uint16), _exact16(ref).view(np.uint16))


@pytest.mark.parametrize("M,N,K,mark", [
    (8192, 64, 512, "f16.tc.bn64.tma.epi_tma"),        # 64 tiles of 8 k-blocks: whole tiles
    (8192, 64, 1024, "f16.tc.bn64.tma.epi_tma.kb2"),   # 16 k-blocks: two per ring stage
    (4096, 32, 2048, "f16.tc.bn64.tma.epi_tma.kb2"),
    (8192, 64, 4096, "f16.tc.bn64.tma.epi_tma.kb2"),
    (4096, 64, 8192, "f16.tc.bn64.tma.epi_tma.sk"),    # 32 tiles of 128: stream-K over every tile
    (512, 64, 16384, "f16.tc.bn64.tma.epi_tma.sk"),    # 4 tiles of 256 k-blocks
])
def test_tall_schedule_choice(M, N, K, mark):
    """64-wide tiles have no half-width units: stream-K is taken only when its
    ranges plus the fix-up of the shared tiles beat one wave of whole-K tiles,
    which stage two k-blocks at a time from 16 k-blocks on."""
    A, B, C0 = operands(1100 + M + N + K, M, N, K, K, N, N, np.float16)
    got, taken = run("f16", A, B, C0, 0.75, -0.25, M, N, K, K, N, N)
    assert taken == mark, taken
    big = M * N * K > 1e9
    check("f16", got, A, B, C0, 0.75, -0.25, M, N, K, K, N, N,
          rows=oracle.sample_rows(M, block=32) if big else None)


# ---------------------------------------------------------------- two k-blocks per ring stage
@pytest.mark.parametrize("M,N,K,ldc,path,kpb,mark", [
    (5000, 64, 1030, 64, AUTO, 0, ".bn64.tma.epi_tma.kb2"),    # 17 k-blocks: the last stage holds one
    (3000, 40, 2100, 48, AUTO, 0, ".bn64.tma.epi_tma.kb2"),    # N < 64, padded C, ragged last k-block
    (8192, 64, 4096, 64, AUTO, 0, ".bn64.tma.epi_tma.kb2"),
    (2000, 2600, 4100, 2600, AUTO, 2, ".pair.bn256.tma.epi_tma.kb2.ktail"),   # forced on pairs
    (600, 1000, 1000, 1000, NO_TAIL, 2, ".pair.bn256.tma.epi_tma.kb2"),
    (700, 64, 900, 64, SK_ALL, 2, ".bn64.tma.epi_tma.kb2.sk"),  # stream-K pieces of odd length
])
@pytest.mark.parametrize("alpha,beta,c_fill", [(0.75, -0.25, "uniform"), (1.0, 0.0, "nan")])
def test_two_kblocks_per_stage_parity(M, N, K, ldc, path, kpb, mark, alpha, beta, c_fill):
    """A ring stage holding two k-blocks (each A part followed by its B part),
    loaded and released as one; a unit with an odd number of k-blocks ends on
    a stage holding one."""
    import dense_gemm_03_gb300 as g
    A, B, C0 = operands(2200 + M + N + K, M, N, K, K, N, ldc, np.float16, c_fill=c_fill)
    prev = g.stage_kblocks(kpb)
    try:
        got, taken = run("f16", A, B, C0, alpha, beta, M, N, K, K, N, ldc, path=path)
    finally:
        g.stage_kblocks(prev)
    assert mark in taken, taken
    big = M * N * K > 1e9
    check("f16", got, A, B, C0, alpha, beta, M, N, K, K, N, ldc,
          rows=oracle.sample_rows(M, block=32) if big else None,
          cols=oracle.sample_cols(N, block=32) if big and N > 64 else None)
    assert padding_untouched(got, C0, N)


@pytest.mark.parametrize("M,N,K,path", [(3000, 64, 2000, AUTO), (1000, 1200, 1100, NO_TAIL)])
def test_two_kblocks_per_stage_bitwise_equal(M, N, K, path):
    """The MMAs run in the same order whatever the stage depth: one and two
    k-blocks per stage give the same bits."""
    import dense_gemm_03_gb300 as g
    A, B, C0 = operands(3300 + M + N + K, M, N, K, K, N, N, np.float16)
    outs = []
    for kpb in (1, 2):
        prev = g.stage_kblocks(kpb)
        try:
            outs.append(run("f16", A, B, C0, 1.5, 0.5, M, N, K, K, N, N, path=path))
        finally:
            g.stage_kblocks(prev)
    assert ".kb2" not in outs[0][1] and ".kb2" in outs[1][1], (outs[0][1], outs[1][1])
    assert np.array_equal(outs[0][0].view(np.uint16), outs[1][0].view(np.uint16))
