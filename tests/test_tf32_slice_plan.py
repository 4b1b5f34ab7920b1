"""Host-side K-slice planning of the fp32 tensor-core path (no GPU needed).

With few 256x256 tiles for the CTA pairs and a long K, every tile is cut into
equal K slices of whole 4-k-block accumulation chunks; the last slice of a
tile to finish adds the slices' partial sums.  These tests check the plans the
library makes: valid partitions of K, one wave of units, and the choice
between slicing and whole-K units for the shapes the GPU tests rely on."""
import itertools

import pytest

import dense_gemm_03_gb300 as g

PAIRS = 76   # CTA pairs resident at once on a GB300


def _plan(tiles, kb, forced=0, pairs=PAIRS):
    return g.plan_tf32_slices(tiles, pairs, kb, forced)


@pytest.mark.parametrize("tiles,kb,forced", list(itertools.product(
    [1, 2, 4, 9, 16, 20, 38], [8, 9, 16, 29, 32, 63, 64, 125, 129, 257, 512, 1000], [0, 2, 3, 7, 16])))
def test_slices_partition_k(tiles, kb, forced):
    p = _plan(tiles, kb, forced)
    s, per = p["splits"], p["kb_per_split"]
    if s == 1:
        assert per == kb
        return
    assert 2 <= s <= 16
    assert per % 4 == 0                       # whole accumulation chunks
    assert (s - 1) * per < kb <= s * per      # every slice non-empty, K covered
    if forced:
        assert s <= forced
    else:
        assert tiles * s <= PAIRS             # one wave of units


@pytest.mark.parametrize("tiles,kb", [(39, 512), (76, 1000), (200, 64)])
def test_many_tiles_never_sliced(tiles, kb):
    for forced in (0, 4):
        assert _plan(tiles, kb, forced)["splits"] == 1


@pytest.mark.parametrize("tiles", [1, 4, 16])
def test_short_k_or_forced_whole_never_sliced(tiles):
    assert _plan(tiles, 7)["splits"] == 1
    assert _plan(tiles, 4096, forced=1)["splits"] == 1


@pytest.mark.parametrize("tiles", [1, 2, 4, 9, 16, 20, 30])
def test_longer_k_keeps_slicing(tiles):
    sliced = [kb for kb in range(8, 1200, 7) if _plan(tiles, kb)["splits"] > 1]
    if sliced:
        first = sliced[0]
        assert all(_plan(tiles, kb)["splits"] > 1 for kb in range(first, 1200, 7))


@pytest.mark.parametrize("M,N,K,expect", [
    (1024, 1024, 1024, 1),    # 16 tiles, 32 k-blocks: half-width whole-K units
    (256, 256, 256, 1),
    (1000, 1100, 900, 1),
    (300, 300, 8200, 11),     # 4 tiles, 257 k-blocks
    (256, 256, 16384, 16),    # 1 tile, 512 k-blocks
    (1000, 1100, 4000, 3),    # 20 tiles, 125 k-blocks
    (600, 700, 4000, 8),      # 9 tiles, 125 k-blocks
    (513, 1025, 4100, 5),     # 15 tiles, 129 k-blocks
])
def test_shape_choices(M, N, K, expect):
    tiles = -(-M // 256) * -(-N // 256)
    kb = -(-K // 32)
    assert _plan(tiles, kb)["splits"] == expect


def test_bad_arguments():
    with pytest.raises(g.GemmError):
        g.plan_tf32_slices(-1, PAIRS, 32, 0)
    with pytest.raises(g.GemmError):
        g.plan_tf32_slices(4, PAIRS, 32, -2)
