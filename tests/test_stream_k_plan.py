"""Host-side stream-K planning of the half-precision path (no GPU needed).

Worker w of W takes k-blocks [w*I/W, (w+1)*I/W) of the I shared ones; the
kernel cuts each range at tile boundaries, finds the first and last worker of
a tile with owner(x) = ((x+1)*W - 1) // I, and lets the last piece of a tile
to finish add up the partial sums.  These tests check the plan the library
makes and the partition arithmetic the kernel relies on."""
import itertools

import pytest

import dense_gemm_03_gb300 as g


def _begin(w, iters, workers):
    return w * iters // workers


def _owner(x, iters, workers):
    return ((x + 1) * workers - 1) // iters


def _pieces(plan, kb):
    """All (tile, worker, kb0, kb1) pieces of the shared region, as the kernel
    walks them."""
    iters = plan["sk_tiles"] * kb
    W = plan["workers"]
    out = []
    for w in range(W):
        x, e = _begin(w, iters, W), _begin(w + 1, iters, W)
        while x < e:
            s = x // kb
            k0 = x - s * kb
            k1 = min(kb, k0 + (e - x))
            out.append((s, w, k0, k1))
            x += k1 - k0
    return out


CASES = list(itertools.product([1, 7, 64, 88, 104, 152, 256, 1000, 1024],   # tiles
                               [74, 76, 148, 152],                          # slots
                               [1, 4, 12, 13, 64, 65, 128]))                # k-blocks per tile


@pytest.mark.parametrize("tiles,slots,kb", CASES)
@pytest.mark.parametrize("all_tiles", [False, True])
def test_partition_covers_every_k_block_once(tiles, slots, kb, all_tiles):
    plan = g.plan_stream_k(tiles, slots, kb, all_tiles)
    if plan["sk_tiles"] == 0:
        return
    W = plan["workers"]
    assert 2 <= W <= slots
    assert plan["dp_tiles"] + plan["sk_tiles"] == tiles
    assert plan["dp_tiles"] % slots == 0          # whole waves of whole tiles first
    iters = plan["sk_tiles"] * kb
    assert iters // W >= 4                        # no worker gets fewer than 4 k-blocks
    covered = [[0] * kb for _ in range(plan["sk_tiles"])]
    per_tile = {}
    for s, w, k0, k1 in _pieces(plan, kb):
        assert 0 <= k0 < k1 <= kb
        for k in range(k0, k1):
            covered[s][k] += 1
        per_tile.setdefault(s, []).append((w, k0))
    assert all(c == 1 for row in covered for c in row)
    for s, ws in per_tile.items():
        first = _owner(s * kb, iters, W)
        last = _owner((s + 1) * kb - 1, iters, W)
        # the workers of a tile are consecutive, in k order, one piece each
        assert [w for w, _ in ws] == list(range(first, last + 1))
        assert [k0 for _, k0 in sorted(ws, key=lambda t: t[1])] == sorted(k for _, k in ws)
        assert last - first + 1 <= plan["max_pieces"]


@pytest.mark.parametrize("iters,workers", [(5632, 76), (8192, 148), (64, 16), (6656, 76),
                                           (100003, 152), (7, 2)])
def test_owner_formula(iters, workers):
    for x in range(0, iters, max(1, iters // 2000)):
        w = _owner(x, iters, workers)
        assert _begin(w, iters, workers) <= x < _begin(w + 1, iters, workers)


def test_headline_plan():
    """4096^3 on 76 CTA pairs: 256 pair tiles = 3.37 waves; two waves stay whole,
    the remaining 104 tiles (6656 k-blocks) are shared, 87-88 per pair."""
    plan = g.plan_stream_k(256, 76, 64)
    assert plan == {"dp_tiles": 152, "sk_tiles": 104, "workers": 76, "max_pieces": 2}


def test_whole_waves_and_small_k_stay_whole():
    assert g.plan_stream_k(152, 76, 64)["sk_tiles"] == 0       # exactly two waves
    assert g.plan_stream_k(64, 76, 12)["sk_tiles"] == 0        # one partial wave, short K
    assert g.plan_stream_k(1024, 76, 4)["sk_tiles"] == 0       # gain below the fix-up cost


def test_few_tiles_share_all_k_blocks():
    """16 x 8192 x 8192 with 128-wide tiles: 64 tiles of 128 k-blocks on 148 SMs."""
    plan = g.plan_stream_k(64, 148, 128, True)
    assert plan["dp_tiles"] == 0 and plan["sk_tiles"] == 64 and plan["workers"] == 148
    assert plan["max_pieces"] == 4


def test_null_out_is_an_error():
    L = g.lib()
    assert L.gemm_plan_stream_k(10, 10, 10, 0, None) == -1


# ---------------------------------------------------------------- stream-K tail (publishers first)

def _tail_pieces(plan, kb):
    """Each worker's pieces as the kernel orders them with sk_order 1: the part
    of its range that does not end a tile first, the part that ends one last.
    Returns {worker: [(tile, kb0, kb1, ends_tile)]} in running order."""
    iters = plan["sk_tiles"] * kb
    W = plan["workers"]
    out = {}
    for w in range(W):
        x0, x1 = _begin(w, iters, W), _begin(w + 1, iters, W)
        tile_end = (x0 // kb + 1) * kb
        seq = []
        if x1 >= tile_end:
            first, last = (tile_end, x1), (x0, tile_end)
        else:
            first, last = (x0, x1), None
        if first[0] < first[1]:
            s = first[0] // kb
            seq.append((s, first[0] - s * kb, first[1] - s * kb, first[1] == (s + 1) * kb))
        if last is not None:
            s = last[0] // kb
            seq.append((s, last[0] - s * kb, last[1] - s * kb, True))
        out[w] = seq
    return out


TAIL_CASES = list(itertools.product([77, 100, 104, 152 + 1, 256, 300, 1000, 1024],   # tiles
                                    [74, 76, 148, 152],                             # slots
                                    [1, 4, 8, 13, 16, 64, 65, 128]))                 # k-blocks


@pytest.mark.parametrize("tiles,slots,kb", TAIL_CASES)
def test_tail_plan_partition(tiles, slots, kb):
    """The tail form shares out exactly the last partial wave; every range is
    no longer than a tile (so it ends at most one tile and starts at most one);
    every k-block is covered once; each tile has one piece that ends it, run
    last by its worker, and every other piece runs first."""
    plan = g.plan_stream_k(tiles, slots, kb, tail=True)
    rem = tiles % slots
    if plan["sk_tiles"] == 0:
        assert rem == 0 or tiles <= slots or kb < 8 or rem * kb < 4 * (rem + 1)
        return
    W = plan["workers"]
    assert plan["sk_tiles"] == rem and plan["dp_tiles"] == tiles - rem
    assert rem < W <= min(slots, 4 * rem)
    iters = rem * kb
    assert -(-iters // W) <= kb                 # no range longer than a tile
    assert iters // W >= 4
    covered = [[0] * kb for _ in range(rem)]
    enders = [0] * rem
    pieces_per_tile = [set() for _ in range(rem)]
    for w, seq in _tail_pieces(plan, kb).items():
        assert 1 <= len(seq) <= 2
        for i, (s, k0, k1, ends) in enumerate(seq):
            assert 0 <= k0 < k1 <= kb
            for k in range(k0, k1):
                covered[s][k] += 1
            pieces_per_tile[s].add(w)
            if ends:
                enders[s] += 1
                assert i == len(seq) - 1      # the finishing piece runs last
            else:
                assert i == 0                 # the others run first
    assert all(c == 1 for row in covered for c in row)
    assert enders == [1] * rem
    assert max(len(x) for x in pieces_per_tile) <= plan["max_pieces"]
