"""The key-tile lists of the block-sparse prefill (built on the host, reported by the library's plan
diagnostics) against the oracle's membership predicate is_key_blocksparse (CPU only).

For every query pair: tiles hold disjoint runs of positions inside the causal range of the pair; the
global-column words mark exactly the global tokens of each tile; every key of every non-global row's key set
lies in a tile its query tile uses; and every used tile holds at least one key of a row of that query tile.
(Global rows are recomputed over their whole prefix by a separate pass.)  A packed tile holds two runs of 64
keys, columns 0..63 and 64..127, neither touching the sinks or the pair's band (its per-row masks have only
random blocks and global tokens)."""
import numpy as np
import pytest

import oracle
import swa_inputs
import sliding_window_softmax_swa_gb300 as swa

BM, BQ = 256, 128


def column_position(pbase, pbase1, c):
    """The key position held by column c of a tile (packed tiles: columns 64.. start again at pbase1)."""
    return pbase + c if pbase1 < 0 or c < 64 else pbase1 + c - 64


def check_pattern(L, w, s, globals_, block, rand):
    """Checks every pair's tile list; returns the number of packed tiles seen."""
    rd = swa_inputs.rand_blocks_dict(rand) if rand is not None else None
    gset = set(globals_)
    m = w - s
    packed = 0
    for pair in range((L + BM - 1) // BM):
        q0, qlast = pair * BM, min(pair * BM + BM, L) - 1
        plan = swa.prefill_blocksparse_plan(L, w, s, globals_, block, rand, pair)
        seen = {}
        for j, (pbase, chi, used, gm, pbase1) in enumerate(plan):
            assert 0 <= chi < 128 and used in (1, 2, 3)
            assert 0 <= pbase and column_position(pbase, pbase1, chi) <= qlast
            if pbase1 >= 0:
                packed += 1
                assert chi == 127
                for first in (pbase, pbase1):  # outside the sinks and the band of every row of the pair
                    assert first >= s and first + 63 < max(0, q0 - m + 1), (pair, first)
            for c in range(chi + 1):
                pos = column_position(pbase, pbase1, c)
                assert pos not in seen, f"position {pos} in two tiles"
                seen[pos] = j
                assert bool(gm >> c & 1) == (pos in gset), f"global mask of column {c} at {pbase}"
            assert gm >> (chi + 1) == 0
        useful = set()
        for t in range(q0, qlast + 1):
            x = (t - q0) // BQ
            if t in gset:
                continue
            for i in range(t + 1):
                if oracle.is_key_blocksparse(t, i, w, s, gset, block, rd):
                    assert i in seen, f"key {i} of row {t} is in no tile"
                    j = seen[i]
                    assert plan[j][2] >> x & 1, f"key {i} of row {t}: its tile is not walked by query tile {x}"
                    useful.add((j, x))
        for j, (_, _, used, _, _) in enumerate(plan):
            for x in range(2):
                if used >> x & 1:
                    # a global row may be the only user; the pass still walks the tile (its rows are overwritten)
                    rows = range(q0 + x * BQ, min(q0 + x * BQ + BQ, qlast + 1))
                    assert (j, x) in useful or any(t in gset for t in rows), f"tile {j} walked by {x} for nothing"
    return packed


def test_hand_pattern():
    rand = np.array([[-1], [-1], [0]], dtype=np.int32)  # query block 2 -> key block 0
    check_pattern(12, 3, 1, [5], 4, rand)


@pytest.mark.parametrize("L,w,s,ng,block,r,seed", [
    (300, 64, 4, 1, 16, 2, 1),
    (700, 40, 0, 0, 64, 2, 2),
    (900, 300, 16, 1, 128, 1, 3),
    (1100, 200, 4, 2, 64, 3, 4),
    (600, 600, 4, 0, 32, 4, 5),
    (520, 129, 4, 0, 7, 5, 6),  # blocks that straddle tiles and query tiles
])
def test_random_patterns(L, w, s, ng, block, r, seed):
    globals_, rand = swa_inputs.bigbird_pattern(L, block, ng, r, seed)
    packed = check_pattern(L, w, s, globals_, block, rand if r else None)
    if block == 64 and r >= 2 and L >= 1000:
        assert packed > 0  # lone random blocks far behind the band share tiles


def test_packed_halves_by_hand():
    # query block 9 (rows 576..639, query tile 4 of pair 2) -> key blocks 0 and 3; w = 64: both lie outside
    # the sinks and the band, serve the same query tile, and so share one tile
    L, block = 700, 64
    rand = np.full((11, 2), -1, dtype=np.int32)
    rand[9] = [3, 1]
    plan = swa.prefill_blocksparse_plan(L, 64, 4, [], block, rand, 2)
    packed = [t for t in plan if t[4] >= 0]
    assert [(t[0], t[1], t[2], t[4]) for t in packed] == [(64, 127, 1, 192)]
    check_pattern(L, 64, 4, [], block, rand)


def test_scattered_globals():
    _, rand = swa_inputs.bigbird_pattern(800, 64, 0, 2, 7)
    check_pattern(800, 100, 4, [0, 7, 300, 301, 555, 799], 64, rand)


def test_without_globals_and_blocks_matches_plain_walk():
    # no global token and no random block: the same key runs as the plain prefill walks
    L, w, s = 1000, 300, 4
    for pair in range((L + BM - 1) // BM):
        q0, q1 = pair * BM, min(pair * BM + BM, L) - 1
        bs = [(p, c, u) for p, c, u, _, _ in swa.prefill_blocksparse_plan(L, w, s, [], 16, None, pair)]
        plain = [(pb, c, u) for _, _, pb, c, u in swa.prefill_tile_plan(q0, q1, 0, w, s)]
        cover = lambda tl: sorted(p for pb, c, _ in tl for p in range(pb, pb + c + 1))
        assert cover(bs) == cover(plain)


def test_pattern_errors():
    with pytest.raises(swa.SwaError):
        swa.prefill_blocksparse_plan(100, 16, 4, [5, 3], 16, None, 0)  # globals not ascending
    with pytest.raises(swa.SwaError):
        swa.prefill_blocksparse_plan(100, 16, 4, [100], 16, None, 0)  # global past L
    with pytest.raises(swa.SwaError):
        swa.prefill_blocksparse_plan(100, 16, 4, [], 16, np.full((7, 1), 7, dtype=np.int32), 0)  # no key block 7
    with pytest.raises(swa.SwaError):
        swa.prefill_blocksparse_plan(100, 16, 4, [], 16, np.full((7, 17), -1, dtype=np.int32), 0)  # r > 16
    with pytest.raises(swa.SwaError):
        swa.prefill_blocksparse_plan(100, 16, 4, [], 16, None, 1)  # only one pair
    # more than 64 tiles for one pair: 65 random blocks of 128 keys are not possible with r <= 16, but 70
    # scattered global tokens 200 apart are
    L = 70 * 200 + 300
    globals_ = [200 * i for i in range(70)]
    with pytest.raises(swa.SwaError):
        swa.prefill_blocksparse_plan(L, 16, 4, globals_, 64, None, (L - 1) // BM)


def test_packed_tiles_with_globals_and_shared_blocks():
    # the pattern of the GPU packed-tile test: blocks used by both query tiles pair first, then within one
    # query tile; global tokens inside packed halves keep their columns
    L, w, s, block = 1300, 64, 4, 64
    rand = np.full(((L + block - 1) // block, 2), -1, dtype=np.int32)
    rand[16] = [1, 5]
    rand[17] = [3, -1]
    rand[18] = [3, 9]
    rand[19] = [11, 0]
    plan = swa.prefill_blocksparse_plan(L, w, s, [200, 330], block, rand, 4)
    packed = [t for t in plan if t[4] >= 0]
    assert [(t[0], t[4], t[2]) for t in packed] == [(192, 320, 3), (576, 704, 2)]
    assert packed[0][3] == (1 << (200 - 192)) | (1 << (64 + 330 - 320))
    assert check_pattern(L, w, s, [200, 330], block, rand) >= 2
