"""The key walks of the bf16 prefill kernels (host-callable, same functions as on the device) cover every
key of every query row exactly once, with the right position in every column (CPU only); and the in-place
dilated prefill computes every row once with exactly its dilated key set.

The plain kernel walks, per 128-row query tile, tiles of up to 128 keys; the RoPE kernel, per 256-row pair of
query tiles, sub-tiles of up to 64; for each the library
reports (source, first row, position of column 0, last valid column, mask of the query tiles that compute
it).  Column c <= last holds source row (first row + c).  For the rolling cache the position stored in a slot comes from the oracle's sequential
replay of the writes; for the call's own rows it is pos0 + row.  Membership of a position in the key set of
row t is the oracle's brute-force predicate.
"""
import random

import numpy as np
import pytest

import oracle
import sliding_window_softmax_swa_gb300 as swa

BN = 128   # keys per tile of the plain kernel's walk
SUB = 64   # keys per sub-tile of the RoPE kernel's walk
BQ = 128   # rows per query tile
BM = 256   # query rows per work item of the RoPE kernel (two query tiles)
PQ = 128   # query rows per work item of the plain kernel (one query tile)


def check_plan(q0, q1, pos0, w, s, L, plan=None, width=BN):
    plan = swa.prefill_tile_plan(q0, q1, pos0, w, s) if plan is None else plan
    holder = oracle.cache_replay(w, s, pos0) if pos0 > 0 else None
    cols, users = [], []
    for src, row0, pbase, chi, used in plan:
        assert 0 <= chi < width
        assert row0 >= 0
        assert used != 0, "a tile no query tile needs"
        for c in range(chi + 1):
            p = pbase + c
            row = row0 + c
            if src == 1:
                assert row < w, "cache column past the cache"
                assert holder[row] == p, f"slot {row} holds {holder[row]}, tile says {p}"
                assert p < pos0
            else:
                assert p >= pos0 and row == p - pos0
                assert row < L or p > q1
            cols.append(p)
            users.append(used)
    cols = np.array(cols, dtype=np.int64)
    users = np.array(users, dtype=np.int64)
    allpos = np.arange(q1 + 1, dtype=np.int64)
    for t in range(q0, q1 + 1):
        x = (t - q0) // BQ  # the query tile of row t
        mine = cols[(users >> x) & 1 == 1]
        got = np.sort(mine[oracle.is_key_many(t, mine, w, s)])
        want = allpos[oracle.is_key_many(t, allpos, w, s)]
        assert np.array_equal(got, want), (q0, q1, pos0, w, s, t)
    return plan


@pytest.mark.parametrize("w,s", [(1024, 4), (4096, 4), (4096, 0), (300, 4), (64, 16), (1, 0), (2, 1), (129, 4),
                                 (300, 200), (256, 130), (17, 16)])
def test_whole_sequence_tiles(w, s):
    L = 3000
    for qt in range(0, (L + PQ - 1) // PQ):
        q0 = qt * PQ
        q1 = min(q0 + PQ, L) - 1
        check_plan(q0, q1, 0, w, s, L)


def test_chunked_tiles_random():
    rng = random.Random(1234)
    for _ in range(300):
        w = rng.choice([8, 40, 100, 128, 129, 300, 513, 1024])
        s = rng.choice([0, 1, 4, min(w - 1, 16), w - 1])
        pos0 = rng.choice([1, 2, s, s + 1, w - 1, w, w + 1, 3 * w + 7, rng.randrange(1, 5 * w + 10)])
        pos0 = max(1, pos0)
        L = rng.randrange(1, 700)
        qt = rng.randrange(0, (L + PQ - 1) // PQ)
        q0 = pos0 + qt * PQ
        q1 = pos0 + min(qt * PQ + PQ, L) - 1
        check_plan(q0, q1, pos0, w, s, L)


def test_chunked_tiles_long_window_boundaries():
    # the chunk shapes of a 131072-token prompt in 4096-token chunks with w = 4096, s = 4
    w, s, C = 4096, 4, 4096
    for pos0 in (C, 2 * C, 7 * C, 31 * C):
        for qt in (0, 1, 7, 8, 15, 16, 31):
            q0 = pos0 + qt * PQ
            plan = check_plan(q0, q0 + PQ - 1, pos0, w, s, C)
            assert len(plan) <= 37


def test_tile_count_is_minimal_for_full_windows():
    # a full-window query tile walks the ceil((m + 127) / 128) band tiles its rows reach plus one sink tile
    for w, s in [(1024, 4), (4096, 4), (4096, 0)]:
        m = w - s
        plan = swa.prefill_tile_plan(8192, 8192 + PQ - 1, 0, w, s)
        assert len(plan) == (m + 127 + BN - 1) // BN + (1 if s else 0)
        assert all(tl[4] == 1 for tl in plan)


def test_rope_sub_tile_count_is_minimal_for_full_windows():
    # the RoPE kernel's walk: ceil((m' + 255) / 64) band sub-tiles (the band starts at s) plus the sinks, and
    # each query tile computes only the ceil((m' + 127) / 64) its own rows reach
    for w, s in [(1024, 4), (4096, 4), (4096, 0)]:
        m = w - s
        plan = swa.prefill_tile_plan_rope(8192, 8192 + BM - 1, 0, w, s)
        assert len(plan) == (m + 255 + SUB - 1) // SUB + (1 if s else 0)
        for x in (0, 1):
            used = sum(1 for tl in plan if (tl[4] >> x) & 1)
            assert used == (m + 127 + SUB - 1) // SUB + (1 if s else 0)


@pytest.mark.parametrize("w,s", [(1024, 4), (4096, 4), (4096, 0), (300, 4), (64, 16), (2, 1), (129, 4), (300, 128),
                                 (256, 100), (17, 16), (1, 0)])
def test_rope_tiles(w, s):
    # RoPE prefill: the sinks [0, min(s, q1 + 1)) are the first tile, alone (their scores use another
    # query rotation); every other tile starts at or after position s; coverage stays exact
    L = 3000
    for qt in range(0, (L + BM - 1) // BM):
        q0 = qt * BM
        q1 = min(q0 + BM, L) - 1
        plan = check_plan(q0, q1, 0, w, s, L, swa.prefill_tile_plan_rope(q0, q1, 0, w, s), SUB)
        ns = sink_prefix(plan, s, min(s, q1 + 1), src=0)
        for src, row0, pbase, chi, used in plan[ns:]:
            assert pbase >= s


def sink_prefix(plan, s, nsink, src):
    """The RoPE walk starts with the sinks [0, nsink) on their own (one or two sub-tiles, consecutive
    positions from 0); returns how many entries they take."""
    if s == 0:
        return 0
    k, p = 0, 0
    while k < len(plan) and plan[k][2] < s:
        e = plan[k]
        assert e[0] == src and e[2] == p and e[2] + e[3] < nsink, e
        p = e[2] + e[3] + 1
        k += 1
    assert p == nsink and 1 <= k <= 2
    return k


def test_rope_chunked_tiles_random():
    # chunked RoPE prefill (pos0 >= s): the sinks come from the cache as the first tile, alone
    rng = random.Random(4321)
    for _ in range(300):
        w = rng.choice([8, 40, 100, 128, 129, 300, 513, 1024])
        s = rng.choice([0, 1, 4, min(w - 1, 16), min(w - 1, 128)])
        pos0 = max(s, 1, rng.choice([1, s, s + 1, w - 1, w, w + 1, 3 * w + 7, rng.randrange(1, 5 * w + 10)]))
        L = rng.randrange(1, 700)
        qt = rng.randrange(0, (L + BM - 1) // BM)
        q0 = pos0 + qt * BM
        q1 = pos0 + min(qt * BM + BM, L) - 1
        plan = check_plan(q0, q1, pos0, w, s, L, swa.prefill_tile_plan_rope(q0, q1, pos0, w, s), SUB)
        ns = sink_prefix(plan, s, s, src=1)
        for src, row0, pbase, chi, used in plan[ns:]:
            assert pbase >= s


def check_dilated(L, w, s, r):
    """The in-place dilated prefill (the library's own split and per-item tile lists): every row of a (b, h) is
    computed exactly once, by the tensor-core pass or the CUDA-core rows, and each row the tensor-core pass
    stores sees exactly the oracle's dilated key set through the virtual positions of its class."""
    m = w - s
    nrows, G, ns, tail0 = swa.prefill_dilated_split(L, s, r)
    done = np.zeros(L, dtype=np.int64)
    done[:ns] += 1
    done[tail0:] += 1
    for c in range(r):
        p0 = s + (c - s) % r  # the first position >= s of class c
        assert p0 % r == c
        for row_start in range(0, nrows, BQ):
            plan = swa.prefill_tile_plan_dilated(L, w, s, r, c, row_start)
            q0 = s + row_start
            qlast = s + min(row_start + BQ, nrows) - 1
            for u in range(q0, qlast + 1):
                p = p0 + (u - s) * r  # real position of virtual row u
                if p >= G * r:
                    continue  # a row past the last whole group: not stored by this pass
                done[p] += 1
                keys = []
                for src, row0, pbase, chi, used in plan:
                    assert used == 1
                    for col in range(chi + 1):
                        vpos = pbase + col  # virtual key position; the kernel's per-row mask rule
                        if vpos > u or not (vpos < s or vpos >= u - m + 1):
                            continue
                        if src == 1:  # plain rows: the sinks
                            assert vpos < s and row0 + col == vpos
                            keys.append(vpos)
                        else:  # groups of the class; groups from G on would read zeros
                            g = row0 + col
                            assert g < G, ("a stored row attends a zero-filled key", L, w, s, r, c, u)
                            keys.append(g * r + c)
                want = [i for i in range(p + 1) if oracle.is_key_dilated(p, i, w, s, r)]
                assert sorted(keys) == want, (L, w, s, r, c, p)
    assert (done == 1).all(), (L, w, s, r, np.flatnonzero(done != 1)[:8])


@pytest.mark.parametrize("L,w,s,r", [(512, 256, 4, 2), (700, 40, 4, 3), (300, 64, 0, 1), (257, 300, 130, 2),
                                     (263, 300, 5, 2), (1000, 64, 4, 64), (50, 20, 4, 7), (11, 16, 8, 2),
                                     (9, 8, 4, 4), (3, 2, 1, 3), (1001, 200, 4, 7)])
def test_dilated_in_place_plan(L, w, s, r):
    check_dilated(L, w, s, r)


def test_dilated_in_place_plan_random():
    rng = random.Random(77)
    for _ in range(25):
        r = rng.choice([1, 2, 3, 4, 5, 8, 16])
        w = rng.choice([2, 8, 40, 100, 129, 300])
        s = min(w - 1, rng.choice([0, 1, 4, 16, w - 1]))
        check_dilated(rng.randrange(1, 700), w, s, r)
