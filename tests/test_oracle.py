"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: hand-derived values, a textbook
library routine on a special case, a closed form, or an invariant. Together they are chosen so that
a plausible slip in the oracle (a window one key too wide or too narrow, sinks counted outside the
window, a transposed operand, a wrong scale, a missing max-subtraction, a wrong slot formula) fails
at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------------------------------------
# Hand-derived worked examples (hyper.ai summary of arXiv 2608.28444, section
# "带 Sink 的滑动窗口注意力": w keys, s sinks inside the window).
# ---------------------------------------------------------------------------------------------
def test_hand_derived_examples():
    g = json.load(open(os.path.join(GOLDEN, "hand_sink_window.json")))
    L = len(g["v"])
    k = np.log(np.array(g["exp_k"], dtype=np.float64)).reshape(1, 1, L, 1)
    v = np.array(g["v"], dtype=np.float64).reshape(1, 1, L, 1)
    q = np.ones((1, 1, L, 1))
    for case in g["cases"]:
        o, lse = oracle.prefill(q, k, v, case["w"], case["s"], 1.0)
        want = np.array([float(Fraction(x)) for x in case["o"]])
        np.testing.assert_allclose(o[0, 0, :, 0], want, rtol=1e-13, atol=0)
        np.testing.assert_allclose(lse[0, 0], np.log(np.array(case["lse_exp"], dtype=np.float64)),
                                   rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Special case w >= L: full causal softmax attention, equation (1) of "模糊窗口注意力" section 2.1,
# computed here with numpy matmul + scipy.special.softmax on an explicit -inf mask.
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("L,d,w,s", [(37, 8, 37, 0), (37, 8, 50, 0), (29, 5, 29, 3), (64, 16, 64, 0)])
def test_full_window_is_causal_attention(L, d, w, s):
    q, k, v = rnd((2, 3, L, d), 1), rnd((2, 3, L, d), 2), rnd((2, 3, L, d), 3)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.prefill(q, k, v, w, s, scale)
    S = np.einsum("bhtc,bhic->bhti", q, k) / math.sqrt(d)
    M = np.where(np.tril(np.ones((L, L), dtype=bool)), 0.0, -np.inf)
    P = scipy.special.softmax(S + M, axis=-1)
    np.testing.assert_allclose(o, P @ v, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(S + M, axis=-1), rtol=0, atol=1e-12)


def test_w1_s0_returns_v():
    # One-term sum of the SWA formula: x_t = v_t exactly.
    q, k, v = rnd((1, 2, 23, 7), 4), rnd((1, 2, 23, 7), 5), rnd((1, 2, 23, 7), 6)
    o, _ = oracle.prefill(q, k, v, 1, 0, 0.37)
    assert np.array_equal(o, v)


def test_w1_s1_is_sink_plus_self_only_through_sink():
    # w = 1, s = 1: m = 0 recent keys, so every query sees only position 0 (and itself only if t = 0).
    q, k, v = rnd((1, 1, 9, 4), 7), rnd((1, 1, 9, 4), 8), rnd((1, 1, 9, 4), 9)
    o, _ = oracle.prefill(q, k, v, 1, 1, 0.5)
    np.testing.assert_array_equal(o[0, 0], np.repeat(v[0, 0, :1], 9, axis=0))


def test_two_key_window_closed_form():
    # s = 0, w = 2: o_t = sigmoid(x_t - x_{t-1}) v_t + sigmoid(x_{t-1} - x_t) v_{t-1}.
    L, d = 31, 6
    q, k, v = rnd((1, 1, L, d), 10), rnd((1, 1, L, d), 11), rnd((1, 1, L, d), 12)
    sc = 0.8
    o, _ = oracle.prefill(q, k, v, 2, 0, sc)
    q0, k0, v0 = q[0, 0], k[0, 0], v[0, 0]
    np.testing.assert_array_equal(o[0, 0, 0], v0[0])
    for t in range(1, L):
        a = sc * q0[t] @ k0[t]
        b = sc * q0[t] @ k0[t - 1]
        want = scipy.special.expit(a - b) * v0[t] + scipy.special.expit(b - a) * v0[t - 1]
        np.testing.assert_allclose(o[0, 0, t], want, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Key-set membership by an independent construction: the union of the sink range [0, s) and the
# recent range [t - m + 1, t], built as Python sets (the StreamingLLM cache of page
# "滑窗与固定稀疏", eq attn-fixed-streaming: k sinks + m recent).
# ---------------------------------------------------------------------------------------------
def keyset(t, w, s):
    m = w - s
    return (set(range(0, min(s, t + 1))) | set(range(max(0, t - m + 1), t + 1)))


@pytest.mark.parametrize("L", [1, 2, 7, 13, 40])
def test_mask_matches_set_construction(L):
    for w in range(1, L + 3):
        for s in range(0, w):
            mk = oracle.mask(L, w, s)
            for t in range(L):
                assert set(np.nonzero(mk[t])[0].tolist()) == keyset(t, w, s), (L, w, s, t)
                assert np.array_equal(oracle.is_key_many(t, np.arange(L), w, s), mk[t].astype(bool))


def test_zero_query_gives_mean_over_keyset():
    # q = 0 makes every score 0, so o_t is the plain mean of v over K(t): pins which keys and how many.
    L, d = 45, 3
    v = rnd((1, 1, L, d), 13)
    for w, s in [(1, 0), (5, 0), (5, 2), (8, 4), (8, 7), (44, 4), (60, 4)]:
        o, lse = oracle.prefill(np.zeros((1, 1, L, d)), rnd((1, 1, L, d), 14), v, w, s, 1.0)
        for t in range(L):
            ks = sorted(keyset(t, w, s))
            np.testing.assert_allclose(o[0, 0, t], v[0, 0, ks].mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[0, 0, t] - math.log(len(ks))) < 1e-13


def test_mask_picture_n32():
    # The N = 32 StreamingLLM picture (recent band + sink bar on the left), drawn from the figure's
    # description by tests/golden/make_golden.py without the oracle, stored as text.
    g = open(os.path.join(GOLDEN, "streaming_mask_n32_w8_s4.txt")).read().split("\n")
    rows = [r for r in g if r and set(r) <= {"#", "."}]
    pic = np.array([[1 if ch == "#" else 0 for ch in r] for r in rows], dtype=np.uint8)
    assert pic.shape == (32, 32)
    np.testing.assert_array_equal(oracle.mask(32, 8, 4), pic)
    # caption facts: lower-triangular, a full left bar of 4 columns below the diagonal, a band of 4
    for t in range(32):
        assert pic[t, t + 1:].sum() == 0
        assert pic[t, :min(4, t + 1)].all()
        assert pic[t, max(0, t - 3):t + 1].all()
        assert pic[t].sum() == min(t + 1, 8)


# ---------------------------------------------------------------------------------------------
# Normalisation, page "滑窗与固定稀疏", eq attn-fixed-softmax-sink: with V = identity the output rows
# are the attention weights; they sum to 1, are >= 0 and vanish outside K(t).
# ---------------------------------------------------------------------------------------------
def test_rows_are_probability_vectors():
    L = 24
    q, k = rnd((1, 1, L, L), 15), rnd((1, 1, L, L), 16)
    v = np.eye(L).reshape(1, 1, L, L)
    for w, s in [(6, 2), (6, 0), (24, 4), (3, 1)]:
        P, _ = oracle.prefill(q, k, v, w, s, 0.3)
        P = P[0, 0]
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert (P >= 0).all()
        for t in range(L):
            outside = [i for i in range(L) if i not in keyset(t, w, s)]
            assert (P[t, outside] == 0).all()
            assert (P[t, sorted(keyset(t, w, s))] > 0).all()


def test_scale_is_applied_once():
    # Scaling q by lam and the softmax scale by 1/lam leaves every score unchanged.
    L, d = 33, 8
    q, k, v = rnd((1, 2, L, d), 17), rnd((1, 2, L, d), 18), rnd((1, 2, L, d), 19)
    o1, l1 = oracle.prefill(q, k, v, 9, 2, 0.25)
    o2, l2 = oracle.prefill(q * 4.0, k, v, 9, 2, 0.0625)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)
    o3, _ = oracle.prefill(q, k, v, 9, 2, 0.5)
    assert np.abs(o3 - o1).max() > 1e-3  # the scale matters


def test_large_sink_logits_stay_finite():
    # Keys at positions 0..3 boosted (x4 and x1000): exp() of the raw scores would overflow in fp64;
    # the max-subtracted softmax must stay finite and match scipy's logsumexp.
    L, d = 40, 16
    q, k, v = rnd((1, 1, L, d), 20) * 30, rnd((1, 1, L, d), 21), rnd((1, 1, L, d), 22)
    k[..., :4, :] *= 1000.0
    o, lse = oracle.prefill(q, k, v, 12, 4, 1.0)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    S = q[0, 0] @ k[0, 0].T
    for t in range(L):
        ks = sorted(keyset(t, 12, 4))
        np.testing.assert_allclose(lse[0, 0, t], scipy.special.logsumexp(S[t, ks]), rtol=1e-14, atol=0)
        P = scipy.special.softmax(S[t, ks])
        np.testing.assert_allclose(o[0, 0, t], P @ v[0, 0, ks], rtol=0, atol=1e-10)


# ---------------------------------------------------------------------------------------------
# Rolling cache: slot replay (page "滑窗与固定稀疏", eq attn-fixed-rolling cache_slot(i) = i mod W,
# and eq attn-fixed-streaming: sinks + recent, k + m slots) and the order-free decode
# ("模糊窗口注意力" section 3: softmax attention is invariant to the order of the keys).
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("w", [1, 2, 5, 16])
def test_slot_replay_s0_is_mod_w(w):
    for npos in range(0, 4 * w + 3):
        h = oracle.cache_replay(w, 0, npos)
        for j in range(w):
            held = [p for p in range(npos) if p % w == j]
            assert h[j] == (held[-1] if held else -1)


@pytest.mark.parametrize("w,s", [(8, 4), (5, 1), (6, 5), (16, 4)])
def test_slot_replay_holds_sinks_and_recent(w, s):
    m = w - s
    for npos in range(0, 5 * w):
        h = oracle.cache_replay(w, s, npos)
        held = sorted(p for p in h.tolist() if p >= 0)
        want = sorted(set(range(min(s, npos))) | set(range(max(s, npos - m), npos)))
        assert held == want
        assert len(h) == w  # constant footprint, k + m slots


@pytest.mark.parametrize("w,s", [(8, 4), (5, 1), (6, 5), (16, 4), (4, 0)])
def test_slot_index_fills_in_order_then_overwrites_oldest(w, s):
    # The cache fills slot p with position p until it is full; from then on each new position takes
    # the slot of the oldest recent position (the rolling buffer overwrites the oldest entry, page
    # "滑窗与固定稀疏", rolling-buffer section), and the s sink slots are never overwritten.
    m = w - s
    for npos in range(0, w + 1):
        h = oracle.cache_replay(w, s, npos)
        assert h.tolist() == list(range(npos)) + [-1] * (w - npos)
    prev = oracle.cache_replay(w, s, w)
    for p in range(w, 6 * w):
        cur = oracle.cache_replay(w, s, p + 1)
        changed = [j for j in range(w) if cur[j] != prev[j]]
        if m == 0:
            assert changed == []
        else:
            oldest = min(x for x in prev.tolist() if x >= s)
            assert changed == [prev.tolist().index(oldest)] and cur[changed[0]] == p
        assert cur[:s].tolist() == list(range(s))
        prev = cur


@pytest.mark.parametrize("w,s,d", [(8, 4, 4), (5, 0, 3), (7, 2, 5), (1, 0, 2)])
def test_cached_decode_equals_history_every_step(w, s, d):
    T = 3 * w + 5
    nh = 2
    q, k, v = rnd((nh, T, d), 30 + w), rnd((nh, T, d), 31 + s), rnd((nh, T, d), 32)
    k[:, :min(4, T), :] *= 4.0
    sc = 1.0 / math.sqrt(d)
    for t in range(T):
        o_hist, l_hist = oracle.decode(q[:, t], k[:, :t + 1], v[:, :t + 1], t, w, s, sc)
        h = oracle.cache_replay(w, s, t + 1)
        slots = [j for j in range(w) if h[j] >= 0]
        kpos = h[slots]
        o_c, l_c = oracle.attend(q[:, t:t + 1], [t], k[:, kpos], v[:, kpos], kpos, w, s, sc)
        np.testing.assert_allclose(o_c[:, 0], o_hist, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l_c[:, 0], l_hist, rtol=0, atol=1e-13)
        # every cached key is in K(t): the cache is exactly the key set
        assert set(kpos.tolist()) == keyset(t, w, s)


def test_cache_footprint_ratio():
    # Rolling buffer of W = 4096 slots vs the full cache: 8x at 32K tokens, 2x at 8K
    # (page "滑窗与固定稀疏", rolling-buffer section).
    for L, ratio in [(32768, 8), (8192, 2)]:
        h = oracle.cache_replay(4096, 0, L)
        assert L / len(h) == ratio


def test_key_order_does_not_matter():
    L, d = 50, 8
    q, k, v = rnd((2, L, d), 40), rnd((2, L, d), 41), rnd((2, L, d), 42)
    pos = np.arange(L)
    perm = np.random.default_rng(3).permutation(L)
    o1, l1 = oracle.attend(q, pos, k, v, pos, 11, 3, 0.4)
    o2, l2 = oracle.attend(q, pos, k[:, perm], v[:, perm], pos[perm], 11, 3, 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_rows_subset_and_threads_agree():
    B, H, L, d = 1, 3, 70, 8
    q, k, v = rnd((B, H, L, d), 50), rnd((B, H, L, d), 51), rnd((B, H, L, d), 52)
    o, lse = oracle.prefill(q, k, v, 13, 4, 0.35, nthreads=1)
    o4, lse4 = oracle.prefill(q, k, v, 13, 4, 0.35, nthreads=4)
    assert np.array_equal(o, o4) and np.array_equal(lse, lse4)
    rows = [0, 5, 12, 13, 14, 69]
    orow, lrow = oracle.prefill_rows(q[0][:, rows], rows, k[0], v[0], 13, 4, 0.35)
    assert np.array_equal(orow, o[0][:, rows]) and np.array_equal(lrow, lse[0][:, rows])


# ---------------------------------------------------------------- RoPE at positions inside the cache
def test_rope_matches_complex_rotation():
    # the rotation written as complex multiplication: (x_i + i x_{i+d/2}) * exp(i * pos * base^(-2i/d))
    rng = np.random.default_rng(11)
    d, n = 16, 9
    x = rng.standard_normal((3, n, d))
    pos = rng.integers(0, 5000, n).astype(np.float64)
    theta = 10000.0 ** (-np.arange(d // 2) * 2.0 / d)
    z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * np.exp(1j * pos[:, None] * theta[None, :])
    want = np.concatenate([z.real, z.imag], axis=-1)
    np.testing.assert_allclose(oracle.rope(x, pos), want, rtol=0, atol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(12)
    d = 32
    q, k = rng.standard_normal((1, 1, d)), rng.standard_normal((1, 1, d))
    for p, pk, shift in [(5.0, 2.0, 100.0), (0.0, 17.0, 3.0), (1000.0, 4.0, 1.0)]:
        a = (oracle.rope(q, [p]) * oracle.rope(k, [pk])).sum()
        b = (oracle.rope(q, [p + shift]) * oracle.rope(k, [pk + shift])).sum()
        assert abs(a - b) < 1e-9


def test_decode_rope_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "rope_cache_positions_d4.json")))
    t, w, s, d = 5, 3, 1, 4
    k = np.zeros((1, t + 1, d))
    v = np.zeros((1, t + 1, d))
    for p in g["filler_positions"]:  # outside K(5): must not matter
        k[0, p] = 100.0
        v[0, p] = -7.0
    for p, row in g["keys"].items():
        k[0, int(p)] = row
    for p, row in g["values"].items():
        v[0, int(p)] = row
    o, lse = oracle.decode_rope(np.array([g["q"]]), k, v, t, w, s, 1.0)
    np.testing.assert_allclose(o[0], g["o"], rtol=0, atol=1e-12)
    assert abs(lse[0] - g["lse"]) < 1e-12


def test_decode_rope_before_the_window_fills_is_plain_rope():
    # while t < w every position is in the cache, in order: cache position == original position
    rng = np.random.default_rng(13)
    nh, d, w, s = 2, 16, 12, 4
    for t in (0, 3, 11):
        q = rng.standard_normal((nh, d))
        k, v = rng.standard_normal((nh, t + 1, d)), rng.standard_normal((nh, t + 1, d))
        pos = np.arange(t + 1, dtype=np.float64)
        o_ref, l_ref = oracle.attend(oracle.rope(q[:, None], [float(t)]), [t], oracle.rope(k, pos), v,
                                     np.arange(t + 1), w, s, 0.25)
        o, lse = oracle.decode_rope(q, k, v, t, w, s, 0.25)
        np.testing.assert_allclose(o, o_ref[:, 0], atol=1e-12)
        np.testing.assert_allclose(lse, l_ref[:, 0], atol=1e-12)


def test_decode_rope_without_sinks_keeps_relative_distances():
    # s = 0: the cache holds the last w positions in order, so re-assigning positions only shifts them by
    # a constant and RoPE at the original positions gives the same result
    rng = np.random.default_rng(14)
    nh, d, w = 2, 16, 6
    for t in (6, 20, 57):
        q = rng.standard_normal((nh, d))
        k, v = rng.standard_normal((nh, t + 1, d)), rng.standard_normal((nh, t + 1, d))
        pos = np.arange(t + 1, dtype=np.float64)
        o_ref, _ = oracle.attend(oracle.rope(q[:, None], [float(t)]), [t], oracle.rope(k, pos), v,
                                 np.arange(t + 1), w, 0, 0.3)
        o, _ = oracle.decode_rope(q, k, v, t, w, 0, 0.3)
        np.testing.assert_allclose(o, o_ref[:, 0], atol=1e-10)


def test_decode_rope_sinks_sit_at_fixed_distance_once_the_window_is_full():
    # with the window full, sink i sits at distance w - 1 - i from the query whatever t is: advancing t
    # with the same window contents and sinks leaves the result unchanged (plain RoPE would not)
    rng = np.random.default_rng(15)
    nh, d, w, s = 1, 16, 8, 2
    m = w - s
    sinks_k, sinks_v = rng.standard_normal((nh, s, d)), rng.standard_normal((nh, s, d))
    win_k, win_v = rng.standard_normal((nh, m, d)), rng.standard_normal((nh, m, d))
    q = rng.standard_normal((nh, d))
    outs = []
    for t in (20, 45):
        k, v = rng.standard_normal((nh, t + 1, d)), rng.standard_normal((nh, t + 1, d))
        k[:, :s], v[:, :s] = sinks_k, sinks_v
        k[:, t - m + 1:], v[:, t - m + 1:] = win_k, win_v
        outs.append(oracle.decode_rope(q, k, v, t, w, s, 0.3)[0])
    np.testing.assert_allclose(outs[0], outs[1], atol=1e-12)
    # and differs from RoPE at the original positions
    t = 45
    k = rng.standard_normal((nh, t + 1, d))
    v = rng.standard_normal((nh, t + 1, d))
    o_new, _ = oracle.decode_rope(q, k, v, t, w, s, 0.3)
    members = np.array([i for i in range(t + 1) if oracle.is_key(t, i, w, s)])
    o_plain, _ = oracle.attend(oracle.rope(q[:, None], [float(t)]), [t],
                               oracle.rope(k[:, members], members.astype(np.float64)), v[:, members], members,
                               w, s, 0.3)
    assert np.abs(o_new - o_plain[:, 0]).max() > 1e-3


def _rope_rows_closed_form(q, k, v, w, s, scale, base=10000.0):
    # the reading of the cache-position rule for a whole sequence, written out directly: query t scores
    # its window keys i at (q at t, k at i), as plain RoPE does, and the sinks at (q at min(t, w - 1),
    # k at i), since a full cache puts the query at position w - 1 and sink i at i
    nh, L, d = q.shape
    m = w - s
    pos = np.arange(L, dtype=np.float64)
    kr = oracle.rope(k, pos, base)
    o = np.empty((nh, L, d))
    lse = np.empty((nh, L))
    for t in range(L):
        win = np.arange(max(s, t - m + 1), t + 1)
        snk = np.arange(0, min(s, t + 1))
        qw = oracle.rope(q[:, t:t + 1], [float(t)], base)[:, 0]
        qs = oracle.rope(q[:, t:t + 1], [float(min(t, w - 1))], base)[:, 0]
        x = np.concatenate([np.einsum("hd,hnd->hn", qs, kr[:, snk]), np.einsum("hd,hnd->hn", qw, kr[:, win])],
                           axis=1) * scale
        idx = np.concatenate([snk, win])
        p = scipy.special.softmax(x, axis=1)
        o[:, t] = np.einsum("hn,hnd->hd", p, v[:, idx])
        lse[:, t] = scipy.special.logsumexp(x, axis=1)
    return o, lse


@pytest.mark.parametrize("L,w,s", [(40, 12, 4), (33, 8, 1), (25, 6, 5), (30, 30, 4), (21, 50, 3), (28, 9, 0)])
def test_prefill_rope_equals_the_closed_form(L, w, s):
    rng = np.random.default_rng(16 + L + w + s)
    nh, d = 2, 16
    q, k, v = (rng.standard_normal((1, nh, L, d)) for _ in range(3))
    o, lse = oracle.prefill_rope(q, k, v, w, s, 0.3)
    o_ref, l_ref = _rope_rows_closed_form(q[0], k[0], v[0], w, s, 0.3)
    np.testing.assert_allclose(o[0], o_ref, atol=1e-10)
    np.testing.assert_allclose(lse[0], l_ref, atol=1e-10)


def test_prefill_rope_without_eviction_is_causal_rope_attention():
    # w >= L: nothing leaves the cache and every position is its own: causal softmax attention on
    # RoPE-rotated q and k (scipy), whatever s is
    rng = np.random.default_rng(17)
    nh, L, d, scale = 2, 24, 16, 0.25
    q, k, v = (rng.standard_normal((1, nh, L, d)) for _ in range(3))
    pos = np.arange(L, dtype=np.float64)
    x = np.einsum("hid,hjd->hij", oracle.rope(q[0], pos), oracle.rope(k[0], pos)) * scale
    x = np.where(np.tril(np.ones((L, L), dtype=bool)), x, -np.inf)
    p = scipy.special.softmax(x, axis=2)
    for s in (0, 3):
        o, lse = oracle.prefill_rope(q, k, v, L + 5, s, scale)
        np.testing.assert_allclose(o[0], np.einsum("hij,hjd->hid", p, v[0]), atol=1e-12)
        np.testing.assert_allclose(lse[0], scipy.special.logsumexp(x, axis=2), atol=1e-12)


def test_prefill_rope_without_sinks_is_the_band_oracle_on_rotated_inputs():
    # s = 0: distances are the original ones, so the plain oracle (C) on RoPE-rotated q, k agrees
    rng = np.random.default_rng(18)
    nh, L, d, w = 2, 50, 16, 7
    q, k, v = (rng.standard_normal((1, nh, L, d)) for _ in range(3))
    pos = np.arange(L, dtype=np.float64)
    o_ref, l_ref = oracle.prefill(oracle.rope(q, pos), oracle.rope(k, pos), v, w, 0, 0.2)
    o, lse = oracle.prefill_rope(q, k, v, w, 0, 0.2, rows=range(0, L, 3))
    np.testing.assert_allclose(o, o_ref[:, :, ::3], atol=1e-10)
    np.testing.assert_allclose(lse, l_ref[:, :, ::3], atol=1e-10)


# ------------------------------------------------------------------ dilated window with sinks
def test_dilated_mask_matches_hand_derived_golden():
    path = os.path.join(GOLDEN, "dilated_mask_L14_w5_s2_r3.txt")
    rows = [l.strip() for l in open(path) if l.strip() and not l.startswith("#")]
    assert len(rows) == 14
    for t in range(14):
        for i in range(14):
            assert (rows[t][i] == "1") == oracle.is_key_dilated(t, i, 5, 2, 3), (t, i)


@pytest.mark.parametrize("w,s", [(5, 2), (8, 0), (3, 2), (40, 4)])
def test_dilation_one_is_the_plain_key_set(w, s):
    for t in range(60):
        for i in range(60):
            assert oracle.is_key_dilated(t, i, w, s, 1) == oracle.is_key(t, i, w, s)


def test_dilated_key_count_closed_form():
    # |K(t)| = min(s, t + 1) + min(m, t // r + 1) - (sinks that are also window keys: i < s, i <= t,
    # t - i divisible by r and (t - i) / r < m), counted without the membership function
    for w, s, r in [(5, 2, 3), (9, 4, 2), (7, 0, 5), (12, 3, 1)]:
        m = w - s
        for t in range(80):
            both = sum(1 for i in range(min(s, t + 1)) if (t - i) % r == 0 and (t - i) // r < m)
            want = min(s, t + 1) + min(m, t // r + 1) - both
            got = sum(oracle.is_key_dilated(t, i, w, s, r) for i in range(t + 1))
            assert got == want, (w, s, r, t)


def test_prefill_dilated_with_dilation_one_equals_the_plain_oracle():
    # independent code paths: numpy per row (dilated) against the C oracle (plain)
    rng = np.random.default_rng(19)
    q, k, v = (rng.standard_normal((1, 2, 45, 16)) for _ in range(3))
    o, lse = oracle.prefill_dilated(q, k, v, 9, 3, 1, 0.3)
    o_ref, l_ref = oracle.prefill(q, k, v, 9, 3, 0.3)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, l_ref, atol=1e-12)


def test_prefill_dilated_zero_query_is_the_mean_over_the_key_set():
    # q = 0: uniform weights, so o = mean of v over K(t) and lse = ln |K(t)| (members from the golden's rule)
    rng = np.random.default_rng(20)
    L, w, s, r = 30, 6, 2, 4
    q = np.zeros((1, 1, L, 8))
    k, v = rng.standard_normal((1, 1, L, 8)), rng.standard_normal((1, 1, L, 8))
    o, lse = oracle.prefill_dilated(q, k, v, w, s, r, 1.0)
    m = w - s
    for t in range(L):
        members = sorted(set(range(min(s, t + 1))) | {t - j * r for j in range(m) if t - j * r >= 0})
        np.testing.assert_allclose(o[0, 0, t], v[0, 0, members].mean(axis=0), atol=1e-12)
        assert abs(lse[0, 0, t] - math.log(len(members))) < 1e-12


def test_prefill_dilated_without_sinks_is_plain_attention_on_each_residue_class():
    # s = 0: row t only meets positions of its own residue class mod r, as a window of m on that
    # subsequence -- the plain oracle on the subsequence gives the same rows
    rng = np.random.default_rng(21)
    L, d, w, r = 41, 8, 5, 3
    q, k, v = (rng.standard_normal((1, 1, L, d)) for _ in range(3))
    o, lse = oracle.prefill_dilated(q, k, v, w, 0, r, 0.5)
    for c in range(r):
        idx = np.arange(c, L, r)
        o_c, l_c = oracle.prefill(q[:, :, idx], k[:, :, idx], v[:, :, idx], w, 0, 0.5)
        np.testing.assert_allclose(o[:, :, idx], o_c, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, idx], l_c, atol=1e-12)


@pytest.mark.parametrize("L,w,s,r", [(60, 9, 3, 4), (41, 6, 2, 3), (25, 5, 0, 2), (30, 7, 4, 1), (10, 6, 4, 3),
                                     (50, 4, 3, 9)])
def test_dilated_window_is_the_plain_window_on_virtual_heads(L, w, s, r):
    # the layout the GPU path uses: virtual head c = the s sinks, then the positions >= s of residue class
    # c (mod r); the plain key set (s sinks, window w) of a row there is the dilated key set of that row
    # in the sequence, and rows t < s are the sink prefix of head 0
    rng = np.random.default_rng(22 + L + r)
    d = 8
    q, k, v = (rng.standard_normal((1, 1, L, d)) for _ in range(3))
    o, lse = oracle.prefill_dilated(q, k, v, w, s, r, 0.4)
    got_o, got_l = np.full_like(o, np.nan), np.full_like(lse, np.nan)
    for c in range(r):
        pos = list(range(min(s, L))) + [p for p in range(s, L) if p % r == c]
        ov, lv = oracle.prefill(q[:, :, pos], k[:, :, pos], v[:, :, pos], w, s, 0.4)
        for u, p in enumerate(pos):
            if p >= s or c == 0:
                got_o[:, :, p], got_l[:, :, p] = ov[:, :, u], lv[:, :, u]
    np.testing.assert_allclose(got_o, o, atol=1e-12)
    np.testing.assert_allclose(got_l, lse, atol=1e-12)


@pytest.mark.parametrize("w,s,r", [(5, 2, 3), (8, 0, 2), (6, 4, 4), (9, 3, 1)])
def test_dilated_class_caches_hold_the_dilated_key_set(w, s, r):
    # the streaming layout: one rolling cache per residue class mod r, holding the sinks and the class's
    # positions >= s at class-local positions s, s + 1, ...; after writing step t, cache t mod r (cache 0
    # for t < s) holds exactly the dilated key set of t (the oracle's own slot replay per class)
    for t in range(70):
        c = 0 if t < s else t % r
        p0 = s + ((c - s) % r)
        local = t if t < s else s + (t - p0) // r
        held = oracle.cache_replay(w, s, local + 1)  # class-local position held by each slot
        orig = {int(x) if x < s else p0 + (int(x) - s) * r for x in held if x >= 0}
        want = {i for i in range(t + 1) if oracle.is_key_dilated(t, i, w, s, r)}
        assert orig == want, (w, s, r, t)


# ------------------------------------------------------------------ BigBird-style union (oracle ahead of its GPU path)
def test_blocksparse_mask_matches_hand_derived_golden():
    path = os.path.join(GOLDEN, "blocksparse_mask_L12_w3_s1_g5_b4.txt")
    rows = [l.strip() for l in open(path) if l.strip() and not l.startswith("#")]
    for t in range(12):
        for i in range(12):
            assert (rows[t][i] == "1") == oracle.is_key_blocksparse(t, i, 3, 1, {5}, 4, {2: [0]}), (t, i)


def test_blocksparse_without_globals_or_random_blocks_is_the_plain_oracle():
    rng = np.random.default_rng(23)
    q, k, v = (rng.standard_normal((1, 2, 40, 16)) for _ in range(3))
    o, lse = oracle.prefill_blocksparse(q, k, v, 9, 3, 0.3)
    o_ref, l_ref = oracle.prefill(q, k, v, 9, 3, 0.3)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, l_ref, atol=1e-12)


def test_blocksparse_every_position_global_is_full_causal_attention():
    rng = np.random.default_rng(24)
    L, d = 20, 8
    q, k, v = (rng.standard_normal((1, 1, L, d)) for _ in range(3))
    o, lse = oracle.prefill_blocksparse(q, k, v, 3, 1, 0.5, globals_=range(L))
    x = np.einsum("id,jd->ij", q[0, 0], k[0, 0]) * 0.5
    x = np.where(np.tril(np.ones((L, L), dtype=bool)), x, -np.inf)
    np.testing.assert_allclose(o[0, 0], scipy.special.softmax(x, axis=1) @ v[0, 0], atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], scipy.special.logsumexp(x, axis=1), atol=1e-12)


def test_blocksparse_random_blocks_add_whole_earlier_blocks():
    # with w = 1, s = 0 a row attends itself and exactly the causal part of its random key blocks
    block = 4
    rand = {2: [0], 3: [1, 3], 1: [1]}
    for t in range(16):
        want = {t} | {i for kb in rand.get(t // block, ()) for i in range(kb * block, kb * block + block) if i <= t}
        got = {i for i in range(t + 1) if oracle.is_key_blocksparse(t, i, 1, 0, (), block, rand)}
        assert got == want, t


def test_rope_and_dilated_single_key_windows_return_v():
    # w = 1, s = 0: every row attends only itself, so o = v and lse = scale q.k of the rotated pair
    # (RoPE: a key at the query's own position has rotation distance 0, so lse = scale q.k)
    rng = np.random.default_rng(25)
    q, k, v = (rng.standard_normal((1, 2, 15, 8)) for _ in range(3))
    o, lse = oracle.prefill_rope(q, k, v, 1, 0, 0.3)
    np.testing.assert_allclose(o, v, atol=1e-12)
    np.testing.assert_allclose(lse, 0.3 * np.einsum("bhld,bhld->bhl", q, k), atol=1e-12)
    for r in (1, 3, 100):
        o, lse = oracle.prefill_dilated(q, k, v, 1, 0, r, 0.3)
        np.testing.assert_allclose(o, v, atol=1e-12)


def test_dilation_past_the_sequence_leaves_sinks_and_self():
    # r >= L: the window holds only t itself, so row t attends the sinks and t
    L, w, s = 20, 5, 2
    for t in range(L):
        got = {i for i in range(t + 1) if oracle.is_key_dilated(t, i, w, s, L + 3)}
        assert got == set(range(min(s, t + 1))) | {t}


# ------------------------------------------------------------------ SWA + linear-attention hybrid (oracle ahead of its GPU path)
def _hybrid_direct(q, k, v, w, s, scale, wf):
    # the same quantity summed directly over the keys outside K(t) (no running state)
    nh, L, d = q.shape
    pq, pk = oracle.hedgehog(q, wf), oracle.hedgehog(k, wf)
    o = np.empty_like(q)
    for t in range(L):
        inside = [i for i in range(t + 1) if oracle.is_key(t, i, w, s)]
        outside = [i for i in range(t + 1) if not oracle.is_key(t, i, w, s)]
        e = np.exp(np.einsum("hd,hnd->hn", q[:, t], k[:, inside]) * scale)
        a = np.einsum("hd,hnd->hn", pq[:, t], pk[:, outside]) if outside else np.zeros((nh, 0))
        num = np.einsum("hn,hnd->hd", e, v[:, inside]) + (np.einsum("hn,hnd->hd", a, v[:, outside]) if outside else 0)
        o[:, t] = num / (e.sum(axis=1) + a.sum(axis=1))[:, None]
    return o


def test_hedgehog_feature_map():
    # phi(x) = (exp(x W), exp(-x W)): positive, so phi(q).phi(k) > 0 (the monotone, positive kernel the page
    # asks for); with W = 0 it is all ones and phi(q).phi(k) = d
    rng = np.random.default_rng(26)
    x, y = rng.standard_normal((5, 8)), rng.standard_normal((7, 8))
    wf = rng.standard_normal((8, 4)) * 0.3
    px, py = oracle.hedgehog(x, wf), oracle.hedgehog(y, wf)
    assert px.shape == (5, 8) and (px > 0).all() and (px @ py.T > 0).all()
    np.testing.assert_allclose(px[:, :4] * px[:, 4:], 1.0, atol=1e-12)  # exp(f) * exp(-f) = 1
    np.testing.assert_allclose(oracle.hedgehog(x, np.zeros((8, 4))) @ oracle.hedgehog(y, np.zeros((8, 4))).T, 8.0)


def test_hybrid_running_state_equals_the_direct_sum():
    # the page's recurrence (s_t, z_t), applied as keys leave the window, against direct summation
    rng = np.random.default_rng(27)
    q, k, v = (rng.standard_normal((2, 40, 8)) for _ in range(3))
    wf = rng.standard_normal((8, 4)) * 0.2
    for w, s in [(6, 2), (5, 0), (9, 4)]:
        np.testing.assert_allclose(oracle.hybrid_linear(q, k, v, w, s, 0.35, wf),
                                   _hybrid_direct(q, k, v, w, s, 0.35, wf), atol=1e-10)


def test_hybrid_without_evicted_keys_is_softmax_attention():
    # w >= L: no key ever leaves the window, so the linear branch is empty
    rng = np.random.default_rng(28)
    q, k, v = (rng.standard_normal((1, 2, 30, 8)) for _ in range(3))
    o = oracle.hybrid_linear(q[0], k[0], v[0], 40, 3, 0.3, rng.standard_normal((8, 4)))
    o_ref, _ = oracle.prefill(q, k, v, 40, 3, 0.3)
    np.testing.assert_allclose(o, o_ref[0], atol=1e-12)


def test_hybrid_with_a_flat_feature_map_in_closed_form():
    # W = 0: every evicted key weighs d, so o = (sum_K e^x v + d sum_R v) / (sum_K e^x + d |R|)
    rng = np.random.default_rng(29)
    L, d, w, s = 25, 8, 6, 2
    q, k, v = (rng.standard_normal((1, L, d)) for _ in range(3))
    o = oracle.hybrid_linear(q, k, v, w, s, 0.4, np.zeros((d, d // 2)))
    for t in range(L):
        K = [i for i in range(t + 1) if oracle.is_key(t, i, w, s)]
        R = [i for i in range(t + 1) if i not in K]
        e = np.exp(0.4 * q[0, t] @ k[0, K].T)
        want = (e @ v[0, K] + d * v[0, R].sum(axis=0)) / (e.sum() + d * len(R))
        np.testing.assert_allclose(o[0, t], want, atol=1e-12)


def test_hybrid_rows_equal_the_running_state():
    # the closed-form state at selected rows (any order, repeats) against the page's recurrence
    rng = np.random.default_rng(30)
    q, k, v = (rng.standard_normal((2, 50, 8)) for _ in range(3))
    wf = rng.standard_normal((8, 4)) * 0.25
    for w, s in [(7, 2), (5, 0), (12, 4)]:
        full = oracle.hybrid_linear(q, k, v, w, s, 0.3, wf)
        rows = [49, 0, 13, 13, 6, 30, 7]
        np.testing.assert_allclose(oracle.hybrid_linear_rows(q, k, v, w, s, 0.3, wf, rows), full[:, rows], atol=1e-10)
