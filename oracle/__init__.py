"""Oracle for causal sliding-window softmax attention with attention sinks (fp64, CPU).

TEST INFRASTRUCTURE. This package is the plain, slow, obviously-correct statement of the
computation, used only by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``. The GPU library never imports it and shares no code with it.

The arithmetic lives in ``swa_oracle.c`` (plain C, fp64, POSIX threads); this module converts
arrays to float64, calls it through ctypes and returns numpy arrays.

Definition (0-indexed positions, m = w - s recent keys):
    K(t) = { i <= t : i < s  or  i >= t - m + 1 }
    o_t  = sum_{i in K(t)} exp(x_i - M) v_i / sum_{i in K(t)} exp(x_i - M),  x_i = scale * q_t.k_i
    lse_t = M + log(sum_{i in K(t)} exp(x_i - M)),  M = max_{i in K(t)} x_i
It follows the SWA formula of the hyper.ai summary of arXiv 2608.28444 (section
"带 Sink 的滑动窗口注意力"; w keys including the query's own, the first s = 4 always attended in
addition to the w - 4 window keys), equation (1) of "模糊窗口注意力" section 2.1 (causal softmax
attention) and eq attn-fixed-softmax-sink of "滑窗与固定稀疏" (row normalisation).

``rope``, ``decode_rope`` and ``prefill_rope`` state the streaming decode and the prefill with
positions re-assigned inside the cache and rotary embedding (StreamingLLM section of "滑窗与固定稀疏").
``hedgehog`` and ``hybrid_linear`` state the SWA + linear-attention hybrid (a stated reading of the
combination); ``hybrid_linear_rows`` evaluates it at selected rows with the state summed in closed form
(pinned against the recurrence), for sampled rows of large cases.
``is_key_blocksparse`` and ``prefill_blocksparse`` state the BigBird-style union (window, global
tokens inside the sequence, given random key blocks) in causal form with sinks: an oracle ahead of its GPU
path.
``is_key_dilated`` and ``prefill_dilated`` state the dilated window with sinks (the dilated sliding
window of "滑窗与固定稀疏", glossary and Longformer section: attended positions skip r - 1 tokens).

Parity status: every function here is pinned by ``tests/test_oracle.py`` against closed forms,
textbook special cases and hand-derived golden values (``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libswa_oracle.so")
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into ``oracle/_build/libswa_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.swa_oracle_is_key.restype = ctypes.c_int
        lib.swa_oracle_is_key.argtypes = [ctypes.c_int64] * 4
        lib.swa_oracle_is_key_many.restype = None
        lib.swa_oracle_is_key_many.argtypes = [ctypes.c_int64, _i64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.POINTER(ctypes.c_uint8)]
        lib.swa_oracle_mask.restype = None
        lib.swa_oracle_mask.argtypes = [ctypes.c_int64] * 3 + [ctypes.POINTER(ctypes.c_uint8)]
        lib.swa_oracle_attend.restype = None
        lib.swa_oracle_attend.argtypes = [_f64p, _i64p, _f64p, _f64p, _i64p] + [ctypes.c_int64] * 6 + [
            ctypes.c_double, _f64p, _f64p, ctypes.c_int]
        lib.swa_oracle_cache_replay.restype = None
        lib.swa_oracle_cache_replay.argtypes = [ctypes.c_int64] * 3 + [_i64p]
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(a) -> np.ndarray:
    """Exact conversion of a numpy array or torch tensor (any float dtype) to contiguous float64."""
    if hasattr(a, "detach"):  # torch tensor: bf16/fp32 -> fp32 (exact) -> fp64 (exact)
        a = a.detach().to("cpu")
        if str(a.dtype) != "torch.float64":
            a = a.float()
        a = a.numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def is_key(t: int, i: int, w: int, s: int) -> bool:
    """Brute-force membership of key position i in the key set of query position t."""
    return bool(_get().swa_oracle_is_key(t, i, w, s))


def is_key_many(t: int, positions, w: int, s: int) -> np.ndarray:
    """Boolean array: membership of each key position in the key set of query position t."""
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    out = np.zeros(pos.shape, dtype=np.uint8)
    _get().swa_oracle_is_key_many(t, pos.ctypes.data_as(_i64p), pos.size, w, s,
                                  out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    return out.astype(bool)


def mask(L: int, w: int, s: int) -> np.ndarray:
    """L x L uint8 matrix, 1 where query t attends key i."""
    out = np.zeros((L, L), dtype=np.uint8)
    _get().swa_oracle_mask(L, w, s, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    return out


def attend(q, qpos, k, v, kpos, w: int, s: int, scale: float, nthreads: int | None = None):
    """Queries against explicitly given keys.

    q: [nh, nq, d]; k, v: [nh, nk, d]; qpos: [nq], kpos: [nk] absolute positions (any order).
    Returns (o [nh, nq, d] float64, lse [nh, nq] float64).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    qpos = np.ascontiguousarray(qpos, dtype=np.int64)
    kpos = np.ascontiguousarray(kpos, dtype=np.int64)
    nh, nq, d = q.shape
    nk = k.shape[1]
    assert k.shape == (nh, nk, d) and v.shape == (nh, nk, d)
    assert qpos.shape == (nq,) and kpos.shape == (nk,)
    o = np.empty((nh, nq, d), dtype=np.float64)
    lse = np.empty((nh, nq), dtype=np.float64)
    _get().swa_oracle_attend(q.ctypes.data_as(_f64p), qpos.ctypes.data_as(_i64p), k.ctypes.data_as(_f64p),
                             v.ctypes.data_as(_f64p), kpos.ctypes.data_as(_i64p), nh, nq, nk, d, w, s,
                             float(scale), o.ctypes.data_as(_f64p), lse.ctypes.data_as(_f64p),
                             int(nthreads or default_threads()))
    return o, lse


def prefill(q, k, v, w: int, s: int, scale: float, nthreads: int | None = None):
    """Whole-sequence prefill: q, k, v [B, H, L, d] -> (o [B, H, L, d], lse [B, H, L]), fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, L, d = q.shape
    pos = np.arange(L, dtype=np.int64)
    o, lse = attend(q.reshape(B * H, L, d), pos, k.reshape(B * H, L, d), v.reshape(B * H, L, d), pos,
                    w, s, scale, nthreads)
    return o.reshape(B, H, L, d), lse.reshape(B, H, L)


def prefill_rows(q_rows, rows, k, v, w: int, s: int, scale: float, nthreads: int | None = None):
    """Selected query rows of a prefill: q_rows [nh, nr, d] at positions ``rows`` against the full key
    history k, v [nh, L, d] (positions 0..L-1)."""
    k, v = _f64(k), _f64(v)
    kpos = np.arange(k.shape[1], dtype=np.int64)
    return attend(q_rows, np.asarray(rows, dtype=np.int64), k, v, kpos, w, s, scale, nthreads)


def decode(q_t, k_hist, v_hist, t: int, w: int, s: int, scale: float, nthreads: int | None = None):
    """Streaming decode at position t from the full, un-cached history.

    q_t: [nh, d]; k_hist, v_hist: [nh, t + 1, d] (positions 0..t). Returns (o [nh, d], lse [nh]).
    The cache is never consulted: the definition is applied to the history.
    """
    q_t = _f64(q_t)
    nh, d = q_t.shape
    kpos = np.arange(t + 1, dtype=np.int64)
    o, lse = attend(q_t.reshape(nh, 1, d), np.array([t], dtype=np.int64), k_hist, v_hist, kpos,
                    w, s, scale, nthreads)
    return o.reshape(nh, d), lse.reshape(nh)


def rope(x, pos, base: float = 10000.0) -> np.ndarray:
    """Rotary position embedding of rows x [..., n, d] at positions pos [n] (fp64).

    The pages name RoPE without printing it (StreamingLLM section of "滑窗与固定稀疏"); this is its plain
    reading in the form of the Llama-2 / Mistral models the pages use: dimension i of the first half and
    dimension i + d/2 form a pair that is rotated by the angle pos * base^(-2i/d), i = 0 .. d/2 - 1.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    theta = base ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]
    c, sn = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * sn, x1 * sn + x2 * c], axis=-1)


def decode_rope(q_t, k_hist, v_hist, t: int, w: int, s: int, scale: float, base: float = 10000.0,
                nthreads: int | None = None):
    """Streaming decode at position t with positions re-assigned inside the cache (StreamingLLM section
    of "滑窗与固定稀疏": the cache holds the s sinks and the m most recent tokens, their positional
    encoding is their consecutive position inside the cache, 0 .. s+m-1, not the original position, and
    RoPE is applied each step to keys kept unrotated).

    q_t: [nh, d] unrotated query; k_hist, v_hist: [nh, t + 1, d] unrotated history (positions 0..t).
    The key set K(t) is decided per key by the brute-force test; its members, in increasing original
    position (the sinks first, then the window), take cache positions 0 .. n-1; the query, whose own
    key is the newest member, takes position n - 1.  Returns (o [nh, d], lse [nh]).
    """
    q_t = _f64(q_t)
    nh, d = q_t.shape
    members = np.array([i for i in range(t + 1) if is_key(t, i, w, s)], dtype=np.int64)
    cpos = np.arange(len(members), dtype=np.float64)
    k_rot = rope(_f64(k_hist)[:, members], cpos, base)
    v_sel = np.ascontiguousarray(_f64(v_hist)[:, members])
    q_rot = rope(q_t[:, None, :], np.array([len(members) - 1.0]), base)
    o, lse = attend(q_rot, np.array([t], dtype=np.int64), k_rot, v_sel, members, w, s, scale, nthreads)
    return o.reshape(nh, d), lse.reshape(nh)


def prefill_rope(q, k, v, w: int, s: int, scale: float, base: float = 10000.0, rows=None,
                 nthreads: int | None = None):
    """Prefill with positions re-assigned inside the cache (StreamingLLM section of "滑窗与固定稀疏"):
    row t is the streaming decode at step t over the same unrotated keys (``decode_rope``), i.e. the
    members of K(t) take cache positions 0 .. |K(t)| - 1 and the query the last of them.

    q, k, v: [B, H, L, d] unrotated; ``rows``: query positions to compute (default all).
    Returns (o [B, H, len(rows), d], lse [B, H, len(rows)]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, L, d = q.shape
    rows = list(range(L)) if rows is None else [int(t) for t in rows]
    o = np.empty((B * H, len(rows), d))
    lse = np.empty((B * H, len(rows)))
    qf, kf, vf = q.reshape(B * H, L, d), k.reshape(B * H, L, d), v.reshape(B * H, L, d)
    for j, t in enumerate(rows):
        o[:, j], lse[:, j] = decode_rope(qf[:, t], kf[:, :t + 1], vf[:, :t + 1], t, w, s, scale, base, nthreads)
    return o.reshape(B, H, len(rows), d), lse.reshape(B, H, len(rows))


def is_key_dilated(t: int, i: int, w: int, s: int, r: int) -> bool:
    """Brute-force membership of key position i in the dilated key set of query t: the s sinks, and the
    m = w - s window keys t, t - r, ..., t - (m-1) r, each skipping r - 1 positions (the dilated window of
    the fixed-sparsity page, in its causal form with sinks)."""
    m = w - s
    if i < 0 or i > t:
        return False
    return i < s or ((t - i) % r == 0 and (t - i) // r < m)


def prefill_dilated(q, k, v, w: int, s: int, r: int, scale: float, rows=None):
    """Whole-sequence prefill over the dilated key sets (fp64, numpy): row t attends
    {i < s} | {t - j r : 0 <= j < m}, restricted to i <= t, softmax of scale * q.k.

    q, k, v: [B, H, L, d]; ``rows``: query positions to compute (default all).
    Returns (o [B, H, len(rows), d], lse [B, H, len(rows)]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, L, d = q.shape
    rows = list(range(L)) if rows is None else [int(t) for t in rows]
    qf, kf, vf = q.reshape(B * H, L, d), k.reshape(B * H, L, d), v.reshape(B * H, L, d)
    o = np.empty((B * H, len(rows), d))
    lse = np.empty((B * H, len(rows)))
    for j, t in enumerate(rows):
        members = np.array([i for i in range(t + 1) if is_key_dilated(t, i, w, s, r)], dtype=np.int64)
        x = np.einsum("hd,hnd->hn", qf[:, t], kf[:, members]) * scale
        mx = x.max(axis=1, keepdims=True)
        e = np.exp(x - mx)
        den = e.sum(axis=1)
        o[:, j] = np.einsum("hn,hnd->hd", e, vf[:, members]) / den[:, None]
        lse[:, j] = mx[:, 0] + np.log(den)
    return o.reshape(B, H, len(rows), d), lse.reshape(B, H, len(rows))


def is_key_blocksparse(t: int, i: int, w: int, s: int, globals_=(), block: int = 1, rand_blocks=None) -> bool:
    """Membership in the BigBird-style key set of query t (the union of local window, global and random
    connections of the fixed-sparsity page, eq attn-fixed-bigbird, with global tokens placed inside the
    sequence (ITC)), in causal form with the sinks: i <= t and one of
      i < s (sink), i >= t - m + 1 (window), i a global position, t a global position (a global query sees
      every earlier key), or key block i // block in rand_blocks[t // block] (the query block's random key
      blocks; the random choice is an input)."""
    m = w - s
    if i < 0 or i > t:
        return False
    if i < s or i >= t - m + 1 or i in globals_ or t in globals_:
        return True
    return rand_blocks is not None and (i // block) in rand_blocks.get(t // block, ())


def prefill_blocksparse(q, k, v, w: int, s: int, scale: float, globals_=(), block: int = 1, rand_blocks=None,
                        rows=None):
    """Whole-sequence prefill over the key sets of ``is_key_blocksparse`` (fp64, numpy per row).
    q, k, v: [B, H, L, d]; globals_: positions of the global tokens; rand_blocks: {query block: key blocks}.
    Returns (o [B, H, len(rows), d], lse [B, H, len(rows)])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, L, d = q.shape
    rows = list(range(L)) if rows is None else [int(t) for t in rows]
    g = set(int(x) for x in globals_)
    qf, kf, vf = q.reshape(B * H, L, d), k.reshape(B * H, L, d), v.reshape(B * H, L, d)
    o = np.empty((B * H, len(rows), d))
    lse = np.empty((B * H, len(rows)))
    for j, t in enumerate(rows):
        members = np.array([i for i in range(t + 1) if is_key_blocksparse(t, i, w, s, g, block, rand_blocks)],
                           dtype=np.int64)
        x = np.einsum("hd,hnd->hn", qf[:, t], kf[:, members]) * scale
        mx = x.max(axis=1, keepdims=True)
        e = np.exp(x - mx)
        den = e.sum(axis=1)
        o[:, j] = np.einsum("hn,hnd->hd", e, vf[:, members]) / den[:, None]
        lse[:, j] = mx[:, 0] + np.log(den)
    return o.reshape(B, H, len(rows), d), lse.reshape(B, H, len(rows))


def hedgehog(x, wf) -> np.ndarray:
    """The Hedgehog feature map of the linear-attention section of the hyper.ai summary of 2608.28444:
    phi(x) = (exp(f(x)), exp(-f(x))) with f(x) = x wf a linear projection from d to d/2 (wf: [d, d/2],
    a given matrix -- the learned one needs weights).  x: [..., d] -> [..., d]."""
    f = np.asarray(x, dtype=np.float64) @ np.asarray(wf, dtype=np.float64)
    return np.concatenate([np.exp(f), np.exp(-f)], axis=-1)


def hybrid_linear(q, k, v, w: int, s: int, scale: float, wf):
    """SWA with sinks plus a linear-attention branch for the keys that left the window (the hybrid of
    the hyper.ai summary of 2608.28444: the SWA branch keeps local detail, the linear branch aggregates
    the rest).  Reading, as in the LoLCATs model that summary discusses: one shared normaliser,
        o_t = (sum_{i in K(t)} e^{x_i} v_i + phi(q_t) s_t) / (sum_{i in K(t)} e^{x_i} + phi(q_t) z_t),
    x_i = scale q_t.k_i, K(t) the sinks + window, and (s_t, z_t) the running state of the keys outside it,
    updated by the page's recurrence s <- s + phi(k)^T v, z <- z + phi(k)^T as each key leaves the window
    (key i leaves at step i + m; the sinks never do).  q, k, v: [nh, L, d]; returns o [nh, L, d] (fp64)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    nh, L, d = q.shape
    m = w - s
    pq, pk = hedgehog(q, wf), hedgehog(k, wf)
    S = np.zeros((nh, d, d))
    z = np.zeros((nh, d))
    o = np.empty((nh, L, d))
    for t in range(L):
        i_out = t - m  # the key that leaves the window at step t (sinks excepted)
        if i_out >= s:
            S += np.einsum("hi,hj->hij", pk[:, i_out], v[:, i_out])
            z += pk[:, i_out]
        members = np.array([i for i in range(t + 1) if is_key(t, i, w, s)], dtype=np.int64)
        e = np.exp(np.einsum("hd,hnd->hn", q[:, t], k[:, members]) * scale)
        num = np.einsum("hn,hnd->hd", e, v[:, members]) + np.einsum("hi,hij->hj", pq[:, t], S)
        den = e.sum(axis=1) + np.einsum("hi,hi->h", pq[:, t], z)
        o[:, t] = num / den[:, None]
    return o


def hybrid_linear_rows(q, k, v, w: int, s: int, scale: float, wf, rows):
    """``hybrid_linear`` at selected rows, with the state in closed form: S_t = sum_{i=s}^{t-m} phi(k_i)^T v_i,
    z_t = sum_{i=s}^{t-m} phi(k_i)^T (the page's recurrence summed out), accumulated between consecutive rows
    in increasing order.  q, k, v: [nh, L, d]; returns o [nh, len(rows), d] (fp64) in the order of ``rows``."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    nh, L, d = q.shape
    m = w - s
    pk = hedgehog(k, wf)
    order = sorted(range(len(rows)), key=lambda j: int(rows[j]))
    S = np.zeros((nh, d, d))
    z = np.zeros((nh, d))
    upto = s  # keys s .. upto-1 are in the state
    o = np.empty((nh, len(rows), d))
    for j in order:
        t = int(rows[j])
        end = t - m + 1  # keys s .. t-m have left the window
        if end > upto:
            S += np.matmul(pk[:, upto:end].transpose(0, 2, 1), v[:, upto:end])
            z += pk[:, upto:end].sum(axis=1)
            upto = end
        members = np.array([i for i in range(t + 1) if is_key(t, i, w, s)], dtype=np.int64)
        e = np.exp(np.einsum("hd,hnd->hn", q[:, t], k[:, members]) * scale)
        pq = hedgehog(q[:, t], wf)
        num = np.einsum("hn,hnd->hd", e, v[:, members]) + np.einsum("hi,hij->hj", pq, S)
        den = e.sum(axis=1) + np.einsum("hi,hi->h", pq, z)
        o[:, j] = num / den[:, None]
    return o


def cache_replay(w: int, s: int, npos: int) -> np.ndarray:
    """Slot -> position held after writing positions 0..npos-1 one by one (-1 = never written)."""
    out = np.empty(w, dtype=np.int64)
    _get().swa_oracle_cache_replay(w, s, npos, out.ctypes.data_as(_i64p))
    return out
