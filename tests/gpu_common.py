"""Shared helpers of the GPU tests: library loading, seeded inputs, oracle comparisons and tolerances."""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs

# Tolerances against the fp64 oracle: bf16 outputs (fp32 accumulation) and the fp32 CUDA-core path.
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
F32_MAX_ABS = 1e-4
LSE_ABS = 1e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for tests marked gpu")
    import sliding_window_softmax_swa_gb300 as swa
    swa.lib(build_if_missing=True)  # the CUDA library must be there; there is no fallback
    return swa


def inputs(B, H, L, d, dtype, seed, sink_boost=False, device="cuda"):
    """Seeded q, k, v [B, H, L, d]; drawn on the CPU for small sizes so the bytes are platform-stable."""
    gen_dev = "cpu" if B * H * L * d <= (1 << 22) else device
    q, k, v = swa_inputs.prefill_inputs(B, H, L, d, seed, dtype, gen_dev, sink_boost)
    return q.to(device), k.to(device), v.to(device)


def compare(name, got, want, dtype, max_abs=None, mean_abs=None):
    got = got.detach().float().cpu().numpy().astype(np.float64) if hasattr(got, "detach") else got
    err = np.abs(got - want)
    assert np.isfinite(got).all(), f"{name}: non-finite output"
    if dtype == torch.float32:
        lim = F32_MAX_ABS if max_abs is None else max_abs
        assert err.max() <= lim, f"{name}: max-abs {err.max():.3e} > {lim}"
    else:
        lim = BF16_MAX_ABS if max_abs is None else max_abs
        lim_mean = BF16_MEAN_ABS if mean_abs is None else mean_abs
        assert err.max() <= lim, f"{name}: max-abs {err.max():.3e} > {lim}"
        assert err.mean() <= lim_mean, f"{name}: mean-abs {err.mean():.3e} > {lim_mean}"
    return float(err.max()), float(err.mean())


def oracle_rows(q, k, v, bh_list, row_blocks, w, s, scale, pos_offset=0):
    """Oracle of selected (head, row-block) pairs of a prefill over q/k/v [B, H, L, d] (any device).

    For a block of rows [r0, r1) only the keys the oracle needs are copied: positions [0, s) and
    [r0 - m, r1), each tagged with its absolute position; the oracle decides membership itself.
    Returns {(bh, r0): (o [r1-r0, d], lse [r1-r0])}.
    """
    B, H, L, d = q.shape
    m = w - s
    qf, kf, vf = q.reshape(B * H, L, d), k.reshape(B * H, L, d), v.reshape(B * H, L, d)
    out = {}
    for bh in bh_list:
        for r0, r1 in row_blocks:
            lo = max(0, r0 - m - 1)
            kpos = np.array(sorted(set(range(min(s, r1))) | set(range(lo, r1))), dtype=np.int64)
            idx = torch.as_tensor(kpos, device=k.device)
            kk = kf[bh].index_select(0, idx)[None]
            vv = vf[bh].index_select(0, idx)[None]
            o, l = oracle.attend(qf[bh, r0:r1][None], np.arange(r0, r1) + pos_offset, kk, vv, kpos + pos_offset,
                                 w, s, scale)
            out[(bh, r0)] = (o[0], l[0])
    return out


# ---------------------------------------------------------------- RoPE prefill: operand rounding and bounds
def rope_operand_reference(qr, qs, kr, vf, rows, w, s, scale):
    """fp64 softmax attention of the selected rows on given rotated operands: the window keys i of row t
    scored with qr[:, t] . kr[:, i], the sinks with qs[:, t] . kr[:, i].  All [nh, ., d] fp64; qr and qs
    hold the selected rows only.  Returns (o [nh, len(rows), d], lse [nh, len(rows)])."""
    nh = vf.shape[0]
    d = vf.shape[2]
    m = w - s
    o = np.empty((nh, len(rows), d))
    lse = np.empty((nh, len(rows)))
    for j, t in enumerate(rows):
        snk = np.arange(0, min(s, t + 1))
        win = np.arange(max(s, t - m + 1), t + 1)
        x = np.concatenate([np.einsum("hd,hnd->hn", qs[:, j], kr[:, snk]),
                            np.einsum("hd,hnd->hn", qr[:, j], kr[:, win])], axis=1) * scale
        idx = np.concatenate([snk, win])
        mx = x.max(axis=1, keepdims=True)
        e = np.exp(x - mx)
        l = e.sum(axis=1)
        o[:, j] = np.einsum("hn,hnd->hd", e, vf[:, idx]) / l[:, None]
        lse[:, j] = mx[:, 0] + np.log(l)
    return o, lse


def rope_score_error_bound(qf, kf, rows, w, scale, base=10000.0):
    """Per (head, row): the largest error the bf16 rounding of the rotated q and k (relative 2^-9 each, so
    2^-8 + 2^-18 per product term, plus fp32 slack) can put on one score: scale (2^-8 + 2^-16)
    max_i sum_j |q~_j k~_i,j| over the keys i <= t, q~ in both of its rotations."""
    top = max(rows) + 1
    kr = np.abs(oracle.rope(kf[:, :top], np.arange(top, dtype=np.float64), base))
    out = np.empty((qf.shape[0], len(rows)))
    for j, t in enumerate(rows):
        qr = np.abs(oracle.rope(qf[:, t:t + 1], [float(t)], base))[:, 0]
        qs = np.abs(oracle.rope(qf[:, t:t + 1], [float(min(t, w - 1))], base))[:, 0]
        worst = np.maximum(np.einsum("hd,hnd->hn", qr, kr[:, :t + 1]).max(axis=1),
                           np.einsum("hd,hnd->hn", qs, kr[:, :t + 1]).max(axis=1))
        out[:, j] = scale * (2.0 ** -8 + 2.0 ** -16) * worst
    return out


def check_rope_prefill(name, o_got, lse_got, ops, qf, kf, vf, rows, w, s, scale, base, o_ref, l_ref):
    """RoPE prefill rows, in three parts.
    (a) The rotation pass: ops = (qr, qs, kr), the kernel's bf16 operands read back from its workspace (qr,
        qs at the selected rows, kr at positions 0..max(rows)), each element within one bf16 ulp (2^-8
        relative) of the oracle's fp64 rotation (q at t, q at min(t, w - 1), k at i), plus 1e-5 of the row's
        largest input magnitude for the fp32 sin/cos (absolute error ~5e-7) where x cos - y sin cancels.
    (b) The attention on those operands: against fp64 attention on the same operands, with the bf16
        tolerances of every path (and 1e-3 on the log-sum-exp).
    (c) The whole against the oracle's exact definition (o_ref, l_ref): the operand rounding moves a score
        by at most eps (rope_score_error_bound), so |d lse| <= LSE_ABS + eps and, since each softmax weight
        then changes by a factor within e^(+-2 eps) and the changes sum to zero,
        |d o| <= BF16_MAX_ABS + (e^(2 eps) - 1) max_i |v_i - o| per element.
    o_got [nh, nr, d], lse_got [nh, nr]: numpy fp64."""
    qr, qs, kr = ops
    top = max(rows) + 1
    pos = np.arange(top, dtype=np.float64)
    rows_f = np.asarray(rows, dtype=np.float64)
    for got, src, want, what in ((qr, qf[:, rows], oracle.rope(qf[:, rows], rows_f, base), "q at t"),
                                 (qs, qf[:, rows], oracle.rope(qf[:, rows], np.minimum(rows_f, w - 1), base),
                                  "q at min(t, w-1)"),
                                 (kr, kf[:, :top], oracle.rope(kf[:, :top], pos, base), "k at i")):
        slack = 1e-5 * np.abs(src).max(axis=-1, keepdims=True)
        assert (np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + slack).all(), f"{name}: rotated {what}"
    o_op, l_op = rope_operand_reference(qr, qs, kr, vf, rows, w, s, scale)
    compare(f"{name} vs attention on its operands", o_got, o_op, torch.bfloat16)
    assert np.abs(lse_got - l_op).max() < LSE_ABS, f"{name}: lse vs attention on its operands"
    eps = rope_score_error_bound(qf, kf, rows, w, scale, base)
    assert (np.abs(lse_got - l_ref) <= LSE_ABS + eps).all(), f"{name}: lse vs oracle"
    m = w - s
    for j, t in enumerate(rows):
        idx = np.concatenate([np.arange(0, min(s, t + 1)), np.arange(max(s, t - m + 1), t + 1)])
        spread = np.abs(vf[:, idx] - o_ref[:, j][:, None, :]).max(axis=1)  # [nh, d]
        lim = BF16_MAX_ABS + np.expm1(2 * eps[:, j])[:, None] * spread
        assert (np.abs(o_got[:, j] - o_ref[:, j]) <= lim).all(), f"{name}: row {t} vs oracle"


def rope_workspace_operands(ws, B, H, L, d, rows):
    """The rotated operands a RoPE prefill left in its workspace (qr | qs | kr, bf16 [B*H, L, d] each):
    qr and qs at the selected rows, kr at positions 0..max(rows), as fp64 numpy."""
    nh = B * H
    t = ws[:3 * nh * L * d * 2].view(torch.bfloat16).reshape(3, nh, L, d)
    top = max(rows) + 1
    ridx = torch.as_tensor(rows, device=ws.device)
    return (t[0][:, ridx].double().cpu().numpy(), t[1][:, ridx].double().cpu().numpy(),
            t[2][:, :top].double().cpu().numpy())
