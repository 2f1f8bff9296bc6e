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


# ---------------------------------------------------------------- RoPE prefill: rotated operands
def check_rope_prefill(name, o_got, lse_got, ops, qf, kf, vf, rows, w, s, scale, base, o_ref, l_ref):
    """RoPE prefill rows, in two parts.
    (a) The rotation pass: ops = (qr, kr, ssink), read back from the kernel's workspace.  qr (at the selected
        rows) and kr (at positions 0..max(rows)) as hi + lo: each element within 2^-16 relative of the oracle's
        fp64 rotation (q at t, k at i; the (hi, lo) bf16 pair keeps ~17 bits), plus 1e-5 of the row's largest
        input magnitude for the fp32 sin/cos (absolute error ~5e-7) where x cos - y sin cancels.
        ssink[row, i], i < s, is the sink score (R(min(t, w - 1)) q_t) . (R(i) k_i): within 1e-5 |R q| |R k| of
        the oracle's fp64 dot product of its fp64 rotations (fp32 rotations and an fp32 sum of 128 terms).
    (b) The result against the oracle's exact definition (o_ref, l_ref) with the bf16 tolerances of every
        path and 1e-3 on the log-sum-exp: the window scores are formed from the (hi, lo) operands with the error
        of fp32 ones, the sink scores in fp32, far below what the bf16 output rounding allows.
    o_got [nh, nr, d], lse_got [nh, nr]: numpy fp64."""
    qr, kr, ssink = ops
    top = max(rows) + 1
    pos = np.arange(top, dtype=np.float64)
    rows_f = np.asarray(rows, dtype=np.float64)
    for got, src, want, what in ((qr, qf[:, rows], oracle.rope(qf[:, rows], rows_f, base), "q at t"),
                                 (kr, kf[:, :top], oracle.rope(kf[:, :top], pos, base), "k at i")):
        slack = 1e-5 * np.abs(src).max(axis=-1, keepdims=True)
        assert (np.abs(got - want) <= 2.0 ** -16 * np.abs(want) + slack).all(), f"{name}: rotated {what}"
    if s > 0:
        qs = oracle.rope(qf[:, rows], np.minimum(rows_f, w - 1), base)   # [nh, nr, d]
        ks = oracle.rope(kf[:, :s], np.arange(s, dtype=np.float64), base)  # [nh, s, d]
        want = np.einsum("hrd,hid->hri", qs, ks)
        bound = 1e-5 * np.linalg.norm(qs, axis=-1)[:, :, None] * np.linalg.norm(ks, axis=-1)[:, None, :]
        assert (np.abs(ssink - want) <= bound).all(), f"{name}: sink scores"
    compare(f"{name} vs oracle", o_got, o_ref, torch.bfloat16)
    assert np.abs(lse_got - l_ref).max() < LSE_ABS, f"{name}: lse vs oracle"


def rope_workspace_operands(ws, B, H, L, d, s, rows):
    """What a RoPE prefill left in its workspace (qr, qr_lo, kr, kr_lo: bf16 [B*H, L, d] each; then the sink
    scores, fp32 [B*H, L, 4 ceil(s/4)]), in fp64: qr as hi + lo at the selected rows, kr as hi + lo at positions
    0..max(rows), and the first s sink scores of the selected rows."""
    nh = B * H
    one = nh * L * d
    t = ws[:4 * one * 2].view(torch.bfloat16).reshape(4, nh, L, d).double()
    top = max(rows) + 1
    ridx = torch.as_tensor(rows, device=ws.device)
    qr, kr = t[0] + t[1], t[2] + t[3]
    sst = (s + 3) // 4 * 4
    ss = ws[4 * one * 2:4 * one * 2 + nh * L * sst * 4].view(torch.float32).reshape(nh, L, sst).double()
    return qr[:, ridx].cpu().numpy(), kr[:, :top].cpu().numpy(), ss[:, ridx, :s].cpu().numpy()
