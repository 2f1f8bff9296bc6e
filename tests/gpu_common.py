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
