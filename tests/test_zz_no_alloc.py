"""The allocation-free decode entry point (swa_sink_decode_step_noalloc) gives the same result as the
regular one (swa_sink_decode_step with a caller workspace), called through the C ABI several times in a row.

It exists for callers that cannot allocate device memory when they run a decode step (a plugin callback
that must not allocate, a server whose pool owns all device memory, a token loop that cannot afford the
synchronisation an allocation may cause); its split-K scratch is an array built into the library. The
shapes below have few (b, h) rows and long windows, so every step is split over several CTAs and really
goes through that scratch. A call with a larger scratch footprint runs first, so the checked calls read a
scratch array that still holds another call's partials: they must be ignored. Both entry points run the
same kernels with the same split count, so their outputs must agree bit for bit; the checked calls are
also compared with the oracle. This file is collected last on purpose.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from gpu_common import BF16_MAX_ABS, BF16_MEAN_ABS, LSE_ABS, require_gpu

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, kc, vc, o, lse, t, w, s):
    B, H, d = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.swa_sink_decode_step_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                            B, H, d, w, s, t, 1.0 / d ** 0.5, 0, stream)


def _cache_at(k, v, t, w, s):
    B, H, _, d = k.shape
    kc = torch.full((B, H, w, d), float("nan"), dtype=k.dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    import sliding_window_softmax_swa_gb300 as swa
    swa.kv_rolling_write(kc, vc, k[:, :, :t + 1].contiguous(), v[:, :, :t + 1].contiguous(), w, s, 0)
    return kc, vc


def test_noalloc_decode_matches_regular_decode_and_oracle():
    swa = require_gpu()
    lib = swa.lib()
    d, s = 128, 4
    # a larger footprint first: 64 (b, h) rows x 16 splits of partials fill ~0.5 MiB of the array
    Bb, Hb, wb = 4, 16, 4096
    assert 0 < lib.swa_sink_decode_workspace_size(Bb, Hb, d, wb) <= (2 << 20)
    qb, kb, vb = swa_inputs.prefill_inputs(Bb, Hb, wb, d, 4141, torch.bfloat16, "cuda", sink_boost=True)
    kcb, vcb = _cache_at(kb, vb, wb - 1, wb, s)
    ob = torch.empty((Bb, Hb, d), dtype=torch.bfloat16, device="cuda")
    lb = torch.empty((Bb, Hb), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, qb[:, :, wb - 1].contiguous(), kcb, vcb, ob, lb, wb - 1, wb, s) == swa.SWA_OK, swa.last_error()
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()

    # then the checked calls, twice in a row on a smaller footprint that still splits
    B, H, w = 1, 2, 2048
    assert lib.swa_sink_decode_workspace_size(B, H, d, w) > 0
    T = 2600
    q, k, v = swa_inputs.prefill_inputs(B, H, T, d, 4242, torch.bfloat16, "cpu", sink_boost=True)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    for call, t in enumerate((2047, 2599)):  # a full cache, then a wrapped ring
        kc, vc = _cache_at(kg, vg, t, w, s)
        qt = qg[:, :, t].contiguous()
        o_ref = torch.empty((B, H, d), dtype=torch.bfloat16, device="cuda")
        l_ref = torch.empty((B, H), dtype=torch.float32, device="cuda")
        swa.swa_sink_decode_step(qt, kc, vc, t, w, s, o=o_ref, lse=l_ref)
        o = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(lib, qt, kc, vc, o, lse, t, w, s)
        assert rc == swa.SWA_OK, swa.last_error()
        assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), f"call {call}: o differs from the regular call"
        assert torch.equal(lse, l_ref), f"call {call}: lse differs from the regular call"
        want, lwant = oracle.decode(q[:, :, t].reshape(B * H, d), k[:, :, :t + 1].reshape(B * H, t + 1, d),
                                    v[:, :, :t + 1].reshape(B * H, t + 1, d), t, w, s, 1.0 / math.sqrt(d))
        err = np.abs(o.float().cpu().numpy().reshape(B * H, d) - want)
        assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS, f"call {call} vs oracle: {err.max():.3e}"
        assert np.abs(lse.cpu().numpy().reshape(B * H) - lwant).max() < LSE_ABS


def test_noalloc_decode_validates_before_launch():
    swa = require_gpu()
    lib = swa.lib()
    f = 1 << 20  # never dereferenced: validation fails first
    assert lib.swa_sink_decode_step_noalloc(f, f, f, f, None, 1, 1, 128, 8, 8, 0, 0.1, 0, None) == swa.SWA_ERR_INVALID
    assert lib.swa_sink_decode_step_noalloc(None, f, f, f, None, 1, 1, 128, 8, 4, 0, 0.1, 0, None) == swa.SWA_ERR_INVALID
