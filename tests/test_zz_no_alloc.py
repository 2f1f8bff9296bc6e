"""The allocation-free decode entry point (swa_sink_decode_step_noalloc) gives the same result as the
regular one (swa_sink_decode_step with a caller workspace), called through the C ABI twice in a row.

It exists for callers that cannot allocate device memory when they run a decode step (a plugin callback
that must not allocate, a server whose pool owns all device memory, a token loop that cannot afford the
synchronisation an allocation may cause); its split-K scratch is an array built into the library. The
shape below has few (b, h) rows and a long window, so the step is split over several CTAs and really goes
through that scratch. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import swa_inputs
from gpu_common import BF16_MAX_ABS, BF16_MEAN_ABS, LSE_ABS, require_gpu

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, kc, vc, o, lse, t, w, s):
    B, H, d = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.swa_sink_decode_step_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                            B, H, d, w, s, t, 1.0 / d ** 0.5, 0, stream)


def test_noalloc_decode_matches_regular_decode_twice():
    swa = require_gpu()
    lib = swa.lib()
    B, H, d, w, s = 1, 2, 128, 2048, 4
    assert lib.swa_sink_decode_workspace_size(B, H, d, w) > 0  # the split path, which needs scratch
    T = 2600
    q, k, v = swa_inputs.prefill_inputs(B, H, T, d, 4242, torch.bfloat16, "cpu", sink_boost=True)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    for call, t in enumerate((2047, 2599)):  # two calls in a row: a full cache, then a wrapped ring
        kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        swa.kv_rolling_write(kc, vc, k[:, :, :t + 1].contiguous(), v[:, :, :t + 1].contiguous(), w, s, 0)
        qt = q[:, :, t].contiguous()
        o_ref = torch.empty((B, H, d), dtype=torch.bfloat16, device="cuda")
        l_ref = torch.empty((B, H), dtype=torch.float32, device="cuda")
        swa.swa_sink_decode_step(qt, kc, vc, t, w, s, o=o_ref, lse=l_ref)
        o = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(lib, qt, kc, vc, o, lse, t, w, s)
        assert rc == swa.SWA_OK, swa.last_error()
        assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
        err = (o.float() - o_ref.float()).abs()
        assert torch.isfinite(o.float()).all()
        assert err.max().item() <= BF16_MAX_ABS and err.mean().item() <= BF16_MEAN_ABS, f"call {call}"
        assert (lse - l_ref).abs().max().item() < LSE_ABS


def test_noalloc_decode_validates_before_launch():
    swa = require_gpu()
    lib = swa.lib()
    f = 1 << 20  # never dereferenced: validation fails first
    assert lib.swa_sink_decode_step_noalloc(f, f, f, f, None, 1, 1, 128, 8, 8, 0, 0.1, 0, None) == swa.SWA_ERR_INVALID
    assert lib.swa_sink_decode_step_noalloc(None, f, f, f, None, 1, 1, 128, 8, 4, 0, 0.1, 0, None) == swa.SWA_ERR_INVALID
