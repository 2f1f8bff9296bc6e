"""GPU parity of the rolling-cache write (bit-exact against the oracle's sequential replay) and of the
streaming decode (against the oracle's un-cached history definition, at every step)."""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from gpu_common import LSE_ABS, compare, require_gpu

pytestmark = pytest.mark.gpu


def position_pattern(B, H, n, d, pos0):
    """fp32 rows that encode (b*H + h, position) exactly: value = bh * 100000 + p (+ c / 1024 per column)."""
    bh = torch.arange(B * H, dtype=torch.float64).reshape(B, H, 1, 1)
    p = torch.arange(pos0, pos0 + n, dtype=torch.float64).reshape(1, 1, n, 1)
    c = torch.arange(d, dtype=torch.float64).reshape(1, 1, 1, d) / 1024.0
    return (bh * 100000 + p + c).float()


@pytest.mark.parametrize("w,s", [(8, 4), (16, 0), (5, 1), (64, 4), (33, 32)])
def test_rolling_write_slots_bit_exact(w, s):
    swa = require_gpu()
    B, H, d = 2, 3, 16
    kc = torch.full((B, H, w, d), -1.0, device="cuda")
    vc = torch.full((B, H, w, d), -2.0, device="cuda")
    batches = [1, 3, w - s, 1, 2 * w + 3, w, 7, 1, 3 * w]  # includes batches longer than the ring
    pos = 0
    for n in batches:
        kn = position_pattern(B, H, n, d, pos).cuda()
        swa.kv_rolling_write(kc, vc, kn, -kn, w, s, pos)
        pos += n
        torch.cuda.synchronize()
        holder = oracle.cache_replay(w, s, pos)
        got = kc.double().cpu().numpy()
        gotv = vc.double().cpu().numpy()
        for bh in range(B * H):
            b, h = divmod(bh, H)
            for j in range(w):
                if holder[j] < 0:
                    assert (got[b, h, j] == -1.0).all()
                    continue
                want = bh * 100000 + holder[j] + np.arange(d) / 1024.0
                assert np.array_equal(got[b, h, j], want.astype(np.float32)), (bh, j, holder[j])
                assert np.array_equal(gotv[b, h, j], -want.astype(np.float32))
    assert swa.swa_device_status() == swa.SWA_OK


def test_rolling_write_bf16_bytes_exact():
    swa = require_gpu()
    B, H, d, w, s = 1, 4, 128, 40, 4
    n = 3 * w + 11
    k, v = swa_inputs.normal((B, H, n, d), 5, 1), swa_inputs.normal((B, H, n, d), 5, 2)
    kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    swa.kv_rolling_write(kc, vc, k.cuda(), v.cuda(), w, s, 0)
    holder = oracle.cache_replay(w, s, n)
    assert (holder >= 0).all()
    want_k = k[:, :, torch.as_tensor(holder)]
    want_v = v[:, :, torch.as_tensor(holder)]
    assert torch.equal(kc.cpu().view(torch.int16), want_k.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), want_v.view(torch.int16))


@pytest.mark.parametrize("dtype,d,w,s", [
    (torch.bfloat16, 128, 40, 4),
    (torch.bfloat16, 64, 24, 0),
    (torch.bfloat16, 16, 17, 16),
    (torch.float32, 16, 16, 4),
    (torch.float32, 128, 9, 1),
])
def test_streaming_decode_every_step(dtype, d, w, s):
    swa = require_gpu()
    B, H = 2, 3
    T = 3 * w + 5
    q, k, v = swa_inputs.prefill_inputs(B, H, T, d, 77 + d, dtype, "cpu", sink_boost=True)
    kc = torch.zeros((B, H, w, d), dtype=dtype, device="cuda")
    vc = torch.zeros_like(kc)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    outs, lses = [], []
    for t in range(T):
        swa.kv_rolling_write(kc, vc, kg[:, :, t:t + 1].contiguous(), vg[:, :, t:t + 1].contiguous(), w, s, t)
        lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
        o = swa.swa_sink_decode_step(qg[:, :, t].contiguous(), kc, vc, t, w, s, lse=lse)
        outs.append(o.cpu())
        lses.append(lse.cpu())
    assert swa.swa_device_status() == swa.SWA_OK
    scale = 1.0 / math.sqrt(d)
    for t in range(T):
        o_ref, l_ref = oracle.decode(q[:, :, t].reshape(B * H, d), k[:, :, :t + 1].reshape(B * H, t + 1, d),
                                     v[:, :, :t + 1].reshape(B * H, t + 1, d), t, w, s, scale)
        compare(f"decode t={t}", outs[t].reshape(B * H, d), o_ref, dtype)
        assert np.abs(lses[t].double().numpy().reshape(-1) - l_ref).max() < LSE_ABS


@pytest.mark.parametrize("t", [0, 1, 255, 256, 1000, 2047, 2048, 2500, 5000])
def test_split_decode_long_window(t):
    # few (b, h) rows and a long window: the cache is split over several CTAs and merged
    swa = require_gpu()
    B, H, d, w, s = 1, 2, 128, 2048, 4
    n = t + 1
    q, k, v = swa_inputs.prefill_inputs(B, H, n, d, 300 + t, torch.bfloat16, "cpu", sink_boost=True)
    kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    swa.kv_rolling_write(kc, vc, k.cuda(), v.cuda(), w, s, 0)  # all positions 0..t in one batch
    ws = torch.empty(swa.swa_sink_decode_workspace_size(B, H, d, w), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_decode_step(q[:, :, t].contiguous().cuda(), kc, vc, t, w, s, lse=lse, workspace=ws)
    assert swa.swa_device_status() == swa.SWA_OK
    o_ref, l_ref = oracle.decode(q[:, :, t].reshape(B * H, d), k.reshape(B * H, n, d), v.reshape(B * H, n, d),
                                 t, w, s, 1.0 / math.sqrt(d))
    compare(f"split decode t={t}", o.cpu().reshape(B * H, d), o_ref, torch.bfloat16)
    assert np.abs(lse.cpu().double().numpy().reshape(-1) - l_ref).max() < LSE_ABS


def test_decode_resume_from_copied_cache():
    # the rolling cache is the whole decode state: a copy taken at step t resumes identically
    swa = require_gpu()
    B, H, d, w, s = 1, 2, 128, 32, 4
    T = 80
    q, k, v = [x.cuda() for x in swa_inputs.prefill_inputs(B, H, T, d, 9, torch.bfloat16, "cpu")]
    kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    outs = []
    snap = None
    for t in range(T):
        swa.kv_rolling_write(kc, vc, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), w, s, t)
        outs.append(swa.swa_sink_decode_step(q[:, :, t].contiguous(), kc, vc, t, w, s))
        if t == 50:
            snap = (kc.clone(), vc.clone())
    kc2, vc2 = snap
    for t in range(51, T):
        swa.kv_rolling_write(kc2, vc2, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), w, s, t)
        o2 = swa.swa_sink_decode_step(q[:, :, t].contiguous(), kc2, vc2, t, w, s)
        assert torch.equal(o2, outs[t])


# ------------------------------------------------- RoPE at the positions the entries have inside the cache
@pytest.mark.parametrize("dtype,d,w,s,base", [
    (torch.bfloat16, 128, 40, 4, 10000.0),
    (torch.bfloat16, 64, 24, 0, 10000.0),
    (torch.bfloat16, 16, 17, 16, 500.0),
    (torch.float32, 16, 16, 4, 10000.0),
    (torch.float32, 128, 9, 1, 10000.0),
])
def test_rope_streaming_decode_every_step(dtype, d, w, s, base):
    # write unrotated keys, decode with positions re-assigned inside the cache, at every step against the
    # oracle's history definition (through the window filling, the ring wrapping and long after)
    swa = require_gpu()
    B, H = 2, 3
    T = 3 * w + 5
    q, k, v = swa_inputs.prefill_inputs(B, H, T, d, 91 + d, dtype, "cpu", sink_boost=True)
    kc = torch.zeros((B, H, w, d), dtype=dtype, device="cuda")
    vc = torch.zeros_like(kc)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    outs, lses = [], []
    for t in range(T):
        swa.kv_rolling_write(kc, vc, kg[:, :, t:t + 1].contiguous(), vg[:, :, t:t + 1].contiguous(), w, s, t)
        lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
        o = swa.swa_sink_decode_step_rope(qg[:, :, t].contiguous(), kc, vc, t, w, s, rope_base=base, lse=lse)
        outs.append(o.cpu())
        lses.append(lse.cpu())
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    scale = 1.0 / math.sqrt(d)
    for t in range(T):
        o_ref, l_ref = oracle.decode_rope(q[:, :, t].reshape(B * H, d), k[:, :, :t + 1].reshape(B * H, t + 1, d),
                                          v[:, :, :t + 1].reshape(B * H, t + 1, d), t, w, s, scale, base)
        compare(f"rope decode t={t}", outs[t].reshape(B * H, d), o_ref, dtype)
        assert np.abs(lses[t].double().numpy().reshape(-1) - l_ref).max() < LSE_ABS


@pytest.mark.parametrize("w,t,base", [(2048, 0, 1e4), (2048, 700, 1e4), (2048, 2047, 1e4), (2048, 2048, 1e4),
                                      (2048, 3000, 1e4), (2048, 9000, 1e4), (16384, 16383, 1e4),
                                      (16384, 40000, 1e4), (8192, 20000, 5e5)])
def test_rope_split_decode_long_window(w, t, base):
    # few (b, h) rows and a long window: split-K over the cache; distances up to w - 1 = 16383 and a base
    # of 500000 check the angle reduction
    swa = require_gpu()
    B, H, d, s = 1, 2, 128, 4
    n = t + 1
    q, k, v = swa_inputs.prefill_inputs(B, H, n, d, 500 + t, torch.bfloat16, "cpu", sink_boost=True)
    kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    swa.kv_rolling_write(kc, vc, k.cuda(), v.cuda(), w, s, 0)
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_decode_step_rope(q[:, :, t].contiguous().cuda(), kc, vc, t, w, s, rope_base=base, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, l_ref = oracle.decode_rope(q[:, :, t].reshape(B * H, d), k.reshape(B * H, n, d), v.reshape(B * H, n, d),
                                      t, w, s, 1.0 / math.sqrt(d), base)
    compare(f"rope split decode t={t}", o.cpu().reshape(B * H, d), o_ref, torch.bfloat16)
    assert np.abs(lse.cpu().double().numpy().reshape(-1) - l_ref).max() < LSE_ABS
