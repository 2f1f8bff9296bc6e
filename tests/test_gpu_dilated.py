"""GPU parity of the prefill over a dilated window with sinks (swa_sink_prefill_dilated) against the oracle's
definition, element by element: bf16 outputs within the tolerances of every bf16 path (one rounding of o),
fp32 within 1e-4, lse within 1e-3.  bf16 with d = 128 runs in place (the tensor-core pass over whole groups of r
positions after the sinks, read through 4-D maps, and a CUDA-core pass over the sink rows and the last L mod r
rows); the other forms gather into virtual heads and scatter back."""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from gpu_common import LSE_ABS, compare, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,L,d,w,s,r,dtype", [
    (1, 2, 700, 128, 256, 4, 2, torch.bfloat16),   # several tiles per virtual head, ragged classes
    (1, 2, 600, 128, 128, 16, 3, torch.bfloat16),
    (2, 1, 300, 128, 64, 0, 4, torch.bfloat16),    # no sinks: independent residue classes
    (1, 1, 1001, 128, 200, 4, 7, torch.bfloat16),  # L not a multiple of r
    (16, 2, 300, 128, 100, 4, 2, torch.bfloat16),  # 64 virtual heads
    (1, 1, 200, 128, 40, 32, 5, torch.bfloat16),   # many sinks
    (1, 1, 3, 128, 2, 1, 3, torch.bfloat16),       # fewer rows than r
    (1, 2, 263, 128, 300, 5, 2, torch.bfloat16),   # classes of 129 and 128 rows: one tile holds a phantom row only
    (1, 2, 700, 128, 300, 130, 2, torch.bfloat16), # more sinks than a key tile
    (1, 2, 1000, 128, 64, 4, 64, torch.bfloat16),  # r = 64: short classes, 40 rows past the last whole group
    (2, 3, 2000, 128, 1024, 4, 3, torch.bfloat16), # several query tiles per class, full windows
    (1, 2, 11, 128, 16, 8, 2, torch.bfloat16),     # one whole group after the sinks, then one row past it
    (1, 2, 300, 64, 100, 4, 3, torch.bfloat16),    # d = 64: the gathered form
    (1, 2, 130, 16, 16, 4, 3, torch.float32),      # the fp32 path
])
def test_dilated_prefill_every_row(B, H, L, d, w, s, r, dtype):
    swa = require_gpu()
    q, k, v = swa_inputs.prefill_inputs(B, H, L, d, 3000 + L + r, dtype, "cpu", sink_boost=True)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill_dilated(q.cuda(), k.cuda(), v.cuda(), w, s, r, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, l_ref = oracle.prefill_dilated(q, k, v, w, s, r, 1.0 / math.sqrt(d))
    compare(f"dilated {B, H, L, d, w, s, r}", o.cpu(), o_ref, dtype)
    assert np.abs(lse.cpu().double().numpy() - l_ref).max() < LSE_ABS


def test_dilation_one_is_the_plain_prefill_bit_for_bit():
    # r = 1 is the plain window: the call runs the plain prefill
    swa = require_gpu()
    q, k, v = (x.cuda() for x in swa_inputs.prefill_inputs(1, 4, 900, 128, 31, torch.bfloat16, "cpu", True))
    la = torch.empty((1, 4, 900), dtype=torch.float32, device="cuda")
    lb = torch.empty_like(la)
    a = swa.swa_sink_prefill_dilated(q, k, v, 300, 4, 1, lse=la)
    b = swa.swa_sink_prefill(q, k, v, 300, 4, lse=lb)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(la, lb)


@pytest.mark.parametrize("dtype,d,w,s,r", [
    (torch.bfloat16, 128, 40, 4, 3),
    (torch.bfloat16, 64, 24, 0, 2),
    (torch.bfloat16, 16, 17, 16, 4),
    (torch.float32, 16, 16, 4, 2),
    (torch.bfloat16, 128, 9, 1, 1),
])
def test_dilated_streaming_decode_every_step(dtype, d, w, s, r):
    # write, then attend, through the per-class caches; every step against the oracle's dilated key set
    swa = require_gpu()
    B, H = 2, 3
    T = 3 * w * r + 5
    q, k, v = swa_inputs.prefill_inputs(B, H, T, d, 400 + d + r, dtype, "cpu", sink_boost=True)
    kc = torch.zeros((r, B, H, w, d), dtype=dtype, device="cuda")
    vc = torch.zeros_like(kc)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    outs, lses = [], []
    for t in range(T):
        swa.swa_sink_dilated_cache_write(kc, vc, kg[:, :, t].contiguous(), vg[:, :, t].contiguous(), s, r, t)
        lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
        outs.append(swa.swa_sink_decode_step_dilated(qg[:, :, t].contiguous(), kc, vc, s, r, t, lse=lse).cpu())
        lses.append(lse.cpu())
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, l_ref = oracle.prefill_dilated(q, k, v, w, s, r, 1.0 / math.sqrt(d))
    for t in range(T):
        compare(f"dilated decode t={t}", outs[t], o_ref[:, :, t], dtype)
        assert np.abs(lses[t].double().numpy() - l_ref[:, :, t]).max() < LSE_ABS


@pytest.mark.parametrize("B,H,L,d,w,s,r,C,dtype", [
    (1, 2, 700, 128, 256, 4, 2, 128, torch.bfloat16),
    (2, 1, 600, 128, 100, 0, 3, 90, torch.bfloat16),
    (16, 1, 300, 128, 64, 4, 2, 64, torch.bfloat16),   # 32 virtual heads: two row groups
    (1, 2, 130, 16, 16, 4, 3, 20, torch.float32),
])
def test_chunked_dilated_prefill_rows_and_caches(B, H, L, d, w, s, r, C, dtype):
    # the rows equal the dilated definition, and the per-class caches end as L streaming writes leave them
    swa = require_gpu()
    q, k, v = swa_inputs.prefill_inputs(B, H, L, d, 5000 + L + r, dtype, "cpu", sink_boost=True)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    kc = torch.full((r, B, H, w, d), float("nan"), dtype=dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill_chunked_dilated(qg, kg, vg, s, r, C, kc, vc, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, l_ref = oracle.prefill_dilated(q, k, v, w, s, r, 1.0 / math.sqrt(d))
    compare(f"chunked dilated {B, H, L, w, s, r, C}", o.cpu(), o_ref, dtype)
    assert np.abs(lse.cpu().double().numpy() - l_ref).max() < LSE_ABS
    kc2 = torch.full_like(kc, float("nan"))
    vc2 = torch.full_like(vc, float("nan"))
    for t in range(L):
        swa.swa_sink_dilated_cache_write(kc2, vc2, kg[:, :, t].contiguous(), vg[:, :, t].contiguous(), s, r, t)
    iv = torch.int16 if dtype == torch.bfloat16 else torch.int32
    assert torch.equal(kc.view(iv), kc2.view(iv))
    assert torch.equal(vc.view(iv), vc2.view(iv))
