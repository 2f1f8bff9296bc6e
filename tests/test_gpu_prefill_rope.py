"""GPU parity of the prefill with RoPE at the positions inside the cache (swa_sink_prefill_rope) against
the oracle's definition (row t = the streaming decode at step t over unrotated keys), element by element.

The rotation pass writes the rotated q and k as bf16 (hi, lo) pairs, from which the kernel forms each window
score with three tensor-core products (hi hi + hi lo + lo hi), and the sink scores (the query rotated at
min(t, w - 1)) as fp32 dot products; so every score carries the error of fp32 operands and the results meet the
same tolerances as every other path (gpu_common.check_rope_prefill): the rotated operands and sink scores
against the oracle's fp64 rotation, and the output and log-sum-exp against the oracle's exact definition.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from gpu_common import check_rope_prefill, compare, require_gpu, rope_workspace_operands

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,L,w,s,base", [
    (1, 2, 700, 256, 4, 1e4),     # several key tiles, rows far past the window, a ragged tail
    (1, 2, 600, 128, 16, 1e4),
    (2, 1, 300, 64, 0, 1e4),      # no sinks: plain RoPE over the band
    (1, 1, 520, 520, 4, 1e4),     # w = L: nothing is evicted
    (1, 1, 1000, 300, 100, 5e5),  # many sinks, another base
    (1, 2, 257, 40, 4, 1e4),      # one row past a query pair
    (1, 1, 3, 2, 1, 1e4),         # fewer rows than sinks + 1
])
def test_rope_prefill_every_row(B, H, L, w, s, base):
    swa = require_gpu()
    d = 128
    q, k, v = swa_inputs.prefill_inputs(B, H, L, d, 900 + L + s, torch.bfloat16, "cpu", sink_boost=True)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    ws = torch.empty(swa.lib().swa_sink_prefill_rope_workspace_size(B, H, L, d, s), dtype=torch.uint8, device="cuda")
    o = swa.swa_sink_prefill_rope(q.cuda(), k.cuda(), v.cuda(), w, s, rope_base=base, lse=lse, workspace=ws)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.prefill_rope(q, k, v, w, s, scale, base)
    nh = B * H
    rows = list(range(L))
    qf, kf, vf = (x.double().numpy().reshape(nh, L, d) for x in (q, k, v))
    check_rope_prefill(f"rope prefill {B, H, L, w, s}", o.cpu().double().numpy().reshape(nh, L, d),
                       lse.cpu().double().numpy().reshape(nh, L), rope_workspace_operands(ws, B, H, L, d, s, rows),
                       qf, kf, vf, rows, w, s, scale, base, o_ref.reshape(nh, L, d), l_ref.reshape(nh, L))


def test_rope_prefill_row_equals_rope_decode_step():
    # the same unrotated keys through the decode path: row t of the prefill is step t of the stream
    swa = require_gpu()
    B, H, L, d, w, s = 1, 2, 400, 128, 96, 4
    q, k, v = (x.cuda() for x in swa_inputs.prefill_inputs(B, H, L, d, 77, torch.bfloat16, "cpu", True))
    o = swa.swa_sink_prefill_rope(q, k, v, w, s)
    kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    for t in range(L):
        swa.kv_rolling_write(kc, vc, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), w, s, t)
        if t in (0, 50, 95, 96, 97, 200, 399):
            od = swa.swa_sink_decode_step_rope(q[:, :, t].contiguous(), kc, vc, t, w, s)
            # both paths form fp32-accurate scores: they agree within the bf16 output tolerance
            compare(f"prefill row {t} vs decode", o[:, :, t].float().cpu().numpy().astype(np.float64),
                    od.float().cpu().numpy().astype(np.float64), torch.bfloat16)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()


def test_rope_prefill_workspace_is_checked():
    swa = require_gpu()
    q = torch.zeros((1, 1, 300, 128), dtype=torch.bfloat16, device="cuda")
    need = swa.lib().swa_sink_prefill_rope_workspace_size(1, 1, 300, 128, 4)
    assert need == 4 * 300 * 128 * 2 + 300 * 4 * 4 + 4 * 128 * 4
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(swa.SwaError):
        swa.swa_sink_prefill_rope(q, q, q, 64, 4, workspace=ws)


@pytest.mark.parametrize("B,H,L,w,s,C", [
    (1, 2, 700, 256, 4, 128),
    (1, 2, 600, 128, 16, 200),
    (2, 1, 300, 64, 0, 50),      # no sinks
    (1, 1, 1000, 300, 100, 256),  # many sinks, chunk >= s
    (1, 2, 3000, 512, 4, 256),   # 12 chunks: the ring wraps several times
    (16, 2, 300, 100, 4, 64),    # 32 (b, h) rows: two row groups on two streams
])
def test_rope_chunked_prefill_every_row(B, H, L, w, s, C):
    # chunked prefill with RoPE equals the whole-sequence definition (the oracle's prefill_rope), and
    # leaves the caller's caches as a plain rolling write of all positions does (unrotated keys)
    swa = require_gpu()
    d = 128
    q, k, v = swa_inputs.prefill_inputs(B, H, L, d, 1300 + L + s, torch.bfloat16, "cpu", sink_boost=True)
    kc = torch.full((B, H, w, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    ws = torch.empty(swa.lib().swa_sink_prefill_chunked_rope_workspace_size(B, H, L, d, w, s), dtype=torch.uint8,
                     device="cuda")
    o = swa.swa_sink_prefill_chunked_rope(q.cuda(), k.cuda(), v.cuda(), w, s, C, kc, vc, lse=lse, workspace=ws)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.prefill_rope(q, k, v, w, s, scale)
    nh = B * H
    rows = list(range(L))
    qf, kf, vf = (x.double().numpy().reshape(nh, L, d) for x in (q, k, v))
    check_rope_prefill(f"rope chunked {B, H, L, w, s, C}", o.cpu().double().numpy().reshape(nh, L, d),
                       lse.cpu().double().numpy().reshape(nh, L), rope_workspace_operands(ws, B, H, L, d, s, rows),
                       qf, kf, vf, rows, w, s, scale, 10000.0, o_ref.reshape(nh, L, d), l_ref.reshape(nh, L))
    kc2 = torch.full_like(kc, float("nan"))
    vc2 = torch.full_like(vc, float("nan"))
    swa.kv_rolling_write(kc2, vc2, k.cuda(), v.cuda(), w, s, 0)
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc2.view(torch.int16))


def test_rope_chunked_prefill_rejects_chunks_shorter_than_the_sinks():
    swa = require_gpu()
    q = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(swa.SwaError):
        swa.swa_sink_prefill_chunked_rope(q, q, q, 32, 8, 4, kc, kc.clone())
