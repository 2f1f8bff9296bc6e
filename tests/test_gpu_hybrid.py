"""GPU parity of the SWA + linear-attention hybrid (swa_hybrid_prefill, swa_hybrid_decode_step) against the
oracle's hybrid_linear / hybrid_linear_rows, element by element, with the sink keys scaled x4."""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from gpu_common import compare, inputs, require_gpu

pytestmark = pytest.mark.gpu
D = 128


def flat(x):
    B, H, L, d = x.shape
    return x.reshape(B * H, L, d)


def wf_for(seed):
    return swa_inputs.hedgehog_weights(D, seed)


@pytest.mark.parametrize("B,H,L,w,s", [
    (1, 2, 600, 128, 4),    # several chunks, ragged tail
    (1, 1, 1000, 200, 0),   # no sinks
    (2, 1, 777, 300, 16),   # m = 284: intra keys across two chunks
    (1, 2, 100, 128, 4),    # L < m: no key leaves the window
    (1, 1, 1300, 129, 4),   # m = 125
    (1, 1, 260, 2, 1),      # a one-key window
])
def test_prefill_parity(B, H, L, w, s):
    swa = require_gpu()
    q, k, v = inputs(B, H, L, D, torch.bfloat16, 300 + L + w, sink_boost=True)
    wf = wf_for(L)
    o = swa.swa_hybrid_prefill(q, k, v, wf.cuda(), w, s)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    ref = oracle.hybrid_linear(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w, s, 1 / math.sqrt(D), wf.double().numpy())
    compare(f"hybrid prefill L{L} w{w} s{s}", flat(o), ref, torch.bfloat16)


def test_prefill_without_evictions_is_the_plain_prefill():
    swa = require_gpu()
    q, k, v = inputs(1, 2, 300, D, torch.bfloat16, 5, sink_boost=True)
    o = swa.swa_hybrid_prefill(q, k, v, wf_for(1).cuda(), 400, 4)
    ref = swa.swa_sink_prefill(q, k, v, 400, 4)
    assert torch.equal(o, ref)


def test_prefill_final_state():
    swa = require_gpu()
    B, H, L, w, s = 1, 2, 900, 160, 4
    q, k, v = inputs(B, H, L, D, torch.bfloat16, 17, sink_boost=True)
    wf = wf_for(2)
    S = torch.empty((B, H, D, D), dtype=torch.float32, device="cuda")
    z = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
    swa.swa_hybrid_prefill(q, k, v, wf.cuda(), w, s, state_s=S, state_z=z)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    m = w - s
    pk = oracle.hedgehog(flat(k).cpu().double().numpy()[:, s:L - m], wf.double().numpy())
    S_ref = np.matmul(pk.transpose(0, 2, 1), flat(v).cpu().double().numpy()[:, s:L - m])
    z_ref = pk.sum(axis=1)
    S_got = S.reshape(B * H, D, D).cpu().double().numpy()
    z_got = z.reshape(B * H, D).cpu().double().numpy()
    # phi(k) enters the product as bf16 (relative 2^-9 per term); z is summed in fp32
    assert np.abs(S_got - S_ref).max() <= 1e-2 * np.abs(S_ref).max()
    assert np.abs(z_got - z_ref).max() <= 1e-5 * np.abs(z_ref).max()


def test_decode_stepwise_from_position_zero():
    swa = require_gpu()
    B, H, L, w, s = 2, 2, 300, 64, 4
    q, k, v = inputs(B, H, L, D, torch.bfloat16, 23, sink_boost=True)
    wf = wf_for(3)
    kc = torch.zeros((B, H, w, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    S = torch.zeros((B, H, D, D), dtype=torch.float32, device="cuda")
    z = torch.zeros((B, H, D), dtype=torch.float32, device="cuda")
    wfc = wf.cuda()
    outs = []
    for t in range(L):
        o = swa.swa_hybrid_decode_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(),
                                       kc, vc, S, z, wfc, w, s, t)
        outs.append(o.clone())
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    got = torch.stack(outs, dim=2)
    ref = oracle.hybrid_linear(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w, s, 1 / math.sqrt(D), wf.double().numpy())
    compare("hybrid decode", flat(got), ref, torch.bfloat16)


def test_prefill_then_decode():
    swa = require_gpu()
    B, H, L0, n, w, s = 1, 2, 500, 40, 96, 4
    L = L0 + n
    q, k, v = inputs(B, H, L, D, torch.bfloat16, 29, sink_boost=True)
    wf = wf_for(4)
    wfc = wf.cuda()
    S = torch.empty((B, H, D, D), dtype=torch.float32, device="cuda")
    z = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
    o0 = swa.swa_hybrid_prefill(q[:, :, :L0].contiguous(), k[:, :, :L0].contiguous(), v[:, :, :L0].contiguous(),
                                wfc, w, s, state_s=S, state_z=z)
    kc = torch.zeros((B, H, w, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    swa.kv_rolling_write(kc, vc, k[:, :, :L0].contiguous(), v[:, :, :L0].contiguous(), w, s, 0)
    outs = []
    for t in range(L0, L):
        outs.append(swa.swa_hybrid_decode_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(),
                                               v[:, :, t].contiguous(), kc, vc, S, z, wfc, w, s, t).clone())
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    ref = oracle.hybrid_linear(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), w, s, 1 / math.sqrt(D), wf.double().numpy())
    compare("hybrid prefill part", flat(o0), ref[:, :L0], torch.bfloat16)
    compare("hybrid decode after prefill", flat(torch.stack(outs, dim=2)), ref[:, L0:], torch.bfloat16)


def test_full_size_sampled_rows():
    # the benchmark's shape (B=1, H=32, L=8192, w=1024, s=4) in the launch configuration the benchmark times,
    # on rows around the first eviction, the chunk and tile boundaries and the last rows
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS["prefill_llama7b_L8192_w1024_s4"]
    q, k, v = inputs(wl.B, wl.H, wl.L, wl.d, torch.bfloat16, wl.seed, sink_boost=True)
    wf = wf_for(8192)
    o = swa.swa_hybrid_prefill(q, k, v, wf.cuda(), wl.w, wl.s)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    rows = [0, 1023, 1024, 1025, 1100, 1151, 1152, 1279, 1280, 2047, 2048, 4095, 5000, 8064, 8190, 8191]
    ref = oracle.hybrid_linear_rows(flat(q).cpu(), flat(k).cpu(), flat(v).cpu(), wl.w, wl.s, wl.scale,
                                    wf.double().numpy(), rows)
    compare("hybrid full size", flat(o)[:, rows], ref, torch.bfloat16)


def test_rejects_bad_arguments():
    swa = require_gpu()
    q = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    wf = torch.zeros((64, 32), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(swa.SwaError):
        swa.swa_hybrid_prefill(q, q, q, wf, 16, 4)  # d = 64
    q = torch.zeros((1, 1, 64, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(swa.SwaError):
        swa.swa_hybrid_prefill(q, q, q, wf_for(1).cuda(), 16, 16)  # s >= w
