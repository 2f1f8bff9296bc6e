"""Parity at the full workload sizes, in the launch configuration the benchmark times (the RoPE forms on
sampled rows): the primary prefill in full; for the two B=2 L=32768 prefills every row of four heads and every row with t < w + 128
in every head; for the chunked prefill every row of chunks 0, 1, 2 and 31 and the rows around every chunk
boundary in every head; for decode every step of 8 (b, h) rows."""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from gpu_common import LSE_ABS, check_rope_prefill, compare, oracle_rows, require_gpu, rope_workspace_operands

pytestmark = pytest.mark.gpu


def check_samples(name, o, lse, q, k, v, wl, heads, blocks):
    B, H, L, d = q.shape
    ref = oracle_rows(q, k, v, heads, blocks, wl.w, wl.s, wl.scale)
    of = o.reshape(B * H, L, d)
    lf = lse.reshape(B * H, L)
    for (bh, r0), (o_ref, l_ref) in ref.items():
        r1 = r0 + o_ref.shape[0]
        compare(f"{name} bh={bh} rows {r0}..{r1 - 1}", of[bh, r0:r1], o_ref, torch.bfloat16)
        assert np.abs(lf[bh, r0:r1].cpu().double().numpy() - l_ref).max() < LSE_ABS


def _full_size_prefill_outputs(swa, wl):
    q, k, v = swa_inputs.workload_inputs(wl, "cuda")
    lse = torch.empty((wl.B, wl.H, wl.L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill(q, k, v, wl.w, wl.s, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    assert torch.isfinite(o).all()
    return q, k, v, o, lse


def test_full_size_prefill_llama7b_every_row():
    # the primary workload in full: every row of every head against the oracle
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS["prefill_llama7b_L8192_w1024_s4"]
    q, k, v, o, lse = _full_size_prefill_outputs(swa, wl)
    check_samples(wl.name, o, lse, q, k, v, wl, list(range(wl.B * wl.H)), [(0, wl.L)])


@pytest.mark.parametrize("name", ["prefill_mistral_B2_L32768_w4096_s0", "prefill_mistral_B2_L32768_w4096_s4"])
def test_full_size_prefill_mistral(name):
    # every row of four heads (both batch entries), and in every head every row with t < w + 128 (the
    # rows whose key set is still growing, plus the first full-window tile)
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS[name]
    q, k, v, o, lse = _full_size_prefill_outputs(swa, wl)
    check_samples(name, o, lse, q, k, v, wl, [0, 21, 42, 63], [(0, wl.L)])
    others = [bh for bh in range(wl.B * wl.H) if bh not in (0, 21, 42, 63)]
    check_samples(name, o, lse, q, k, v, wl, others, [(0, wl.w + 128)])


def test_full_size_chunked_prefill():
    # every row of chunks 0, 1, 2 and 31 in every head, and the rows around every chunk boundary
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS["chunked_mistral_L131072_w4096_s4_C4096"]
    q, k, v = swa_inputs.workload_inputs(wl, "cuda")
    kc = torch.full((wl.B, wl.H, wl.w, wl.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    lse = torch.empty((wl.B, wl.H, wl.L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill_chunked(q, k, v, wl.w, wl.s, wl.chunk, kc, vc, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    assert torch.isfinite(o).all()
    C = wl.chunk
    nch = wl.L // C
    blocks = [(0, 3 * C), ((nch - 1) * C, nch * C)] + [(c * C - 4, c * C + 4) for c in range(3, nch - 1)]
    check_samples("chunked", o, lse, q, k, v, wl, list(range(wl.B * wl.H)), blocks)


def test_full_size_streaming_decode():
    # 20480 steps of write + decode at B=64, H=40, 4 sink + 1020 recent slots; 8 (b, h) pairs are checked
    # against the oracle's history definition at every step
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS["decode_llama13b_B64_w1024_s4_20480"]
    B, H, d, w, s, T = wl.B, wl.H, wl.d, wl.w, wl.s, wl.L
    qs = swa_inputs.normal((T, B, H, d), wl.seed, swa_inputs.TID_Q, torch.bfloat16, "cuda")
    ks = swa_inputs.normal((T, B, H, d), wl.seed, swa_inputs.TID_K, torch.bfloat16, "cuda")
    vs = swa_inputs.normal((T, B, H, d), wl.seed, swa_inputs.TID_V, torch.bfloat16, "cuda")
    ks[:4] *= 4.0
    kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pairs = torch.tensor([0, 1, 39, 40, 777, 1300, 2000, B * H - 1], device="cuda")
    outs = torch.empty((T, len(pairs), d), dtype=torch.bfloat16, device="cuda")
    lses = torch.empty((T, len(pairs)), dtype=torch.float32, device="cuda")
    o = torch.empty((B, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    for t in range(T):
        swa.kv_rolling_write(kc, vc, ks[t].unsqueeze(2), vs[t].unsqueeze(2), w, s, t)
        swa.swa_sink_decode_step(qs[t], kc, vc, t, w, s, o=o, lse=lse)
        outs[t] = o.reshape(B * H, d).index_select(0, pairs)
        lses[t] = lse.reshape(B * H).index_select(0, pairs)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    pos = np.arange(T)
    for j, bh in enumerate(pairs.tolist()):
        b, h = divmod(bh, H)
        qh, kh, vh = (x[:, b, h].float().cpu().numpy()[None] for x in (qs, ks, vs))
        o_ref, l_ref = oracle.attend(qh, pos, kh, vh, pos, w, s, wl.scale)
        compare(f"decode bh={bh}", outs[:, j], o_ref[0], torch.bfloat16)
        assert np.abs(lses[:, j].cpu().double().numpy() - l_ref[0]).max() < LSE_ABS


def test_full_size_streaming_decode_rope():
    # the same 20480-step stream with RoPE at the positions inside the cache; 8 (b, h) rows are checked
    # against the oracle's history definition at sampled steps (window filling, first wraps, deep in)
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS["decode_llama13b_B64_w1024_s4_20480"]
    B, H, d, w, s, T = wl.B, wl.H, wl.d, wl.w, wl.s, wl.L
    qs = swa_inputs.normal((T, B, H, d), wl.seed, swa_inputs.TID_Q, torch.bfloat16, "cuda")
    ks = swa_inputs.normal((T, B, H, d), wl.seed, swa_inputs.TID_K, torch.bfloat16, "cuda")
    vs = swa_inputs.normal((T, B, H, d), wl.seed, swa_inputs.TID_V, torch.bfloat16, "cuda")
    ks[:4] *= 4.0
    kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pairs = torch.tensor([0, 1, 39, 40, 777, 1300, 2000, B * H - 1], device="cuda")
    steps = sorted({0, 1, 3, 4, 5, 100, 1019, 1022, 1023, 1024, 1025, 1026, 2045, 2046, 2047, 3070, 4099, 7777,
                    10000, 15000, T - 2, T - 1} | set(range(997, T, 997)))
    outs = torch.empty((len(steps), len(pairs), d), dtype=torch.bfloat16, device="cuda")
    lses = torch.empty((len(steps), len(pairs)), dtype=torch.float32, device="cuda")
    o = torch.empty((B, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(swa.lib().swa_sink_decode_rope_workspace_size(B, H, d, w), dtype=torch.uint8, device="cuda")
    k_at = {t: i for i, t in enumerate(steps)}
    for t in range(T):
        swa.kv_rolling_write(kc, vc, ks[t].unsqueeze(2), vs[t].unsqueeze(2), w, s, t)
        swa.swa_sink_decode_step_rope(qs[t], kc, vc, t, w, s, o=o, lse=lse, workspace=ws)
        if t in k_at:
            outs[k_at[t]] = o.reshape(B * H, d).index_select(0, pairs)
            lses[k_at[t]] = lse.reshape(B * H).index_select(0, pairs)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    for j, bh in enumerate(pairs.tolist()):
        b, h = divmod(bh, H)
        qh, kh, vh = (x[:, b, h].float().cpu().numpy() for x in (qs, ks, vs))
        for i, t in enumerate(steps):
            o_ref, l_ref = oracle.decode_rope(qh[t][None], kh[None, :t + 1], vh[None, :t + 1], t, w, s, wl.scale)
            compare(f"rope decode bh={bh} t={t}", outs[i, j][None], o_ref, torch.bfloat16)
            assert abs(float(lses[i, j]) - l_ref[0]) < LSE_ABS


def test_full_size_prefill_rope_sampled_rows():
    # the primary shape with RoPE at the positions inside the cache: every head at rows around the tile,
    # pair and window boundaries, the last rows and a few random ones, against the oracle's definition;
    # checked as in tests/test_gpu_prefill_rope.py (rotated operands, then the exact definition)
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS["prefill_llama7b_L8192_w1024_s4"]
    q, k, v = swa_inputs.workload_inputs(wl, "cuda")
    lse = torch.empty((wl.B, wl.H, wl.L), dtype=torch.float32, device="cuda")
    ws = torch.empty(swa.lib().swa_sink_prefill_rope_workspace_size(wl.B, wl.H, wl.L, wl.d, wl.s), dtype=torch.uint8,
                     device="cuda")
    o = swa.swa_sink_prefill_rope(q, k, v, wl.w, wl.s, lse=lse, workspace=ws)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    rng = np.random.default_rng(5)
    rows = sorted({0, 1, 3, 4, 127, 128, 255, 256, 1022, 1023, 1024, 1025, 1026, 1279, 1280, 2047, 2048, 4095,
                   4096, 8190, 8191} | set(int(x) for x in rng.integers(0, wl.L, 12)))
    qc, kc_, vc_ = q.cpu(), k.cpu(), v.cpu()
    o_ref, l_ref = oracle.prefill_rope(qc, kc_, vc_, wl.w, wl.s, wl.scale, rows=rows)
    nh, d = wl.B * wl.H, wl.d
    qf, kf, vf = (x.double().numpy().reshape(nh, wl.L, d) for x in (qc, kc_, vc_))
    check_rope_prefill("rope prefill llama7b sampled rows",
                       o[:, :, rows].reshape(nh, len(rows), d).cpu().double().numpy(),
                       lse[:, :, rows].reshape(nh, len(rows)).cpu().double().numpy(),
                       rope_workspace_operands(ws, wl.B, wl.H, wl.L, d, wl.s, rows), qf, kf, vf, rows, wl.w, wl.s,
                       wl.scale, 10000.0, o_ref.reshape(nh, len(rows), d), l_ref.reshape(nh, len(rows)))


def test_full_size_chunked_prefill_rope_sampled_rows():
    # the chunked workload (L = 131072 in 4096-token chunks, w = 4096, s = 4) with RoPE at the positions
    # inside the cache, in the launch configuration the benchmark times: every head at rows of the first
    # three chunks around the chunk boundaries (the ring has wrapped by the third) and random rows there
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS["chunked_mistral_L131072_w4096_s4_C4096"]
    q, k, v = swa_inputs.workload_inputs(wl, "cuda")
    kc = torch.zeros((wl.B, wl.H, wl.w, wl.d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    lse = torch.empty((wl.B, wl.H, wl.L), dtype=torch.float32, device="cuda")
    ws = torch.empty(swa.lib().swa_sink_prefill_chunked_rope_workspace_size(wl.B, wl.H, wl.L, wl.d, wl.w, wl.s),
                     dtype=torch.uint8, device="cuda")
    o = swa.swa_sink_prefill_chunked_rope(q, k, v, wl.w, wl.s, wl.chunk, kc, vc, lse=lse, workspace=ws)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    rng = np.random.default_rng(6)
    C = wl.chunk
    rows = sorted({0, 3, 4, C - 1, C, C + 1, 2 * C - 1, 2 * C, 2 * C + 1, 3 * C - 1}
                  | set(int(x) for x in rng.integers(0, 3 * C, 6)))
    top = max(rows) + 1
    qc, kc_, vc_ = (x[:, :, :top].cpu() for x in (q, k, v))
    o_ref, l_ref = oracle.prefill_rope(qc, kc_, vc_, wl.w, wl.s, wl.scale, rows=rows)
    nh, d = wl.B * wl.H, wl.d
    qf, kf, vf = (x.double().numpy().reshape(nh, top, d) for x in (qc, kc_, vc_))
    ops = rope_workspace_operands(ws, wl.B, wl.H, wl.L, d, wl.s, rows)
    check_rope_prefill("rope chunked L131072 sampled rows",
                       o[:, :, rows].reshape(nh, len(rows), d).cpu().double().numpy(),
                       lse[:, :, rows].reshape(nh, len(rows)).cpu().double().numpy(), ops, qf, kf, vf, rows, wl.w,
                       wl.s, wl.scale, 10000.0, o_ref.reshape(nh, len(rows), d), l_ref.reshape(nh, len(rows)))


def test_full_size_prefill_dilated_sampled_rows():
    # the primary shape with dilation 2 (window reaching 2 * 1019 + 1 positions back), in the launch
    # configuration the benchmark times: every head at rows around the window, tile and class boundaries
    swa = require_gpu()
    wl = swa_inputs.WORKLOADS["prefill_llama7b_L8192_w1024_s4"]
    r = 2
    q, k, v = swa_inputs.workload_inputs(wl, "cuda")
    lse = torch.empty((wl.B, wl.H, wl.L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill_dilated(q, k, v, wl.w, wl.s, r, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    rng = np.random.default_rng(7)
    rows = sorted({0, 1, 3, 4, 5, 255, 256, 1023, 2041, 2042, 2043, 2044, 2045, 4096, 4097, 8190, 8191}
                  | set(int(x) for x in rng.integers(0, wl.L, 10)))
    o_ref, l_ref = oracle.prefill_dilated(q.cpu(), k.cpu(), v.cpu(), wl.w, wl.s, r, wl.scale, rows=rows)
    nh, d = wl.B * wl.H, wl.d
    compare("dilated llama7b sampled rows", o[:, :, rows].reshape(nh, len(rows), d), o_ref.reshape(nh, len(rows), d),
            torch.bfloat16)
    assert np.abs(lse[:, :, rows].cpu().double().numpy() - l_ref).max() < LSE_ABS
