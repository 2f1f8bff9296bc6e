"""GPU parity of prefill and chunked prefill against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from gpu_common import LSE_ABS, compare, inputs, oracle_rows, require_gpu

pytestmark = pytest.mark.gpu


def run_and_check(B, H, L, d, w, s, dtype, seed, sink_boost=False):
    swa = require_gpu()
    q, k, v = inputs(B, H, L, d, dtype, seed, sink_boost)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill(q, k, v, w, s, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, l_ref = oracle.prefill(q, k, v, w, s, 1.0 / math.sqrt(d))
    compare(f"prefill B{B} H{H} L{L} d{d} w{w} s{s}", o, o_ref, dtype)
    assert np.abs(lse.cpu().double().numpy() - l_ref).max() < LSE_ABS
    return o


@pytest.mark.parametrize("name", ["prefill_tiny_f32_w16_s4", "prefill_tiny_f32_w16_s0", "prefill_tiny_f32_w64_s0"])
def test_tiny_fp32_workloads(name):
    wl = swa_inputs.WORKLOADS[name]
    swa = require_gpu()
    q, k, v = [x.cuda() for x in swa_inputs.workload_inputs(wl, "cpu")]
    o = swa.swa_sink_prefill(q, k, v, wl.w, wl.s)
    o_ref, _ = oracle.prefill(q, k, v, wl.w, wl.s, wl.scale)
    compare(name, o, o_ref, torch.float32)


@pytest.mark.parametrize("L,d,w,s", [(100, 16, 16, 4), (77, 64, 9, 2), (300, 128, 64, 4), (50, 32, 1, 0)])
def test_fp32_shapes(L, d, w, s):
    run_and_check(1, 2, L, d, w, s, torch.float32, 11 + L)


# bf16 tensor-core path: shapes spanning several 128-row tiles, ragged tails, w < 128, w > L,
# s = 0, s = 1, s >= 128, w = 1, and single-row problems.
BF16_SHAPES = [
    (1, 2, 700, 300, 4),
    (1, 1, 1000, 1024, 4),
    (2, 1, 513, 128, 0),
    (1, 2, 257, 64, 16),
    (1, 1, 384, 1, 0),
    (1, 1, 384, 2, 1),
    (1, 1, 130, 129, 4),
    (1, 1, 128, 128, 4),
    (1, 1, 1, 8, 4),
    (1, 3, 5, 3, 1),
    (1, 1, 2048, 1536, 4),
    (1, 1, 900, 300, 200),
    (1, 1, 9000, 7296, 4),   # the largest window the 64-entry key-tile list takes at s = 4
    (8, 300, 64, 16, 4),     # 2400 (b, h) rows of one short query pair: many rounds of the persistent grid
    (1, 1, 640, 256, 130),
    (1, 2, 600, 14, 4),      # band of 137 keys per query tile: a 9-key narrow tile (N = 16 product) after each full one
    (1, 1, 700, 300, 17),    # a sink tile of 17 keys: just past the narrow-tile limit, on the full-width path
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,H,L,w,s", BF16_SHAPES)
def test_bf16_tensor_core_prefill(B, H, L, w, s, d):
    run_and_check(B, H, L, d, w, s, torch.bfloat16, 1000 + L + w + s + d)


def test_bf16_sink_boost_stability():
    # keys at positions 0..3 x4 and a large query norm: large logits must not overflow the online softmax
    swa = require_gpu()
    B, H, L, d, w, s = 1, 2, 600, 128, 200, 4
    q, k, v = inputs(B, H, L, d, torch.bfloat16, 5, sink_boost=True)
    q = (q.float() * 6).to(torch.bfloat16)
    o = swa.swa_sink_prefill(q, k, v, w, s)
    o_ref, _ = oracle.prefill(q, k, v, w, s, 1.0 / math.sqrt(d))
    compare("sink boost", o, o_ref, torch.bfloat16)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
@pytest.mark.parametrize("L,w,s,pos0", [(300, 100, 4, 257), (200, 64, 0, 1000), (150, 300, 4, 2), (129, 40, 8, 64)])
def test_prefill_with_cache(dtype, d, L, w, s, pos0):
    # rows pos0..pos0+L-1 against the rolling cache of positions < pos0 plus their own keys
    swa = require_gpu()
    B, H = 1, 2
    q, k, v = inputs(B, H, pos0 + L, d, dtype, 40 + pos0, sink_boost=True)
    kc = torch.full((B, H, w, d), float("nan"), dtype=dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    swa.kv_rolling_write(kc, vc, k[:, :, :pos0].contiguous(), v[:, :, :pos0].contiguous(), w, s, 0)
    qc, kk, vv = (x[:, :, pos0:].contiguous() for x in (q, k, v))
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill(qc, kk, vv, w, s, lse=lse, k_cache=kc, v_cache=vc, pos0=pos0)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, l_ref = oracle.prefill(q, k, v, w, s, 1.0 / math.sqrt(d))
    compare("cached prefill", o, o_ref[:, :, pos0:], dtype)
    assert np.abs(lse.cpu().double().numpy() - l_ref[:, :, pos0:]).max() < LSE_ABS


@pytest.mark.parametrize("L,w,s,chunk,H", [(1000, 300, 4, 256, 2), (1000, 300, 4, 300, 2), (777, 64, 4, 100, 2),
                                           (640, 128, 0, 128, 2), (500, 200, 4, 1000, 2), (1024, 512, 4, 96, 2),
                                           # sink rescales make softmax warps drift a tile apart: a race here
                                           # once mixed P-ready arrivals of two tiles on one barrier
                                           (8192, 1024, 4, 1024, 4), (6144, 2048, 4, 2048, 2),
                                           # 17 (b, h) rows: split into two uneven row groups that walk the
                                           # chunks on separate streams
                                           (700, 256, 4, 200, 17)])
def test_chunked_prefill(L, w, s, chunk, H):
    swa = require_gpu()
    B, d = 1, 128
    q, k, v = inputs(B, H, L, d, torch.bfloat16, 60 + chunk, sink_boost=True)
    # the scratch cache starts as NaN: slots not yet written must never reach the result
    kc = torch.full((B, H, w, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill_chunked(q, k, v, w, s, chunk, kc, vc, lse=lse)
    o_full = swa.swa_sink_prefill(q, k, v, w, s)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, l_ref = oracle.prefill(q, k, v, w, s, 1.0 / math.sqrt(d))
    compare("chunked", o, o_ref, torch.bfloat16)
    assert np.abs(lse.cpu().double().numpy() - l_ref).max() < LSE_ABS
    # chunked equals un-chunked (both against the oracle, and to each other within bf16 rounding)
    assert (o.float() - o_full.float()).abs().max().item() <= 2e-2
    # the cache left behind is the state after position L-1
    holder = torch.as_tensor(oracle.cache_replay(w, s, L))
    held = holder >= 0
    assert torch.equal(kc.cpu()[:, :, held], k.cpu()[:, :, holder[held]])
    assert torch.equal(vc.cpu()[:, :, held], v.cpu()[:, :, holder[held]])


@pytest.mark.parametrize("L,w,s,chunk,H", [(1000, 300, 4, 256, 2), (2048, 1024, 4, 512, 17)])
def test_chunked_prefill_d64(L, w, s, chunk, H):
    swa = require_gpu()
    B, d = 1, 64
    q, k, v = inputs(B, H, L, d, torch.bfloat16, 90 + chunk, sink_boost=True)
    kc = torch.full((B, H, w, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill_chunked(q, k, v, w, s, chunk, kc, vc, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, l_ref = oracle.prefill(q, k, v, w, s, 1.0 / math.sqrt(d))
    compare("chunked d64", o, o_ref, torch.bfloat16)
    assert np.abs(lse.cpu().double().numpy() - l_ref).max() < LSE_ABS
    holder = torch.as_tensor(oracle.cache_replay(w, s, L))
    held = holder >= 0
    assert torch.equal(kc.cpu()[:, :, held], k.cpu()[:, :, holder[held]])


def test_chunked_prefill_fp32():
    swa = require_gpu()
    B, H, L, d, w, s = 1, 1, 200, 16, 16, 4
    q, k, v = inputs(B, H, L, d, torch.float32, 3)
    kc = torch.full((B, H, w, d), float("nan"), device="cuda")
    vc = torch.full_like(kc, float("nan"))
    o = swa.swa_sink_prefill_chunked(q, k, v, w, s, 37, kc, vc)
    o_ref, _ = oracle.prefill(q, k, v, w, s, 0.25)
    compare("chunked fp32", o, o_ref, torch.float32)


def test_prefill_from_host_buffers():
    # the host-buffer entry point (copies pipelined over row groups) gives exactly the device-buffer
    # result, row group by row group, including a ragged last tile and lse
    swa = require_gpu()
    B, H, L, d, w, s = 1, 13, 1000, 128, 256, 4
    q, k, v = inputs(B, H, L, d, torch.bfloat16, 777, sink_boost=True)
    lse_ref = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    o_ref = swa.swa_sink_prefill(q, k, v, w, s, lse=lse_ref)
    qh, kh, vh = (x.cpu().pin_memory() for x in (q, k, v))
    qd, kd, vd = (torch.full_like(x, float("nan")) for x in (q, k, v))
    od = torch.empty_like(q)
    lse_d = torch.empty_like(lse_ref)
    lse_h = torch.empty((B, H, L), dtype=torch.float32).pin_memory()
    o_h = swa.swa_sink_prefill_host(qh, kh, vh, w, s, qd, kd, vd, od, lse_h=lse_h, lse_d=lse_d)
    torch.cuda.synchronize()
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    assert torch.equal(o_h, o_ref.cpu())
    assert torch.equal(lse_h, lse_ref.cpu())
    o_or, _ = oracle.prefill(q, k, v, w, s, 1.0 / math.sqrt(d))
    compare("host-buffer prefill", o_h, o_or, torch.bfloat16)


def test_multi_stream_calls_capture_into_a_cuda_graph():
    # the chunked and the host-buffer prefill fork work onto library streams and join it back with
    # events; both must capture into a CUDA graph and replay to the same result as a direct call
    swa = require_gpu()
    B, H, L, d, w, s, chunk = 1, 17, 600, 128, 256, 4, 200
    q, k, v = inputs(B, H, L, d, torch.bfloat16, 4321, sink_boost=True)
    kc = torch.zeros((B, H, w, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    o_direct = swa.swa_sink_prefill_chunked(q, k, v, w, s, chunk, kc, vc)
    qh, kh, vh = (x.cpu().pin_memory() for x in (q, k, v))
    qd, kd, vd, od = (torch.empty_like(x) for x in (q, k, v, q))
    oh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    o_g = torch.empty_like(q)
    kc2, vc2 = torch.zeros_like(kc), torch.zeros_like(vc)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        swa.swa_sink_prefill_chunked(q, k, v, w, s, chunk, kc2, vc2, o=o_g)
        swa.swa_sink_prefill_host(qh, kh, vh, w, s, qd, kd, vd, od, o_h=oh)
    for _ in range(2):
        o_g.fill_(float("nan"))
        oh.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
        assert torch.equal(o_g, o_direct)
        assert torch.equal(kc2, kc) and torch.equal(vc2, vc)
        assert torch.equal(oh, swa.swa_sink_prefill(q, k, v, w, s).cpu())
