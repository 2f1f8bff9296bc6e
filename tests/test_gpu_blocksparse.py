"""GPU parity of the block-sparse prefill (BigBird-style union of window, sinks, global tokens and random key
blocks, causal; swa_sink_prefill_blocksparse) against the oracle's prefill_blocksparse, element by element."""
import math

import numpy as np
import pytest
import torch

import oracle
import swa_inputs
from gpu_common import LSE_ABS, compare, inputs, require_gpu

pytestmark = pytest.mark.gpu


def run(B, H, L, w, s, globals_, block, rand, seed, rows=None):
    swa = require_gpu()
    d = 128
    q, k, v = inputs(B, H, L, d, torch.bfloat16, seed, sink_boost=True)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    o = swa.swa_sink_prefill_blocksparse(q, k, v, w, s, globals_, block, rand, lse=lse)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    rd = swa_inputs.rand_blocks_dict(rand) if rand is not None else None
    o_ref, l_ref = oracle.prefill_blocksparse(q, k, v, w, s, 1.0 / math.sqrt(d), globals_, block, rd, rows=rows)
    sel = list(range(L)) if rows is None else rows
    compare(f"blocksparse L{L} w{w} s{s} g{len(globals_)} b{block}", o[:, :, sel], o_ref, torch.bfloat16)
    assert np.abs(lse[:, :, sel].cpu().double().numpy() - l_ref).max() < LSE_ABS
    return o


def test_hand_pattern():
    # the pattern of tests/golden/blocksparse_mask_L12_w3_s1_g5_b4.txt: global token 5, query block 2 -> key block 0
    rand = np.full((3, 1), -1, dtype=np.int32)
    rand[2, 0] = 0
    run(1, 2, 12, 3, 1, [5], 4, rand, 31)


@pytest.mark.parametrize("L,w,s,ng,block,r", [
    (300, 64, 4, 1, 16, 2),     # several tiles, ragged tail, small blocks
    (1000, 256, 4, 2, 64, 3),   # the BigBird shape at a small size
    (700, 40, 0, 0, 64, 2),     # no globals, no sinks
    (900, 300, 16, 1, 128, 1),  # tile-sized blocks
    (2600, 512, 4, 2, 64, 3),   # several query pairs per head, far rows
    (513, 129, 4, 0, 32, 0),    # no random blocks, no globals: the plain key set
])
def test_random_patterns(L, w, s, ng, block, r):
    globals_, rand = swa_inputs.bigbird_pattern(L, block, ng, r, seed=L + block)
    run(1, 2, L, w, s, globals_, block, rand if r else None, 100 + L)


def test_scattered_globals():
    # global tokens anywhere in the sequence (not only a leading block), some inside windows, one at the end
    L, w, s = 1200, 200, 4
    globals_ = [0, 7, 300, 301, 777, 1100, 1199]
    _, rand = swa_inputs.bigbird_pattern(L, 64, 0, 2, seed=5)
    run(2, 1, L, w, s, globals_, 64, rand, 71)


def test_all_global_is_causal_attention():
    swa = require_gpu()
    L, d = 260, 128
    q, k, v = inputs(1, 1, L, d, torch.bfloat16, 9)
    o = swa.swa_sink_prefill_blocksparse(q, k, v, 4, 1, list(range(L)), 64, None)
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    o_ref, _ = oracle.prefill(q, k, v, L, 0, 1.0 / math.sqrt(d))  # w >= L, s = 0: full causal attention
    compare("all global", o, o_ref, torch.bfloat16)


def test_full_size_bigbird_sampled_rows():
    # the benchmark's pattern (B=1, H=32, L=8192, w=1024, s=4, block 64, 2 global blocks, 3 random blocks per
    # query block) in the launch configuration the benchmark times, on rows around the global, window and
    # tile boundaries and the last rows
    wl = swa_inputs.WORKLOADS["prefill_llama7b_L8192_w1024_s4"]
    globals_, rand = swa_inputs.bigbird_pattern(wl.L, 64, 2, 3, seed=2024)
    rows = [0, 5, 127, 128, 129, 255, 256, 1023, 1024, 1025, 1151, 1152, 4095, 4096, 6000, 8190, 8191]
    run(wl.B, wl.H, wl.L, wl.w, wl.s, globals_, 64, rand, wl.seed, rows=rows)


def test_rejects_bad_patterns():
    swa = require_gpu()
    q = torch.zeros((1, 1, 100, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(swa.SwaError):
        swa.swa_sink_prefill_blocksparse(q, q, q, 16, 4, [5, 3], 16, None)  # not ascending
    with pytest.raises(swa.SwaError):
        swa.swa_sink_prefill_blocksparse(q, q, q, 16, 4, [100], 16, None)  # past L
    bad = np.full((7, 1), 9, dtype=np.int32)  # key block 9 does not exist (7 blocks of 16)
    with pytest.raises(swa.SwaError):
        swa.swa_sink_prefill_blocksparse(q, q, q, 16, 4, [], 16, bad)


def test_packed_tiles():
    # query pair 4 (rows 1024..1279, w = 64): query tile 0 takes key blocks 1, 3, 5, query tile 1 blocks 3, 9, 11
    # and 0 (with the sinks); the global tokens 200 and 330 sit in blocks 3 and 5.  Blocks 3 and 5 (both query
    # tiles) share one packed tile, each half with a global column, and so do blocks 9 and 11 (query tile 1)
    swa = require_gpu()
    L, w, s, block = 1300, 64, 4, 64
    rand = np.full(((L + block - 1) // block, 2), -1, dtype=np.int32)
    rand[16] = [1, 5]
    rand[17] = [3, -1]
    rand[18] = [3, 9]
    rand[19] = [11, 0]
    globals_ = [200, 330]
    packed = [(t[0], t[4], t[2]) for t in swa.prefill_blocksparse_plan(L, w, s, globals_, block, rand, 4) if t[4] >= 0]
    assert packed == [(192, 320, 3), (576, 704, 2)], packed
    run(1, 2, L, w, s, globals_, block, rand, 77)
