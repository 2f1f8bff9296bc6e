"""The C-ABI library: builds, loads without a GPU, exports every symbol include/swa_sink.h declares, and
rejects bad arguments before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import sliding_window_softmax_swa_gb300 as swa
from sliding_window_softmax_swa_gb300 import build as swa_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "swa_sink.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    swa_build.build()
    return swa.lib()


def test_header_declares_the_three_path_calls():
    names = declared_functions()
    for n in ("swa_sink_prefill", "swa_sink_decode_step", "kv_rolling_write"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(swa.SIGNATURES), "binding signatures out of sync with the header"


def test_library_has_no_dynamic_cuda_dependency():
    # the runtime is linked statically, so the library loads on a host without a GPU driver
    ctypes.CDLL(swa_build.LIB)
    needed = os.popen(f"readelf -d {swa_build.LIB}").read()
    assert "libcudart" not in needed and "libcuda.so" not in needed


@pytest.mark.parametrize("args,msg", [
    (dict(w=4, s=4), "s < w"),
    (dict(w=0, s=0), "w="),
    (dict(d=96), "d=96"),
    (dict(B=0), "B=0"),
    (dict(dtype=7), "dtype"),
    (dict(L=-1), "L=-1"),
    (dict(scale=0.0), "scale"),
    (dict(pos0=-3), "pos0"),
])
def test_prefill_rejects_bad_arguments(lib, args, msg):
    a = dict(B=1, H=1, L=16, d=128, w=8, s=4, scale=0.1, dtype=0, pos0=0)
    a.update(args)
    fake = 1 << 20  # never dereferenced: validation fails first
    rc = lib.swa_sink_prefill(fake, fake, fake, fake, None, None, None, a["pos0"], a["B"], a["H"], a["L"], a["d"],
                              a["w"], a["s"], a["scale"], a["dtype"], None)
    assert rc in (swa.SWA_ERR_INVALID, swa.SWA_ERR_UNSUPPORTED)
    assert msg in swa.last_error()


def test_prefill_null_and_misaligned(lib):
    rc = lib.swa_sink_prefill(None, None, None, None, None, None, None, 0, 1, 1, 16, 128, 8, 4, 0.1, 0, None)
    assert rc == swa.SWA_ERR_INVALID and "non-null" in swa.last_error()
    rc = lib.swa_sink_prefill(1 << 20 | 8, 1 << 20, 1 << 20, 1 << 20, None, None, None, 0, 1, 1, 16, 128, 8, 4, 0.1,
                              0, None)
    assert rc == swa.SWA_ERR_INVALID and "aligned" in swa.last_error()
    # chunked prefill with pos0 > 0 needs the cache
    rc = lib.swa_sink_prefill(1 << 20, 1 << 20, 1 << 20, 1 << 20, None, None, None, 5, 1, 1, 16, 128, 8, 4, 0.1, 0,
                              None)
    assert rc == swa.SWA_ERR_INVALID and "cache" in swa.last_error()
    # L == 0 is a no-op that succeeds without touching anything
    assert lib.swa_sink_prefill(None, None, None, None, None, None, None, 0, 1, 1, 0, 128, 8, 4, 0.1, 0, None) == 0


def test_bf16_prefill_takes_d64_and_d128_only(lib):
    # the tensor-core path runs at d = 64 and d = 128; other head dimensions are refused before any launch
    f = 1 << 20
    for d in (16, 32):
        rc = lib.swa_sink_prefill(f, f, f, f, None, None, None, 0, 1, 1, 16, d, 8, 4, 0.1, 0, None)
        assert rc == swa.SWA_ERR_UNSUPPORTED, d


def test_decode_and_write_reject_bad_arguments(lib):
    f = 1 << 20
    assert lib.swa_sink_decode_step(f, f, f, f, None, 1, 1, 128, 8, 8, 0, 0.1, None, 0, 0, None) == swa.SWA_ERR_INVALID
    assert lib.swa_sink_decode_step(f, f, f, f, None, 1, 1, 128, 8, 4, -1, 0.1, None, 0, 0, None) == swa.SWA_ERR_INVALID
    assert lib.kv_rolling_write(f, f, f, f, 1, 1, 128, 8, 4, -1, 1, 0, None) == swa.SWA_ERR_INVALID
    assert lib.kv_rolling_write(None, None, None, None, 1, 1, 128, 8, 4, 0, 0, 0, None) == swa.SWA_OK  # n = 0
    # a workspace smaller than required is refused
    need = lib.swa_sink_decode_workspace_size(1, 2, 128, 4096)
    assert need > 0
    rc = lib.swa_sink_decode_step(f, f, f, f, None, 1, 2, 128, 4096, 4, 5000, 0.1, f, need - 1, 0, None)
    assert rc == swa.SWA_ERR_INVALID and "workspace" in swa.last_error()


def test_workspace_size_shapes(lib):
    # a full GPU of (b, h) rows needs no split; few rows with a long window split the cache
    assert lib.swa_sink_decode_workspace_size(64, 40, 128, 1024) == 0
    assert lib.swa_sink_decode_workspace_size(1, 32, 128, 4096) == 32 * 16 * 130 * 4
    assert lib.swa_sink_decode_workspace_size(0, 32, 128, 4096) == 0


def test_selftests_validate(lib):
    assert lib.swa_selftest_wait_timeout(0, None) == swa.SWA_ERR_INVALID
    assert lib.swa_selftest_umma(None, None, None, 0, None) == swa.SWA_ERR_INVALID


def test_host_prefill_validates_before_any_cuda_call(lib):
    f = 1 << 20  # never dereferenced: validation fails first
    args = [f, f, f, f, None, f, f, f, f, None, 1, 1, 128, 128, 64, 4, 0.1, 0, None]
    bad = list(args)
    bad[0] = None  # no host q
    assert lib.swa_sink_prefill_host(*bad) == swa.SWA_ERR_INVALID
    bad = list(args)
    bad[4] = f  # host lse without a device lse
    assert lib.swa_sink_prefill_host(*bad) == swa.SWA_ERR_INVALID
    bad = list(args)
    bad[15] = 64  # s >= w
    assert lib.swa_sink_prefill_host(*bad) == swa.SWA_ERR_INVALID


def test_bf16_prefill_rejects_windows_past_the_tile_list(lib):
    f = 1 << 20  # never dereferenced: the window check comes first
    rc = lib.swa_sink_prefill(f, f, f, f, None, None, None, 0, 1, 1, 9000, 128, 7400, 4, 0.1, swa.SWA_BF16, None)
    assert rc == swa.SWA_ERR_UNSUPPORTED


def test_rope_decode_validates_before_launch(lib):
    f = 1 << 20  # never dereferenced: validation fails first
    need = lib.swa_sink_decode_rope_workspace_size(1, 1, 128, 4096)
    assert need == lib.swa_sink_decode_workspace_size(1, 1, 128, 4096) > 0  # split-K partials only
    ok = [f, f, f, f, None, 1, 1, 128, 4096, 4, 5000, 0.1, 10000.0, f << 8, need, 0, None]
    bad = list(ok)
    bad[12] = 1.0  # base must be > 1
    assert lib.swa_sink_decode_step_rope(*bad) == swa.SWA_ERR_INVALID
    bad = list(ok)
    bad[14] = need - 1  # workspace too small
    assert lib.swa_sink_decode_step_rope(*bad) == swa.SWA_ERR_INVALID
    bad = list(ok)
    bad[10] = 1 << 31  # t past 2^31 - 1
    assert lib.swa_sink_decode_step_rope(*bad) == swa.SWA_ERR_INVALID
    bad = list(ok)
    bad[8], bad[10] = 70000, 80000  # window past 2^16
    bad[14] = lib.swa_sink_decode_rope_workspace_size(1, 1, 128, 70000)
    assert lib.swa_sink_decode_step_rope(*bad) == swa.SWA_ERR_UNSUPPORTED


def test_rope_prefills_validate_before_launch(lib):
    f = 1 << 20  # never dereferenced: validation fails first
    need = lib.swa_sink_prefill_rope_workspace_size(1, 2, 300, 128, 4)
    # rotated q and k as (hi, lo) bf16 pairs, the sink scores (fp32, 4 per row) and the rotated sink keys (fp32)
    assert need == 4 * (2 * 300 * 128 * 2) + 2 * 300 * 4 * 4 + 2 * 4 * 128 * 4
    assert lib.swa_sink_prefill_rope_workspace_size(1, 2, 300, 128, 5) == 4 * (2 * 300 * 128 * 2) + 2 * 300 * 8 * 4 + 2 * 5 * 128 * 4
    assert lib.swa_sink_prefill_rope_workspace_size(1, 2, 300, 128, 129) == 0
    assert lib.swa_sink_prefill_rope_workspace_size(1, 2, 300, 64, 4) == 0
    ok = [f, f, f, f, None, 1, 2, 300, 128, 64, 4, 0.1, 10000.0, f << 8, need, swa.SWA_BF16, None]
    bad = list(ok)
    bad[15] = swa.SWA_F32  # the RoPE prefill runs on the tensor cores only
    assert lib.swa_sink_prefill_rope(*bad) == swa.SWA_ERR_UNSUPPORTED
    bad = list(ok)
    bad[9], bad[10] = 300, 129  # more sinks than one key tile
    assert lib.swa_sink_prefill_rope(*bad) == swa.SWA_ERR_UNSUPPORTED
    bad = list(ok)
    bad[12] = 0.5  # base must be > 1
    assert lib.swa_sink_prefill_rope(*bad) == swa.SWA_ERR_INVALID
    bad = list(ok)
    bad[14] = need - 1
    assert lib.swa_sink_prefill_rope(*bad) == swa.SWA_ERR_INVALID
    # chunked: chunks shorter than the sinks are refused, and the workspace adds a rotated-key cache
    cneed = lib.swa_sink_prefill_chunked_rope_workspace_size(1, 2, 300, 128, 64, 8)
    # + the rotated-key cache (hi, lo)
    assert cneed == lib.swa_sink_prefill_rope_workspace_size(1, 2, 300, 128, 8) + 2 * 2 * 64 * 128 * 2
    cok = [f, f, f, f, None, f, f, 1, 2, 300, 128, 64, 8, 0.1, 32, 10000.0, f << 8, cneed, swa.SWA_BF16, None]
    bad = list(cok)
    bad[14] = 4  # chunk < s
    assert lib.swa_sink_prefill_chunked_rope(*bad) == swa.SWA_ERR_INVALID
    bad = list(cok)
    bad[17] = cneed - 256
    assert lib.swa_sink_prefill_chunked_rope(*bad) == swa.SWA_ERR_INVALID
    # the RoPE tile plan refuses a chunk start inside the sinks
    buf = (ctypes.c_int * (5 * 64))()
    assert lib.swa_prefill_tile_plan_rope(8, 300, 3, 64, 8, buf, 64) == swa.SWA_ERR_UNSUPPORTED


def test_dilated_prefill_validates_before_launch(lib):
    # the workspace rules of the gathered form (fp32 here; bf16 with d = 128 runs in place and reads none)
    f = 1 << 20
    need = lib.swa_sink_prefill_dilated_workspace_size(1, 2, 300, 128, 4, 3, swa.SWA_F32)
    rows = 2 * 3 * (4 + (300 - 4 + 2) // 3)  # virtual heads x (sinks + the longest residue class)
    assert need >= 4 * rows * 128 * 4 + rows * 4
    ok = [f, f, f, f, None, 1, 2, 300, 128, 64, 4, 3, 0.1, f << 8, need, swa.SWA_F32, None]
    bad = list(ok)
    bad[11] = 0  # dilation >= 1
    assert lib.swa_sink_prefill_dilated(*bad) == swa.SWA_ERR_INVALID
    bad = list(ok)
    bad[14] = need - 1
    assert lib.swa_sink_prefill_dilated(*bad) == swa.SWA_ERR_INVALID
    bad = list(ok)
    bad[5], bad[6], bad[11] = 65535, 32, 2  # B * H * r past the supported virtual heads
    bad[14] = lib.swa_sink_prefill_dilated_workspace_size(65535, 32, 300, 128, 4, 2, swa.SWA_F32)
    assert lib.swa_sink_prefill_dilated(*bad) == swa.SWA_ERR_UNSUPPORTED
    assert lib.swa_sink_prefill_dilated_workspace_size(1, 2, 300, 128, 4, 0, swa.SWA_BF16) == 0
