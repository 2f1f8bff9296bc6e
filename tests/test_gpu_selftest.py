"""GPU diagnostics: the bounded device waits report a timeout instead of hanging, and the tensor-core
building blocks (TMA tiles with the 128-byte swizzle, shared-memory descriptors, tcgen05.mma into TMEM,
tcgen05.ld back) compute 128 x 128 x 128 bf16 products exactly like a plain fp32 matmul."""
import pytest
import torch

from gpu_common import require_gpu

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    swa = require_gpu()
    L = swa.lib()
    assert swa.swa_device_status() == swa.SWA_OK
    stream = torch.cuda.current_stream().cuda_stream
    assert L.swa_selftest_wait_timeout(2_000_000, stream) == swa.SWA_OK  # 2 ms limit, nothing arrives
    assert swa.swa_device_status() == swa.SWA_ERR_TIMEOUT
    assert "wait ran out" in swa.last_error()
    assert swa.swa_device_status() == swa.SWA_OK  # cleared on read
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0  # the context is still usable


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_umma_tile_matches_matmul(mode):
    swa = require_gpu()
    g = torch.Generator(device="cpu").manual_seed(7 + mode)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    c = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    rc = swa.lib().swa_selftest_umma(a.data_ptr(), b.data_ptr(), c.data_ptr(), mode,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == swa.SWA_OK, swa.last_error()
    assert swa.swa_device_status() == swa.SWA_OK, swa.last_error()
    want = a.double() @ (b.double().T if mode == 0 else b.double())
    err = (c.double() - want).abs().max().item()
    assert err < 1e-3, f"mode {mode}: max-abs {err}"
