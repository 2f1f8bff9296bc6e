"""ctypes binding of the C ABI in include/swa_sink.h.

Argument marshalling only: each function checks shapes/dtypes/devices of torch tensors, passes their
device pointers and the current CUDA stream to the library, and raises on a non-zero status. Every
step of the computation runs in the library's CUDA kernels; there is no CPU or PyTorch fallback. If
the library is not built the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SWA_OK, SWA_ERR_INVALID, SWA_ERR_UNSUPPORTED, SWA_ERR_CUDA, SWA_ERR_TIMEOUT = 0, -1, -2, -3, -4
SWA_BF16, SWA_F32 = 0, 1
_STATUS_NAMES = {0: "SWA_OK", -1: "SWA_ERR_INVALID", -2: "SWA_ERR_UNSUPPORTED", -3: "SWA_ERR_CUDA",
                 -4: "SWA_ERR_TIMEOUT"}

_vp, _i, _i64, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/swa_sink.h
SIGNATURES = {
    "swa_sink_prefill": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i, _i, _i64, _i, _i, _i, _f, _i, _vp]),
    "swa_sink_prefill_chunked": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _i, _f, _i64, _i,
                                      _vp]),
    "swa_sink_prefill_host": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _i, _f,
                                   _i, _vp]),
    "kv_rolling_write": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i64, _i64, _i, _vp]),
    "swa_sink_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i64, _f, _vp, _sz, _i, _vp]),
    "swa_sink_decode_step_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i64, _f, _i, _vp]),
    "swa_sink_decode_workspace_size": (_sz, [_i, _i, _i, _i]),
    "swa_sink_decode_step_rope": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i64, _f, ctypes.c_double, _vp,
                                       _sz, _i, _vp]),
    "swa_sink_decode_rope_workspace_size": (_sz, [_i, _i, _i, _i]),
    "swa_last_error_string": (ctypes.c_char_p, []),
    "swa_device_status": (_i, [_vp]),
    "swa_selftest_wait_timeout": (_i, [_i64, _vp]),
    "swa_selftest_umma": (_i, [_vp, _vp, _vp, _i, _vp]),
    "swa_prefill_tile_plan": (_i, [_i64, _i64, _i64, _i, _i, ctypes.POINTER(ctypes.c_int), _i]),
    "swa_prefill_tile_plan_rope": (_i, [_i64, _i64, _i64, _i, _i, ctypes.POINTER(ctypes.c_int), _i]),
    "swa_prefill_dilated_split": (_i, [_i64, _i, _i, ctypes.POINTER(ctypes.c_int64)]),
    "swa_prefill_tile_plan_dilated": (_i, [_i64, _i, _i, _i, _i, _i64, ctypes.POINTER(ctypes.c_int), _i]),
    "swa_prefill_blocksparse_plan": (_i, [_i64, _i, _i, _vp, _i, _i, _vp, _i, _i64, ctypes.POINTER(ctypes.c_int), _i]),
    "swa_sink_prefill_dilated": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _i, _i, _f, _vp, _sz, _i, _vp]),
    "swa_sink_prefill_chunked_dilated": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _i, _i, _f, _i64,
                                              _vp, _sz, _i, _vp]),
    "swa_sink_dilated_cache_write": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i64, _i, _vp]),
    "swa_sink_decode_step_dilated": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i64, _f, _vp, _sz, _i,
                                          _vp]),
    "swa_sink_prefill_dilated_workspace_size": (_sz, [_i, _i, _i64, _i, _i, _i, _i]),
    "swa_sink_prefill_chunked_rope": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _i, _f, _i64,
                                           ctypes.c_double, _vp, _sz, _i, _vp]),
    "swa_sink_prefill_chunked_rope_workspace_size": (_sz, [_i, _i, _i64, _i, _i, _i]),
    "swa_sink_prefill_rope": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _i, _f, ctypes.c_double, _vp,
                                   _sz, _i, _vp]),
    "swa_sink_prefill_rope_workspace_size": (_sz, [_i, _i, _i64, _i, _i]),
    "swa_sink_prefill_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _i, _f, _vp, _i, _i, _vp, _i,
                                          _vp, _sz, _i, _vp]),
    "swa_sink_prefill_blocksparse_workspace_size": (_sz, [_i64, _i, _i, _i]),
    "swa_hybrid_prefill": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i64, _i, _i, _i, _f, _vp, _sz, _i, _vp]),
    "swa_hybrid_prefill_workspace_size": (_sz, [_i, _i, _i64, _i]),
    "swa_hybrid_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i64, _f, _vp, _sz,
                                    _i, _vp]),
    "swa_hybrid_decode_workspace_size": (_sz, [_i, _i, _i, _i]),
}

_lib = None


class SwaError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with {_STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = False):
    """The loaded library (ctypes.CDLL with typed entry points)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"the CUDA library {path} is not built; run __graft_entry__.build() or "
                               "python -m sliding_window_softmax_swa_gb300.build")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().swa_last_error_string().decode()


def _check(fn: str, rc: int):
    if rc != SWA_OK:
        raise SwaError(fn, rc, last_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SWA_BF16
    if t.dtype == torch.float32:
        return SWA_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _dev(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _ptr(t):
    return None if t is None else t.data_ptr()


def swa_sink_prefill(q, k, v, w: int, s: int, scale: float | None = None, o=None, lse=None,
                     k_cache=None, v_cache=None, pos0: int = 0, stream=None):
    """Prefill of q, k, v [B, H, L, d] at absolute positions pos0..pos0+L-1 -> o [B, H, L, d].
    With ``lse`` (a [B, H, L] float32 tensor) the log-sum-exp of each row is written too."""
    B, H, L, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and k.dtype == q.dtype and v.dtype == q.dtype
    if o is None:
        o = torch.empty_like(q)
    _dev(q, k, v, o, lse, k_cache, v_cache)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_prefill", lib().swa_sink_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(k_cache), _ptr(v_cache), pos0, B, H, L, d, w, s,
        scale, _dtype_code(q), _stream(stream)))
    return o


def swa_sink_prefill_chunked_dilated(q, k, v, s: int, r: int, chunk: int, k_cache, v_cache,
                                     scale: float | None = None, o=None, lse=None, workspace=None, stream=None):
    """Chunked prefill over the dilated window through the per-class caches [r, B, H, w, d] (overwritten)."""
    B, H, L, d = q.shape
    w = k_cache.shape[3]
    assert k_cache.shape == (r, B, H, w, d)
    if o is None:
        o = torch.empty_like(q)
    nws = lib().swa_sink_prefill_dilated_workspace_size(B, H, L, d, s, r, _dtype_code(q))
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    _dev(q, k, v, o, lse, k_cache, v_cache, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_prefill_chunked_dilated", lib().swa_sink_prefill_chunked_dilated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(k_cache), _ptr(v_cache), B, H, L, d, w, s, r, scale,
        chunk, _ptr(workspace), workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return o


def swa_sink_dilated_cache_write(k_cache, v_cache, k_new, v_new, s: int, r: int, t: int, stream=None):
    """Write position t's key/value ([B, H, d]) into the dilated caches [r, B, H, w, d] (write, then attend)."""
    r_, B, H, w, d = k_cache.shape
    assert r_ == r and k_new.shape == (B, H, d) and v_new.shape == (B, H, d)
    _dev(k_cache, v_cache, k_new, v_new)
    _check("swa_sink_dilated_cache_write", lib().swa_sink_dilated_cache_write(
        _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), B, H, d, w, s, r, t, _dtype_code(k_cache),
        _stream(stream)))


def swa_sink_decode_step_dilated(q, k_cache, v_cache, s: int, r: int, t: int, scale: float | None = None, o=None,
                                 lse=None, workspace=None, stream=None):
    """Decode step at position t over the dilated window with sinks (caches [r, B, H, w, d])."""
    B, H, d = q.shape
    r_, _, _, w, _ = k_cache.shape
    assert r_ == r
    if o is None:
        o = torch.empty_like(q)
    nws = lib().swa_sink_decode_workspace_size(B, H, d, w)
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    _dev(q, k_cache, v_cache, o, lse, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_decode_step_dilated", lib().swa_sink_decode_step_dilated(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, H, d, w, s, r, t, scale, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return o


def swa_sink_prefill_dilated(q, k, v, w: int, s: int, r: int, scale: float | None = None, o=None, lse=None,
                             workspace=None, stream=None):
    """Prefill over the dilated window with sinks: row t attends the s sinks and t, t - r, ..., t - (m-1) r.
    bf16 with d = 128 (and any r = 1 call) runs in place and takes no workspace."""
    B, H, L, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and k.dtype == q.dtype and v.dtype == q.dtype
    if o is None:
        o = torch.empty_like(q)
    in_place = r == 1 or (q.dtype == torch.bfloat16 and d == 128)
    if workspace is None and not in_place:
        nws = lib().swa_sink_prefill_dilated_workspace_size(B, H, L, d, s, r, _dtype_code(q))
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    _dev(q, k, v, o, lse, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("swa_sink_prefill_dilated", lib().swa_sink_prefill_dilated(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, L, d, w, s, r, scale, _ptr(workspace), nbytes,
        _dtype_code(q), _stream(stream)))
    return o


def swa_sink_prefill_rope(q, k, v, w: int, s: int, rope_base: float = 10000.0, scale: float | None = None, o=None,
                          lse=None, workspace=None, stream=None):
    """Prefill of unrotated q, k (bf16 [B, H, L, 128]) with RoPE at the positions inside the cache."""
    B, H, L, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and k.dtype == q.dtype and v.dtype == q.dtype
    if o is None:
        o = torch.empty_like(q)
    nws = lib().swa_sink_prefill_rope_workspace_size(B, H, L, d, s)
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    _dev(q, k, v, o, lse, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_prefill_rope", lib().swa_sink_prefill_rope(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, L, d, w, s, scale, float(rope_base), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return o


def swa_sink_prefill_chunked_rope(q, k, v, w: int, s: int, chunk: int, k_cache, v_cache, rope_base: float = 10000.0,
                                  scale: float | None = None, o=None, lse=None, workspace=None, stream=None):
    """Chunked prefill with RoPE at the positions inside the cache (unrotated q, k; the caches end up
    holding unrotated keys and the values)."""
    B, H, L, d = q.shape
    w_ = k_cache.shape[2]
    if o is None:
        o = torch.empty_like(q)
    nws = lib().swa_sink_prefill_chunked_rope_workspace_size(B, H, L, d, w_, s)
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    _dev(q, k, v, o, lse, k_cache, v_cache, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_prefill_chunked_rope", lib().swa_sink_prefill_chunked_rope(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(k_cache), _ptr(v_cache), B, H, L, d, w, s, scale, chunk,
        float(rope_base), _ptr(workspace), workspace.numel() * workspace.element_size(), _dtype_code(q),
        _stream(stream)))
    return o


def _pattern(globals_, rand_blocks):
    """Host int32 arrays of a block-sparse pattern, as given (the library checks them): (globals, r, rand)."""
    import numpy as np
    g = np.ascontiguousarray([int(x) for x in globals_], dtype=np.int32)
    if rand_blocks is None:
        return g, 0, np.zeros((0,), dtype=np.int32)
    rb = np.ascontiguousarray(rand_blocks, dtype=np.int32)
    return g, (rb.shape[1] if rb.ndim == 2 else 0), rb


def swa_sink_prefill_blocksparse(q, k, v, w: int, s: int, globals_=(), block: int = 64, rand_blocks=None,
                                 scale: float | None = None, o=None, lse=None, workspace=None, stream=None):
    """Prefill over the BigBird-style union (window + sinks + global tokens + random key blocks), causal.
    globals_: positions of the global tokens; rand_blocks: int array [ceil(L / block), r] of key blocks per query
    block (-1 = none), or None."""
    B, H, L, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and k.dtype == q.dtype and v.dtype == q.dtype
    if o is None:
        o = torch.empty_like(q)
    g, r, rb = _pattern(globals_, rand_blocks)
    nws = lib().swa_sink_prefill_blocksparse_workspace_size(L, g.size, block, r)
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    _dev(q, k, v, o, lse, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_prefill_blocksparse", lib().swa_sink_prefill_blocksparse(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, L, d, w, s, scale,
        g.ctypes.data if g.size else None, g.size, block, rb.ctypes.data if r else None, r, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return o


def swa_hybrid_prefill(q, k, v, wf, w: int, s: int, scale: float | None = None, o=None, state_s=None,
                       state_z=None, workspace=None, stream=None):
    """SWA with sinks + a Hedgehog linear-attention branch over the keys that left the window (one shared
    normaliser).  q, k, v [B, H, L, 128] bf16, wf [128, 64] bf16.  With state_s/state_z (fp32 [B, H, 128, 128]
    and [B, H, 128]) the state after the last row is written there."""
    B, H, L, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    if o is None:
        o = torch.empty_like(q)
    nws = lib().swa_hybrid_prefill_workspace_size(B, H, L, d)
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    _dev(q, k, v, o, wf, state_s, state_z, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_hybrid_prefill", lib().swa_hybrid_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(wf), _ptr(o), _ptr(state_s), _ptr(state_z), B, H, L, d, w, s, scale,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return o


def swa_hybrid_decode_step(q, k_new, v_new, k_cache, v_cache, state_s, state_z, wf, w: int, s: int, t: int,
                           scale: float | None = None, o=None, workspace=None, stream=None):
    """One decode step of the hybrid at position t: fold the evicted key into the state, write k_new/v_new
    into the rolling cache, attend, combine.  q, k_new, v_new [B, H, 128] bf16; caches [B, H, w, 128]."""
    B, H, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    nws = lib().swa_hybrid_decode_workspace_size(B, H, d, w)
    if workspace is None:
        workspace = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    _dev(q, k_new, v_new, k_cache, v_cache, state_s, state_z, wf, o, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_hybrid_decode_step", lib().swa_hybrid_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(state_s), _ptr(state_z), _ptr(wf),
        _ptr(o), B, H, d, w, s, t, scale, _ptr(workspace), workspace.numel() * workspace.element_size(),
        _dtype_code(q), _stream(stream)))
    return o


def swa_sink_prefill_chunked(q, k, v, w: int, s: int, chunk: int, k_cache, v_cache, scale: float | None = None,
                             o=None, lse=None, stream=None):
    """Chunked prefill through the rolling cache (k_cache/v_cache [B, H, w, d] are overwritten)."""
    B, H, L, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    _dev(q, k, v, o, lse, k_cache, v_cache)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_prefill_chunked", lib().swa_sink_prefill_chunked(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(k_cache), _ptr(v_cache), B, H, L, d, w, s, scale,
        chunk, _dtype_code(q), _stream(stream)))
    return o


def swa_sink_prefill_host(q_h, k_h, v_h, w: int, s: int, q_d, k_d, v_d, o_d, o_h=None, lse_h=None, lse_d=None,
                          scale: float | None = None, stream=None):
    """Prefill of host tensors q_h, k_h, v_h [B, H, L, d] (pinned for overlap) through the caller's device
    buffers q_d, k_d, v_d, o_d; the output lands in o_h (host).  Copies and compute are pipelined by the
    library over groups of (b, h) rows.  Asynchronous: synchronise the stream before reading o_h."""
    B, H, L, d = q_h.shape
    for t in (q_h, k_h, v_h):
        assert t.device.type == "cpu" and t.is_contiguous() and t.shape == q_h.shape and t.dtype == q_h.dtype
    if o_h is None:
        o_h = torch.empty(q_h.shape, dtype=q_h.dtype, pin_memory=q_h.is_pinned())
    assert o_h.device.type == "cpu" and o_h.is_contiguous() and o_h.shape == q_h.shape
    if lse_h is not None:
        assert lse_h.device.type == "cpu" and lse_h.is_contiguous() and lse_d is not None
    for t in (q_d, k_d, v_d, o_d):
        assert t.shape == q_h.shape and t.dtype == q_h.dtype
    _dev(q_d, k_d, v_d, o_d, lse_d)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_prefill_host", lib().swa_sink_prefill_host(
        q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), o_h.data_ptr(), lse_h.data_ptr() if lse_h is not None else None,
        _ptr(q_d), _ptr(k_d), _ptr(v_d), _ptr(o_d), _ptr(lse_d), B, H, L, d, w, s, scale, _dtype_code(q_h),
        _stream(stream)))
    return o_h


def kv_rolling_write(k_cache, v_cache, k_new, v_new, w: int, s: int, pos0: int, stream=None):
    """Write k_new/v_new [B, H, n, d] (positions pos0..pos0+n-1) into the caches [B, H, w, d]."""
    B, H, n, d = k_new.shape
    assert k_cache.shape == (B, H, w, d) and v_cache.shape == (B, H, w, d)
    _dev(k_cache, v_cache, k_new, v_new)
    _check("kv_rolling_write", lib().kv_rolling_write(
        _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), B, H, d, w, s, pos0, n, _dtype_code(k_new),
        _stream(stream)))


def swa_sink_decode_step_rope(q, k_cache, v_cache, t: int, w: int, s: int, rope_base: float = 10000.0,
                              scale: float | None = None, o=None, lse=None, workspace=None, stream=None):
    """Decode step at position t with RoPE at the positions inside the cache (unrotated q and keys)."""
    B, H, d = q.shape
    assert k_cache.shape == (B, H, w, d) and v_cache.shape == (B, H, w, d)
    if o is None:
        o = torch.empty_like(q)
    nws = lib().swa_sink_decode_rope_workspace_size(B, H, d, w)
    if workspace is None:
        workspace = torch.empty(nws, dtype=torch.uint8, device=q.device)
    _dev(q, k_cache, v_cache, o, lse, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    _check("swa_sink_decode_step_rope", lib().swa_sink_decode_step_rope(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, H, d, w, s, t, scale, float(rope_base),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return o


def swa_sink_decode_workspace_size(B: int, H: int, d: int, w: int) -> int:
    return int(lib().swa_sink_decode_workspace_size(B, H, d, w))


def swa_sink_decode_step(q, k_cache, v_cache, t: int, w: int, s: int, scale: float | None = None, o=None,
                         lse=None, workspace=None, stream=None):
    """Decode for q [B, H, d] at position t against the caches [B, H, w, d] -> o [B, H, d]."""
    B, H, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    need = swa_sink_decode_workspace_size(B, H, d, w)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _dev(q, k_cache, v_cache, o, lse, workspace)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("swa_sink_decode_step", lib().swa_sink_decode_step(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, H, d, w, s, t, scale, _ptr(workspace),
        wbytes, _dtype_code(q), _stream(stream)))
    return o


def prefill_tile_plan(q0: int, q1: int, pos0: int, w: int, s: int):
    """The key tiles the bf16 prefill walks for query rows q0..q1 (one CTA: two 128-row query tiles):
    list of (src, row0, pbase, chi, used_by_mask)."""
    buf = (ctypes.c_int * (5 * 256))()
    n = lib().swa_prefill_tile_plan(q0, q1, pos0, w, s, buf, 256)
    if n < 0:
        raise SwaError("swa_prefill_tile_plan", n, last_error())
    return [tuple(buf[5 * i:5 * i + 5]) for i in range(min(n, 256))]


def prefill_tile_plan_rope(q0: int, q1: int, pos0: int, w: int, s: int):
    """The key tiles of the RoPE prefills for query rows q0..q1 of a call at pos0, as prefill_tile_plan."""
    buf = (ctypes.c_int * (5 * 256))()
    n = lib().swa_prefill_tile_plan_rope(q0, q1, pos0, w, s, buf, 256)
    if n < 0:
        raise SwaError("swa_prefill_tile_plan_rope", n, last_error())
    return [tuple(buf[5 * i:5 * i + 5]) for i in range(min(n, 256))]


def prefill_dilated_split(L: int, s: int, r: int):
    """How the in-place dilated prefill splits the rows of a (b, h): (nrows, G, ns, tail0)."""
    out = (ctypes.c_int64 * 4)()
    _check("swa_prefill_dilated_split", lib().swa_prefill_dilated_split(L, s, r, out))
    return tuple(out)


def prefill_tile_plan_dilated(L: int, w: int, s: int, r: int, cls: int, row_start: int):
    """The key tiles of the in-place dilated prefill's work item (class cls, query tile at virtual row
    s + row_start): list of (src, row0, pbase, chi, used_by_mask); src 1 = plain rows, src 0 = groups."""
    buf = (ctypes.c_int * (5 * 256))()
    n = lib().swa_prefill_tile_plan_dilated(L, w, s, r, cls, row_start, buf, 256)
    if n < 0:
        raise SwaError("swa_prefill_tile_plan_dilated", n, last_error())
    return [tuple(buf[5 * i:5 * i + 5]) for i in range(min(n, 256))]


def prefill_blocksparse_plan(L: int, w: int, s: int, globals_, block: int, rand_blocks, pair: int):
    """The key tiles of the block-sparse prefill for query pair ``pair`` (rows 256*pair ..): list of
    (pbase, chi, used_by_mask, global-column mask as one 128-bit int, pbase1).  pbase1 is -1, or for a packed
    tile the position of column 64 (columns 64..127 hold pbase1 .. pbase1 + 63)."""
    g, r, rb = _pattern(globals_, rand_blocks)
    buf = (ctypes.c_int * (8 * 64))()
    n = lib().swa_prefill_blocksparse_plan(L, w, s, g.ctypes.data if g.size else None, g.size, block,
                                           rb.ctypes.data if r else None, r, pair, buf, 64)
    if n < 0:
        raise SwaError("swa_prefill_blocksparse_plan", n, last_error())
    out = []
    for i in range(min(n, 64)):
        rec = buf[8 * i:8 * i + 8]
        gm = sum((rec[3 + k] & 0xFFFFFFFF) << (32 * k) for k in range(4))
        out.append((rec[0], rec[1], rec[2], gm, rec[7]))
    return out


def swa_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status (0 = fine)."""
    return lib().swa_device_status(_stream(stream))
