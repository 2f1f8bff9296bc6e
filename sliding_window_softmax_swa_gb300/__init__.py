"""GB300 (sm_103a) library for causal sliding-window softmax attention with attention sinks.

Prefill (TMA + tcgen05 tensor cores), chunked prefill through a rolling KV cache, and streaming decode
(split-K over the cache), with or without RoPE at the positions inside the cache, the dilated and the
block-sparse (global tokens + random key blocks) variants and the SWA + linear-attention hybrid, behind the C ABI of
include/swa_sink.h. This package is the thin Python binding of that ABI; the kernels live in csrc/ and are
built with ``build.build()``.
"""
from ._binding import (SWA_BF16, SWA_ERR_CUDA, SWA_ERR_INVALID, SWA_ERR_TIMEOUT, SWA_ERR_UNSUPPORTED, SWA_F32,
                       SWA_OK, SIGNATURES, SwaError, kv_rolling_write, last_error, lib, library_path,
                       prefill_tile_plan, prefill_tile_plan_rope, prefill_tile_plan_dilated, prefill_dilated_split,
                       swa_device_status, swa_sink_decode_step,
                       swa_sink_decode_step_dilated, swa_sink_dilated_cache_write,
                       swa_sink_decode_step_rope, swa_sink_decode_workspace_size, swa_sink_prefill,
                       swa_sink_prefill_chunked, swa_sink_prefill_chunked_dilated, swa_sink_prefill_chunked_rope,
                       swa_sink_prefill_dilated, swa_sink_prefill_blocksparse, prefill_blocksparse_plan,
                       swa_hybrid_prefill, swa_hybrid_decode_step,
                       swa_sink_prefill_host, swa_sink_prefill_rope)

__all__ = ["swa_sink_prefill", "swa_sink_prefill_chunked", "swa_sink_prefill_host", "swa_sink_prefill_rope",
           "swa_sink_prefill_chunked_rope", "swa_sink_prefill_dilated", "swa_sink_prefill_chunked_dilated",
           "kv_rolling_write", "swa_sink_decode_step", "swa_sink_decode_step_rope", "swa_sink_dilated_cache_write",
           "swa_sink_decode_step_dilated", "swa_sink_prefill_blocksparse", "prefill_blocksparse_plan",
           "swa_hybrid_prefill", "swa_hybrid_decode_step",
           "swa_sink_decode_workspace_size", "swa_device_status", "prefill_tile_plan", "prefill_tile_plan_rope",
           "prefill_tile_plan_dilated", "prefill_dilated_split",
           "last_error", "lib", "library_path", "SwaError", "SIGNATURES", "SWA_OK", "SWA_ERR_INVALID",
           "SWA_ERR_UNSUPPORTED", "SWA_ERR_CUDA", "SWA_ERR_TIMEOUT", "SWA_BF16", "SWA_F32"]
