/*
 * swa_sink.h -- C ABI of the GB300 (sm_103a) library for causal sliding-window softmax attention
 * with attention sinks: prefill, chunked prefill through a rolling KV cache, streaming decode.
 *
 * The operation.  For query position t (0-indexed) with window w and s sink tokens (m = w - s recent
 * keys), the key set is
 *     K(t) = { i <= t : i < s  or  i >= t - m + 1 }
 * and the output is o_t = sum_{i in K(t)} softmax_i(scale * q_t.k_i) v_i.
 *   - SWA formula (window of w keys ending at t) and sinks (the first s = 4 tokens attended in
 *     addition to the w - 4 window tokens): hyper.ai summary of arXiv 2608.28444, section
 *     "带 Sink 的滑动窗口注意力".
 *   - Causal softmax attention: "模糊窗口注意力" (Blurry Window Attention), section 2.1, equation (1).
 *   - Rolling cache and chunk-based prefill: "滑窗与固定稀疏", eq attn-fixed-rolling and the
 *     paragraph after it; sink + recent cache of k + m slots: eq attn-fixed-streaming.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns every buffer.  No entry
 *     point allocates or frees device memory.
 *   - Tensors are contiguous, row-major, innermost dimension last ([B, H, L, d]: d contiguous), and
 *     16-byte aligned.  bf16 storage (SWA_BF16) or fp32 storage (SWA_F32).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously on it.
 *   - Argument errors return SWA_ERR_INVALID / SWA_ERR_UNSUPPORTED synchronously, before anything
 *     is launched; a failed launch returns SWA_ERR_CUDA.  swa_last_error_string() explains the most
 *     recent failure of the calling host thread.
 *   - Every device-side wait in the library is bounded in time.  A wait that runs out records an
 *     error word on the device and the kernel returns; swa_device_status() reports it.
 *   - All batch rows share one position: one pos0 in prefill, one t in decode.
 *   - Multi-head layout is one K/V head per query head (H_kv = H).
 */
#ifndef SWA_SINK_H
#define SWA_SINK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SWA_OK = 0,
    SWA_ERR_INVALID = -1,     /* bad argument (null pointer, s >= w, misaligned, ...)          */
    SWA_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. bf16 with d != 128)          */
    SWA_ERR_CUDA = -3,        /* a CUDA runtime call or kernel launch failed                 */
    SWA_ERR_TIMEOUT = -4      /* a bounded device-side wait ran out (see swa_device_status)   */
} swa_status;

typedef enum { SWA_BF16 = 0, SWA_F32 = 1 } swa_dtype;

/*
 * swa_sink_prefill -- attention of L consecutive queries at absolute positions pos0 .. pos0+L-1.
 *
 *   q, k, v : [B, H, L, d], the queries and the keys/values of the same L positions.
 *   o       : [B, H, L, d] output, same dtype as q.
 *   lse     : optional [B, H, L] fp32 output, natural log of sum_{i in K(t)} exp(scale * q_t.k_i);
 *             NULL to skip.
 *   k_cache, v_cache : used only when pos0 > 0: [B, H, w, d] rolling cache holding the keys/values
 *             of positions < pos0 in the layout kv_rolling_write produces (slot p for p < s, slot
 *             s + ((p - s) mod m) otherwise), i.e. the cache state after positions 0..pos0-1 were
 *             written.  May be NULL when pos0 == 0.  Not modified.
 *   pos0    : absolute position of row 0 (0 = a whole-sequence prefill; > 0 = one chunk of a chunked
 *             prefill, see the chunk-based prefill of "滑窗与固定稀疏").
 *   B, H, L, d, w, s : batch, heads, rows, head dim, window (keys per query, sinks included), sinks.
 *             Requires 0 <= s < w, L >= 0 (L == 0 is a no-op), pos0 + L < 2^31.
 *   scale   : softmax scale (1/sqrt(d) for the usual attention).
 *   dtype   : SWA_BF16 requires d in {64, 128} (tensor-core path: TMA + tcgen05 + TMEM);
 *             SWA_F32 accepts d in {16, 32, 64, 128} (CUDA-core path).
 */
int swa_sink_prefill(const void *q, const void *k, const void *v, void *o, float *lse,
                     const void *k_cache, const void *v_cache, int64_t pos0,
                     int B, int H, int64_t L, int d, int w, int s, float scale,
                     int dtype, void *stream);

/*
 * swa_sink_prefill_host -- swa_sink_prefill (pos0 = 0) of q, k, v held in host memory, with the output
 * copied back to host memory: the end-to-end form of the prefill of "带 Sink 的滑动窗口注意力".  The
 * (b, h) rows are independent, so they are split into groups whose host-to-device copies, prefill and
 * device-to-host copies are pipelined on streams of the library (created once per device, forked from
 * and joined back to `stream` with events); per row the result is the same as swa_sink_prefill's.
 *
 *   q_h, k_h, v_h : host [B, H, L, d] inputs; o_h : host [B, H, L, d] output; lse_h : optional host
 *             [B, H, L] fp32 output (NULL to skip).  Page-locked (pinned) host memory lets the copies
 *             overlap the compute; pageable memory is correct but serialises them.
 *   q_d, k_d, v_d, o_d : caller-owned device buffers of [B, H, L, d]; lse_d : device [B, H, L] fp32,
 *             required when lse_h is given.  The library allocates nothing.
 *   Other arguments as swa_sink_prefill.  Asynchronous on `stream`: the host buffers must stay valid
 *   and unchanged until `stream` has reached this point.
 */
int swa_sink_prefill_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                          void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d,
                          int B, int H, int64_t L, int d, int w, int s, float scale, int dtype, void *stream);

/*
 * swa_sink_prefill_rope -- swa_sink_prefill (pos0 = 0) with rotary position embedding at the positions
 * the keys have inside the cache of the StreamingLLM section of "滑窗与固定稀疏": for query t the cache holds
 * K(t), sinks first and then the window in order, at positions 0 .. |K(t)| - 1, and the query is the
 * newest entry.  This equals plain RoPE (q at t, key i at i) for the window keys and puts the query at
 * min(t, w - 1) for the sink scores.  RoPE rotates dimension pair (i, i + d/2) by position *
 * rope_base^(-2i/d).  Row t equals swa_sink_decode_step_rope at step t over the same keys.
 *
 *   q, k, v, o, lse : as swa_sink_prefill, with q and k unrotated; bf16, d = 128, contiguous.
 *   rope_base : finite and > 1.
 *   workspace : caller-owned device scratch of swa_sink_prefill_rope_workspace_size(B, H, L, d, s) bytes,
 *             256-byte aligned: the rotated q and k (4 x B*H*L*d bf16: each as a bf16 pair hi + lo whose sum
 *             is the fp32 rotation), the sink scores (B*H*L rows of s rounded up to a multiple of 4, fp32)
 *             and the rotated sink keys (B*H*s*d fp32).
 *   s <= 128, pos0 = 0 only (SWA_ERR_UNSUPPORTED otherwise).  Each window score is formed from three
 *   tensor-core products of the pairs (hi.hi + hi.lo + lo.hi), so the rotation adds about fp32 rounding, not
 *   bf16 rounding, to the scores; the sink scores (the query rotated at min(t, w - 1)) are fp32 dot products
 *   of fp32 rotations made by the rotation pass.  Other arguments and errors as swa_sink_prefill.
 */
int swa_sink_prefill_rope(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                          int64_t L, int d, int w, int s, float scale, double rope_base, void *workspace,
                          size_t workspace_bytes, int dtype, void *stream);
/* The workspace of swa_sink_prefill_rope in bytes; 0 for arguments it does not take (d != 128, s > 128). */
size_t swa_sink_prefill_rope_workspace_size(int B, int H, int64_t L, int d, int s);

/*
 * swa_sink_prefill_chunked_rope -- swa_sink_prefill_chunked with RoPE at the positions inside the cache
 * (as swa_sink_prefill_rope): chunk c attends the cache state left by the earlier chunks plus its own keys,
 * then its keys/values are written into the cache.  The result equals swa_sink_prefill_rope of the whole
 * sequence, and k_cache / v_cache end up holding the unrotated keys and the values, as
 * swa_sink_prefill_chunked leaves them (ready for swa_sink_decode_step_rope).
 *
 *   q, k, v, o, lse, k_cache, v_cache, chunk : as swa_sink_prefill_chunked; q and k unrotated; bf16,
 *             d = 128; chunk >= max(1, s).
 *   rope_base : finite and > 1.
 *   workspace : caller-owned device scratch of swa_sink_prefill_chunked_rope_workspace_size(B, H, L, d, w, s)
 *             bytes, 256-byte aligned: what swa_sink_prefill_rope keeps for the whole sequence (one rotation
 *             pass serves every chunk: rotations depend on absolute positions only) and two [B, H, w, d] bf16
 *             caches of rotated keys (hi and lo).
 *   s <= 128 (SWA_ERR_UNSUPPORTED otherwise).  Scores as swa_sink_prefill_rope; other arguments and errors as
 *   swa_sink_prefill_chunked.
 */
int swa_sink_prefill_chunked_rope(const void *q, const void *k, const void *v, void *o, float *lse, void *k_cache,
                                  void *v_cache, int B, int H, int64_t L, int d, int w, int s, float scale,
                                  int64_t chunk, double rope_base, void *workspace, size_t workspace_bytes, int dtype,
                                  void *stream);
/* The workspace of swa_sink_prefill_chunked_rope in bytes; 0 for arguments it does not take. */
size_t swa_sink_prefill_chunked_rope_workspace_size(int B, int H, int64_t L, int d, int w, int s);

/*
 * swa_sink_prefill_dilated -- whole-sequence prefill over a dilated window with sinks: the dilated sliding
 * window of "滑窗与固定稀疏" (glossary and Longformer section: attended window positions skip r - 1 tokens),
 * causal and with the sinks of the StreamingLLM section.  Row t attends
 *     {i < s}  |  {t - j r : 0 <= j < m},  m = w - s,  restricted to i <= t  (each key once),
 * so the window reaches (m - 1) r + 1 positions back at the cost of m keys; r = 1 is swa_sink_prefill (and
 * runs it).  Each residue class of positions mod r, after the sinks, is a virtual head with the plain band.
 * bf16 with d = 128 runs in place: the tensor-core prefill reads every class straight from q, k, v through
 * 4-D tensor maps and writes each row at its own position, for the rows [s, (L / r) r); a CUDA-core pass
 * does the sink rows and the last L mod r rows.  The other forms (fp32, bf16 d = 64) gather q, k, v into r
 * virtual heads per (b, h) (class-major), run the prefill of swa_sink_prefill on them and scatter o back.
 *
 *   q, k, v, o, lse : as swa_sink_prefill (pos0 = 0), bf16 with d = 64 or 128 (tensor cores) or fp32.
 *   r       : dilation, 1 <= r <= 65536, B * H * r <= 65535 * 32.
 *   workspace : caller-owned device scratch of swa_sink_prefill_dilated_workspace_size(B, H, L, d, s, r,
 *             dtype) bytes, 256-byte aligned (q, k, v, o of the virtual heads and their lse); not read (may
 *             be NULL with 0 bytes) for bf16 with d = 128 and for r = 1.
 *   Other arguments and errors as swa_sink_prefill.
 */
int swa_sink_prefill_dilated(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                             int64_t L, int d, int w, int s, int r, float scale, void *workspace,
                             size_t workspace_bytes, int dtype, void *stream);
size_t swa_sink_prefill_dilated_workspace_size(int B, int H, int64_t L, int d, int s, int r, int dtype);

/*
 * swa_sink_prefill_chunked_dilated -- swa_sink_prefill_dilated through the per-class rolling caches of
 * swa_sink_decode_step_dilated: the virtual heads (class-major) go through the chunk loop of
 * swa_sink_prefill_chunked, chunk / r class-local rows at a time.  The rows equal swa_sink_prefill_dilated's,
 * and k_cache / v_cache ([r, B, H, w, d], overwritten) end up as L calls of swa_sink_dilated_cache_write
 * leave them, ready for swa_sink_decode_step_dilated at t = L.  workspace as swa_sink_prefill_dilated.
 */
int swa_sink_prefill_chunked_dilated(const void *q, const void *k, const void *v, void *o, float *lse, void *k_cache,
                                     void *v_cache, int B, int H, int64_t L, int d, int w, int s, int r, float scale,
                                     int64_t chunk, void *workspace, size_t workspace_bytes, int dtype, void *stream);

/*
 * swa_sink_prefill_blocksparse -- whole-sequence prefill over the BigBird-style union of the fixed-sparsity page
 * ("滑窗与固定稀疏", Longformer and BigBird sections, eq attn-fixed-bigbird: a local window, global tokens and
 * random key blocks, at block granularity), in causal form with the sinks of the StreamingLLM section.  Row t
 * attends the keys i <= t with
 *     i < s (sink)  or  i >= t - (w - s) + 1 (window)  or  i a global token  or  t a global token
 *     or  i in one of the random key blocks given for t's query block (block index t / block),
 * each key once; with no global token and no random block it is swa_sink_prefill.  Global tokens sit inside the
 * sequence (a global row sees every earlier key; every later row sees a global key).  One pattern serves every
 * (b, h).  Rows run on the tensor cores (per-pair key-tile lists built on the host, per-row column masks); the
 * global rows are recomputed over their whole causal prefix by a CUDA-core pass.
 *
 *   q, k, v, o, lse : as swa_sink_prefill (pos0 = 0); bf16, d = 128.
 *   globals   : HOST int32 array of n_globals distinct positions in [0, L), ascending (NULL if n_globals = 0).
 *   block     : block size of the random key blocks, >= 1.
 *   rand_blocks : HOST int32 [ceil(L / block), r]: the key blocks (index i covers positions i*block ..
 *             i*block + block - 1) attended by each query block, -1 for an unused entry; 0 <= r <= 16.  The random
 *             choice is the caller's: the library draws nothing.
 *   workspace : caller-owned device scratch of swa_sink_prefill_blocksparse_workspace_size(L, n_globals, block, r)
 *             bytes, 256-byte aligned.  The tile lists and the pattern are built on the host into one of two
 *             pinned staging buffers the library keeps per device (allocated on first use, grown as needed) and
 *             uploaded with one cudaMemcpyAsync on `stream`; a buffer is reused only after its copy has completed
 *             (an event wait), so the host may prepare the next call while the device runs this one.  The call
 *             is not capturable into a CUDA graph (the copy's source changes from call to call).
 *   A query pair (256 rows) whose keys need more than 64 tiles of 128 keys is refused with SWA_ERR_UNSUPPORTED.
 *   Other arguments and errors as swa_sink_prefill.
 */
int swa_sink_prefill_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                                 int64_t L, int d, int w, int s, float scale, const int32_t *globals, int n_globals,
                                 int block, const int32_t *rand_blocks, int r, void *workspace, size_t workspace_bytes,
                                 int dtype, void *stream);
size_t swa_sink_prefill_blocksparse_workspace_size(int64_t L, int n_globals, int block, int r);

/*
 * swa_hybrid_prefill -- sliding-window softmax attention with sinks plus a linear-attention branch for the
 * keys that have left the window: the SWA / linear-attention hybrid of the hyper.ai summary of arXiv
 * 2608.28444 (linear-attention section: running state s_t = s_{t-1} + phi(k_t)^T v_t, z_t = z_{t-1} + phi(k_t)^T,
 * Hedgehog feature map phi(x) = (exp(x wf), exp(-x wf))).  Both branches share one normaliser (the LoLCATs
 * reading that summary discusses):
 *     o_t = (sum_{i in K(t)} e^{x_i} v_i + phi(q_t) S_t) / (sum_{i in K(t)} e^{x_i} + phi(q_t) z_t)
 * with x_i = scale q_t.k_i, K(t) the sinks + window of swa_sink_prefill, and S_t = sum phi(k_i)^T v_i,
 * z_t = sum phi(k_i)^T over the keys s <= i <= t - (w - s) that have left the window (the sinks never leave).
 *
 *   q, k, v, o : [B, H, L, d] bf16, d = 128, 16-byte aligned.
 *   wf        : [d, d/2] bf16 row-major, the feature projection (f(x) = x wf); phi has d components.
 *   state_s, state_z : NULL, or fp32 [B, H, d, d] and [B, H, d] (16-byte aligned) that receive S and z after
 *             row L-1 (the state swa_hybrid_decode_step continues from at t = L).
 *   workspace : device scratch of swa_hybrid_prefill_workspace_size(B, H, L, d) bytes, 256-byte aligned
 *             (the SWA branch's lse and the linear branch's per-chunk states).
 * Launches the SWA prefill, the chunk states, their scan, the linear branch with the combination (in place
 * over o) and, with state_s, the final state; asynchronous on `stream`, no allocation, capturable.
 */
int swa_hybrid_prefill(const void *q, const void *k, const void *v, const void *wf, void *o, float *state_s,
                       float *state_z, int B, int H, int64_t L, int d, int w, int s, float scale, void *workspace,
                       size_t workspace_bytes, int dtype, void *stream);
size_t swa_hybrid_prefill_workspace_size(int B, int H, int64_t L, int d);

/*
 * swa_hybrid_decode_step -- one streaming-decode step of the hybrid of swa_hybrid_prefill at position t.
 * In order: the key that leaves the window at this step (position t - (w - s), when >= s) is read from its
 * rolling-cache slot and folded into the state (S += phi(k)^T v, z += phi(k)^T); k_new, v_new (the key and
 * value of position t) are written into that slot (kv_rolling_write's slot rule); the SWA decode step attends
 * the cache; the result is combined with phi(q_t) S_t and phi(q_t) z_t.
 *
 *   q, k_new, v_new : [B, H, d] bf16 (q 16-byte aligned); k_cache, v_cache : [B, H, w, d] bf16, updated.
 *   state_s, state_z : fp32 [B, H, d, d] and [B, H, d], updated in place (zeros before position 0, or the
 *             state swa_hybrid_prefill returned).
 *   wf        : [d, d/2] bf16 as swa_hybrid_prefill.   o : [B, H, d] bf16.
 *   workspace : device scratch of swa_hybrid_decode_workspace_size(B, H, d, w) bytes, 256-byte aligned.
 * bf16, d = 128.  Three launches on `stream`, no allocation, capturable.  Other errors as swa_sink_decode_step.
 */
int swa_hybrid_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                           float *state_s, float *state_z, const void *wf, void *o, int B, int H, int d, int w, int s,
                           int64_t t, float scale, void *workspace, size_t workspace_bytes, int dtype, void *stream);
size_t swa_hybrid_decode_workspace_size(int B, int H, int d, int w);

/*
 * swa_sink_prefill_chunked -- the chunk-based prefill of "滑窗与固定稀疏" (rolling-buffer section):
 * the L positions are processed in chunks of `chunk` rows; chunk c attends the rolling cache as it was
 * before the chunk plus its own keys (swa_sink_prefill with pos0 = c*chunk), then its keys/values are
 * written into the cache (kv_rolling_write).  The result equals a whole-sequence prefill.
 *
 *   q, k, v, o, lse : whole-sequence tensors [B, H, L, d] (lse [B, H, L] or NULL).
 *   k_cache, v_cache : [B, H, w, d] scratch cache owned by the caller; contents on entry are ignored,
 *             on exit it holds the cache state after position L-1 (ready for streaming decode).
 *   chunk   : rows per chunk, >= 1.
 * Asynchronous on `stream`.  The (b, h) rows are independent, so the library may split them into up
 * to 2 groups that walk the chunks on streams of its own (created once per device), forked from and
 * joined back to `stream` with events: the call allocates no device memory and can be captured into a
 * CUDA graph like a single-stream call.
 */
int swa_sink_prefill_chunked(const void *q, const void *k, const void *v, void *o, float *lse,
                             void *k_cache, void *v_cache,
                             int B, int H, int64_t L, int d, int w, int s, float scale,
                             int64_t chunk, int dtype, void *stream);

/*
 * kv_rolling_write -- write the keys/values of positions pos0 .. pos0+n-1 into the rolling cache:
 * position p goes to slot p if p < s, else to slot s + ((p - s) mod m), m = w - s (with s = 0 this is
 * the rolling buffer cache_slot(i) = i mod W of "滑窗与固定稀疏", eq attn-fixed-rolling; the sink
 * block + recent block layout is eq attn-fixed-streaming).  When n > m several positions share a
 * slot; only the last of them is written, so the result equals writing the positions one by one.
 *
 *   k_cache, v_cache : [B, H, w, d], updated in place.
 *   k_new, v_new     : [B, H, n, d].
 *   pos0 >= 0, n >= 0 (n == 0 is a no-op).  Bytes are copied exactly.
 */
int kv_rolling_write(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                     int B, int H, int d, int w, int s, int64_t pos0, int64_t n,
                     int dtype, void *stream);

/*
 * swa_sink_decode_step -- one streaming-decode step for the query at absolute position t, whose key
 * and value are already in the cache (write, then attend).  The valid slots are 0 .. min(t+1, w)-1
 * and they hold exactly K(t) (eq attn-fixed-streaming of "滑窗与固定稀疏": sinks + recent window).
 *
 *   q, o      : [B, H, d].
 *   k_cache, v_cache : [B, H, w, d] as written by kv_rolling_write for positions 0..t.
 *   lse       : optional [B, H] fp32 output (NULL to skip).
 *   workspace : caller-owned device scratch of at least swa_sink_decode_workspace_size(B,H,d,w)
 *               bytes, 256-byte aligned (split-K partial results); may be NULL if that size is 0.
 *   dtype     : SWA_BF16 or SWA_F32; d in {16, 32, 64, 128}.
 */
int swa_sink_decode_step(const void *q, const void *k_cache, const void *v_cache, void *o,
                         float *lse, int B, int H, int d, int w, int s, int64_t t, float scale,
                         void *workspace, size_t workspace_bytes, int dtype, void *stream);

/*
 * swa_sink_decode_step_noalloc -- the same decode step as swa_sink_decode_step, for callers that cannot
 * allocate device memory when they run it (an engine's plugin callback that must not allocate while it
 * enqueues work, a server whose memory pool owns all device memory, a token loop that cannot afford the
 * device synchronisation an allocation may cause).  It takes no workspace: the split-K partial results go
 * to a fixed array of 2 MiB built into the library, which every GPU that loads the library keeps until the
 * process exits.  The pages have no counterpart of this entry point; it is an interface convenience.
 *
 *   Arguments are those of swa_sink_decode_step without workspace/workspace_bytes; same layouts, same
 *   results.  A shape whose split-K scratch (swa_sink_decode_workspace_size) exceeds 2 MiB is refused with
 *   SWA_ERR_UNSUPPORTED and a message; nothing is launched.
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress) with that
 *   device current and keeps it for the life of the process; make that first call before any stream
 *   capture, and do not keep using the library on a device after cudaDeviceReset (the kept address
 *   would then be stale).
 *   Every call uses the same array and overwrites what the previous call left there (nothing in it needs
 *   to start at zero).  Calls that run at the same time on the GPU -- on different streams, or from
 *   several host threads -- overwrite each other's partials: serialise them.
 */
int swa_sink_decode_step_noalloc(const void *q, const void *k_cache, const void *v_cache, void *o,
                                 float *lse, int B, int H, int d, int w, int s, int64_t t, float scale,
                                 int dtype, void *stream);

/* Bytes of workspace swa_sink_decode_step needs for this shape (host-only, no CUDA call). */
size_t swa_sink_decode_workspace_size(int B, int H, int d, int w);

/*
 * swa_sink_dilated_cache_write / swa_sink_decode_step_dilated -- streaming decode over the dilated window
 * with sinks (as swa_sink_prefill_dilated: step t attends the s sinks and t, t - r, ..., t - (m-1) r).
 * The cache is r rolling caches, one per residue class of positions mod r, class-major
 * [r, B, H, w, d]: cache c holds the sinks in slots 0..s-1 and a ring of m slots for the positions p >= s
 * with p = c (mod r).  Per step, write then attend: swa_sink_dilated_cache_write(t) puts the new key/value
 * ([B, H, d]) into cache t mod r (a sink into all r caches), and swa_sink_decode_step_dilated(t) runs the
 * decode of swa_sink_decode_step on cache t mod r: it reads w rows per (b, h), as the plain decode does.
 *
 *   k_cache, v_cache : [r, B, H, w, d], zero-initialised or never read before written.
 *   r       : dilation, 1 <= r <= 65536; r = 1 is the plain rolling cache and decode.
 *   workspace / workspace_bytes : as swa_sink_decode_step (swa_sink_decode_workspace_size(B, H, d, w)).
 *   Other arguments and errors as kv_rolling_write (one position) and swa_sink_decode_step.
 */
int swa_sink_dilated_cache_write(void *k_cache, void *v_cache, const void *k_new, const void *v_new, int B, int H,
                                 int d, int w, int s, int r, int64_t t, int dtype, void *stream);
int swa_sink_decode_step_dilated(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                                 int B, int H, int d, int w, int s, int r, int64_t t, float scale, void *workspace,
                                 size_t workspace_bytes, int dtype, void *stream);

/*
 * swa_sink_decode_step_rope -- swa_sink_decode_step with rotary position embedding applied at the
 * positions the entries have inside the cache, as the StreamingLLM section of "滑窗与固定稀疏" describes:
 * the cache keeps the keys unrotated; at every step its valid entries, sinks first and then the window
 * from oldest to newest, take the consecutive positions 0 .. n-1 (n = min(t + 1, w)), and the query, whose
 * own key is the newest entry, takes position n - 1.  RoPE rotates dimension pair (i, i + d/2) by
 * position * rope_base^(-2i/d) (the half-split form of the Llama-2 / Mistral models; the pages name
 * RoPE without printing it).
 *
 *   q       : [B, H, d] unrotated query at position t; k_cache / v_cache as for swa_sink_decode_step,
 *             with unrotated keys.
 *   rope_base : the RoPE base (10000 for Llama-2), finite and > 1.
 *   workspace : caller-owned device scratch of at least swa_sink_decode_rope_workspace_size(B,H,d,w)
 *             bytes (the split-K partials; 0 bytes when the step runs unsplit, and then it may be NULL),
 *             256-byte aligned.
 *   t < 2^31 and w <= 65536 (SWA_ERR_UNSUPPORTED otherwise).  The per-pair rate theta_i / 2 pi is
 *   evaluated on the host in double and split in two fp32 parts so that whole turns drop out exactly
 *   for every distance inside the cache; sin and cos are fp32.  Other arguments and errors as
 *   swa_sink_decode_step.
 */
int swa_sink_decode_step_rope(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                              int B, int H, int d, int w, int s, int64_t t, float scale, double rope_base,
                              void *workspace, size_t workspace_bytes, int dtype, void *stream);
size_t swa_sink_decode_rope_workspace_size(int B, int H, int d, int w);

/* Human-readable reason of the calling host thread's most recent failure ("" if none). */
const char *swa_last_error_string(void);

/*
 * swa_device_status -- synchronise `stream`, then read and clear the current device's error word.
 * Returns SWA_OK, SWA_ERR_TIMEOUT (a bounded device wait ran out) or SWA_ERR_CUDA.
 */
int swa_device_status(void *stream);

/*
 * swa_selftest_wait_timeout -- diagnostics for the bounded waits: launches one small kernel whose
 * thread waits on an mbarrier that nothing ever arrives on, with a limit of `timeout_ns`
 * nanoseconds (1 .. 10^9).  The wait runs out, the kernel records the timeout and returns; a following
 * swa_device_status() returns SWA_ERR_TIMEOUT.  No GPU fault, trap or hang is involved.
 */
int swa_selftest_wait_timeout(int64_t timeout_ns, void *stream);

/*
 * swa_selftest_umma -- diagnostics for the tensor-core building blocks of the bf16 prefill kernel:
 * one CTA computes C = A * op(B) for 128 x 128 bf16 tiles with TMA loads, tcgen05.mma and a TMEM
 * accumulator read back with tcgen05.ld.
 *   a : [128, 128] bf16 row-major (M x K).
 *   b : mode 0: [128, 128] (N x K), C = A * B^T  (both operands K-major, as in Q K^T)
 *       mode 1: [128, 128] (K x N), C = A * B    (B MN-major, as in P V)
 *       mode 2: as mode 1, but A is staged into shared memory by threads instead of TMA.
 *       mode 3: as mode 1, but A is read by the MMA from tensor memory (staged there with tcgen05.st).
 *   c : [128, 128] fp32 row-major output.
 */
int swa_selftest_umma(const void *a, const void *b, float *c, int mode, void *stream);

/*
 * swa_prefill_tile_plan -- diagnostics (host only, no CUDA call): the key tiles the bf16 prefill kernel
 * walks for the query rows at absolute positions q0..q1 (one or two query tiles of 128 rows, rows
 * q0..q0+127 and q0+128..q1; a work item of the kernel is one of them) of a call starting at pos0.  For tile i, tiles[5i..5i+4] = {source (0 = the
 * call's k/v, 1 = rolling cache), first source row, absolute position of column 0, last valid column,
 * bit mask of the query tiles that use it}; columns c <= last valid column hold position
 * (column-0 position + c).  Writes at most max_tiles entries; returns the tile count or a negative
 * swa_status.
 */
int swa_prefill_tile_plan(int64_t q0, int64_t q1, int64_t pos0, int w, int s, int *tiles, int max_tiles);
/* The same for the RoPE prefills (pos0 = 0, or pos0 >= s in chunked prefill): the sinks form the first
 * tile on their own, the band starts at position s.  s <= 128. */
int swa_prefill_tile_plan_rope(int64_t q0, int64_t q1, int64_t pos0, int w, int s, int *tiles, int max_tiles);
/* The same for the in-place dilated prefill of swa_sink_prefill_dilated (bf16, d = 128; host only, no CUDA
 * call).  swa_prefill_dilated_split writes out[0..3] = {nrows, G, ns, tail0}: the tensor-core pass runs every
 * residue class c over its virtual rows s .. s + nrows - 1 (virtual row s + i is position p0(c) + i r with
 * p0(c) = s + ((c - s) mod r), and is stored when that position is below G r, G = L / r); the CUDA-core pass
 * takes the rows [0, ns) and [tail0, L).  swa_prefill_tile_plan_dilated lists the key tiles of the work item
 * of class cls whose query tile starts at virtual row s + row_start (row_start a multiple of 128 below nrows),
 * as swa_prefill_tile_plan does, in virtual positions: a tile of source 1 holds plain rows (the sinks; column
 * c is row first-row + c), a tile of source 0 holds groups of the class (column c is group first-row + c,
 * position (first-row + c) r + cls; groups from G on are zero-filled by the tensor map).  Errors as
 * swa_prefill_tile_plan. */
int swa_prefill_dilated_split(int64_t L, int s, int r, int64_t *out);
int swa_prefill_tile_plan_dilated(int64_t L, int w, int s, int r, int cls, int64_t row_start, int *tiles,
                                  int max_tiles);
/* The same for swa_sink_prefill_blocksparse (host only, no CUDA call): the key tiles of query pair `pair`
 * (rows 256*pair .. 256*pair + 255) for the pattern (globals, block, rand_blocks, r) of a sequence of L
 * positions.  For tile i, tiles[8i..8i+7] = {absolute position of column 0, last valid column, bit mask of
 * the query tiles that use it, four 32-bit words whose bit c (of word c / 32) marks a column holding a global
 * token, and -1 or, for a packed tile, the absolute position of column 64}.  A packed tile holds two runs of 64
 * keys outside the sinks and the pair's band: columns 0..63 are positions first .. first + 63 and columns
 * 64..127 positions second .. second + 63.  `tiles` holds 8 * max_tiles ints.  Pattern arguments and errors
 * as swa_sink_prefill_blocksparse. */
int swa_prefill_blocksparse_plan(int64_t L, int w, int s, const int32_t *globals, int n_globals, int block,
                                 const int32_t *rand_blocks, int r, int64_t pair, int *tiles, int max_tiles);

#ifdef __cplusplus
}
#endif

#endif /* SWA_SINK_H */
