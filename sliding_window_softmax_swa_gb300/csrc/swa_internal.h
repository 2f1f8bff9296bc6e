// swa_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace swa {

// Record the calling thread's error message (printf-style); returns `code` for convenience.
int fail(int code, const char *fmt, ...);

// Device error word of the current device (nullptr if it could not be resolved; the error is set).
unsigned *device_status_word();
// First-timeout record of the current device (nullptr if it could not be resolved).
unsigned long long *device_timeout_info();

// cuTensorMapEncodeTiled, resolved once through the runtime's driver entry point (no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// A prefill over L rows whose (b, h) blocks lie seq_stride rows apart in q/k/v/o (and lse).
struct PrefillArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;
    const void *k_cache, *v_cache;  // [BH, w, d]; used when pos0 > 0
    int64_t pos0;
    int BH;
    int64_t L;
    int d, w, s;
    float scale;
    int64_t seq_stride;  // rows between consecutive (b, h) blocks (== L for contiguous tensors)
    cudaStream_t stream;
    // RoPE at the positions inside the cache (bf16 tensor-core prefill, d = 128): q and k are the rotated
    // rows (their bf16 hi parts); the sinks get their own key tile, whose scores are read ready-made from
    // rope_ssink (fp32, row (b, h) * seq_stride + local row, rope_sstride floats per row), and the band starts
    // at position s.  Every rotated operand comes as a (hi, lo) bf16 pair whose sum is the fp32 rotation:
    // q_lo, k_lo, and k_cache_lo for the rotated keys of the cache (pos0 > 0)
    bool rope = false;
    const float *rope_ssink = nullptr;
    int rope_sstride = 0;
    const void *q_lo = nullptr, *k_lo = nullptr, *k_cache_lo = nullptr;
};

int launch_prefill_f32(const PrefillArgs &a);
// The bf16 tensor-core prefill: the sub-tile kernel for RoPE (hi/lo operands) and d = 64, the 128-key-tile
// kernel for plain d = 128.
int launch_prefill_bf16_tc(const PrefillArgs &a);
int launch_prefill_bf16_tc_plain(const PrefillArgs &a);
// Block-sparse prefill (bf16, d = 128, pos0 = 0): the host-built tile lists of every 256-row query pair (see
// blocksparse_build_lists) and the random key blocks of every query block, all in device memory.
struct BlockSparseDev {
    const void *tiles, *gmask;
    const int *count;
    const int *rand;
    int block, r;
};
int launch_prefill_bf16_tc_blocksparse(const PrefillArgs &a, const BlockSparseDev &bs);
size_t blocksparse_tile_list_bytes(int64_t L);  // tiles and global-key masks of all query pairs
int blocksparse_build_lists(int64_t L, int w, int s, const int32_t *globals, int n_globals, int block,
                            const int32_t *rand, int r, void *tiles_out, void *gmask_out, int *count_out);
int launch_prefill_bf16_tc_sub(const PrefillArgs &a);
// Dilated-window prefill in place (bf16, d = 128, pos0 = 0, contiguous [BH, L, d]): the tensor-core pass over the
// rows [s, (L / r) r), every residue class a virtual head read through 4-D maps, and the CUDA-core pass over the
// other rows (the sinks t < s and the last L mod r rows).
int launch_prefill_bf16_tc_dilated(const PrefillArgs &a, int r);
int launch_dilated_rows(const PrefillArgs &a, int r);
struct DilatedSplit {
    int64_t nrows;  // virtual rows after the sinks that every class runs over in the tensor-core pass
    int64_t G;      // whole groups of r positions
    int64_t ns;     // the CUDA-core pass: rows [0, ns) and [tail0, L)
    int64_t tail0;
};
DilatedSplit dilated_split(int64_t L, int s, int r);
// the key tiles of one dilated-mode work item (as prefill_tile_plan; source 0 rows are groups of the class)
int prefill_tile_plan_dilated(int64_t L, int w, int s, int r, int cls, int row_start, int *out, int max_tiles);
// Layout passes of the dilated-window prefill: rows of one virtual head (sinks + one residue class), the
// gather of q, k, v into the virtual heads [BH * r, Lv, d] and the scatter of o (and lse) back.
int64_t dilated_rows(int64_t L, int s, int r);
int launch_dilate_gather(const void *q, const void *k, const void *v, void *qv, void *kv, void *vv, int BH, int64_t L,
                         int d, int esize, int s, int r, cudaStream_t stream);
int launch_dilate_scatter(const void *ov, const float *lsev, void *o, float *lse, int BH, int64_t L, int d, int esize,
                          int s, int r, cudaStream_t stream);
// The rotation pass of RoPE prefill: for the rows of [BH, L, d] (d = 128, bf16) qr = R(t) q and kr = R(t) k, each
// written as a bf16 (hi, lo) pair with hi + lo the fp32 rotation, and the sink scores
// ssink[t][i] = (R(min(t, w - 1)) q_t) . (R(i) k_i), i < s, in fp32 (sstride floats per row); ks holds the
// rotated sink keys (fp32 [BH, s, d]) the scores are made from.
struct RopeParts {
    void *qr, *qr_lo, *kr, *kr_lo;
    float *ssink, *ks;
    int sstride;
};
int rope_sink_stride(int s);
size_t rope_prefill_workspace_bytes(int BH, int64_t L, int d, int s);
RopeParts rope_parts(void *workspace, int BH, int64_t L, int d, int s);
int launch_rope_prep(const void *q, const void *k, const RopeParts &out, int BH, int64_t L, int d, int w, int s,
                     double base, cudaStream_t stream);

// Rolling-cache write of positions pos0..pos0+n-1; source rows of (b, h) start at bh*src_stride.  With
// v_new == nullptr only the keys are written.
int launch_kv_write(void *k_cache, void *v_cache, const void *k_new, const void *v_new, int BH, int d, int w,
                    int s, int64_t pos0, int64_t n, int64_t src_stride, int esize, cudaStream_t stream);
// The same rows into nclass caches of [BH, w, d] that lie one after the other (one launch).
int launch_kv_write_classes(void *k_cache, void *v_cache, const void *k_new, const void *v_new, int BH, int d, int w,
                            int s, int64_t pos0, int64_t n, int64_t src_stride, int esize, int nclass,
                            cudaStream_t stream);

struct DecodeArgs {
    const void *q, *k_cache, *v_cache;
    void *o;
    float *lse;
    int BH, d, w, s;
    int64_t t;
    float scale;
    void *workspace;
    size_t workspace_bytes;
    int esize;  // 2 = bf16, 4 = fp32
    cudaStream_t stream;
};
int decode_num_splits(int BH, int nvalid);
size_t decode_workspace_bytes(int BH, int d, int w);
int launch_decode(const DecodeArgs &a);
// The same decode with rotary embedding at positions inside the cache; the workspace also holds the
// d/2 per-pair angle steps (in turns, split into an exactly-multipliable high part and a remainder).
size_t decode_rope_workspace_bytes(int BH, int d, int w);
int launch_decode_rope(const DecodeArgs &a, double base);
// The same decode with its split-K scratch in a built-in device array (no workspace argument).
size_t decode_noalloc_scratch_bytes();
int launch_decode_noalloc(DecodeArgs a);

// Key walks of the prefill kernels (host): the plain kernel's 128-key tiles, or (rope) the sub-tile kernel's
// 64-key sub-tiles.
int prefill_tile_plan(int q0, int q1, int pos0, int w, int s, int rope, int *out, int max_tiles);
int prefill_tile_plan_sub(int q0, int q1, int pos0, int w, int s, int rope, int *out, int max_tiles);
int launch_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream);
int launch_selftest_umma(const void *a, const void *b, float *c, int mode, cudaStream_t stream);

}  // namespace swa
