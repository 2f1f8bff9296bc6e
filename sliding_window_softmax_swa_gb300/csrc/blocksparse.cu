// blocksparse.cu -- prefill over the BigBird-style union of the fixed-sparsity page ("滑窗与固定稀疏", Longformer
// and BigBird sections, eq attn-fixed-bigbird: local window + global tokens + random key blocks, block-level),
// in causal form with the sinks of the StreamingLLM section.  Row t attends the keys i <= t that are a sink
// (i < s), in its window (i >= t - m + 1), a global token, or in one of the random key blocks given for its query
// block; a global row (t itself a global token) attends every key i <= t.
//
// The tensor-core prefill does every row in block-sparse mode: the host builds the key-tile list of every
// 256-row query pair (band + sinks + global keys + random blocks, merged into disjoint runs, cut into tiles of
// up to 128 keys, with the global-key columns of each tile), and the kernel's per-row column masks add the
// global keys and the row's random blocks to its band and sinks.  The global rows, whose key set is the whole
// causal prefix, are then recomputed by full_rows_kernel and overwrite what the tiled pass wrote for them (a
// global row t < w needs no second pass: its sinks and window already cover [0, t]).
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {

// One row of softmax attention over all keys 0..t of its (b, h): one CTA of 128 threads per (row, (b, h)),
// thread c owning output column c.  Keys go in chunks of 128, one key per thread for the score (fp32 dot
// product of the bf16 row with q), an online softmax across chunks, P.V accumulated in fp32.
__global__ void __launch_bounds__(128) full_rows_kernel(const __nv_bfloat16 *__restrict__ q,
                                                        const __nv_bfloat16 *__restrict__ k,
                                                        const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *o,
                                                        float *lse, const int *__restrict__ rows, int64_t L, float sl2) {
    constexpr int D = 128;
    __shared__ float qs[D];
    __shared__ float ps[128];
    __shared__ float red[4];
    const int t = rows[blockIdx.x];
    const int64_t bh = blockIdx.y;
    const int c = threadIdx.x, lane = c & 31, wid = c >> 5;
    qs[c] = __bfloat162float(q[(bh * L + t) * D + c]);
    __syncthreads();
    float m = -INFINITY, l = 0.f, acc = 0.f;
    for (int c0 = 0; c0 <= t; c0 += 128) {
        const int key = c0 + c;
        float sc = -INFINITY;
        if (key <= t) {
            const uint4 *kr = reinterpret_cast<const uint4 *>(k + (bh * L + key) * D);
            float dot = 0.f;
#pragma unroll 4
            for (int i = 0; i < D / 8; ++i) {
                const uint4 u = __ldg(kr + i);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    dot = fmaf(__uint_as_float(w4[h] << 16), qs[8 * i + 2 * h], dot);
                    dot = fmaf(__uint_as_float(w4[h] & 0xFFFF0000u), qs[8 * i + 2 * h + 1], dot);
                }
            }
            sc = dot * sl2;
        }
        float mx = sc;
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        if (lane == 0) red[wid] = mx;
        __syncthreads();
        mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
        __syncthreads();
        const float mnew = fmaxf(m, mx);  // finite: key 0 <= t is always valid
        const float alpha = exp2f(m - mnew);
        const float p = (key <= t) ? exp2f(sc - mnew) : 0.f;
        ps[c] = p;
        float sum = p;
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
        if (lane == 0) red[wid] = sum;
        __syncthreads();
        l = l * alpha + ((red[0] + red[1]) + (red[2] + red[3]));
        acc *= alpha;
        m = mnew;
        const int nk = (t - c0 + 1) < 128 ? (t - c0 + 1) : 128;
        const __nv_bfloat16 *vr = v + (bh * L + c0) * D + c;
        for (int j = 0; j < nk; ++j) acc = fmaf(ps[j], __bfloat162float(vr[static_cast<int64_t>(j) * D]), acc);
        __syncthreads();
    }
    o[(bh * L + t) * D + c] = __float2bfloat16_rn(acc / l);
    if (lse && c == 0) lse[bh * L + t] = (m + log2f(l)) * 0.69314718055994531f;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace swa

using namespace swa;

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The host-side checks of a block-sparse pattern, shared by the prefill and the plan diagnostics.
static int check_pattern(int64_t L, int w, int s, const int32_t *globals, int n_globals, int block,
                         const int32_t *rand_blocks, int r) {
    if (w < 1 || s < 0 || s >= w) return fail(SWA_ERR_INVALID, "need 0 <= s < w (s=%d, w=%d)", s, w);
    if (L < 0 || L >= (int64_t(1) << 31)) return fail(SWA_ERR_INVALID, "L=%lld out of range", (long long)L);
    if (block < 1 || r < 0 || r > 16 || n_globals < 0)
        return fail(SWA_ERR_INVALID, "need block >= 1, 0 <= r <= 16, n_globals >= 0");
    if (n_globals > 0 && !globals) return fail(SWA_ERR_INVALID, "globals must be non-null when n_globals > 0");
    for (int i = 0; i < n_globals; ++i)
        if (globals[i] < 0 || globals[i] >= L || (i > 0 && globals[i] <= globals[i - 1]))
            return fail(SWA_ERR_INVALID, "globals must be distinct positions in [0, L), ascending");
    const int64_t kblocks = ceil_div(L, block);
    if (r > 0 && !rand_blocks) return fail(SWA_ERR_INVALID, "rand_blocks must be non-null when r > 0");
    for (int64_t i = 0; i < kblocks * r; ++i)
        if (rand_blocks[i] < -1 || rand_blocks[i] >= kblocks)
            return fail(SWA_ERR_INVALID, "rand_blocks entries must be -1 or a key block in [0, %lld)", (long long)kblocks);
    return SWA_OK;
}

// The tile lists of every query pair, built on the host: records of 16 bytes (row0, pbase, chi | flags, row1)
// for all pairs, then their 16-byte global-key column masks.
struct HostLists {
    static constexpr size_t kRecord = 16;
    static constexpr int kPacked = 8;  // flags bit: two 64-key blocks, columns 64..127 from row1
    std::vector<unsigned char> bytes;
    std::vector<int> count;
    size_t tiles_bytes = 0;
    int per_pair = 0;
    int build(int64_t L, int w, int s, const int32_t *globals, int n_globals, int block, const int32_t *rand_blocks,
              int r) {
        const int64_t pairs = ceil_div(L, 256);
        const size_t list_bytes = blocksparse_tile_list_bytes(L);
        tiles_bytes = list_bytes / (kRecord + 16) * kRecord;
        per_pair = static_cast<int>(tiles_bytes / kRecord / pairs);
        bytes.assign(list_bytes, 0);
        count.assign(static_cast<size_t>(pairs), 0);
        return blocksparse_build_lists(L, w, s, globals, n_globals, block, rand_blocks, r, bytes.data(),
                                       bytes.data() + tiles_bytes, count.data());
    }
};

// Pinned staging of what a call uploads (its tile lists, counts, random blocks and global positions, in the
// workspace's layout): two slots per device, used in turn.  A slot is written again only once the copy that read
// it has completed (its event), so the host builds a call's lists while the device still runs the previous call,
// and the whole upload is one asynchronous copy.
struct StageSlot {
    void *host = nullptr;
    size_t cap = 0;
    cudaEvent_t done = nullptr;
    bool pending = false;
};
constexpr int kStageDevices = 64;
static std::mutex g_stage_mu;
static StageSlot g_stage[kStageDevices][2];
static unsigned g_stage_turn[kStageDevices];

// Takes the next slot of the current device with room for `bytes` (waiting for its previous copy), or null with
// the error set.  The caller holds g_stage_mu until it has recorded the slot's event.
static StageSlot *stage_slot(size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kStageDevices) {
        fail(SWA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    StageSlot &sl = g_stage[dev][g_stage_turn[dev]++ & 1];
    if (!sl.done && (e = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming)) != cudaSuccess) {
        sl.done = nullptr;
        fail(SWA_ERR_CUDA, "staging event: %s", cudaGetErrorString(e));
        return nullptr;
    }
    if (sl.pending) {
        if ((e = cudaEventSynchronize(sl.done)) != cudaSuccess) {
            fail(SWA_ERR_CUDA, "staging wait: %s", cudaGetErrorString(e));
            return nullptr;
        }
        sl.pending = false;
    }
    if (sl.cap < bytes) {
        if (sl.host) cudaFreeHost(sl.host);
        sl.host = nullptr;
        sl.cap = 0;
        const size_t cap = bytes + bytes / 4;
        if ((e = cudaHostAlloc(&sl.host, cap, cudaHostAllocDefault)) != cudaSuccess) {
            sl.host = nullptr;
            fail(SWA_ERR_CUDA, "pinned staging of %zu bytes: %s", cap, cudaGetErrorString(e));
            return nullptr;
        }
        sl.cap = cap;
    }
    return &sl;
}

extern "C" int swa_prefill_blocksparse_plan(int64_t L, int w, int s, const int32_t *globals, int n_globals,
                                            int block, const int32_t *rand_blocks, int r, int64_t pair, int *tiles,
                                            int max_tiles) {
    fail(SWA_OK, "%s", "");
    if (int rc = check_pattern(L, w, s, globals, n_globals, block, rand_blocks, r)) return rc;
    const int64_t pairs = ceil_div(L, 256);
    if (pair < 0 || pair >= pairs)
        return fail(SWA_ERR_INVALID, "pair %lld outside [0, %lld)", (long long)pair, (long long)pairs);
    if (!tiles || max_tiles < 0) return fail(SWA_ERR_INVALID, "tiles must be non-null");
    HostLists hl;
    if (int rc = hl.build(L, w, s, globals, n_globals, block, rand_blocks, r)) return rc;
    const int n = hl.count[static_cast<size_t>(pair)];
    for (int i = 0; i < n && i < max_tiles; ++i) {
        const size_t idx = static_cast<size_t>(pair) * hl.per_pair + i;
        int32_t rec[4];  // row0, pbase, chi (low half) | flags (high half), row1
        std::memcpy(rec, hl.bytes.data() + idx * HostLists::kRecord, HostLists::kRecord);
        uint32_t gm[4];
        std::memcpy(gm, hl.bytes.data() + hl.tiles_bytes + idx * 16, 16);
        const int flags = static_cast<int16_t>(static_cast<uint32_t>(rec[2]) >> 16);
        int *out = tiles + 8 * static_cast<int64_t>(i);
        out[0] = rec[1];
        out[1] = static_cast<int16_t>(rec[2] & 0xFFFF);
        out[2] = (flags >> 1) & 3;
        for (int k = 0; k < 4; ++k) out[3 + k] = static_cast<int>(gm[k]);
        out[7] = (flags & HostLists::kPacked) ? rec[3] : -1;
    }
    return n;
}

extern "C" size_t swa_sink_prefill_blocksparse_workspace_size(int64_t L, int n_globals, int block, int r) {
    if (L < 1 || n_globals < 0 || block < 1 || r < 0) return 0;
    const int64_t pairs = ceil_div(L, 256), qblocks = ceil_div(L, block);
    return align256(blocksparse_tile_list_bytes(L)) + align256(static_cast<size_t>(pairs) * 4) +
           align256(static_cast<size_t>(qblocks) * r * 4 + 4) + align256(static_cast<size_t>(n_globals) * 4 + 4);
}

extern "C" int swa_sink_prefill_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                                            int H, int64_t L, int d, int w, int s, float scale, const int32_t *globals,
                                            int n_globals, int block, const int32_t *rand_blocks, int r,
                                            void *workspace, size_t workspace_bytes, int dtype, void *stream) {
    fail(SWA_OK, "%s", "");  // clear the thread's error text
    if (dtype != SWA_BF16 || d != 128) return fail(SWA_ERR_UNSUPPORTED, "block-sparse prefill runs on bf16 with d = 128");
    if (B < 1 || H < 1 || static_cast<int64_t>(B) * H > 65535) return fail(SWA_ERR_INVALID, "need 1 <= B*H <= 65535");
    if (!(scale == scale) || scale <= 0.f || scale > 1e30f)
        return fail(SWA_ERR_INVALID, "scale must be a positive finite number");
    if (int rc = check_pattern(L, w, s, globals, n_globals, block, rand_blocks, r)) return rc;
    if (L == 0) return SWA_OK;
    if (!q || !k || !v || !o) return fail(SWA_ERR_INVALID, "q, k, v and o must be non-null");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(o)) & 15u)
        return fail(SWA_ERR_INVALID, "q, k, v and o must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SWA_ERR_INVALID, "lse must be 4-byte aligned");
    const int64_t qblocks = ceil_div(L, block);
    const size_t need = swa_sink_prefill_blocksparse_workspace_size(L, n_globals, block, r);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");

    // the tile lists, built on the host into a pinned slot laid out as the workspace, then one copy:
    // [tiles | global-column words] [counts] [random blocks] [global positions], each part 256-byte aligned
    const int64_t pairs = ceil_div(L, 256);
    const size_t list_bytes = blocksparse_tile_list_bytes(L);
    const size_t tiles_bytes = list_bytes / (HostLists::kRecord + 16) * HostLists::kRecord;
    const size_t off_count = align256(list_bytes);
    const size_t off_rand = off_count + align256(static_cast<size_t>(pairs) * 4);
    const size_t off_glob = off_rand + align256(static_cast<size_t>(qblocks) * r * 4 + 4);
    const size_t upload = off_glob + static_cast<size_t>(n_globals) * 4;
    char *ws = static_cast<char *>(workspace);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    {
        std::lock_guard<std::mutex> lk(g_stage_mu);
        StageSlot *sl = stage_slot(upload);
        if (!sl) return SWA_ERR_CUDA;
        char *h = static_cast<char *>(sl->host);
        if (int rc = blocksparse_build_lists(L, w, s, globals, n_globals, block, rand_blocks, r, h, h + tiles_bytes,
                                             reinterpret_cast<int *>(h + off_count)))
            return rc;
        if (r > 0) std::memcpy(h + off_rand, rand_blocks, static_cast<size_t>(qblocks) * r * 4);
        if (n_globals > 0) std::memcpy(h + off_glob, globals, static_cast<size_t>(n_globals) * 4);
        cudaError_t e = cudaMemcpyAsync(ws, h, upload, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaEventRecord(sl->done, st);
        if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "block-sparse pattern upload: %s", cudaGetErrorString(e));
        sl->pending = true;
    }
    char *d_lists = ws;
    int *d_count = reinterpret_cast<int *>(ws + off_count);
    int *d_rand = reinterpret_cast<int *>(ws + off_rand);
    int *d_glob = reinterpret_cast<int *>(ws + off_glob);
    PrefillArgs a{q, k, v, o, lse, nullptr, nullptr, 0, B * H, L, d, w, s, scale, L, st};
    const BlockSparseDev bs{d_lists, d_lists + tiles_bytes, d_count, d_rand, block, r};
    if (int rc = launch_prefill_bf16_tc_blocksparse(a, bs)) return rc;
    // The global rows attend their whole causal prefix.  For a global row t < w that prefix is already its sinks
    // and window ([0, s) and [t - m + 1, t] cover [0, t]), which the tiled pass computed: only the rows t >= w
    // are recomputed.
    const int n_near = static_cast<int>(std::lower_bound(globals, globals + n_globals, w) - globals);
    if (n_globals > n_near) {
        full_rows_kernel<<<dim3(static_cast<unsigned>(n_globals - n_near), static_cast<unsigned>(B * H)), 128, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
            static_cast<const __nv_bfloat16 *>(v), static_cast<__nv_bfloat16 *>(o), lse, d_glob + n_near, L,
            scale * 1.4426950408889634f);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "global rows launch: %s", cudaGetErrorString(e));
    }
    return SWA_OK;
}
