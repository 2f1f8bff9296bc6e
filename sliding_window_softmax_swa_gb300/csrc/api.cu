// api.cu -- the C ABI of include/swa_sink.h: argument validation, dispatch to the kernels' launchers,
// the per-device error word, the thread-local error string and the tensor-map encoder lookup.
#include <stdarg.h>
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {

// One error word per device.  Kernels receive its address; swa_device_status() reads and clears it.
// (with where the first bounded wait of the device ran out, cleared together with the word)
__device__ DeviceStatus g_swa_status;

static thread_local char t_err[512];

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
    return code;
}

unsigned *device_status_word() {
    static std::mutex mu;
    static unsigned *ptrs[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        fail(SWA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_swa_status);
        if (e != cudaSuccess) {
            fail(SWA_ERR_CUDA, "cudaGetSymbolAddress(status word): %s", cudaGetErrorString(e));
            return nullptr;
        }
        ptrs[dev] = static_cast<unsigned *>(p);
    }
    return ptrs[dev];
}

unsigned long long *device_timeout_info() {
    static std::mutex mu;
    static unsigned long long *ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_swa_status) != cudaSuccess) return nullptr;
        ptrs[dev] = &static_cast<DeviceStatus *>(p)->info;
    }
    return ptrs[dev];
}

int launch_prefill_bf16_tc(const PrefillArgs &a) {
    if (a.rope || a.d == 64) return launch_prefill_bf16_tc_sub(a);
    return launch_prefill_bf16_tc_plain(a);
}

EncodeTiledFn encode_tiled_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace swa

using namespace swa;

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int esize_of(int dtype) { return dtype == SWA_BF16 ? 2 : dtype == SWA_F32 ? 4 : 0; }

static int check_common(int B, int H, int d, int w, int s, int dtype) {
    if (esize_of(dtype) == 0) return fail(SWA_ERR_INVALID, "dtype %d is neither SWA_BF16 nor SWA_F32", dtype);
    if (B < 1 || H < 1) return fail(SWA_ERR_INVALID, "B=%d, H=%d must be >= 1", B, H);
    if ((int64_t)B * H > 65535 * 32)
        return fail(SWA_ERR_UNSUPPORTED, "B*H=%lld exceeds the supported %d", (long long)B * H, 65535 * 32);
    if (w < 1) return fail(SWA_ERR_INVALID, "w=%d must be >= 1", w);
    if (s < 0 || s >= w) return fail(SWA_ERR_INVALID, "need 0 <= s < w (s=%d, w=%d)", s, w);
    if (!(d == 16 || d == 32 || d == 64 || d == 128))
        return fail(SWA_ERR_UNSUPPORTED, "d=%d not in {16, 32, 64, 128}", d);
    return SWA_OK;
}

extern "C" const char *swa_last_error_string(void) { return t_err; }

extern "C" int swa_device_status(void *stream) {
    t_err[0] = 0;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    unsigned word = 0;
    e = cudaMemcpyFromSymbol(&word, g_swa_status, sizeof(word), offsetof(DeviceStatus, word));
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
    if (word != 0) {
        unsigned zero = 0;
        unsigned long long info = 0, zero64 = 0;
        cudaMemcpyFromSymbol(&info, g_swa_status, sizeof(info), offsetof(DeviceStatus, info));
        cudaMemcpyToSymbol(g_swa_status, &zero, sizeof(zero), offsetof(DeviceStatus, word));
        cudaMemcpyToSymbol(g_swa_status, &zero64, sizeof(zero64), offsetof(DeviceStatus, info));
        if (word & kDevTimeout)
            return fail(SWA_ERR_TIMEOUT,
                        "a bounded device wait ran out (error word 0x%08x; first: site %u, tag %u, warp %u, "
                        "block (%u, %u))",
                        word, unsigned(info & 0xFF), unsigned((info >> 8) & 0xFFF), unsigned((info >> 20) & 0xFFF),
                        unsigned((info >> 32) & 0xFFFF), unsigned((info >> 48) & 0xFFFF));
        return fail(SWA_ERR_CUDA, "device consistency check failed (error word 0x%08x)", word);
    }
    return SWA_OK;
}

static int prefill_impl(const void *q, const void *k, const void *v, void *o, float *lse, const void *k_cache,
                        const void *v_cache, int64_t pos0, int B, int H, int64_t L, int d, int w, int s, float scale,
                        int dtype, int64_t seq_stride, cudaStream_t stream) {
    if (L == 0) return SWA_OK;
    PrefillArgs a{q, k, v, o, lse, k_cache, v_cache, pos0, B * H, L, d, w, s, scale, seq_stride, stream};
    if (dtype == SWA_BF16) {
        if (d != 64 && d != 128) return fail(SWA_ERR_UNSUPPORTED, "bf16 prefill needs d = 64 or 128 (got %d)", d);
        return launch_prefill_bf16_tc(a);
    }
    return launch_prefill_f32(a);
}

static int check_prefill(const void *q, const void *k, const void *v, const void *o, const float *lse,
                         int64_t pos0, int B, int H, int64_t L, int d, int w, int s, float scale, int dtype) {
    int rc = check_common(B, H, d, w, s, dtype);
    if (rc) return rc;
    if (L < 0) return fail(SWA_ERR_INVALID, "L=%lld must be >= 0", (long long)L);
    if (pos0 < 0) return fail(SWA_ERR_INVALID, "pos0=%lld must be >= 0", (long long)pos0);
    if (pos0 + L >= (int64_t(1) << 31))
        return fail(SWA_ERR_UNSUPPORTED, "pos0 + L = %lld must be < 2^31", (long long)(pos0 + L));
    if (!(scale == scale) || scale <= 0.f || scale > 1e30f)
        return fail(SWA_ERR_INVALID, "scale must be a positive finite number");
    if (L == 0) return SWA_OK;
    if (!q || !k || !v || !o) return fail(SWA_ERR_INVALID, "q, k, v and o must be non-null");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return fail(SWA_ERR_INVALID, "q, k, v and o must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SWA_ERR_INVALID, "lse must be 4-byte aligned");
    return SWA_OK;
}

extern "C" int swa_sink_prefill(const void *q, const void *k, const void *v, void *o, float *lse,
                                const void *k_cache, const void *v_cache, int64_t pos0, int B, int H, int64_t L,
                                int d, int w, int s, float scale, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_prefill(q, k, v, o, lse, pos0, B, H, L, d, w, s, scale, dtype);
    if (rc) return rc;
    if (L == 0) return SWA_OK;
    if (pos0 > 0) {
        if (!k_cache || !v_cache) return fail(SWA_ERR_INVALID, "pos0 > 0 needs k_cache and v_cache");
        if (!aligned16(k_cache) || !aligned16(v_cache))
            return fail(SWA_ERR_INVALID, "k_cache and v_cache must be 16-byte aligned");
    }
    return prefill_impl(q, k, v, o, lse, k_cache, v_cache, pos0, B, H, L, d, w, s, scale, dtype, L,
                        static_cast<cudaStream_t>(stream));
}

// Streams and events of the chunked prefill's row groups: created once per device and kept (no
// allocation of device memory; a chunked prefill call only records and waits on events).
constexpr int kChunkGroups = 2;
constexpr int kChunkGroupMinRows = 8;  // (b, h) rows per group at least
struct ChunkStreams {
    cudaStream_t stream[kChunkGroups];
    cudaEvent_t fork;
    cudaEvent_t join[kChunkGroups];
};
static ChunkStreams *chunk_streams() {
    static std::mutex mu;
    static ChunkStreams *per_dev[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!per_dev[dev]) {
        ChunkStreams *c = new ChunkStreams();
        bool ok = cudaEventCreateWithFlags(&c->fork, cudaEventDisableTiming) == cudaSuccess;
        for (int g = 0; ok && g < kChunkGroups; ++g) {
            ok = cudaStreamCreateWithFlags(&c->stream[g], cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&c->join[g], cudaEventDisableTiming) == cudaSuccess;
        }
        if (!ok) {  // fall back to one stream (the caller's); nothing is released on this rare path
            delete c;
            return nullptr;
        }
        per_dev[dev] = c;
    }
    return per_dev[dev];
}

// RoPE mode of the chunk loop: q and k passed to it are the rotated rows (hi parts); these are the rest.
struct ChunkRope {
    const void *q_lo;                  // [BH, L, d] lo parts of the rotated query rows
    const float *ssink;                // [BH, L, sstride] the sink scores of every row (fp32)
    int sstride;
    const void *k_lo;                  // [BH, L, d] lo parts of the rotated keys
    const void *k_raw;                 // [BH, L, d] unrotated keys: they go into the caller's cache
    void *kc_rot, *kc_rot_lo;          // [BH, w, d] scratch cache of rotated keys (hi, lo), read by the
                                       // prefill for positions < pos0
};

// The chunk loop of chunked prefill (validated arguments, L > 0): L rows per (b, h), consecutive (b, h)
// blocks of q/k/v/o (and lse) `stride` rows apart.
static int chunk_loop(const void *q, const void *k, const void *v, void *o, float *lse, void *k_cache, void *v_cache,
                      int B, int H, int64_t L, int64_t stride, int d, int w, int s, float scale, int64_t chunk,
                      int dtype, cudaStream_t st, const ChunkRope *rp) {
    const int es = esize_of(dtype);
    const size_t row_bytes = static_cast<size_t>(d) * es;
    int rc = SWA_OK;
    // The (b, h) rows are independent; only the chunks of one row depend on each other, through its
    // cache.  The rows are split into groups, each walking all chunks on its own stream, so that one
    // group's next chunk fills the SMs that another group's chunk leaves idle at its end (a chunk of one
    // group alone is a few waves of work items, the last one partly empty).
    const int BH = B * H;
    ChunkStreams *cs = chunk_streams();
    const int groups = (cs && BH >= 2 * kChunkGroupMinRows) ? (BH / kChunkGroupMinRows < kChunkGroups ? BH / kChunkGroupMinRows : kChunkGroups) : 1;
    if (groups > 1) {
        cudaError_t e = cudaEventRecord(cs->fork, st);
        for (int g = 0; e == cudaSuccess && g < groups; ++g) e = cudaStreamWaitEvent(cs->stream[g], cs->fork, 0);
        if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "chunked prefill fork: %s", cudaGetErrorString(e));
    }
    for (int g = 0; g < groups; ++g) {
        const int r0 = static_cast<int>(static_cast<int64_t>(BH) * g / groups);
        const int r1 = static_cast<int>(static_cast<int64_t>(BH) * (g + 1) / groups);
        cudaStream_t gs = groups > 1 ? cs->stream[g] : st;
        const size_t seq_off = static_cast<size_t>(r0) * static_cast<size_t>(stride) * row_bytes;  // q, k, v, o
        const size_t cache_off = static_cast<size_t>(r0) * static_cast<size_t>(w) * row_bytes;
        void *kcg = static_cast<char *>(k_cache) + cache_off;
        void *vcg = static_cast<char *>(v_cache) + cache_off;
        void *krg = rp ? static_cast<char *>(rp->kc_rot) + cache_off : nullptr;
        void *krg_lo = rp ? static_cast<char *>(rp->kc_rot_lo) + cache_off : nullptr;
        for (int64_t c0 = 0; c0 < L; c0 += chunk) {
            const int64_t n = (L - c0 < chunk) ? (L - c0) : chunk;
            const size_t off = seq_off + static_cast<size_t>(c0) * row_bytes;
            const char *qc = static_cast<const char *>(q) + off;
            const char *kc = static_cast<const char *>(k) + off;
            const char *vc = static_cast<const char *>(v) + off;
            char *oc = static_cast<char *>(o) + off;
            float *lc = lse ? lse + static_cast<int64_t>(r0) * stride + c0 : nullptr;
            if (!rp) {
                // prefill_impl treats its B as the number of (b, h) rows when H = 1
                rc = prefill_impl(qc, kc, vc, oc, lc, kcg, vcg, c0, r1 - r0, 1, n, d, w, s, scale, dtype, stride, gs);
                if (rc) return rc;
                rc = launch_kv_write(kcg, vcg, kc, vc, r1 - r0, d, w, s, c0, n, stride, es, gs);
                if (rc) return rc;
            } else {
                // rotated rows against the rotated cache; then the chunk's rotated keys (hi and lo) into the
                // scratch caches, its unrotated keys and its values into the caller's
                PrefillArgs a{qc, kc, vc, oc, lc, krg, vcg, c0, r1 - r0, n, d, w, s, scale, stride, gs};
                a.rope = true;
                a.rope_ssink = rp->ssink + (static_cast<size_t>(r0) * static_cast<size_t>(stride) + static_cast<size_t>(c0)) *
                                               static_cast<size_t>(rp->sstride);
                a.rope_sstride = rp->sstride;
                a.q_lo = static_cast<const char *>(rp->q_lo) + off;
                a.k_lo = static_cast<const char *>(rp->k_lo) + off;
                a.k_cache_lo = krg_lo;
                rc = launch_prefill_bf16_tc(a);
                if (rc) return rc;
                rc = launch_kv_write(krg, krg_lo, kc, static_cast<const char *>(rp->k_lo) + off, r1 - r0, d, w, s, c0, n,
                                     stride, es, gs);
                if (rc) return rc;
                rc = launch_kv_write(kcg, vcg, static_cast<const char *>(rp->k_raw) + off, vc, r1 - r0, d, w, s, c0,
                                     n, stride, es, gs);
                if (rc) return rc;
            }
        }
    }
    if (groups > 1) {
        for (int g = 0; g < groups; ++g) {
            cudaError_t e = cudaEventRecord(cs->join[g], cs->stream[g]);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(st, cs->join[g], 0);
            if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "chunked prefill join: %s", cudaGetErrorString(e));
        }
    }
    return SWA_OK;
}

extern "C" int swa_sink_prefill_chunked(const void *q, const void *k, const void *v, void *o, float *lse,
                                        void *k_cache, void *v_cache, int B, int H, int64_t L, int d, int w, int s,
                                        float scale, int64_t chunk, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_prefill(q, k, v, o, lse, 0, B, H, L, d, w, s, scale, dtype);
    if (rc) return rc;
    if (chunk < 1) return fail(SWA_ERR_INVALID, "chunk=%lld must be >= 1", (long long)chunk);
    if (L == 0) return SWA_OK;
    if (!k_cache || !v_cache) return fail(SWA_ERR_INVALID, "k_cache and v_cache must be non-null");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(SWA_ERR_INVALID, "k_cache and v_cache must be 16-byte aligned");
    return chunk_loop(q, k, v, o, lse, k_cache, v_cache, B, H, L, L, d, w, s, scale, chunk, dtype,
                      static_cast<cudaStream_t>(stream), nullptr);
}

extern "C" size_t swa_sink_prefill_chunked_rope_workspace_size(int B, int H, int64_t L, int d, int w, int s) {
    if (B < 1 || H < 1 || L < 0 || d != 128 || w < 1 || s < 0 || s > 128) return 0;
    return rope_prefill_workspace_bytes(B * H, L, d, s) + 2 * static_cast<size_t>(B) * H * w * d * 2;
}

extern "C" int swa_sink_prefill_chunked_rope(const void *q, const void *k, const void *v, void *o, float *lse,
                                             void *k_cache, void *v_cache, int B, int H, int64_t L, int d, int w,
                                             int s, float scale, int64_t chunk, double rope_base, void *workspace,
                                             size_t workspace_bytes, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_prefill(q, k, v, o, lse, 0, B, H, L, d, w, s, scale, dtype);
    if (rc) return rc;
    if (dtype != SWA_BF16 || d != 128) return fail(SWA_ERR_UNSUPPORTED, "RoPE prefill runs on bf16 with d = 128");
    if (s > 128) return fail(SWA_ERR_UNSUPPORTED, "RoPE prefill needs s <= 128 (s=%d)", s);
    if (chunk < 1 || chunk < s)
        return fail(SWA_ERR_INVALID, "chunk=%lld must be >= max(1, s) with RoPE", (long long)chunk);
    if (!(rope_base == rope_base) || rope_base <= 1.0 || rope_base > 1e30)
        return fail(SWA_ERR_INVALID, "rope_base must be a finite number > 1");
    const size_t need = swa_sink_prefill_chunked_rope_workspace_size(B, H, L, d, w, s);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (L == 0) return SWA_OK;
    if (!k_cache || !v_cache) return fail(SWA_ERR_INVALID, "k_cache and v_cache must be non-null");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(SWA_ERR_INVALID, "k_cache and v_cache must be 16-byte aligned");
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const RopeParts rpt = rope_parts(ws, B * H, L, d, s);
    char *kc_rot = ws + rope_prefill_workspace_bytes(B * H, L, d, s);
    char *kc_rot_lo = kc_rot + static_cast<size_t>(B) * H * w * d * 2;
    // the rotations depend on absolute positions only, so one pass serves every chunk
    rc = launch_rope_prep(q, k, rpt, B * H, L, d, w, s, rope_base, st);
    if (rc) return rc;
    const ChunkRope rp{rpt.qr_lo, rpt.ssink, rpt.sstride, rpt.kr_lo, k, kc_rot, kc_rot_lo};
    return chunk_loop(rpt.qr, rpt.kr, v, o, lse, k_cache, v_cache, B, H, L, L, d, w, s, scale, chunk, dtype, st, &rp);
}

// Streams and events of the host-buffer prefill pipeline (copies in, compute, copies out), created once
// per device.
constexpr int kHostGroups = 8;
struct HostPipe {
    cudaStream_t in, comp, out;
    cudaEvent_t fork, join_out;
    cudaEvent_t copied[kHostGroups], computed[kHostGroups];
};
static HostPipe *host_pipe() {
    static std::mutex mu;
    static HostPipe *per_dev[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!per_dev[dev]) {
        HostPipe *h = new HostPipe();
        bool ok = cudaStreamCreateWithFlags(&h->in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h->comp, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h->out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h->join_out, cudaEventDisableTiming) == cudaSuccess;
        for (int g = 0; ok && g < kHostGroups; ++g)
            ok = cudaEventCreateWithFlags(&h->copied[g], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h->computed[g], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            delete h;
            return nullptr;
        }
        per_dev[dev] = h;
    }
    return per_dev[dev];
}

extern "C" int swa_sink_prefill_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                                     void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d, int B, int H,
                                     int64_t L, int d, int w, int s, float scale, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_prefill(q_d, k_d, v_d, o_d, lse_d, 0, B, H, L, d, w, s, scale, dtype);
    if (rc) return rc;
    if (L == 0) return SWA_OK;
    if (!q_h || !k_h || !v_h || !o_h) return fail(SWA_ERR_INVALID, "q_h, k_h, v_h and o_h must be non-null");
    if (lse_h && !lse_d) return fail(SWA_ERR_INVALID, "lse_h needs a device lse_d");
    HostPipe *hp = host_pipe();
    if (!hp) return fail(SWA_ERR_CUDA, "cannot create the streams of the host-buffer pipeline");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int BH = B * H;
    const int groups = BH < kHostGroups ? BH : kHostGroups;
    const size_t row_bytes = static_cast<size_t>(d) * esize_of(dtype);
    const size_t bh_bytes = static_cast<size_t>(L) * row_bytes;  // one (b, h) block of q, k, v or o
    cudaError_t e = cudaEventRecord(hp->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->comp, hp->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->fork, 0);
    for (int g = 0; e == cudaSuccess && g < groups; ++g) {
        const int r0 = static_cast<int>(static_cast<int64_t>(BH) * g / groups);
        const int r1 = static_cast<int>(static_cast<int64_t>(BH) * (g + 1) / groups);
        const size_t off = static_cast<size_t>(r0) * bh_bytes, bytes = static_cast<size_t>(r1 - r0) * bh_bytes;
        // inputs of the group: three contiguous blocks
        cudaStream_t in = hp->in;
        e = cudaMemcpyAsync(static_cast<char *>(q_d) + off, static_cast<const char *>(q_h) + off, bytes,
                            cudaMemcpyHostToDevice, in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char *>(k_d) + off, static_cast<const char *>(k_h) + off, bytes,
                                cudaMemcpyHostToDevice, in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char *>(v_d) + off, static_cast<const char *>(v_h) + off, bytes,
                                cudaMemcpyHostToDevice, in);
        if (e == cudaSuccess) e = cudaEventRecord(hp->copied[g], in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->comp, hp->copied[g], 0);
        if (e != cudaSuccess) break;
        float *lg = lse_d ? lse_d + static_cast<int64_t>(r0) * L : nullptr;
        rc = prefill_impl(static_cast<char *>(q_d) + off, static_cast<char *>(k_d) + off,
                          static_cast<char *>(v_d) + off, static_cast<char *>(o_d) + off, lg, nullptr, nullptr, 0,
                          r1 - r0, 1, L, d, w, s, scale, dtype, L, hp->comp);
        if (rc) return rc;
        e = cudaEventRecord(hp->computed[g], hp->comp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->computed[g], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char *>(o_h) + off, static_cast<char *>(o_d) + off, bytes,
                                cudaMemcpyDeviceToHost, hp->out);
        if (e == cudaSuccess && lse_h)
            e = cudaMemcpyAsync(lse_h + static_cast<int64_t>(r0) * L, lg, static_cast<size_t>(r1 - r0) * L * 4,
                                cudaMemcpyDeviceToHost, hp->out);
    }
    // the output stream finishes last (it waited for every group's compute); the caller's stream joins it
    if (e == cudaSuccess) e = cudaEventRecord(hp->join_out, hp->out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->join_out, 0);
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "host-buffer prefill pipeline: %s", cudaGetErrorString(e));
    return SWA_OK;
}

extern "C" int kv_rolling_write(void *k_cache, void *v_cache, const void *k_new, const void *v_new, int B, int H,
                                int d, int w, int s, int64_t pos0, int64_t n, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_common(B, H, d, w, s, dtype);
    if (rc) return rc;
    if (pos0 < 0 || n < 0) return fail(SWA_ERR_INVALID, "pos0=%lld and n=%lld must be >= 0", (long long)pos0,
                                       (long long)n);
    if (n == 0) return SWA_OK;
    if (!k_cache || !v_cache || !k_new || !v_new)
        return fail(SWA_ERR_INVALID, "k_cache, v_cache, k_new and v_new must be non-null");
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
        return fail(SWA_ERR_INVALID, "cache and new tensors must be 16-byte aligned");
    return launch_kv_write(k_cache, v_cache, k_new, v_new, B * H, d, w, s, pos0, n, n, esize_of(dtype),
                           static_cast<cudaStream_t>(stream));
}

extern "C" size_t swa_sink_decode_workspace_size(int B, int H, int d, int w) {
    if (B < 1 || H < 1 || d < 1 || w < 1) return 0;
    return decode_workspace_bytes(B * H, d, w);
}

extern "C" int swa_sink_decode_step(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                                    int B, int H, int d, int w, int s, int64_t t, float scale, void *workspace,
                                    size_t workspace_bytes, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_common(B, H, d, w, s, dtype);
    if (rc) return rc;
    if (t < 0 || t >= (int64_t(1) << 62)) return fail(SWA_ERR_INVALID, "t=%lld out of range", (long long)t);
    if (!(scale == scale) || scale <= 0.f || scale > 1e30f)
        return fail(SWA_ERR_INVALID, "scale must be a positive finite number");
    if (!q || !k_cache || !v_cache || !o) return fail(SWA_ERR_INVALID, "q, caches and o must be non-null");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
        return fail(SWA_ERR_INVALID, "q, caches and o must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SWA_ERR_INVALID, "lse must be 4-byte aligned");
    const size_t need = decode_workspace_bytes(B * H, d, w);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");
    DecodeArgs a{q, k_cache, v_cache, o, lse, B * H, d, w, s, t, scale, workspace, workspace_bytes,
                 esize_of(dtype), static_cast<cudaStream_t>(stream)};
    return launch_decode(a);
}

// The dilated window in streaming form.  r rolling caches, one per residue class of positions mod r, laid
// out class-major [r, B, H, w, d]: cache c holds the s sinks in slots 0..s-1 and a ring of m slots for the
// positions p >= s with p = c (mod r), each at its class-local position s + (p - p0(c)) / r, p0(c) the first
// such position.  At step t cache (t mod r) then holds exactly the dilated key set of t, so the plain
// rolling write and decode run on it at t's class-local position.  Rows t < s use cache 0.
static int64_t dilated_local(int64_t t, int s, int r, int *cls) {
    if (t < s) {
        *cls = 0;
        return t;
    }
    const int c = static_cast<int>(t % r);
    const int64_t p0 = s + ((c - s) % r + r) % r;
    *cls = c;
    return s + (t - p0) / r;
}

extern "C" int swa_sink_dilated_cache_write(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                                            int B, int H, int d, int w, int s, int r, int64_t t, int dtype,
                                            void *stream) {
    t_err[0] = 0;
    int rc = check_common(B, H, d, w, s, dtype);
    if (rc) return rc;
    if (r < 1 || r > 65536) return fail(SWA_ERR_INVALID, "dilation r=%d must be in [1, 65536]", r);
    if (t < 0 || t >= (int64_t(1) << 62)) return fail(SWA_ERR_INVALID, "t=%lld out of range", (long long)t);
    if (!k_cache || !v_cache || !k_new || !v_new)
        return fail(SWA_ERR_INVALID, "k_cache, v_cache, k_new and v_new must be non-null");
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
        return fail(SWA_ERR_INVALID, "cache and new tensors must be 16-byte aligned");
    const int es = esize_of(dtype);
    const size_t slab = static_cast<size_t>(B) * H * w * d * es;  // one class's cache
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int c = 0;
    const int64_t local = dilated_local(t, s, r, &c);
    // a sink goes into every class's cache (one launch over the r caches), any other position into its own
    const size_t first = t < s ? 0 : static_cast<size_t>(c) * slab;
    return launch_kv_write_classes(static_cast<char *>(k_cache) + first, static_cast<char *>(v_cache) + first, k_new,
                                   v_new, B * H, d, w, s, local, 1, 1, es, t < s ? r : 1, st);
}

extern "C" int swa_sink_decode_step_dilated(const void *q, const void *k_cache, const void *v_cache, void *o,
                                            float *lse, int B, int H, int d, int w, int s, int r, int64_t t,
                                            float scale, void *workspace, size_t workspace_bytes, int dtype,
                                            void *stream) {
    t_err[0] = 0;
    if (r < 1 || r > 65536) return fail(SWA_ERR_INVALID, "dilation r=%d must be in [1, 65536]", r);
    if (t < 0 || t >= (int64_t(1) << 62)) return fail(SWA_ERR_INVALID, "t=%lld out of range", (long long)t);
    int rc = check_common(B, H, d, w, s, dtype);
    if (rc) return rc;
    if (!k_cache || !v_cache) return fail(SWA_ERR_INVALID, "caches must be non-null");
    int c = 0;
    const int64_t local = dilated_local(t, s, r, &c);
    const size_t slab = static_cast<size_t>(B) * H * w * d * esize_of(dtype);
    return swa_sink_decode_step(q, static_cast<const char *>(k_cache) + c * slab,
                                static_cast<const char *>(v_cache) + c * slab, o, lse, B, H, d, w, s, local, scale,
                                workspace, workspace_bytes, dtype, stream);
}

extern "C" int swa_sink_decode_step_rope(const void *q, const void *k_cache, const void *v_cache, void *o,
                                         float *lse, int B, int H, int d, int w, int s, int64_t t, float scale,
                                         double rope_base, void *workspace, size_t workspace_bytes, int dtype,
                                         void *stream) {
    t_err[0] = 0;
    int rc = check_common(B, H, d, w, s, dtype);
    if (rc) return rc;
    if (t < 0 || t >= (int64_t(1) << 31)) return fail(SWA_ERR_INVALID, "t=%lld out of range", (long long)t);
    if (!(scale == scale) || scale <= 0.f || scale > 1e30f)
        return fail(SWA_ERR_INVALID, "scale must be a positive finite number");
    if (!(rope_base == rope_base) || rope_base <= 1.0 || rope_base > 1e30)
        return fail(SWA_ERR_INVALID, "rope_base must be a finite number > 1");
    if (!q || !k_cache || !v_cache || !o) return fail(SWA_ERR_INVALID, "q, caches and o must be non-null");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
        return fail(SWA_ERR_INVALID, "q, caches and o must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SWA_ERR_INVALID, "lse must be 4-byte aligned");
    const size_t need = decode_rope_workspace_bytes(B * H, d, w);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");
    DecodeArgs a{q, k_cache, v_cache, o, lse, B * H, d, w, s, t, scale, workspace, workspace_bytes,
                 esize_of(dtype), static_cast<cudaStream_t>(stream)};
    return launch_decode_rope(a, rope_base);
}

extern "C" size_t swa_sink_decode_rope_workspace_size(int B, int H, int d, int w) {
    if (B < 1 || H < 1 || w < 1 || (d != 16 && d != 32 && d != 64 && d != 128)) return 0;
    return decode_rope_workspace_bytes(B * H, d, w);
}

extern "C" int swa_selftest_wait_timeout(int64_t timeout_ns, void *stream) {
    t_err[0] = 0;
    if (timeout_ns < 1 || timeout_ns > 1000000000LL)
        return fail(SWA_ERR_INVALID, "timeout_ns=%lld not in [1, 1e9]", (long long)timeout_ns);
    return launch_selftest_wait_timeout(static_cast<uint64_t>(timeout_ns), static_cast<cudaStream_t>(stream));
}

extern "C" int swa_selftest_umma(const void *a, const void *b, float *c, int mode, void *stream) {
    t_err[0] = 0;
    if (!a || !b || !c) return fail(SWA_ERR_INVALID, "a, b and c must be non-null");
    if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return fail(SWA_ERR_INVALID, "a, b, c must be 16-byte aligned");
    if (mode < 0 || mode > 3) return fail(SWA_ERR_INVALID, "mode=%d not in {0, 1, 2, 3}", mode);
    return launch_selftest_umma(a, b, c, mode, static_cast<cudaStream_t>(stream));
}

extern "C" int swa_prefill_tile_plan(int64_t q0, int64_t q1, int64_t pos0, int w, int s, int *tiles, int max_tiles) {
    t_err[0] = 0;
    if (w < 1 || s < 0 || s >= w) return fail(SWA_ERR_INVALID, "need 0 <= s < w (s=%d, w=%d)", s, w);
    if (pos0 < 0 || q0 < pos0 || q1 < q0 || q1 >= (int64_t(1) << 31))
        return fail(SWA_ERR_INVALID, "need 0 <= pos0 <= q0 <= q1 < 2^31");
    if (!tiles || max_tiles < 0) return fail(SWA_ERR_INVALID, "tiles must be non-null");
    return prefill_tile_plan(static_cast<int>(q0), static_cast<int>(q1), static_cast<int>(pos0), w, s, 0, tiles,
                             max_tiles);
}

extern "C" int swa_prefill_tile_plan_rope(int64_t q0, int64_t q1, int64_t pos0, int w, int s, int *tiles,
                                          int max_tiles) {
    t_err[0] = 0;
    if (w < 1 || s < 0 || s >= w) return fail(SWA_ERR_INVALID, "need 0 <= s < w (s=%d, w=%d)", s, w);
    if (s > 128) return fail(SWA_ERR_UNSUPPORTED, "RoPE prefill needs s <= 128");
    if (pos0 > 0 && pos0 < s) return fail(SWA_ERR_UNSUPPORTED, "RoPE prefill needs pos0 = 0 or pos0 >= s");
    if (pos0 < 0 || q0 < pos0 || q1 < q0 || q1 >= (int64_t(1) << 31))
        return fail(SWA_ERR_INVALID, "need 0 <= pos0 <= q0 <= q1 < 2^31");
    if (!tiles || max_tiles < 0) return fail(SWA_ERR_INVALID, "tiles must be non-null");
    return prefill_tile_plan(static_cast<int>(q0), static_cast<int>(q1), static_cast<int>(pos0), w, s, 1, tiles,
                             max_tiles);
}

extern "C" int swa_prefill_dilated_split(int64_t L, int s, int r, int64_t *out) {
    t_err[0] = 0;
    if (L < 0 || L >= (int64_t(1) << 31) || s < 0 || r < 1 || r > 65536)
        return fail(SWA_ERR_INVALID, "need 0 <= L < 2^31, s >= 0, 1 <= r <= 65536");
    if (!out) return fail(SWA_ERR_INVALID, "out must be non-null");
    const DilatedSplit d = dilated_split(L, s, r);
    out[0] = d.nrows;
    out[1] = d.G;
    out[2] = d.ns;
    out[3] = d.tail0;
    return SWA_OK;
}

extern "C" int swa_prefill_tile_plan_dilated(int64_t L, int w, int s, int r, int cls, int64_t row_start, int *tiles,
                                             int max_tiles) {
    t_err[0] = 0;
    if (w < 1 || s < 0 || s >= w) return fail(SWA_ERR_INVALID, "need 0 <= s < w (s=%d, w=%d)", s, w);
    if (L < 1 || L >= (int64_t(1) << 31) || r < 1 || r > 65536 || cls < 0 || cls >= r)
        return fail(SWA_ERR_INVALID, "need 1 <= L < 2^31, 1 <= r <= 65536, 0 <= cls < r");
    if (row_start < 0 || row_start >= (int64_t(1) << 31)) return fail(SWA_ERR_INVALID, "row_start out of range");
    if (!tiles || max_tiles < 0) return fail(SWA_ERR_INVALID, "tiles must be non-null");
    return prefill_tile_plan_dilated(L, w, s, r, cls, static_cast<int>(row_start), tiles, max_tiles);
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

extern "C" size_t swa_sink_prefill_dilated_workspace_size(int B, int H, int64_t L, int d, int s, int r, int dtype) {
    const int es = esize_of(dtype);
    if (B < 1 || H < 1 || L < 0 || s < 0 || r < 1 || es == 0 || !(d == 16 || d == 32 || d == 64 || d == 128)) return 0;
    const size_t rows = static_cast<size_t>(B) * H * r * static_cast<size_t>(dilated_rows(L, s, r));
    return 4 * align256(rows * d * es) + align256(rows * sizeof(float));
}

extern "C" int swa_sink_prefill_dilated(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                                        int64_t L, int d, int w, int s, int r, float scale, void *workspace,
                                        size_t workspace_bytes, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_prefill(q, k, v, o, lse, 0, B, H, L, d, w, s, scale, dtype);
    if (rc) return rc;
    if (r < 1 || r > 65536) return fail(SWA_ERR_INVALID, "dilation r=%d must be in [1, 65536]", r);
    if (static_cast<int64_t>(B) * H * r > 65535 * 32)
        return fail(SWA_ERR_UNSUPPORTED, "B*H*r=%lld exceeds the supported %d", (long long)B * H * r, 65535 * 32);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (r == 1)  // the plain window: the prefill itself (no workspace)
        return prefill_impl(q, k, v, o, lse, nullptr, nullptr, 0, B, H, L, d, w, s, scale, dtype, L, st);
    if (dtype == SWA_BF16 && d == 128) {
        // in place: the tensor-core pass over the whole groups of r positions after the sinks, then the
        // CUDA-core pass over the sink rows and the last L mod r rows (no workspace)
        if (L == 0) return SWA_OK;
        const PrefillArgs a{q, k, v, o, lse, nullptr, nullptr, 0, B * H, L, d, w, s, scale, L, st};
        rc = launch_prefill_bf16_tc_dilated(a, r);
        if (rc) return rc;
        return launch_dilated_rows(a, r);
    }
    const size_t need = swa_sink_prefill_dilated_workspace_size(B, H, L, d, s, r, dtype);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (L == 0) return SWA_OK;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");
    const int es = esize_of(dtype);
    const int VH = B * H * r;
    const int64_t Lv = dilated_rows(L, s, r);
    const size_t one = align256(static_cast<size_t>(VH) * Lv * d * es);
    char *ws = static_cast<char *>(workspace);
    void *qv = ws, *kv = ws + one, *vv = ws + 2 * one, *ov = ws + 3 * one;
    float *lsev = reinterpret_cast<float *>(ws + 4 * one);
    rc = launch_dilate_gather(q, k, v, qv, kv, vv, B * H, L, d, es, s, r, st);
    if (rc) return rc;
    // the virtual heads as (b, h) rows of a plain prefill: s sinks, window w
    rc = prefill_impl(qv, kv, vv, ov, lsev, nullptr, nullptr, 0, VH, 1, Lv, d, w, s, scale, dtype, Lv, st);
    if (rc) return rc;
    return launch_dilate_scatter(ov, lsev, o, lse, B * H, L, d, es, s, r, st);
}

extern "C" int swa_sink_prefill_chunked_dilated(const void *q, const void *k, const void *v, void *o, float *lse,
                                                void *k_cache, void *v_cache, int B, int H, int64_t L, int d, int w,
                                                int s, int r, float scale, int64_t chunk, void *workspace,
                                                size_t workspace_bytes, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_prefill(q, k, v, o, lse, 0, B, H, L, d, w, s, scale, dtype);
    if (rc) return rc;
    if (r < 1 || r > 65536) return fail(SWA_ERR_INVALID, "dilation r=%d must be in [1, 65536]", r);
    if (chunk < 1) return fail(SWA_ERR_INVALID, "chunk=%lld must be >= 1", (long long)chunk);
    if (static_cast<int64_t>(B) * H * r > 65535 * 32)
        return fail(SWA_ERR_UNSUPPORTED, "B*H*r=%lld exceeds the supported %d", (long long)B * H * r, 65535 * 32);
    const size_t need = swa_sink_prefill_dilated_workspace_size(B, H, L, d, s, r, dtype);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (L == 0) return SWA_OK;
    if (!k_cache || !v_cache) return fail(SWA_ERR_INVALID, "k_cache and v_cache must be non-null");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(SWA_ERR_INVALID, "k_cache and v_cache must be 16-byte aligned");
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int es = esize_of(dtype);
    const int VH = B * H * r;
    const int64_t Lv = dilated_rows(L, s, r);
    const size_t one = align256(static_cast<size_t>(VH) * Lv * d * es);
    char *ws = static_cast<char *>(workspace);
    void *qv = ws, *kv = ws + one, *vv = ws + 2 * one, *ov = ws + 3 * one;
    float *lsev = reinterpret_cast<float *>(ws + 4 * one);
    rc = launch_dilate_gather(q, k, v, qv, kv, vv, B * H, L, d, es, s, r, st);
    if (rc) return rc;
    // The virtual heads (class-major, as the per-class caches [r, B, H, w, d]) through the plain chunk loop,
    // chunk / r class-local rows at a time.  Each class runs at its own length (the sinks + its positions
    // >= s; the classes differ by at most one row), so that no padding row is ever written into a cache:
    // runs of classes of equal length share one loop (the longer classes form one cyclic run, so at most
    // three loops).
    const int64_t vchunk = chunk / r > 0 ? chunk / r : 1;
    const int64_t head = L < s ? L : s;
    const size_t rb = static_cast<size_t>(d) * es;
    auto class_rows = [&](int c) -> int64_t {  // rows of virtual head class c
        if (L <= s) return head;
        const int64_t p0 = s + ((c - s) % r + r) % r;
        return head + (p0 < L ? (L - 1 - p0) / r + 1 : 0);
    };
    const int BH = B * H;
    for (int ca = 0; ca < r;) {
        const int64_t n = class_rows(ca);
        int cb = ca + 1;
        while (cb < r && class_rows(cb) == n) ++cb;
        const size_t vo = static_cast<size_t>(ca) * BH * Lv, co = static_cast<size_t>(ca) * BH * w;
        rc = chunk_loop(static_cast<char *>(qv) + vo * rb, static_cast<char *>(kv) + vo * rb,
                        static_cast<char *>(vv) + vo * rb, static_cast<char *>(ov) + vo * rb, lsev + vo,
                        static_cast<char *>(k_cache) + co * rb, static_cast<char *>(v_cache) + co * rb, (cb - ca) * BH, 1,
                        n, Lv, d, w, s, scale, vchunk, dtype, st, nullptr);
        if (rc) return rc;
        ca = cb;
    }
    return launch_dilate_scatter(ov, lsev, o, lse, B * H, L, d, es, s, r, st);
}

extern "C" size_t swa_sink_prefill_rope_workspace_size(int B, int H, int64_t L, int d, int s) {
    if (B < 1 || H < 1 || L < 0 || d != 128 || s < 0 || s > 128) return 0;
    return rope_prefill_workspace_bytes(B * H, L, d, s);
}

extern "C" int swa_sink_prefill_rope(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                                     int64_t L, int d, int w, int s, float scale, double rope_base, void *workspace,
                                     size_t workspace_bytes, int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_prefill(q, k, v, o, lse, 0, B, H, L, d, w, s, scale, dtype);
    if (rc) return rc;
    if (dtype != SWA_BF16 || d != 128) return fail(SWA_ERR_UNSUPPORTED, "RoPE prefill runs on bf16 with d = 128");
    if (s > 128) return fail(SWA_ERR_UNSUPPORTED, "RoPE prefill needs s <= 128 (s=%d)", s);
    if (!(rope_base == rope_base) || rope_base <= 1.0 || rope_base > 1e30)
        return fail(SWA_ERR_INVALID, "rope_base must be a finite number > 1");
    const size_t need = rope_prefill_workspace_bytes(B * H, L, d, s);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (L == 0) return SWA_OK;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const RopeParts rpt = rope_parts(workspace, B * H, L, d, s);
    rc = launch_rope_prep(q, k, rpt, B * H, L, d, w, s, rope_base, st);
    if (rc) return rc;
    PrefillArgs a{rpt.qr, rpt.kr, v, o, lse, nullptr, nullptr, 0, B * H, L, d, w, s, scale, L, st};
    a.rope = true;
    a.rope_ssink = rpt.ssink;
    a.rope_sstride = rpt.sstride;
    a.q_lo = rpt.qr_lo;
    a.k_lo = rpt.kr_lo;
    return launch_prefill_bf16_tc(a);
}

extern "C" int swa_sink_decode_step_noalloc(const void *q, const void *k_cache, const void *v_cache, void *o,
                                            float *lse, int B, int H, int d, int w, int s, int64_t t, float scale,
                                            int dtype, void *stream) {
    t_err[0] = 0;
    int rc = check_common(B, H, d, w, s, dtype);
    if (rc) return rc;
    if (t < 0 || t >= (int64_t(1) << 62)) return fail(SWA_ERR_INVALID, "t=%lld out of range", (long long)t);
    if (!(scale == scale) || scale <= 0.f || scale > 1e30f)
        return fail(SWA_ERR_INVALID, "scale must be a positive finite number");
    if (!q || !k_cache || !v_cache || !o) return fail(SWA_ERR_INVALID, "q, caches and o must be non-null");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
        return fail(SWA_ERR_INVALID, "q, caches and o must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SWA_ERR_INVALID, "lse must be 4-byte aligned");
    DecodeArgs a{q, k_cache, v_cache, o, lse, B * H, d, w, s, t, scale, nullptr, 0,
                 esize_of(dtype), static_cast<cudaStream_t>(stream)};
    return launch_decode_noalloc(a);
}
