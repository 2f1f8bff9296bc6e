// decode.cu -- swa_sink_decode_step: one streaming-decode query per (b, h) against the rolling cache.
//
// After positions 0..t have been written, the cache slots 0..min(t+1, w)-1 hold exactly the key set
// K(t) = sinks + the last m positions (page "滑窗与固定稀疏", eq attn-fixed-streaming), and softmax
// attention does not depend on the order of its keys ("模糊窗口注意力", section 3 introduction), so the
// kernel attends every valid slot in slot order without looking at positions.
//
// The work is HBM-bound: every step reads the whole valid cache (2 * nvalid * d * esize bytes per
// (b, h)) once.  Design:
//   * grid (nsplit, B*H); a split covers a contiguous slot range (split-K over the cache);
//   * a row of the cache is read by LPR = d*esize/16 lanes with one 16-byte streaming load each
//     (ld.global.cs: read once, evict first), so a warp reads RPW = 32/LPR whole rows per load and
//     every load instruction is fully coalesced;
//   * each lane issues U key loads and U value loads before using any of them (memory-level
//     parallelism), then the partial dot products are summed over the LPR lanes of a row with
//     xor-shuffles, and an online softmax (running max m, sum l, accumulator) is kept per row group;
//   * the row groups of a CTA are merged through shared memory; with nsplit > 1 the CTA writes its
//     partial (acc, m, l) to the caller's workspace and a second kernel merges the splits with the
//     log-sum-exp identity  o = sum_j 2^(m_j - M) acc_j / sum_j 2^(m_j - M) l_j,  M = max_j m_j.
// Scores are kept in log2 units (x = scale * log2(e) * q.k) so exp is a single exp2.
#include <math.h>

#include <cmath>

#include <mutex>

#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxSplits = 64;
constexpr int kMinSlotsPerSplit = 256;

__device__ __forceinline__ void unpack16(const uint4 &u, float (&f)[8], __nv_bfloat16) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4 &u, float (&f)[4], float) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }

// Rotary embedding at positions inside the cache (StreamingLLM section of "滑窗与固定稀疏": the cache's
// entries take the consecutive positions 0 .. n-1, sinks first, then the window in order; keys are kept
// unrotated and rotated at every step).  Dimensions i and i + D/2 form a pair rotated by pos * theta_i.
// With relative position delta = c_key - c_query the score of a pair is
//     q_i (k_i cos - k_{i+D/2} sin) + q_{i+D/2} (k_i sin + k_{i+D/2} cos),  angle = delta * theta_i,
// so the query stays unrotated and each key row meets cos/sin of its own delta.
constexpr int kMaxRopePairs = 64;         // d <= 128
constexpr int kMaxRopeWindowBits = 16;     // w <= 2^16
struct RopeArgs {
    // theta_i / (2 pi) in turns as hi + lo (fp32).  hi keeps 24 - k significant bits, where every distance
    // inside the cache is below 2^k (k = ceil(log2 w)), so distance * hi is exact in fp32 and its whole
    // turns drop out exactly; lo is the rest, and distance * lo rounds to within theta_i 2^(2k-47) turns.
    float2 theta[kMaxRopePairs];
    int s, m;  // sinks, ring slots
    int t;     // position of the query
};

// sin and cos of the angle a * theta_i, reduced to [-pi, pi] as above
__device__ __forceinline__ void rope_sincos(int a, float2 th, float &sn, float &c) {
    const float fa = static_cast<float>(a);
    float turns = fa * th.x;
    turns -= rintf(turns);
    turns = fmaf(fa, th.y, turns);
    __sincosf(turns * 6.283185307179586f, &sn, &c);
}

// Blocks per SM in the launch bounds (measured): the plain form compiled for 1 keeps every load of a
// block in flight in its 80 registers (7 % faster than the compiler's default of 60); the RoPE form
// compiled for 3 stays at 80 registers, so three 256-thread blocks still fit on an SM.
template <typename T, int D, int U, bool ROPE>
__global__ void __launch_bounds__(kDecThreads, ROPE ? 3 : 1) decode_kernel(const T *__restrict__ q, const T *__restrict__ kc,
                                                             const T *__restrict__ vc, T *__restrict__ o,
                                                             float *__restrict__ lse, float *__restrict__ part,
                                                             int w, int nvalid, int per_split, int nsplit,
                                                             float scale_log2, const __grid_constant__ RopeArgs ra) {
    constexpr int EPL = 16 / sizeof(T);  // elements per 16-byte chunk
    constexpr int LPR = D / EPL;         // lanes per cache row
    constexpr int RPW = 32 / LPR;        // rows per warp per load
    constexpr int G = kDecWarps * RPW;   // row groups per CTA
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must map onto a power-of-two lane group");

    __shared__ float sm_m[G], sm_l[G];
    __shared__ float sm_acc[G][D];

    const int split = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR;
    const int grp = warp * RPW + lane / LPR;
    const int j0 = split * per_split;
    const int j1 = min(nvalid, j0 + per_split);

    // Without rotary embedding a lane holds one 16-byte chunk of q and of each key row: elements
    // sub*EPL .. sub*EPL+EPL-1.  With it (half-split pairs (i, i + D/2)) a lane holds both halves of
    // its EPL/2 pairs: elements sub*EPL/2 + p in qf[p] and D/2 + sub*EPL/2 + p in qf[EPL/2 + p], read as
    // two 8-byte halves (each half of a row still coalesces into LPR * 8 contiguous bytes).
    constexpr int HPL = EPL / 2;  // pairs per lane
    float qf[EPL];
    {
        uint4 qu;
        if constexpr (ROPE) {
            const uint2 *q2 = reinterpret_cast<const uint2 *>(q + bh * D);
            const uint2 a = __ldg(q2 + sub), b = __ldg(q2 + LPR + sub);
            qu = make_uint4(a.x, a.y, b.x, b.y);
        } else {
            qu = __ldg(reinterpret_cast<const uint4 *>(q + bh * D) + sub);
        }
        unpack16(qu, qf, T());
#pragma unroll
        for (int e = 0; e < EPL; ++e) qf[e] *= scale_log2;
    }
    float2 th[ROPE ? HPL : 1];  // theta / (2 pi) of the lane's pairs, hi + lo
    int cq = 0;                 // cache position of the query
    int jnew = 0;               // ring slot of the newest position (t), once the ring is full
    bool full = false;
    if constexpr (ROPE) {
        full = ra.t >= ra.s + ra.m - 1;
        if (full) jnew = ra.s + (ra.t - ra.s) % ra.m;
        cq = nvalid - 1;  // the query's own key is the newest entry of the cache
#pragma unroll
        for (int p = 0; p < HPL; ++p) th[p] = ra.theta[sub * HPL + p];
        // pin the rates in registers: re-reading them per row from the parameter bank, at 16 addresses per
        // warp, serialises
#pragma unroll
        for (int p = 0; p < HPL; ++p) asm volatile("" : "+f"(th[p].x), "+f"(th[p].y));
    }
    const uint4 *kb = reinterpret_cast<const uint4 *>(kc + bh * w * D) + sub;
    const uint2 *kb2 = reinterpret_cast<const uint2 *>(kc + bh * w * D) + sub;
    const uint4 *vb = reinterpret_cast<const uint4 *>(vc + bh * w * D) + sub;

    float m = -INFINITY, l = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;

    for (int jblk = j0; jblk < j1; jblk += G * U) {  // uniform over the CTA: shuffles stay converged
        uint4 kr[U], vr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = jblk + u * G + grp;
            if (j < j1) {
                if constexpr (ROPE) {
                    const uint2 a = __ldcs(kb2 + static_cast<int64_t>(j) * (2 * LPR));
                    const uint2 b = __ldcs(kb2 + static_cast<int64_t>(j) * (2 * LPR) + LPR);
                    kr[u] = make_uint4(a.x, a.y, b.x, b.y);
                } else {
                    kr[u] = __ldcs(kb + static_cast<int64_t>(j) * LPR);
                }
                vr[u] = __ldcs(vb + static_cast<int64_t>(j) * LPR);
            } else {
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
            }
        }
        float x[U];
        float mt = -INFINITY;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float kf[EPL];
            unpack16(kr[u], kf, T());
            float dot = 0.f;
            if constexpr (ROPE) {
                const int j = min(jblk + u * G + grp, j1 - 1);  // rows past j1 are masked below
                // |delta| = cache position of the query - that of slot j.  Before the ring is full every
                // valid slot j holds position j at cache position j, and the query sits at t.  Once it is
                // full the query sits at w - 1, a sink j at j, and a ring slot at w - 1 - its age (how many
                // ring writes ago it was written, counted back from the slot of position t).
                const int ad = !full ? ra.t - j : (j < ra.s ? cq - j : (j <= jnew ? jnew - j : jnew - j + ra.m));
#pragma unroll
                for (int p = 0; p < HPL; ++p) {
                    float sn, c;
                    rope_sincos(ad, th[p], sn, c);
                    // q . R(delta theta) k over the pair, with sin(delta theta) = -sin(|delta| theta):
                    // k_i (q_i c - q_{i+D/2} sn) + k_{i+D/2} (q_{i+D/2} c + q_i sn)
                    const float qa = qf[p], qb = qf[HPL + p];
                    dot = fmaf(fmaf(qa, c, -qb * sn), kf[p], dot);
                    dot = fmaf(fmaf(qb, c, qa * sn), kf[HPL + p], dot);
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) dot = fmaf(qf[e], kf[e], dot);
            }
#pragma unroll
            for (int off = LPR / 2; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
            x[u] = (jblk + u * G + grp < j1) ? dot : -INFINITY;
            mt = fmaxf(mt, x[u]);
        }
        const float mn = fmaxf(m, mt);
        if (mn == -INFINITY) continue;  // this group had no valid row in the block
        const float alpha = exp2f(m - mn);  // m == -inf -> 0
        l *= alpha;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= alpha;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float p = exp2f(x[u] - mn);  // invalid rows: exp2(-inf) = 0
            float vf[EPL];
            unpack16(vr[u], vf, T());
            l += p;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = fmaf(p, vf[e], acc[e]);
        }
        m = mn;
    }

#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_acc[grp][sub * EPL + e] = acc[e];
    if (sub == 0) {
        sm_m[grp] = m;
        sm_l[grp] = l;
    }
    __syncthreads();
    if (threadIdx.x < D) {
        const int c = threadIdx.x;
        float M = -INFINITY;
        for (int g = 0; g < G; ++g) M = fmaxf(M, sm_m[g]);
        float L = 0.f, a = 0.f;
        if (M != -INFINITY) {
            for (int g = 0; g < G; ++g) {
                const float f = exp2f(sm_m[g] - M);
                L = fmaf(sm_l[g], f, L);
                a = fmaf(sm_acc[g][c], f, a);
            }
        }
        if (nsplit == 1) {
            store_out(o + bh * D + c, a / L);
            if (c == 0 && lse) lse[bh] = (M + log2f(L)) * 0.69314718055994531f;
        } else {
            float *pp = part + (bh * nsplit + split) * (D + 2);
            pp[c] = a;
            if (c == 0) {
                pp[D] = M;
                pp[D + 1] = L;
            }
        }
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const float *__restrict__ part, T *__restrict__ o,
                                                         float *__restrict__ lse, int nsplit) {
    const int64_t bh = blockIdx.x;
    const int c = threadIdx.x;
    const float *pp = part + bh * nsplit * (D + 2);
    float M = -INFINITY;
    for (int j = 0; j < nsplit; ++j) M = fmaxf(M, pp[j * (D + 2) + D]);
    float L = 0.f, a = 0.f;
    for (int j = 0; j < nsplit; ++j) {
        const float mj = pp[j * (D + 2) + D];
        if (mj == -INFINITY) continue;  // a split without a valid slot
        const float f = exp2f(mj - M);
        L = fmaf(pp[j * (D + 2) + D + 1], f, L);
        a = fmaf(pp[j * (D + 2) + c], f, a);
    }
    store_out(o + bh * D + c, a / L);
    if (c == 0 && lse) lse[bh] = (M + log2f(L)) * 0.69314718055994531f;
}

int decode_num_splits(int BH, int nvalid) {
    const int target = 152 * 8;  // CTAs that keep every SM of a GB300 busy (8 x 256 threads per SM)
    int ns = (target + BH - 1) / BH;
    const int by_work = (nvalid + kMinSlotsPerSplit - 1) / kMinSlotsPerSplit;
    if (ns > by_work) ns = by_work;
    if (ns > kMaxSplits) ns = kMaxSplits;
    if (ns < 1) ns = 1;
    return ns;
}

size_t decode_workspace_bytes(int BH, int d, int w) {
    const int ns = decode_num_splits(BH, w);  // the split count only grows with the valid slots (<= w)
    if (ns <= 1) return 0;
    return static_cast<size_t>(BH) * ns * (d + 2) * sizeof(float);
}

template <typename T, int D>
static int launch_typed(const DecodeArgs &a, int nvalid, int ns, int per_split, float sl2, const RopeArgs *ra) {
    constexpr int U = (sizeof(T) == 2 && D >= 64) ? 4 : 2;
    const dim3 grid(ns, a.BH), block(kDecThreads);
    float *part = static_cast<float *>(a.workspace);
    if (ra)
        decode_kernel<T, D, U, true><<<grid, block, 0, a.stream>>>(
            static_cast<const T *>(a.q), static_cast<const T *>(a.k_cache), static_cast<const T *>(a.v_cache),
            static_cast<T *>(a.o), a.lse, part, a.w, nvalid, per_split, ns, sl2, *ra);
    else
        decode_kernel<T, D, U, false><<<grid, block, 0, a.stream>>>(
            static_cast<const T *>(a.q), static_cast<const T *>(a.k_cache), static_cast<const T *>(a.v_cache),
            static_cast<T *>(a.o), a.lse, part, a.w, nvalid, per_split, ns, sl2, RopeArgs{});
    if (ns > 1)
        decode_merge_kernel<T, D><<<a.BH, D, 0, a.stream>>>(part, static_cast<T *>(a.o), a.lse, ns);
    return 0;
}

static int dispatch_decode(const DecodeArgs &a, int nvalid, int ns, int per_split, float sl2, const RopeArgs *ra) {
    if (a.esize == 2) {
        switch (a.d) {
            case 16: launch_typed<__nv_bfloat16, 16>(a, nvalid, ns, per_split, sl2, ra); break;
            case 32: launch_typed<__nv_bfloat16, 32>(a, nvalid, ns, per_split, sl2, ra); break;
            case 64: launch_typed<__nv_bfloat16, 64>(a, nvalid, ns, per_split, sl2, ra); break;
            case 128: launch_typed<__nv_bfloat16, 128>(a, nvalid, ns, per_split, sl2, ra); break;
            default: return fail(SWA_ERR_UNSUPPORTED, "decode: d=%d", a.d);
        }
    } else {
        switch (a.d) {
            case 16: launch_typed<float, 16>(a, nvalid, ns, per_split, sl2, ra); break;
            case 32: launch_typed<float, 32>(a, nvalid, ns, per_split, sl2, ra); break;
            case 64: launch_typed<float, 64>(a, nvalid, ns, per_split, sl2, ra); break;
            case 128: launch_typed<float, 128>(a, nvalid, ns, per_split, sl2, ra); break;
            default: return fail(SWA_ERR_UNSUPPORTED, "decode: d=%d", a.d);
        }
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

int launch_decode(const DecodeArgs &a) {
    const int nvalid = static_cast<int>(a.t + 1 < a.w ? a.t + 1 : a.w);
    const int ns = decode_num_splits(a.BH, nvalid);
    const int per_split = (nvalid + ns - 1) / ns;
    const float sl2 = a.scale * 1.4426950408889634f;
    if (ns > 1 && (!a.workspace || a.workspace_bytes < static_cast<size_t>(a.BH) * ns * (a.d + 2) * sizeof(float)))
        return fail(SWA_ERR_INVALID, "decode needs %d splits but the workspace is too small", ns);
    return dispatch_decode(a, nvalid, ns, per_split, sl2, nullptr);
}

size_t decode_rope_workspace_bytes(int BH, int d, int w) { return decode_workspace_bytes(BH, d, w); }

int launch_decode_rope(const DecodeArgs &a, double base) {
    if (a.t >= (int64_t(1) << 31)) return fail(SWA_ERR_UNSUPPORTED, "rope decode: t must be < 2^31");
    if (a.d / 2 > kMaxRopePairs) return fail(SWA_ERR_UNSUPPORTED, "rope decode: d=%d", a.d);
    if (a.w > (1 << kMaxRopeWindowBits))
        return fail(SWA_ERR_UNSUPPORTED, "rope decode: w = %d > %d", a.w, 1 << kMaxRopeWindowBits);
    const int nvalid = static_cast<int>(a.t + 1 < a.w ? a.t + 1 : a.w);
    const int ns = decode_num_splits(a.BH, nvalid);
    const int per_split = (nvalid + ns - 1) / ns;
    const float sl2 = a.scale * 1.4426950408889634f;
    if (ns > 1 && (!a.workspace || a.workspace_bytes < static_cast<size_t>(a.BH) * ns * (a.d + 2) * sizeof(float)))
        return fail(SWA_ERR_INVALID, "rope decode needs %d splits but the workspace is too small", ns);
    RopeArgs ra{};
    int k = 0;  // distances are 0 .. w - 1 < 2^k
    while ((1 << k) < a.w) ++k;
    // theta_i / (2 pi) = base^(-2i/d) / (2 pi), evaluated in double; hi = its leading 24 - k bits
    for (int i = 0; i < a.d / 2; ++i) {
        const double f = std::pow(base, -2.0 * i / a.d) / 6.283185307179586476925286766559;
        int ex = 0;
        const double mant = std::frexp(f, &ex);  // f = mant 2^ex, mant in [0.5, 1)
        const double hi = std::ldexp(std::floor(std::ldexp(mant, 24 - k)), ex - (24 - k));
        ra.theta[i] = make_float2(static_cast<float>(hi), static_cast<float>(f - hi));
    }
    ra.s = a.s;
    ra.m = a.w - a.s;
    ra.t = static_cast<int>(a.t);
    return dispatch_decode(a, nvalid, ns, per_split, sl2, &ra);
}

}  // namespace swa

// ------------------------------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the moment they run a decode step: an inference
// engine's plugin or custom-op callback is often forbidden to allocate while it enqueues work, a server
// whose device memory is handed out up front by its own pool allocator has nothing to give to a
// library, and cudaMalloc may synchronise the device, which a latency-bound token loop cannot afford.
// For them the split-K partial results go to this fixed, file-scope array instead.  Every GPU that
// loads the library keeps it (kNoAllocScratchBytes) until the process exits.
//
// Every call shares the one array.  A call writes every partial it later reads, so nothing has to be
// cleared between calls, but two calls that run at the same time on the GPU (on different streams, or
// on the same device from several threads) overwrite each other's partials: serialise them.
namespace swa {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch on the current device.  In host code the array's name is only a
// host-side stand-in, so the address is looked up once per device (with that device current) and kept.
static void *decode_scratch_address() {
    static std::mutex mu;
    static void *ptrs[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        fail(SWA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            fail(SWA_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
            return nullptr;
        }
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

size_t decode_noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

int launch_decode_noalloc(DecodeArgs a) {
    const size_t need = decode_workspace_bytes(a.BH, a.d, a.w);
    if (need > kNoAllocScratchBytes)
        return fail(SWA_ERR_UNSUPPORTED,
                    "this shape needs %zu bytes of split-K scratch, more than the %zu bytes of the built-in array; "
                    "use swa_sink_decode_step with a workspace",
                    need, kNoAllocScratchBytes);
    void *scratch = decode_scratch_address();
    if (!scratch) return SWA_ERR_CUDA;
    a.workspace = scratch;
    a.workspace_bytes = kNoAllocScratchBytes;
    return launch_decode(a);
}

}  // namespace swa
