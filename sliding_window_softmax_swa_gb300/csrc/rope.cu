// rope.cu -- the rotation pass of prefill with RoPE at the positions inside the cache.
//
// The StreamingLLM section of "滑窗与固定稀疏" gives every entry of the cache its position inside the cache
// (sinks 0..s-1, then the recent keys in order) rather than its position in the text.  For a whole
// sequence that rule differs from plain RoPE in one place only: the query of row t scores its window keys
// at distance t - i, as plain RoPE does, but the sinks at distance min(t, w - 1) - i, because once the
// cache is full the query sits at position w - 1.  So the tensor-core prefill runs on
//     Qr = R(t) q_t,  Kr = R(i) k_i                              (the band)
// and takes the sink scores ready-made:
//     Ssink[t, i] = (R(min(t, w - 1)) q_t) . (R(i) k_i),  i < s   (fp32 dot products of fp32 rotations),
// all written by this pass into the caller's workspace.  R(a) rotates the half-split pair (x_i, x_{i+d/2})
// by a * base^(-2i/d): (x cos - y sin, x sin + y cos).  Each rotated value x (fp32) of Qr and Kr is written as
// two bf16 numbers, hi = bf16(x) and lo = bf16(x - hi), so hi + lo holds x to about 2^-17 relative and the
// prefill's three products hi hi + hi lo + lo hi give scores with the error of fp32 operands.
//
// Angles are reduced exactly for every position < 2^31: theta_i / (2 pi) is held as the 64-bit fraction
// F_i = round(2^64 theta_i / (2 pi)) (host, double), and the fraction of a turn of a * theta_i is
// (a F_i) mod 2^64, whose top 32 bits are a * F_hi + umulhi(a, F_lo).  The error is that of F_i, at most
// a * 2^-65 turns; sin and cos are fp32.  The pass is HBM-bound: per row it reads q and k and writes four
// bf16 rows and s fp32 scores, 16 lanes per row, each lane holding both halves of its 4 pairs.
#include <cuda_bf16.h>

#include <cmath>

#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {

constexpr int kRopeD = 128;
constexpr int kRopeLanes = 16;               // lanes per row
constexpr int kRopePpl = kRopeD / 2 / kRopeLanes;  // pairs per lane (4)

struct RopePrep {
    uint2 frac[kRopeD / 2];  // F_i as (low 32 bits, high 32 bits)
};

__device__ __forceinline__ void turn_sincos(uint32_t a, uint2 f, float &sn, float &c) {
    const uint32_t top = a * f.y + __umulhi(a, f.x);                                        // (a F) >> 32, mod 2^32
    const float turns = static_cast<float>(static_cast<int32_t>(top)) * 2.3283064365386963e-10f;  // [-1/2, 1/2)
    __sincosf(turns * 6.283185307179586f, &sn, &c);
}

__device__ __forceinline__ void unpack4(uint2 u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xFFFF0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The pairs (a[p], b[p]) rotated by the angles (sn[p], c[p]): x = a cos - b sin, y = a sin + b cos (fp32).
__device__ __forceinline__ void rotate(const float (&a)[4], const float (&b)[4], const float (&sn)[4],
                                       const float (&c)[4], float (&x)[4], float (&y)[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        x[p] = fmaf(a[p], c[p], -b[p] * sn[p]);
        y[p] = fmaf(a[p], sn[p], b[p] * c[p]);
    }
}

// Both halves (elements ia and ib, 4 each) of one rotated row as (hi, lo) bf16 pairs.
__device__ __forceinline__ void store_hilo(const float (&x)[4], const float (&y)[4], uint2 *hi, uint2 *lo, int64_t ia,
                                           int64_t ib) {
    uint32_t xh[2], yh[2], xl[2], yl[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        xh[p] = pack2(x[2 * p], x[2 * p + 1]);
        yh[p] = pack2(y[2 * p], y[2 * p + 1]);
        // the rounding residues x - bf16(x), exact in fp32, rounded to bf16 in turn
        xl[p] = pack2(x[2 * p] - __uint_as_float(xh[p] << 16), x[2 * p + 1] - __uint_as_float(xh[p] & 0xFFFF0000u));
        yl[p] = pack2(y[2 * p] - __uint_as_float(yh[p] << 16), y[2 * p + 1] - __uint_as_float(yh[p] & 0xFFFF0000u));
    }
    hi[ia] = make_uint2(xh[0], xh[1]);
    hi[ib] = make_uint2(yh[0], yh[1]);
    lo[ia] = make_uint2(xl[0], xl[1]);
    lo[ib] = make_uint2(yl[0], yl[1]);
}

// The s sink keys of every (b, h) rotated at their own positions, in fp32: ks[bh][i][.] = R(i) k_i.
// 16 lanes per key row; lane `sub` holds elements 4 sub .. 4 sub + 3 and 64 + 4 sub .. 64 + 4 sub + 3.
__global__ void __launch_bounds__(256) rope_sink_keys_kernel(const uint2 *__restrict__ k, float4 *__restrict__ ks,
                                                             int BH, int64_t L, int s,
                                                             const __grid_constant__ RopePrep rp) {
    const int sub = threadIdx.x % kRopeLanes;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / kRopeLanes) + threadIdx.x / kRopeLanes;
    if (row >= static_cast<int64_t>(BH) * s) return;
    const int64_t bh = row / s;
    const int i = static_cast<int>(row % s);
    const int64_t src = (bh * L + i) * 32 + sub;
    float ka[4], kb[4], sn[4], c[4], x[4], y[4];
    unpack4(__ldg(k + src), ka);
    unpack4(__ldg(k + src + 16), kb);
#pragma unroll
    for (int p = 0; p < kRopePpl; ++p) turn_sincos(static_cast<uint32_t>(i), rp.frac[sub * kRopePpl + p], sn[p], c[p]);
    rotate(ka, kb, sn, c, x, y);
    ks[row * 32 + sub] = make_float4(x[0], x[1], x[2], x[3]);
    ks[row * 32 + 16 + sub] = make_float4(y[0], y[1], y[2], y[3]);
}

// Rows of [BH, L, 128] bf16 viewed as 32 uint2 each: lane `sub` of a row holds elements 4 sub .. 4 sub + 3
// (uint2 index sub) and their partners 64 + 4 sub .. (uint2 index 16 + sub).
struct RopeOut {
    uint2 *qr, *qr_lo, *kr, *kr_lo;
    float *ssink;      // [BH, L, sstride] (s > 0)
    const float4 *ks;  // [BH, s, 128] rotated sink keys (s > 0)
    int s, sstride;
};
__global__ void __launch_bounds__(256) rope_prep_kernel(const uint2 *__restrict__ q, const uint2 *__restrict__ k,
                                                        const RopeOut out, int64_t rows, int64_t L, int w,
                                                        const __grid_constant__ RopePrep rp) {
    const int sub = threadIdx.x % kRopeLanes;
    uint2 f[kRopePpl];
#pragma unroll
    for (int p = 0; p < kRopePpl; ++p) {
        f[p] = rp.frac[sub * kRopePpl + p];
        asm volatile("" : "+r"(f[p].x), "+r"(f[p].y));  // keep them in registers, not re-read per row
    }
    // the sink rotation of every row t >= w - 1: angle (w - 1) theta_i
    float sw[kRopePpl], cw[kRopePpl];
#pragma unroll
    for (int p = 0; p < kRopePpl; ++p) turn_sincos(static_cast<uint32_t>(w - 1), f[p], sw[p], cw[p]);

    const int rows_per_cta = blockDim.x / kRopeLanes;
    const int64_t step = static_cast<int64_t>(gridDim.x) * rows_per_cta;
    // A warp holds two rows (lanes 0-15 and 16-31).  Both halves walk the loop together, a half whose row is
    // past the end only idling, so that the 16-lane shuffles below always have the whole warp.
    // Each pass of the loop takes two row pairs, `step` apart, and issues the loads of both before working on
    // either, so that twice the bytes are in flight per thread.
    const int64_t first = static_cast<int64_t>(blockIdx.x) * rows_per_cta + (threadIdx.x / 32) * 2;
    for (int64_t pair0 = first; pair0 < rows; pair0 += 2 * step) {
      uint2 ld[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int64_t row = pair0 + u * step + (threadIdx.x / kRopeLanes) % 2;
        const int64_t ia = row * 32 + sub, ib = ia + 16;
        if (row < rows) {
            ld[u][0] = __ldg(q + ia);
            ld[u][1] = __ldg(q + ib);
            ld[u][2] = __ldg(k + ia);
            ld[u][3] = __ldg(k + ib);
        } else {
            ld[u][0] = ld[u][1] = ld[u][2] = ld[u][3] = make_uint2(0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int64_t row = pair0 + u * step + (threadIdx.x / kRopeLanes) % 2;
        const bool valid = row < rows;
        const int64_t t = row % L;
        const int64_t ia = row * 32 + sub, ib = ia + 16;
        float x[4] = {0.f, 0.f, 0.f, 0.f}, y[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid) {
            float qa[4], qb[4], ka[4], kb[4];
            unpack4(ld[u][0], qa);
            unpack4(ld[u][1], qb);
            unpack4(ld[u][2], ka);
            unpack4(ld[u][3], kb);
            float sn[kRopePpl], c[kRopePpl];
#pragma unroll
            for (int p = 0; p < kRopePpl; ++p) turn_sincos(static_cast<uint32_t>(t), f[p], sn[p], c[p]);
            rotate(ka, kb, sn, c, x, y);
            store_hilo(x, y, out.kr, out.kr_lo, ia, ib);
            rotate(qa, qb, sn, c, x, y);
            store_hilo(x, y, out.qr, out.qr_lo, ia, ib);
            // the query at min(t, w - 1) for the sink scores: the same rotation below w - 1
            if (t >= w - 1) rotate(qa, qb, sw, cw, x, y);
        }
        if (out.s > 0) {
            // the query against each rotated sink key: dot products over the 16 lanes of the row, four sinks at a
            // time, reduced by halving the four values across the lanes (5 shuffles for 4 sums): after the steps
            // over lane bits 3 and 2 each lane keeps the partial of sink 2 b3 + b2, and after bits 1 and 0 lanes
            // 0, 4, 8, 12 hold the sums of sinks 0, 1, 2, 3
            const float4 *ksr = out.ks + (valid ? row / L : 0) * out.s * 32;
            for (int i0 = 0; i0 < out.s; i0 += 4) {
                float p[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    p[u] = 0.f;
                    if (valid && i0 + u < out.s) {
                        const float4 a = ksr[(i0 + u) * 32 + sub], b = ksr[(i0 + u) * 32 + 16 + sub];
                        float part = x[0] * a.x;
                        part = fmaf(x[1], a.y, part);
                        part = fmaf(x[2], a.z, part);
                        part = fmaf(x[3], a.w, part);
                        part = fmaf(y[0], b.x, part);
                        part = fmaf(y[1], b.y, part);
                        part = fmaf(y[2], b.z, part);
                        part = fmaf(y[3], b.w, part);
                        p[u] = part;
                    }
                }
                // lane bit 3: the lower half keeps sinks 0, 1, the upper half sinks 2, 3
                const bool hi3 = (sub & 8) != 0;
                const float s0 = __shfl_xor_sync(0xFFFFFFFFu, hi3 ? p[0] : p[2], 8, kRopeLanes);
                const float s1 = __shfl_xor_sync(0xFFFFFFFFu, hi3 ? p[1] : p[3], 8, kRopeLanes);
                const float q0 = (hi3 ? p[2] : p[0]) + s0;
                const float q1 = (hi3 ? p[3] : p[1]) + s1;
                // lane bit 2: keep the first or the second of the two
                const bool hi2 = (sub & 4) != 0;
                float v = (hi2 ? q1 : q0) + __shfl_xor_sync(0xFFFFFFFFu, hi2 ? q0 : q1, 4, kRopeLanes);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 2, kRopeLanes);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 1, kRopeLanes);
                const int i = i0 + (sub >> 2);
                if (valid && (sub & 3) == 0 && i < out.s) out.ssink[row * out.sstride + i] = v;
            }
        }
      }
    }
}

int rope_sink_stride(int s) { return (s + 3) & ~3; }

// Workspace: Qr, Qr_lo, Kr, Kr_lo ([BH, L, d] bf16 each), the sink scores ([BH, L, sstride] fp32) and the rotated
// sink keys ([BH, s, d] fp32), one after the other.
size_t rope_prefill_workspace_bytes(int BH, int64_t L, int d, int s) {
    const size_t rows = static_cast<size_t>(BH) * static_cast<size_t>(L);
    const size_t one = rows * static_cast<size_t>(d) * 2;
    return 4 * one + rows * rope_sink_stride(s) * 4 + static_cast<size_t>(BH) * s * d * 4;
}

RopeParts rope_parts(void *workspace, int BH, int64_t L, int d, int s) {
    char *ws = static_cast<char *>(workspace);
    const size_t rows = static_cast<size_t>(BH) * static_cast<size_t>(L);
    const size_t one = rows * static_cast<size_t>(d) * 2;
    char *ssink = ws + 4 * one;
    char *ks = ssink + rows * rope_sink_stride(s) * 4;
    return RopeParts{ws, ws + one, ws + 2 * one, ws + 3 * one, reinterpret_cast<float *>(ssink),
                     reinterpret_cast<float *>(ks), rope_sink_stride(s)};
}

int launch_rope_prep(const void *q, const void *k, const RopeParts &o, int BH, int64_t L, int d, int w, int s,
                     double base, cudaStream_t stream) {
    if (d != kRopeD) return fail(SWA_ERR_UNSUPPORTED, "rope prefill needs d = %d", kRopeD);
    RopePrep rp{};
    // theta_i / (2 pi) = base^(-2i/d) / (2 pi) < 1/6 in double, rounded to a 64-bit fraction in two 32-bit
    // steps (each exact in double; a carry out of the low step is absorbed by the 64-bit sum)
    for (int i = 0; i < d / 2; ++i) {
        const double fr = std::pow(base, -2.0 * i / d) / 6.283185307179586476925286766559;
        const double hi = std::floor(std::ldexp(fr, 32));
        const double lo = std::nearbyint(std::ldexp(std::ldexp(fr, 32) - hi, 32));
        const uint64_t F = (static_cast<uint64_t>(hi) << 32) + static_cast<uint64_t>(lo);
        rp.frac[i] = make_uint2(static_cast<uint32_t>(F), static_cast<uint32_t>(F >> 32));
    }
    const int rows_per_cta = 256 / kRopeLanes;
    if (s > 0) {
        const int64_t krows = static_cast<int64_t>(BH) * s;
        rope_sink_keys_kernel<<<static_cast<unsigned>((krows + rows_per_cta - 1) / rows_per_cta), 256, 0, stream>>>(
            static_cast<const uint2 *>(k), reinterpret_cast<float4 *>(o.ks), BH, L, s, rp);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "rope sink keys launch: %s", cudaGetErrorString(e));
    }
    const int64_t rows = static_cast<int64_t>(BH) * L;
    const int64_t ctas_needed = (rows + rows_per_cta - 1) / rows_per_cta;
    // one wave: as many CTAs as the SMs hold at once (the loop strides over the rest)
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rope_prep_kernel, 256, 0) != cudaSuccess || per_sm < 1)
        return fail(SWA_ERR_CUDA, "rope prefill pass: device attributes");
    const int64_t wave = static_cast<int64_t>(sms) * per_sm;
    const int ctas = static_cast<int>(ctas_needed < wave ? ctas_needed : wave);
    const RopeOut out{static_cast<uint2 *>(o.qr), static_cast<uint2 *>(o.qr_lo), static_cast<uint2 *>(o.kr),
                      static_cast<uint2 *>(o.kr_lo), o.ssink, reinterpret_cast<const float4 *>(o.ks), s, o.sstride};
    rope_prep_kernel<<<ctas, 256, 0, stream>>>(static_cast<const uint2 *>(q), static_cast<const uint2 *>(k), out,
                                               rows, L, w, rp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "rope prefill pass launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

}  // namespace swa
