// prefill_f32.cu -- fp32 prefill on CUDA cores (the SWA_F32 path of swa_sink_prefill).
//
// One CTA of 128 threads per (query row, b*h).  The key set of query position t is enumerated
// directly as two position ranges: the sinks [0, min(s, t+1)) and the recent window
// [max(s, t-m+1), t] (hyper.ai summary of arXiv 2608.28444, section "带 Sink 的滑动窗口注意力":
// w keys, the first s always attended in addition to the w - s window keys).  Keys are processed
// in blocks of 128: each thread scores one key (dot product in fp32), the block keeps an online
// softmax (running max in log2 units, running sum), and thread c < d accumulates output column c.
//
// A position p < pos0 (chunked prefill) is read from the rolling cache: slot p for a sink, slot
// s + ((p - s) mod m) otherwise; positions >= pos0 come from this call's k/v rows.  This path is
// meant for the small fp32 shapes; the bf16 tensor-core kernel is the fast path.
#include <math.h>

#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {

constexpr int kF32Threads = 128;

__device__ __forceinline__ float block_reduce_max(float x, float *red) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, off));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kF32Threads / 32; ++i) r = fmaxf(r, red[i]);
    return r;
}
__device__ __forceinline__ float block_reduce_sum(float x, float *red) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    float r = 0.f;
#pragma unroll
    for (int i = 0; i < kF32Threads / 32; ++i) r += red[i];
    return r;
}

template <int D>
__global__ void __launch_bounds__(kF32Threads) prefill_f32_kernel(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v, float *__restrict__ o,
    float *__restrict__ lse, const float *__restrict__ kc, const float *__restrict__ vc, int64_t pos0, int w, int s,
    float scale_log2, int64_t seq_stride) {
    __shared__ float qs[D];
    __shared__ float ps[kF32Threads];
    __shared__ int64_t rows[kF32Threads];  // element offset of each key's row (k and v share it)
    __shared__ unsigned char from_cache[kF32Threads];
    __shared__ float red[kF32Threads / 32];

    const int64_t r = blockIdx.x;
    const int64_t bh = blockIdx.y;
    const int64_t t = pos0 + r;
    const int m = w - s;
    const int tid = threadIdx.x;
    const int64_t qrow = (bh * seq_stride + r) * D;
    if (tid < D) qs[tid] = q[qrow + tid] * scale_log2;

    // key set: sinks [0, ns) and the window [blo, t]
    const int64_t ns = (s < t + 1) ? s : t + 1;
    int64_t blo = t - m + 1;
    if (blo < s) blo = s;
    const int64_t nb = (t >= blo) ? (t - blo + 1) : 0;
    const int64_t nkeys = ns + nb;

    float mrun = -INFINITY, lrun = 0.f, acc = 0.f;
    for (int64_t base = 0; base < nkeys; base += kF32Threads) {
        __syncthreads();
        float x = -INFINITY;
        const int64_t j = base + tid;
        if (j < nkeys) {
            const int64_t p = (j < ns) ? j : blo + (j - ns);
            int64_t off;
            bool cache;
            if (p >= pos0) {
                off = (bh * seq_stride + (p - pos0)) * D;
                cache = false;
            } else {
                const int64_t slot = (p < s) ? p : s + (p - s) % m;
                off = (bh * w + slot) * D;
                cache = true;
            }
            rows[tid] = off;
            from_cache[tid] = cache;
            const float *kr = (cache ? kc : k) + off;
            float dot = 0.f;
#pragma unroll 16
            for (int c = 0; c < D; ++c) dot = fmaf(qs[c], kr[c], dot);
            x = dot;
        }
        const float mx = block_reduce_max(x, red);
        const float mn = fmaxf(mrun, mx);
        const float alpha = exp2f(mrun - mn);
        const float p = (j < nkeys) ? exp2f(x - mn) : 0.f;
        ps[tid] = p;
        const float psum = block_reduce_sum(p, red);  // also publishes ps/rows (barriers inside)
        lrun = lrun * alpha + psum;
        mrun = mn;
        if (tid < D) {
            float a = acc * alpha;
            const int64_t cnt = (nkeys - base < kF32Threads) ? nkeys - base : kF32Threads;
            for (int i = 0; i < cnt; ++i) {
                const float *vr = (from_cache[i] ? vc : v) + rows[i];
                a = fmaf(ps[i], vr[tid], a);
            }
            acc = a;
        }
    }
    if (tid < D) o[qrow + tid] = acc / lrun;
    if (tid == 0 && lse) lse[bh * seq_stride + r] = (mrun + log2f(lrun)) * 0.69314718055994531f;
}

int launch_prefill_f32(const PrefillArgs &a) {
    if (a.L > 0x7FFFFFFF) return fail(SWA_ERR_UNSUPPORTED, "fp32 prefill: L too large");
    if (a.BH > 65535) return fail(SWA_ERR_UNSUPPORTED, "fp32 prefill: B*H=%d > 65535", a.BH);
    const dim3 grid(static_cast<unsigned>(a.L), a.BH), block(kF32Threads);
    const float sl2 = a.scale * 1.4426950408889634f;
    const float *q = static_cast<const float *>(a.q), *k = static_cast<const float *>(a.k),
                *v = static_cast<const float *>(a.v), *kc = static_cast<const float *>(a.k_cache),
                *vc = static_cast<const float *>(a.v_cache);
    float *o = static_cast<float *>(a.o);
    switch (a.d) {
        case 16: prefill_f32_kernel<16><<<grid, block, 0, a.stream>>>(q, k, v, o, a.lse, kc, vc, a.pos0, a.w, a.s, sl2, a.seq_stride); break;
        case 32: prefill_f32_kernel<32><<<grid, block, 0, a.stream>>>(q, k, v, o, a.lse, kc, vc, a.pos0, a.w, a.s, sl2, a.seq_stride); break;
        case 64: prefill_f32_kernel<64><<<grid, block, 0, a.stream>>>(q, k, v, o, a.lse, kc, vc, a.pos0, a.w, a.s, sl2, a.seq_stride); break;
        case 128: prefill_f32_kernel<128><<<grid, block, 0, a.stream>>>(q, k, v, o, a.lse, kc, vc, a.pos0, a.w, a.s, sl2, a.seq_stride); break;
        default: return fail(SWA_ERR_UNSUPPORTED, "fp32 prefill: d=%d", a.d);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "fp32 prefill launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

}  // namespace swa
