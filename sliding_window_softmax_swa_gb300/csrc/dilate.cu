// dilate.cu -- the dilated-window prefill's passes outside the tensor-core kernel.
//
// The dilated sliding window of "滑窗与固定稀疏" (glossary and Longformer section) lets the attended window
// positions skip r - 1 tokens: causal, with the sinks of the StreamingLLM section, row t attends
//     K_r(t) = {i < s} | {t - j r : 0 <= j < m},  m = w - s,  restricted to i <= t.
// Re-laid out, this is the plain band with sinks.  Virtual head (c, b, h), c = 0 .. r-1, is the sequence
// positions 0 .. s-1 (the sinks), then the positions p >= s with p = c (mod r), increasing.  A row t >= s of
// class c = t mod r sits in it after the sinks, and its plain key set there -- the sinks and the m rows back
// from it -- holds exactly the sinks and t, t - r, ..., t - (m-1) r (those below s are sinks anyway).  A row
// t < s attends {0 .. t}.
//
// bf16 with d = 128 runs in place: the tensor-core prefill reads the virtual heads straight from q, k, v through
// 4-D tensor maps (d, class, group, (b, h)), position = group * r + class, and writes every row at its own
// position; it covers the rows [s, G r), G = L / r, and dilated_rows_kernel below the others (the sink rows and
// the last L mod r rows, whose group is not whole).  Every other form (fp32, d = 64, the chunked prefill that
// fills the per-class caches) gathers q, k, v into the virtual heads, runs the plain prefill on them and
// scatters o back: two HBM-bound passes of 16-byte copies; the rows past the end of a shorter class are zero
// and, lying after every real row, are never attended.
#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {

// Rows of one virtual head: the s sinks (or all L rows when L <= s) and the longest residue class >= s.
int64_t dilated_rows(int64_t L, int s, int r) {
    const int64_t head = L < s ? L : s;
    const int64_t tail = L > s ? (L - s + r - 1) / r : 0;
    return head + tail;
}

// How the in-place dilated prefill splits the rows of a (b, h): the tensor-core pass over the whole groups of r
// positions after the sinks ([s, G r), G = L / r; every class runs over the rows of the longest class), the
// CUDA-core pass over [0, ns) and [tail0, L).
DilatedSplit dilated_split(int64_t L, int s, int r) {
    DilatedSplit d;
    d.G = L / r;
    d.nrows = d.G * r > s ? (d.G * r - s + r - 1) / r : 0;
    d.ns = L < s ? L : s;
    d.tail0 = d.G * r > d.ns ? d.G * r : d.ns;
    return d;
}

// Original position of row u of virtual head class c, or -1 past the end of the sequence.
__device__ __forceinline__ int64_t dilated_source(int64_t u, int c, int s, int r, int64_t L) {
    if (u < s) return u < L ? u : -1;
    const int64_t p0 = s + ((c - s) % r + r) % r;  // the first position >= s of class c
    const int64_t p = p0 + (u - s) * r;
    return p < L ? p : -1;
}

__global__ void __launch_bounds__(256) dilate_gather_kernel(const uint4 *__restrict__ q, const uint4 *__restrict__ k,
                                                            const uint4 *__restrict__ v, uint4 *__restrict__ qv,
                                                            uint4 *__restrict__ kv, uint4 *__restrict__ vv, int BH,
                                                            int64_t L, int64_t Lv, int s, int r, int chunks) {
    const int64_t total = static_cast<int64_t>(BH) * r * Lv * chunks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int ch = static_cast<int>(i % chunks);
        const int64_t row = i / chunks;  // (vh, u), vh = c * BH + bh
        const int64_t u = row % Lv;
        const int64_t vh = row / Lv;
        const int c = static_cast<int>(vh / BH);
        const int64_t bh = vh % BH;
        const int64_t p = dilated_source(u, c, s, r, L);
        uint4 a = make_uint4(0, 0, 0, 0), b = a, e = a;
        if (p >= 0) {
            const int64_t src = (bh * L + p) * chunks + ch;
            a = __ldg(q + src);
            b = __ldg(k + src);
            e = __ldg(v + src);
        }
        qv[i] = a;
        kv[i] = b;
        vv[i] = e;
    }
}

__global__ void __launch_bounds__(256) dilate_scatter_kernel(const uint4 *__restrict__ ov,
                                                             const float *__restrict__ lsev, uint4 *__restrict__ o,
                                                             float *__restrict__ lse, int BH, int64_t L, int64_t Lv,
                                                             int s, int r, int chunks) {
    const int64_t total = static_cast<int64_t>(BH) * L * chunks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int ch = static_cast<int>(i % chunks);
        const int64_t row = i / chunks;  // (bh, t)
        const int64_t t = row % L;
        const int64_t bh = row / L;
        int c = 0;
        int64_t u = t;
        if (t >= s) {
            c = static_cast<int>(t % r);
            const int64_t p0 = s + ((c - s) % r + r) % r;
            u = s + (t - p0) / r;
        }
        const int64_t src_row = (static_cast<int64_t>(c) * BH + bh) * Lv + u;
        o[i] = __ldg(ov + src_row * chunks + ch);
        if (lse && ch == 0) lse[row] = __ldg(lsev + src_row);
    }
}

// Rows of the dilated prefill outside the tensor-core pass (bf16, d = 128): rows [0, ns) and [tail0, L) of
// every (b, h), one CTA of 128 threads per row at a time.  Row t attends the sinks [0, min(s, t + 1)) and, when
// t >= s, the positions t, t - r, ... that stay >= s, at most m of them.  The keys go in chunks of 128, one
// key per thread for the fp32 score (bf16 row times the fp32 query), with an online softmax across chunks;
// thread c accumulates output column c in fp32.
__global__ void __launch_bounds__(128) dilated_rows_kernel(const __nv_bfloat16 *__restrict__ q,
                                                           const __nv_bfloat16 *__restrict__ k,
                                                           const __nv_bfloat16 *__restrict__ v,
                                                           __nv_bfloat16 *__restrict__ o, float *__restrict__ lse,
                                                           int BH, int64_t L, int ns, int64_t tail0, int s, int m,
                                                           int r, float sl2) {
    constexpr int D = 128;
    __shared__ float qs[D];
    __shared__ float ps[128];
    __shared__ int64_t pos[128];
    __shared__ float red[4];
    const int c = threadIdx.x, lane = c & 31, wid = c >> 5;
    const int64_t per_bh = ns + (L - tail0);
    const int64_t total = per_bh * BH;
    for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
        const int64_t bh = item / per_bh, i = item % per_bh;
        const int64_t t = i < ns ? i : tail0 + (i - ns);
        const int64_t nsink = t + 1 < s ? t + 1 : s;
        const int64_t nband = t >= s ? ((t - s) / r + 1 < m ? (t - s) / r + 1 : m) : 0;
        const int64_t nk = nsink + nband;
        const __nv_bfloat16 *kb = k + bh * L * D, *vb = v + bh * L * D;
        __syncthreads();  // the previous row is done with qs, pos and ps
        qs[c] = __bfloat162float(q[(bh * L + t) * D + c]);
        float mrun = -INFINITY, l = 0.f, acc = 0.f;
        for (int64_t c0 = 0; c0 < nk; c0 += 128) {
            const int64_t kk = c0 + c;
            const int64_t p = kk < nsink ? kk : t - (kk - nsink) * r;
            pos[c] = p;
            __syncthreads();
            float sc = -INFINITY;
            if (kk < nk) {
                const uint4 *kr = reinterpret_cast<const uint4 *>(kb + p * D);
                float dot = 0.f;
#pragma unroll 4
                for (int j = 0; j < D / 8; ++j) {
                    const uint4 u = __ldg(kr + j);
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        dot = fmaf(__uint_as_float(w4[h] << 16), qs[8 * j + 2 * h], dot);
                        dot = fmaf(__uint_as_float(w4[h] & 0xFFFF0000u), qs[8 * j + 2 * h + 1], dot);
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
            const float mnew = fmaxf(mrun, mx);  // finite: every chunk holds at least one key
            const float alpha = exp2f(mrun - mnew);
            const float pr = kk < nk ? exp2f(sc - mnew) : 0.f;
            ps[c] = pr;
            float sum = pr;
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
            if (lane == 0) red[wid] = sum;
            __syncthreads();
            l = l * alpha + ((red[0] + red[1]) + (red[2] + red[3]));
            acc *= alpha;
            mrun = mnew;
            const int n = nk - c0 < 128 ? static_cast<int>(nk - c0) : 128;
            for (int j = 0; j < n; ++j) acc = fmaf(ps[j], __bfloat162float(vb[pos[j] * D + c]), acc);
            __syncthreads();
        }
        o[(bh * L + t) * D + c] = __float2bfloat16_rn(acc / l);
        if (lse && c == 0) lse[bh * L + t] = (mrun + log2f(l)) * 0.69314718055994531f;
    }
}

static int grid_for(int64_t work) {
    const int64_t ctas = (work + 255) / 256;
    return static_cast<int>(ctas < 152 * 16 ? (ctas < 1 ? 1 : ctas) : 152 * 16);
}

int launch_dilate_gather(const void *q, const void *k, const void *v, void *qv, void *kv, void *vv, int BH, int64_t L,
                         int d, int esize, int s, int r, cudaStream_t stream) {
    const int chunks = d * esize / 16;
    const int64_t Lv = dilated_rows(L, s, r);
    dilate_gather_kernel<<<grid_for(static_cast<int64_t>(BH) * r * Lv * chunks), 256, 0, stream>>>(
        static_cast<const uint4 *>(q), static_cast<const uint4 *>(k), static_cast<const uint4 *>(v),
        static_cast<uint4 *>(qv), static_cast<uint4 *>(kv), static_cast<uint4 *>(vv), BH, L, Lv, s, r, chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "dilated gather launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

int launch_dilate_scatter(const void *ov, const float *lsev, void *o, float *lse, int BH, int64_t L, int d, int esize,
                          int s, int r, cudaStream_t stream) {
    const int chunks = d * esize / 16;
    const int64_t Lv = dilated_rows(L, s, r);
    dilate_scatter_kernel<<<grid_for(static_cast<int64_t>(BH) * L * chunks), 256, 0, stream>>>(
        static_cast<const uint4 *>(ov), lsev, static_cast<uint4 *>(o), lse, BH, L, Lv, s, r, chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "dilated scatter launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

int launch_dilated_rows(const PrefillArgs &a, int r) {
    const int64_t L = a.L;
    const DilatedSplit sp = dilated_split(L, a.s, r);
    const int ns = static_cast<int>(sp.ns);
    const int64_t tail0 = sp.tail0;
    const int64_t rows = static_cast<int64_t>(a.BH) * (ns + (L - tail0));
    if (rows == 0) return SWA_OK;
    const int grid = static_cast<int>(rows < 152 * 16 ? rows : 152 * 16);
    dilated_rows_kernel<<<grid, 128, 0, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
        static_cast<const __nv_bfloat16 *>(a.v), static_cast<__nv_bfloat16 *>(a.o), a.lse, a.BH, L, ns, tail0, a.s,
        a.w - a.s, r, a.scale * 1.4426950408889634f);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "dilated rows launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

}  // namespace swa
