// dilate.cu -- the layout passes of prefill over a dilated window with sinks.
//
// The dilated sliding window of "滑窗与固定稀疏" (glossary and Longformer section) lets the attended window
// positions skip r - 1 tokens: causal, with the sinks of the StreamingLLM section, row t attends
//     K_r(t) = {i < s} | {t - j r : 0 <= j < m},  m = w - s, restricted to i <= t.
// Re-laid out, this is the plain band with sinks of the tensor-core prefill.  Virtual head (c, b, h),
// c = 0 .. r-1 (class-major: the layout of the streaming decode's per-class caches), is the sequence
//     positions 0 .. s-1 (the sinks), then the positions p >= s with p = c (mod r), increasing.
// A row t >= s of class c = t mod r sits in it after the sinks, and its plain key set there -- the sinks
// and the m rows back from it -- holds exactly the sinks and t, t - r, ..., t - (m-1) r (those below s
// are sinks anyway).  A row t < s attends {0 .. t} = the sink prefix of any virtual head, so head c = 0
// supplies it.  So: gather q, k, v into the virtual heads, run the prefill unchanged (s sinks, window
// w), and scatter the rows back.  Both passes are HBM-bound 16-byte copies; the rows past the end of a
// shorter class are zero and, lying after every real row, are never attended.
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

}  // namespace swa
