// kv_write.cu -- kv_rolling_write: copy the keys/values of positions pos0..pos0+n-1 into the rolling
// cache of w = s + m slots.  Position p goes to slot p if p < s (the sink block) and to slot
// s + ((p - s) mod m) otherwise (the recent ring), the layout of the StreamingLLM cache
// (page "滑窗与固定稀疏", eq attn-fixed-streaming; with s = 0 the rolling buffer i mod W of eq
// attn-fixed-rolling).
//
// Only the last writer of each slot is copied: of the positions >= s in the batch only the last m can
// survive, and those map to m distinct slots.  So every (slot, 16-byte chunk) is written at most once
// per call and no ordering between threads is needed; the result equals writing the positions one by
// one.  The copy is a grid-stride loop of 16-byte vector loads/stores (HBM-bound, trivially small in
// decode: one row per (b, h) per step).
#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {

template <int CHUNKS>  // 16-byte chunks per row: d * esize / 16
__global__ void __launch_bounds__(256) kv_write_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                                                       const uint4 *__restrict__ kn, const uint4 *__restrict__ vn,
                                                       int BH, int w, int s, int64_t pos0, int64_t src_stride,
                                                       int64_t n_sink, int64_t ring_first, int64_t count, int nclass,
                                                       int64_t class_stride) {
    const int64_t m = w - s;
    const int64_t total = static_cast<int64_t>(BH) * count * CHUNKS;
    // grid.y walks the caches that receive the same rows (nclass > 1: the per-class caches of the dilated
    // window, class_stride 16-byte chunks apart, each getting a sink)
    for (int cls = static_cast<int>(blockIdx.y); cls < nclass; cls += static_cast<int>(gridDim.y)) {
        const int64_t cbase = static_cast<int64_t>(cls) * class_stride;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
             i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const int c = static_cast<int>(i % CHUNKS);
            const int64_t r = i / CHUNKS;
            const int64_t j = r % count;
            const int64_t bh = r / count;
            const int64_t p = (j < n_sink) ? pos0 + j : ring_first + (j - n_sink);
            const int64_t slot = (p < s) ? p : s + (p - s) % m;
            const int64_t src = (bh * src_stride + (p - pos0)) * CHUNKS + c;
            const int64_t dst = cbase + (bh * w + slot) * CHUNKS + c;
            const uint4 kx = __ldg(kn + src);
            kc[dst] = kx;
            if (vn != nullptr) vc[dst] = __ldg(vn + src);  // keys only when no values are given
        }
    }
}

int launch_kv_write_classes(void *k_cache, void *v_cache, const void *k_new, const void *v_new, int BH, int d, int w,
                            int s, int64_t pos0, int64_t n, int64_t src_stride, int esize, int nclass,
                            cudaStream_t stream) {
    if (n <= 0 || nclass <= 0) return SWA_OK;
    const int64_t m = w - s;
    // sinks among the new positions: [pos0, min(s, pos0 + n))
    const int64_t n_sink = (pos0 < s) ? ((s < pos0 + n ? s : pos0 + n) - pos0) : 0;
    // ring positions that survive: the last m positions >= s of the batch
    int64_t ring_first = pos0 + n - m;
    if (ring_first < s) ring_first = s;
    if (ring_first < pos0) ring_first = pos0;
    const int64_t n_ring = (pos0 + n > ring_first) ? (pos0 + n - ring_first) : 0;
    const int64_t count = n_sink + n_ring;
    if (count == 0) return SWA_OK;
    const int chunks = d * esize / 16;
    const int64_t total = static_cast<int64_t>(BH) * count * chunks;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    int64_t ycls = nclass;
    while (ycls > 1 && blocks * ycls > 152 * 32) ycls = (ycls + 1) / 2;  // bound the grid; y loops over the rest
    const int64_t class_stride = static_cast<int64_t>(BH) * w * chunks;  // one cache, in 16-byte chunks
    uint4 *kc = static_cast<uint4 *>(k_cache);
    uint4 *vc = static_cast<uint4 *>(v_cache);
    const uint4 *kn = static_cast<const uint4 *>(k_new);
    const uint4 *vn = static_cast<const uint4 *>(v_new);
    const dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(ycls)), block(256);
#define SWA_KVW(C)                                                                                                 \
    kv_write_kernel<C><<<grid, block, 0, stream>>>(kc, vc, kn, vn, BH, w, s, pos0, src_stride, n_sink, ring_first, \
                                                   count, nclass, class_stride)
    switch (chunks) {
        case 2: SWA_KVW(2); break;
        case 4: SWA_KVW(4); break;
        case 8: SWA_KVW(8); break;
        case 16: SWA_KVW(16); break;
        case 32: SWA_KVW(32); break;
        default: return fail(SWA_ERR_UNSUPPORTED, "kv_rolling_write: row of %d bytes", d * esize);
    }
#undef SWA_KVW
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "kv_rolling_write launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

int launch_kv_write(void *k_cache, void *v_cache, const void *k_new, const void *v_new, int BH, int d, int w, int s,
                    int64_t pos0, int64_t n, int64_t src_stride, int esize, cudaStream_t stream) {
    return launch_kv_write_classes(k_cache, v_cache, k_new, v_new, BH, d, w, s, pos0, n, src_stride, esize, 1, stream);
}

}  // namespace swa
