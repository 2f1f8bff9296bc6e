// hybrid.cu -- sliding-window softmax attention with sinks plus a linear-attention branch for the keys that
// have left the window (the SWA / linear-attention hybrid of the hyper.ai summary of arXiv 2608.28444, its
// linear-attention section: running state s_t = s_{t-1} + phi(k_t)^T v_t, z_t = z_{t-1} + phi(k_t)^T, and the
// Hedgehog feature map phi(x) = (exp(f(x)), exp(-f(x))), f(x) = x wf with wf a d x d/2 projection).  The two
// branches share one normaliser (the LoLCATs reading that summary discusses):
//     o_t = (sum_{i in K(t)} e^{x_i} v_i + phi(q_t) S_t) / (sum_{i in K(t)} e^{x_i} + phi(q_t) z_t),
// K(t) the sinks + window, S_t, z_t the sums over the keys s <= i <= t - m that left it (the sinks never do).
// With the SWA prefill's output o' and lse the first terms are o' e^{lse} and e^{lse}, so
//     o_t = (o'_t + phi(q_t) S_t e^{-lse_t}) / (1 + phi(q_t) z_t e^{-lse_t}).
//
// Prefill (bf16, d = 128), all contractions on the tensor cores (tcgen05, operands in 128-byte-swizzled
// shared memory, fp32 accumulators in TMEM), with W2 = [wf^T ; -wf^T] (128 x d) so that one product gives
// both halves of f and phi is exp of it:
//   1. chunk states, per (head, key chunk j of 128 keys): f(K_j)^T = W2 K_j^T, phi(K_j)^T = exp(.) with the
//      sinks and the keys past the end zeroed (kept, bf16, for step 3), D_j = phi(K_j)^T V_j (d x d, stored as
//      bf16) and z_j = phi(K_j)^T 1 (fp32);
//   2. an exclusive scan over j in place, summed in fp32: P_j = sum_{j' < j} D_j' (the state of the keys before
//      chunk j, bf16: it enters the tensor cores as an operand);
//   3. per (head, query tile of 128 rows at a): J = floor((a - m + 1) / 128) (every key below 128 J has left
//      the window of every row of the tile), then
//          num = phi(Q) P_J + sum over the <= 2 key tiles from 128 J: (phi(Q) phi(K)^T masked to i <= t - m,
//                i >= s) V,   den = phi(Q) z_J + the masked row sums,
//      and the combination above, in place over the SWA prefill's output.
// Decode: per (b, h) one pass over the state: fold the key that leaves the window at this step (it sits in
// the rolling slot the new key goes to) into S and z, write the new key and value into that slot, and form
// phi(q) S and phi(q) z; the SWA decode step with lse follows, then the combination.
#include <cuda_bf16.h>
#include <math.h>

#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {
namespace hy {

constexpr int D = 128;                      // head dimension (and feature dimension of phi)
constexpr int C = 128;                      // keys per chunk / rows per query tile
constexpr uint32_t HALF = 128 * 128;        // one 64-column half of a [128 x 128] bf16 tile
constexpr uint32_t TILE = 2 * HALF;
constexpr uint32_t IDESC_KK = idesc_bf16_f32(128, 128, false, false);  // A K-major, B K-major (A B^T)
constexpr uint32_t IDESC_KM = idesc_bf16_f32(128, 128, false, true);   // A K-major, B MN-major (A B)
constexpr float LOG2E = 1.4426950408889634f;

// D (+)= A B^T: A and B [128 x 128] tiles whose rows are M (resp. N) and whose columns are K.
__device__ __forceinline__ void mma_abt(uint32_t d, uint32_t a, uint32_t b, bool acc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
        umma_ss(d, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), IDESC_KK, (acc || kk) ? 1u : 0u);
    }
}
// D (+)= A B: A [128 x 128] with rows M and columns K, B [128 x 128] with rows K and columns N.
__device__ __forceinline__ void mma_ab(uint32_t d, uint32_t a, uint32_t b, bool acc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a_off = (kk >> 2) * HALF + (kk & 3) * 32;
        umma_ss(d, sdesc_sw128(a + a_off, 16, 1024), sdesc_sw128(b + kk * 2048, HALF, 1024), IDESC_KM,
                (acc || kk) ? 1u : 0u);
    }
}

// Row r, columns c0..c0+31 of a [128 x 128] bf16 tile in the swizzled two-half layout, from 32 floats.
__device__ __forceinline__ void st_row32(uint32_t tile, int r, int c0, const float (&x)[32]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int c = c0 + 8 * g;
        st_shared_v4(tile + (c >> 6) * HALF + sw128_offset(r, c & 63), pack_bf16x2(x[8 * g], x[8 * g + 1]),
                     pack_bf16x2(x[8 * g + 2], x[8 * g + 3]), pack_bf16x2(x[8 * g + 4], x[8 * g + 5]),
                     pack_bf16x2(x[8 * g + 6], x[8 * g + 7]));
    }
}

// W2 = [wf^T ; -wf^T] as a row-major [128 x d] bf16 image in global memory (TMA-loaded by the kernels below);
// grid 128 (row j = feature j) x 128 threads (column x).
__global__ void __launch_bounds__(128) w2_kernel(const __nv_bfloat16 *__restrict__ wf, __nv_bfloat16 *w2) {
    const int j = blockIdx.x, x = threadIdx.x;
    const uint16_t sign = j >= 64 ? 0x8000u : 0u;
    w2[j * D + x] = __ushort_as_bfloat16(__bfloat16_as_ushort(wf[x * (D / 2) + (j & 63)]) ^ sign);
}

// TMEM address of this warp's 32 lanes (warp w may access lanes 32 (w mod 4) .. +31) at column col.
__device__ __forceinline__ uint32_t lane_addr(uint32_t tmem, int col) {
    return tmem + (static_cast<uint32_t>(((threadIdx.x >> 5) & 3) * 32) << 16) + col;
}

// Shared state of one CTA: barriers, TMEM base, abort flag.
struct Ctl {
    uint64_t load_bar, mma_bar;
    uint32_t tmem;
    int abort_flag;
};

// TMA of a [128 rows x 128] bf16 tile (two 64-column boxes) of (bh, row0); one thread.
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *m, uint64_t *bar, int row0, int bh) {
    tma_load_3d(dst, m, bar, 0, row0, bh);
    tma_load_3d(dst + HALF, m, bar, 64, row0, bh);
}

// Wait for the MMAs committed to mma_bar (phase `ph`) on every thread; false once any wait of the CTA gave up.
__device__ __forceinline__ bool wait_mma(Ctl *ctl, int ph, const WaitCtl &wc, unsigned site) {
    const bool ok = __syncthreads_and(mbar_wait(&ctl->mma_bar, ph & 1, wc, site));
    tc_fence_after();
    return ok;
}

// Issue (thread 0) after shared-memory operand writes by all threads.
__device__ __forceinline__ void operands_written() {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// ---- 1. chunk states ------------------------------------------------------------------------------
// grid (chunks, BH), 128 threads.  Key chunk j: keys j*C .. j*C + C - 1; a key counts when s <= key < key_end.
// Writes, per (bh, j): dmat = D_j = phi(K_j)^T V_j (bf16, row = feature, column = value column), zst = z_j
// (fp32) and phik = phi(K_j)^T (bf16, row = feature, column = key of the chunk), each [BH][chunks][128][...].
// Final mode (fin_s != nullptr): one chunk per head (index chunk0); the scanned prefix of that chunk (dmat,
// zst after the scan) is added to its D and z, and the sums go to fin_s [BH][d][d] and fin_z [BH][d] (fp32).
__global__ void __launch_bounds__(128, 1) chunk_state_kernel(const __grid_constant__ CUtensorMap mk,
                                                             const __grid_constant__ CUtensorMap mv,
                                                             const __grid_constant__ CUtensorMap mw2,
                                                             __nv_bfloat16 *dmat, float *zst, __nv_bfloat16 *phik,
                                                             float *fin_s, float *fin_z, int chunk0, int nchunks,
                                                             int s, int64_t key_end, DeviceStatus *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *Tw = sm, *Tk = sm + TILE, *Tv = sm + 2 * TILE;
    Ctl *ctl = reinterpret_cast<Ctl *>(sm + 3 * TILE);
    const int j = chunk0 + static_cast<int>(blockIdx.x), bh = blockIdx.y, r = threadIdx.x;
    const bool fin = fin_s != nullptr;
    const int64_t rec = static_cast<int64_t>(bh) * nchunks + j;  // (bh, chunk) record index
    if (r == 0) {
        ctl->abort_flag = 0;
        mbar_init(&ctl->load_bar, 1);
        mbar_init(&ctl->mma_bar, 1);
        mbar_init_fence();
    }
    if (r < 32) {
        tmem_alloc(&ctl->tmem, 256);
        tmem_relinquish();
    }
    operands_written();
    const uint32_t tmem = ctl->tmem;
    const WaitCtl wc{smem_u32(&ctl->abort_flag), kWaitTimeoutUs, status};
    if (r == 0) {
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        mbar_arrive_expect_tx(&ctl->load_bar, 3 * TILE);
        load_tile(Tw, &mw2, &ctl->load_bar, 0, 0);
        load_tile(Tk, &mk, &ctl->load_bar, j * C, bh);
        load_tile(Tv, &mv, &ctl->load_bar, j * C, bh);
        if (mbar_wait(&ctl->load_bar, 0, wc, 40)) {
            tc_fence_after();
            mma_abt(tmem, smem_u32(Tw), smem_u32(Tk), false);  // f(K)^T: [feature][key]
        } else {
            mbar_wait_drain(&ctl->load_bar, 0);
        }
        umma_commit(&ctl->mma_bar);
    }
    bool fine = wait_mma(ctl, 0, wc, 41);
    float z = 0.f;
    if (fine) {
        // phi(K)^T row r (feature r) over the 128 keys; uncounted keys are zero
        const int64_t k0 = static_cast<int64_t>(j) * C;
        uint4 *prow = reinterpret_cast<uint4 *>(phik + (rec * D + r) * C);
        for (int c0 = 0; c0 < C; c0 += 32) {
            float x[32];
            tmem_ld32(lane_addr(tmem, c0), x);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int64_t key = k0 + c0 + i;
                x[i] = (key >= s && key < key_end) ? exp2f(x[i] * LOG2E) : 0.f;
                z += x[i];
            }
            st_row32(smem_u32(Tk), r, c0, x);
            if (!fin) {
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    prow[c0 / 8 + g] = make_uint4(pack_bf16x2(x[8 * g], x[8 * g + 1]), pack_bf16x2(x[8 * g + 2], x[8 * g + 3]),
                                                  pack_bf16x2(x[8 * g + 4], x[8 * g + 5]), pack_bf16x2(x[8 * g + 6], x[8 * g + 7]));
            }
        }
    }
    operands_written();
    if (r == 0) {
        if (fine) mma_ab(tmem + 128, smem_u32(Tk), smem_u32(Tv), false);  // phi(K)^T V: [feature][column]
        umma_commit(&ctl->mma_bar);
    }
    fine = wait_mma(ctl, 1, wc, 42) && fine;
    if (fine) {
        const __nv_bfloat16 *pre = dmat + (rec * D + r) * D;
        for (int c0 = 0; c0 < D; c0 += 32) {
            float x[32];
            tmem_ld32(lane_addr(tmem, 128 + c0), x);
            if (fin) {  // + the prefix, to fp32
                const uint4 *pp = reinterpret_cast<const uint4 *>(pre + c0);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint4 u = pp[g];
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        x[8 * g + 2 * h] += __uint_as_float(w4[h] << 16);
                        x[8 * g + 2 * h + 1] += __uint_as_float(w4[h] & 0xFFFF0000u);
                    }
                }
                float4 *p4 = reinterpret_cast<float4 *>(fin_s + (static_cast<int64_t>(bh) * D + r) * D + c0);
#pragma unroll
                for (int i = 0; i < 8; ++i) p4[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
            } else {
                uint4 *pd = reinterpret_cast<uint4 *>(dmat + (rec * D + r) * D + c0);
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    pd[g] = make_uint4(pack_bf16x2(x[8 * g], x[8 * g + 1]), pack_bf16x2(x[8 * g + 2], x[8 * g + 3]),
                                       pack_bf16x2(x[8 * g + 4], x[8 * g + 5]), pack_bf16x2(x[8 * g + 6], x[8 * g + 7]));
            }
        }
        if (fin)
            fin_z[static_cast<int64_t>(bh) * D + r] = z + zst[rec * D + r];
        else
            zst[rec * D + r] = z;
    }
    tc_fence_before();
    __syncthreads();
    if (r < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ---- 2. exclusive scan over the chunks, in place: per (bh, pair of matrix entries) in bf16 with an fp32
// running sum, per (bh, feature) for z in fp32 ---------------------------------------------------------------
__global__ void __launch_bounds__(256) scan_kernel(uint32_t *dmat, float *zst, int nchunks, int64_t npairs,
                                                   int64_t nz) {
    const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    constexpr int PAIRS = D * D / 2;  // bf16 pairs per record
    if (e < npairs) {
        const int64_t bh = e / PAIRS, k = e % PAIRS;
        uint32_t *p = dmat + bh * nchunks * PAIRS + k;
        float r0 = 0.f, r1 = 0.f;
        for (int j0 = 0; j0 < nchunks; j0 += 16) {  // 16 independent loads in flight, then their prefix
            uint32_t x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (j0 + i < nchunks) x[i] = p[static_cast<int64_t>(j0 + i) * PAIRS];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (j0 + i < nchunks) {
                    p[static_cast<int64_t>(j0 + i) * PAIRS] = pack_bf16x2(r0, r1);
                    r0 += __uint_as_float(x[i] << 16);
                    r1 += __uint_as_float(x[i] & 0xFFFF0000u);
                }
        }
    } else if (e < npairs + nz) {
        const int64_t f = e - npairs, bh = f / D, k = f % D;
        float *p = zst + bh * nchunks * D + k;
        float run = 0.f;
        for (int j0 = 0; j0 < nchunks; j0 += 16) {
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (j0 + i < nchunks) x[i] = p[static_cast<int64_t>(j0 + i) * D];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (j0 + i < nchunks) {
                    p[static_cast<int64_t>(j0 + i) * D] = run;
                    run += x[i];
                }
        }
    }
}

// ---- 3. linear branch + combination ----------------------------------------------------------------------
// Persistent: one CTA per SM walks the work items (query tile, bh) with item = tile * BH + bh, from blockIdx.x
// in steps of gridDim.x, skipping the tiles whose rows have no key outside their window yet.  256 threads;
// thread r (mod 128) owns query row a + r (TMEM lane r) and the column half h = warp / 4 of it.  Per item: the Q
// tile, phi(K)^T and V of the <= 2 key chunks from 128 J, and the prefix state P_J (bf16, from the scan); W2 is
// loaded once per CTA.  The next item's Q, phi(K) and P_J are loaded as soon as this item's products that read
// them are done (before its masking, PV products and combination), and its V tiles once this item's PV
// products are: the loads overlap the rest of the item.  TMEM: f(Q), then the scores of chunk J, columns
// [0, 128); the scores of chunk J + 1, [128, 256); the numerator, [256, 384).  The masked scores go back over
// their own TMEM columns as bf16 pairs, the A operand of their product with V.  o holds the SWA prefill's output
// on entry and the hybrid output on exit; lse is the SWA prefill's.
// A from TMEM: keys 0..63 as bf16 pairs in columns [0, 32), keys 64..127 in columns [64, 96) (each key half is
// written by the threads that read that half of the scores).
__device__ __forceinline__ void mma_tv(uint32_t d, uint32_t a_tmem, uint32_t b, bool acc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        umma_ts(d, a_tmem + kk * 8 + (kk >= 4 ? 32 : 0), sdesc_sw128(b + kk * 2048, HALF, 1024), IDESC_KM,
                (acc || kk) ? 1u : 0u);
}

// The shape of one work item of the linear pass.
struct LinItem {
    int64_t a, last, J;  // first row, last row, first key chunk
    int bh;
    bool two, has_p;     // the rows reach into chunk J + 1; a prefix state before chunk J
};
__device__ __forceinline__ bool lin_item(int item, int BH, int64_t L, int m, int s, LinItem &it) {
    it.a = static_cast<int64_t>(item / BH) * C;
    it.bh = item % BH;
    it.last = (it.a + C < L ? it.a + C : L) - 1;
    if (it.last - m < s) return false;  // no row of the tile has a key outside its window yet
    it.J = it.a - m + 1 > 0 ? (it.a - m + 1) / C : 0;
    it.two = it.J * C + C <= it.last - m;
    it.has_p = it.J > 0;
    return true;
}
// The next item of this CTA with work from item on (n_items if none).
__device__ __forceinline__ int lin_next(int item, int n_items, int BH, int64_t L, int m, int s, LinItem &it) {
    for (; item < n_items; item += static_cast<int>(gridDim.x))
        if (lin_item(item, BH, L, m, s, it)) return item;
    return n_items;
}

__global__ void __launch_bounds__(256, 1) linear_kernel(const __grid_constant__ CUtensorMap mq,
                                                        const __grid_constant__ CUtensorMap mv,
                                                        const __grid_constant__ CUtensorMap mpk,
                                                        const __grid_constant__ CUtensorMap mpj,
                                                        const __grid_constant__ CUtensorMap mw2,
                                                        const float *__restrict__ zst, __nv_bfloat16 *o,
                                                        const float *__restrict__ lse, int64_t L, int m, int s,
                                                        int nchunks, int BH, DeviceStatus *status) {
    const int r = threadIdx.x & (C - 1), hh = threadIdx.x >> 7;
    const int n_items = nchunks * BH;
    LinItem cur;
    int item = lin_next(static_cast<int>(blockIdx.x), n_items, BH, L, m, s, cur);
    if (item >= n_items) return;  // uniform: no work for this CTA
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *Tq = sm, *Tw = sm + TILE, *Tk0 = sm + 2 * TILE, *Tk1 = sm + 3 * TILE, *Tv0 = sm + 4 * TILE,
            *Tv1 = sm + 5 * TILE, *Tp = sm + 6 * TILE;
    Ctl *ctl = reinterpret_cast<Ctl *>(sm + 7 * TILE);
    uint64_t *k_bar = reinterpret_cast<uint64_t *>(sm + 7 * TILE + 64);  // phi(K) tiles and P_J of an item
    uint64_t *v_bar = k_bar + 1;                                           // V tiles of an item
    float *dx = reinterpret_cast<float *>(sm + 7 * TILE + 128);  // [2][128] the halves' parts of the denominators
    const bool t0 = threadIdx.x == 0;
    if (t0) {
        ctl->abort_flag = 0;
        mbar_init(&ctl->load_bar, 1);
        mbar_init(&ctl->mma_bar, 1);
        mbar_init(k_bar, 1);
        mbar_init(v_bar, 1);
        mbar_init_fence();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(&ctl->tmem, 512);
        tmem_relinquish();
    }
    __syncthreads();
    int lq = 0, lv = 0;  // thread 0: Q / phi(K) loads and V loads issued (the phase each barrier is in)
    auto load_qk = [&](const LinItem &it, bool with_w2) {  // thread 0: Q (and W2), then phi(K) and P_J
        ++lq;
        mbar_arrive_expect_tx(&ctl->load_bar, (with_w2 ? 2 : 1) * TILE);
        load_tile(Tq, &mq, &ctl->load_bar, static_cast<int>(it.a), it.bh);
        if (with_w2) load_tile(Tw, &mw2, &ctl->load_bar, 0, 0);
        mbar_arrive_expect_tx(k_bar, (1 + (it.two ? 1 : 0) + (it.has_p ? 1 : 0)) * TILE);
        load_tile(Tk0, &mpk, k_bar, static_cast<int>(it.J * C), it.bh);
        if (it.two) load_tile(Tk1, &mpk, k_bar, static_cast<int>(it.J * C + C), it.bh);
        if (it.has_p) load_tile(Tp, &mpj, k_bar, static_cast<int>(it.J * C), it.bh);
    };
    auto load_v = [&](const LinItem &it) {  // thread 0: the V tiles
        ++lv;
        mbar_arrive_expect_tx(v_bar, (1 + (it.two ? 1 : 0)) * TILE);
        load_tile(Tv0, &mv, v_bar, static_cast<int>(it.J * C), it.bh);
        if (it.two) load_tile(Tv1, &mv, v_bar, static_cast<int>(it.J * C + C), it.bh);
    };
    if (t0) {
        load_qk(cur, true);
        load_v(cur);
    }
    operands_written();
    const uint32_t tmem = ctl->tmem;
    const uint32_t T_S0 = tmem, T_S1 = tmem + 128, T_NUM = tmem + 256;
    const WaitCtl wc{smem_u32(&ctl->abort_flag), kWaitTimeoutUs, status};
    int mph = 0;  // mma_bar phases waited so far
    bool fine = true;
    for (int n = 0; fine && item < n_items; ++n) {
        LinItem nxt;
        const int next = lin_next(item + static_cast<int>(gridDim.x), n_items, BH, L, m, s, nxt);
        const float *zJ = zst + (static_cast<int64_t>(cur.bh) * nchunks + cur.J) * D;
        if (t0) {
            if (mbar_wait(&ctl->load_bar, n & 1, wc, 43)) {
                tc_fence_after();
                mma_abt(T_S0, smem_u32(Tq), smem_u32(Tw), false);  // f(Q): [row][feature]
            } else {
                mbar_wait_drain(&ctl->load_bar, n & 1);
            }
            umma_commit(&ctl->mma_bar);
        }
        fine = wait_mma(ctl, mph++, wc, 44);
        float den = 0.f;
        if (fine) {  // phi(Q) (bf16, over the Q tile) and phi(q) z_J (fp32), this thread's half of the features
            for (int c0 = 64 * hh; c0 < 64 * hh + 64; c0 += 32) {
                float x[32];
                tmem_ld32(lane_addr(T_S0, c0), x);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    x[i] = exp2f(x[i] * LOG2E);
                    den = fmaf(x[i], zJ[c0 + i], den);
                }
                st_row32(smem_u32(Tq), r, c0, x);
            }
        }
        operands_written();
        if (t0) {
            if (fine && mbar_wait(k_bar, n & 1, wc, 45)) {
                tc_fence_after();
                mma_ab(T_S0, smem_u32(Tq), smem_u32(Tk0), false);                  // phi(Q) phi(K_J)^T: [row][key]
                if (cur.two) mma_ab(T_S1, smem_u32(Tq), smem_u32(Tk1), false);     // chunk J + 1
                if (cur.has_p) mma_ab(T_NUM, smem_u32(Tq), smem_u32(Tp), false);   // phi(Q) P_J
            } else {
                mbar_wait_drain(k_bar, n & 1);
            }
            umma_commit(&ctl->mma_bar);
        }
        fine = wait_mma(ctl, mph++, wc, 46) && fine;
        // Q, phi(K) and P_J are read: the next item's go in now
        if (t0 && fine && next < n_items) load_qk(nxt, false);
        const int64_t t = cur.a + r;  // this thread's query row
        if (fine) {  // keep s <= key <= t - m; fp32 row sums into the denominator, bf16 pairs back into TMEM
            for (int u = 0; u < (cur.two ? 2 : 1); ++u) {
                const uint32_t ts = u ? T_S1 : T_S0;
                const int64_t kt = cur.J * C + u * C;
                {  // this thread's half of the keys; its bf16 pairs go to the first 32 of its own 64 columns
                    float x[64];
                    tmem_ld64(lane_addr(ts, 64 * hh), x);
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int64_t k0 = kt + 64 * hh + 2 * i;
                        const float p0 = (k0 >= s && k0 <= t - m) ? x[2 * i] : 0.f;
                        const float p1 = (k0 + 1 >= s && k0 + 1 <= t - m) ? x[2 * i + 1] : 0.f;
                        den += p0 + p1;
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32u_nowait(lane_addr(ts, 64 * hh), pk);
                }
            }
            tmem_wait_st();
        }
        dx[hh * C + r] = den;  // this half's part of the row's denominator
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        den += dx[(hh ^ 1) * C + r];
        if (t0) {
            if (fine && mbar_wait(v_bar, n & 1, wc, 47)) {
                tc_fence_after();
                mma_tv(T_NUM, T_S0, smem_u32(Tv0), cur.has_p);  // masked scores of chunk J x V_J
                if (cur.two) mma_tv(T_NUM, T_S1, smem_u32(Tv1), true);
            } else {
                mbar_wait_drain(v_bar, n & 1);
            }
            umma_commit(&ctl->mma_bar);
        }
        fine = wait_mma(ctl, mph++, wc, 48) && fine;
        // the V tiles are read: the next item's go in now
        if (t0 && fine && next < n_items) load_v(nxt);
        if (fine) {
            // tcgen05.ld is warp-collective: every thread loads, only rows t < L read o', lse and write o
            const bool live = t < L;
            const int64_t row = static_cast<int64_t>(cur.bh) * L + (live ? t : 0);
            const float e = live ? exp2f(-lse[row] * LOG2E) : 0.f;  // e^{-lse}
            const float inv = 1.f / fmaf(den, e, 1.f);
            __nv_bfloat16 *orow = o + row * D;
            for (int c0 = 64 * hh; c0 < 64 * hh + 64; c0 += 32) {
                float x[32];
                tmem_ld32(lane_addr(T_NUM, c0), x);
                if (!live) continue;
                uint4 *p = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint4 ov = p[g];
                    const uint32_t w4[4] = {ov.x, ov.y, ov.z, ov.w};
                    uint32_t res[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float lo = __uint_as_float(w4[h] << 16), hi = __uint_as_float(w4[h] & 0xFFFF0000u);
                        res[h] = pack_bf16x2(fmaf(x[8 * g + 2 * h], e, lo) * inv, fmaf(x[8 * g + 2 * h + 1], e, hi) * inv);
                    }
                    p[g] = make_uint4(res[0], res[1], res[2], res[3]);
                }
            }
        }
        item = next;
        cur = nxt;
    }
    if (t0 && !fine) {  // no copy may still be landing when the CTA exits: the last loads issued on each barrier
        mbar_wait_drain(&ctl->load_bar, (lq - 1) & 1);
        mbar_wait_drain(k_bar, (lq - 1) & 1);
        mbar_wait_drain(v_bar, (lv - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---- decode ----------------------------------------------------------------------------------------
// grid BH, 128 threads (thread c: feature c / value column c).  Folds the key leaving the window at step t
// (position t - m >= s, in the slot key t goes to) into S, z; writes k_new, v_new into that slot; writes
// lin[bh] = (phi(q) S_t [d], phi(q) z_t).
__global__ void __launch_bounds__(128) decode_state_kernel(const __nv_bfloat16 *__restrict__ q,
                                                           const __nv_bfloat16 *__restrict__ k_new,
                                                           const __nv_bfloat16 *__restrict__ v_new,
                                                           __nv_bfloat16 *k_cache, __nv_bfloat16 *v_cache, float *S,
                                                           float *z, const __nv_bfloat16 *__restrict__ wf, float *lin,
                                                           int w, int s, int64_t t) {
    __shared__ float kev[D], vev[D], qs[D], phk[D], phq[D], red[4];
    const int bh = blockIdx.x, c = threadIdx.x;
    const int m = w - s;
    const int64_t slot = t < s ? t : s + (t - s) % m;
    const bool evict = t - m >= s;
    const int64_t crow = (static_cast<int64_t>(bh) * w + slot) * D;
    kev[c] = __bfloat162float(k_cache[crow + c]);
    vev[c] = __bfloat162float(v_cache[crow + c]);
    qs[c] = __bfloat162float(q[static_cast<int64_t>(bh) * D + c]);
    __syncthreads();
    k_cache[crow + c] = k_new[static_cast<int64_t>(bh) * D + c];
    v_cache[crow + c] = v_new[static_cast<int64_t>(bh) * D + c];
    {  // f = x wf for the evicted key and the query; thread c < 64 computes column c of both
        const int col = c & 63;
        const float *x = c < 64 ? kev : qs;
        float f = 0.f;
        for (int i = 0; i < D; ++i) f = fmaf(x[i], __bfloat162float(wf[i * (D / 2) + col]), f);
        float *dst = c < 64 ? phk : phq;
        dst[col] = exp2f(f * LOG2E);
        dst[col + 64] = exp2f(-f * LOG2E);
    }
    __syncthreads();
    float *Sh = S + static_cast<int64_t>(bh) * D * D;
    float num = 0.f;
    const float vc = evict ? vev[c] : 0.f;
    for (int j = 0; j < D; ++j) {
        float x = Sh[j * D + c];
        if (evict) {
            x = fmaf(phk[j], vc, x);
            Sh[j * D + c] = x;
        }
        num = fmaf(phq[j], x, num);
    }
    float zc = z[static_cast<int64_t>(bh) * D + c];
    if (evict) {
        zc += phk[c];
        z[static_cast<int64_t>(bh) * D + c] = zc;
    }
    float dn = phq[c] * zc;
    for (int off = 16; off > 0; off >>= 1) dn += __shfl_xor_sync(0xFFFFFFFFu, dn, off);
    if ((c & 31) == 0) red[c >> 5] = dn;
    __syncthreads();
    lin[static_cast<int64_t>(bh) * (D + 1) + c] = num;
    if (c == 0) lin[static_cast<int64_t>(bh) * (D + 1) + D] = (red[0] + red[1]) + (red[2] + red[3]);
}

// o = (o' + num e^{-lse}) / (1 + den e^{-lse}) per (b, h) row; grid BH, 128 threads.
__global__ void __launch_bounds__(128) combine_kernel(__nv_bfloat16 *o, const float *__restrict__ lse,
                                                      const float *__restrict__ lin) {
    const int bh = blockIdx.x, c = threadIdx.x;
    const float e = exp2f(-lse[bh] * LOG2E);
    const float *l = lin + static_cast<int64_t>(bh) * (D + 1);
    const float inv = 1.f / fmaf(l[D], e, 1.f);
    const int64_t i = static_cast<int64_t>(bh) * D + c;
    o[i] = __float2bfloat16_rn(fmaf(l[c], e, __bfloat162float(o[i])) * inv);
}

}  // namespace hy

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static bool encode_tile_map(CUtensorMap *m, const void *base, int64_t L, int BH) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(hy::D), static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {hy::D * 2, static_cast<cuuint64_t>(L) * hy::D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int64_t n_chunks(int64_t L) { return (L + hy::C - 1) / hy::C; }

}  // namespace swa

using namespace swa;

extern "C" size_t swa_hybrid_prefill_workspace_size(int B, int H, int64_t L, int d) {
    if (B < 1 || H < 1 || L < 1 || d != hy::D) return 0;
    const int64_t BH = static_cast<int64_t>(B) * H, recs = BH * n_chunks(L);
    // lse, the chunk states (bf16) and their z (fp32), phi(K)^T of every chunk (bf16)
    return align256(static_cast<size_t>(BH * L) * 4) + 2 * align256(static_cast<size_t>(recs) * hy::D * hy::D * 2) +
           align256(static_cast<size_t>(recs) * hy::D * 4) + align256(hy::D * hy::D * 2);
}

extern "C" int swa_hybrid_prefill(const void *q, const void *k, const void *v, const void *wf, void *o, float *state_s,
                                  float *state_z, int B, int H, int64_t L, int d, int w, int s, float scale,
                                  void *workspace, size_t workspace_bytes, int dtype, void *stream) {
    fail(SWA_OK, "%s", "");
    if (dtype != SWA_BF16 || d != hy::D) return fail(SWA_ERR_UNSUPPORTED, "hybrid prefill runs on bf16 with d = 128");
    if (B < 1 || H < 1 || static_cast<int64_t>(B) * H > 65535) return fail(SWA_ERR_INVALID, "need 1 <= B*H <= 65535");
    if (w < 1 || s < 0 || s >= w) return fail(SWA_ERR_INVALID, "need 0 <= s < w (s=%d, w=%d)", s, w);
    if (L < 0 || L >= (int64_t(1) << 31)) return fail(SWA_ERR_INVALID, "L=%lld out of range", (long long)L);
    if (!(scale == scale) || scale <= 0.f || scale > 1e30f)
        return fail(SWA_ERR_INVALID, "scale must be a positive finite number");
    if ((state_s == nullptr) != (state_z == nullptr))
        return fail(SWA_ERR_INVALID, "state_s and state_z are given together or not at all");
    const int BH = B * H;
    const int m = w - s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L == 0) {
        if (state_s) {
            cudaError_t e = cudaMemsetAsync(state_s, 0, static_cast<size_t>(BH) * hy::D * hy::D * 4, st);
            if (e == cudaSuccess) e = cudaMemsetAsync(state_z, 0, static_cast<size_t>(BH) * hy::D * 4, st);
            if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "state reset: %s", cudaGetErrorString(e));
        }
        return SWA_OK;
    }
    if (!q || !k || !v || !o || !wf) return fail(SWA_ERR_INVALID, "q, k, v, wf and o must be non-null");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(o)) & 15u)
        return fail(SWA_ERR_INVALID, "q, k, v and o must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(wf) & 1u) return fail(SWA_ERR_INVALID, "wf must be 2-byte aligned");
    if ((reinterpret_cast<uintptr_t>(state_s) | reinterpret_cast<uintptr_t>(state_z)) & 15u)
        return fail(SWA_ERR_INVALID, "state_s and state_z must be 16-byte aligned");
    const size_t need = swa_hybrid_prefill_workspace_size(B, H, L, d);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");
    unsigned *status = device_status_word();
    if (!status) return SWA_ERR_CUDA;
    const int nch = static_cast<int>(n_chunks(L));
    const size_t recs = static_cast<size_t>(BH) * nch;
    char *wsp = static_cast<char *>(workspace);
    float *lse = reinterpret_cast<float *>(wsp);
    wsp += align256(static_cast<size_t>(BH) * L * 4);
    __nv_bfloat16 *dmat = reinterpret_cast<__nv_bfloat16 *>(wsp);
    wsp += align256(recs * hy::D * hy::D * 2);
    __nv_bfloat16 *phik = reinterpret_cast<__nv_bfloat16 *>(wsp);
    wsp += align256(recs * hy::D * hy::D * 2);
    float *zst = reinterpret_cast<float *>(wsp);
    wsp += align256(recs * hy::D * 4);
    __nv_bfloat16 *w2img = reinterpret_cast<__nv_bfloat16 *>(wsp);

    // the SWA branch: o' and lse
    PrefillArgs a{q, k, v, o, lse, nullptr, nullptr, 0, BH, L, d, w, s, scale, L, st};
    if (int rc = launch_prefill_bf16_tc(a)) return rc;

    CUtensorMap mq, mk, mv, mpk, mpj, mw2;
    if (!encode_tile_map(&mq, q, L, BH) || !encode_tile_map(&mk, k, L, BH) || !encode_tile_map(&mv, v, L, BH))
        return fail(SWA_ERR_INVALID, "cuTensorMapEncodeTiled rejected q, k or v");
    // phi(K)^T and the scanned states as [BH][chunks * 128 rows][128] tiles
    if (!encode_tile_map(&mpk, phik, static_cast<int64_t>(nch) * hy::C, BH) ||
        !encode_tile_map(&mpj, dmat, static_cast<int64_t>(nch) * hy::C, BH) || !encode_tile_map(&mw2, w2img, hy::D, 1))
        return fail(SWA_ERR_INVALID, "cuTensorMapEncodeTiled rejected the workspace");
    const __nv_bfloat16 *wfb = static_cast<const __nv_bfloat16 *>(wf);
    DeviceStatus *ds = reinterpret_cast<DeviceStatus *>(status);
    const uint32_t smem_a = 3 * hy::TILE + 1024 + 64, smem_b = 7 * hy::TILE + 1024 + 128 + 1024;
    static bool attr_done = false;  // per process; the attribute is per function and idempotent
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(hy::chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_a);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(hy::linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_b);
        if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "hybrid kernels: %s", cudaGetErrorString(e));
        attr_done = true;
    }
    // the linear branch: W2, chunk states, their exclusive scan, then per query tile
    hy::w2_kernel<<<hy::D, hy::D, 0, st>>>(wfb, w2img);
    hy::chunk_state_kernel<<<dim3(nch, BH), 128, smem_a, st>>>(mk, mv, mw2, dmat, zst, phik, nullptr, nullptr, 0,
                                                               nch, s, L, ds);
    const int64_t npairs = static_cast<int64_t>(BH) * hy::D * hy::D / 2, nz = static_cast<int64_t>(BH) * hy::D;
    hy::scan_kernel<<<static_cast<unsigned>((npairs + nz + 255) / 256), 256, 0, st>>>(
        reinterpret_cast<uint32_t *>(dmat), zst, nch, npairs, nz);
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return fail(SWA_ERR_CUDA, "cannot read the multiprocessor count");
    const int n_lin = nch * BH;  // persistent: one CTA per SM over the (query tile, bh) items
    hy::linear_kernel<<<n_lin < sms ? n_lin : sms, 256, smem_b, st>>>(mq, mv, mpk, mpj, mw2, zst,
                                                                      static_cast<__nv_bfloat16 *>(o), lse, L, m, s,
                                                                      nch, BH, ds);
    if (state_s) {
        // the state after the last row (keys s .. L-1-m): the prefix of chunk jf plus its keys below L - m
        const int64_t jf = L - m > 0 ? (L - m) / hy::C : 0;
        hy::chunk_state_kernel<<<dim3(1, BH), 128, smem_a, st>>>(mk, mv, mw2, dmat, zst, phik, state_s, state_z,
                                                                 static_cast<int>(jf), nch, s, L - m, ds);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "hybrid prefill launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

extern "C" size_t swa_hybrid_decode_workspace_size(int B, int H, int d, int w) {
    if (B < 1 || H < 1 || d != hy::D || w < 1) return 0;
    const int BH = B * H;
    return align256(decode_workspace_bytes(BH, d, w)) + align256(static_cast<size_t>(BH) * 4) +
           align256(static_cast<size_t>(BH) * (hy::D + 1) * 4);
}

extern "C" int swa_hybrid_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                      float *state_s, float *state_z, const void *wf, void *o, int B, int H, int d,
                                      int w, int s, int64_t t, float scale, void *workspace, size_t workspace_bytes,
                                      int dtype, void *stream) {
    fail(SWA_OK, "%s", "");
    if (dtype != SWA_BF16 || d != hy::D) return fail(SWA_ERR_UNSUPPORTED, "hybrid decode runs on bf16 with d = 128");
    if (B < 1 || H < 1 || static_cast<int64_t>(B) * H > 65535) return fail(SWA_ERR_INVALID, "need 1 <= B*H <= 65535");
    if (w < 1 || s < 0 || s >= w) return fail(SWA_ERR_INVALID, "need 0 <= s < w (s=%d, w=%d)", s, w);
    if (t < 0) return fail(SWA_ERR_INVALID, "t must be >= 0");
    if (!(scale == scale) || scale <= 0.f || scale > 1e30f)
        return fail(SWA_ERR_INVALID, "scale must be a positive finite number");
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !state_s || !state_z || !wf || !o)
        return fail(SWA_ERR_INVALID, "every tensor argument must be non-null");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
         reinterpret_cast<uintptr_t>(o)) & 15u)
        return fail(SWA_ERR_INVALID, "q, k_cache, v_cache and o must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) | reinterpret_cast<uintptr_t>(wf)) & 1u)
        return fail(SWA_ERR_INVALID, "k_new, v_new and wf must be 2-byte aligned");
    if ((reinterpret_cast<uintptr_t>(state_s) | reinterpret_cast<uintptr_t>(state_z)) & 3u)
        return fail(SWA_ERR_INVALID, "state_s and state_z must be 4-byte aligned");
    const size_t need = swa_hybrid_decode_workspace_size(B, H, d, w);
    if (workspace_bytes < need)
        return fail(SWA_ERR_INVALID, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(SWA_ERR_INVALID, "workspace must be non-null and 256-byte aligned");
    const int BH = B * H;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const size_t dec_bytes = align256(decode_workspace_bytes(BH, d, w));
    float *lse = reinterpret_cast<float *>(ws + dec_bytes);
    float *lin = reinterpret_cast<float *>(ws + dec_bytes + align256(static_cast<size_t>(BH) * 4));
    hy::decode_state_kernel<<<BH, 128, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k_new),
        static_cast<const __nv_bfloat16 *>(v_new), static_cast<__nv_bfloat16 *>(k_cache),
        static_cast<__nv_bfloat16 *>(v_cache), state_s, state_z, static_cast<const __nv_bfloat16 *>(wf), lin, w, s, t);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "hybrid decode state launch: %s", cudaGetErrorString(e));
    DecodeArgs da{q, k_cache, v_cache, o, lse, BH, d, w, s, t, scale, ws, dec_bytes, 2, st};
    if (int rc = launch_decode(da)) return rc;
    hy::combine_kernel<<<BH, 128, 0, st>>>(static_cast<__nv_bfloat16 *>(o), lse, lin);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "hybrid combine launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}
