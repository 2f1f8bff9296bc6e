// prefill_tc.cu -- bf16 prefill of causal sliding-window attention with sinks on the sm_103a tensor
// cores (TMA + tcgen05.mma + TMEM), plus two diagnostics kernels (bounded-wait timeout, UMMA tile).
//
// The computation (hyper.ai summary of arXiv 2608.28444, section "带 Sink 的滑动窗口注意力"; causal
// softmax attention of "模糊窗口注意力" section 2.1, eq (1)): query t attends
//     K(t) = { i <= t : i < s  or  i >= t - m + 1 },  m = w - s,
// with softmax over scale * q.k.  A fixed sparsity pattern known from positions alone ("滑窗与固定稀疏":
// O(n^2) -> O(n k), banded patterns are hardware friendly), so each CTA walks only the key tiles that
// intersect the band or the sink block of its query tile; no skipped tile is ever loaded.
//
// Work item = two query tiles of 128 rows (256 consecutive rows) of one (b, h).  The kernel is
// persistent: one CTA per SM walks the items blockIdx.x, blockIdx.x + gridDim.x, ..., ordered
// longest-first (the last query pairs of every head, whose windows are full, come first), so the short
// items fall in the last rounds and the CTAs finish together.  352 threads in five roles:
//   warps 0-3 / 4-7  softmax + epilogue of query tile 0 / 1: thread r owns row r of its tile
//              (= TMEM lane r);
//   warp 10    per item: builds the key-tile list into one of two buffers, one item ahead, loads Q_0 and
//              Q_1 as soon as the previous item's last QK product is done, and prefetches the next
//              item's Q into L2;
//   warp 8     TMA producer: K tiles into a 2-stage ring and V tiles into a 2-stage ring (128 rows x
//              128 bf16 each, two 64-column boxes with the 128-byte swizzle), as one stream over all
//              items of the CTA.  A K slot frees as soon as the QK products that read it complete, a V
//              slot after its PV products, so K loads run up to two tiles ahead, also into the next
//              item;
//   warp 9     MMA issuer (one thread).  Per key tile j: PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1), where
//              QK_x(j) is S_x = Q_x K_j^T and PV_x(j) is O_x += P_x V_j with P_x (bf16) read by the MMA
//              straight from tensor memory.  While the tensor cores work on one query tile, the softmax
//              warpgroup of the other turns its S into P (ping-pong), and each K/V tile loaded from L2
//              serves 256 query rows.  The next item's first QK products follow the current item's last
//              PV products, so they overlap its epilogue; the next item's first PV_x waits until the
//              epilogue has read O_x.
// TMEM (512 columns): S_0, S_1 = [0,128), [128,256); O_0, O_1 = [256,384), [384,512) (fp32, lane = row).
// The softmax threads overwrite the first 64 columns of S_x with P_x (two bf16 per column) after
// reading them.  The online softmax keeps a running max in log2 units and only rescales O (TMEM load,
// multiply, store) when the max grows by more than 8 (a factor 256), so p <= 256 always fits
// bf16/fp32 and the rescale is rare; O and l always share the same reference max.  With one S buffer
// per query tile, S_x(j) complete implies PV_x of the previous tile complete (tcgen05 MMAs of a thread
// complete in order), so neither the P store nor the rescale needs another wait.
//
// Key tiles.  For the query rows [q0, q1] of a CTA the key positions needed are the sinks [0, min(s, blo)) and
// the band [blo, q1] with blo = max(0, q0 - m + 1).  Positions >= pos0 are rows of this call's k/v;
// positions < pos0 (chunked prefill) live in the rolling cache: slot p for p < s, slot
// s + ((p - s) mod m) for the rest ("滑窗与固定稀疏", eq attn-fixed-rolling and eq attn-fixed-streaming).
// A contiguous position range maps to at most two contiguous slot runs (the ring wraps once), so every
// range becomes a list of 128-row tiles, each with: source, first row, position of its column 0, and
// the last valid column.  Columns past the range end, positions past t and positions outside the
// window are masked per row; interior tiles need no mask at all.  Every key position appears in
// exactly one tile.  TMA zero-fills rows outside the source tensor.
//
// Every mbarrier wait is bounded (1 s).  A wait that runs out records the timeout in the device error
// word and sets a CTA-wide abort flag; all roles leave their loops, the producer waits (bounded) for
// its copies in flight, the MMA thread waits for its MMAs, and TMEM is freed before the CTA exits.
#include <math.h>

#include <algorithm>
#include <utility>
#include <vector>

#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {
namespace tc {

constexpr int BH_ROWS = 128;               // query rows per query tile (= TMEM lanes)
constexpr int BM = 2 * BH_ROWS;            // query rows per CTA: two query tiles
constexpr int BN = 128;                    // keys per key tile
constexpr int HD = 128;                    // head dimension
constexpr int NK = 2;                      // K tile stages (a slot frees after its QK products)
constexpr int NV = 2;                      // V tile stages (a slot frees after its PV products)
constexpr uint32_t HALF_BYTES = 128 * 128;  // one 64-column half of a 128-row bf16 tile (16 KB)
constexpr uint32_t TILE_BYTES = 2 * HALF_BYTES;
constexpr int MAX_TILES = 64;
constexpr int kThreads = 352;  // warps 0-3 / 4-7: softmax of query tile 0 / 1; 8: TMA; 9: MMA; 10: tile lists
constexpr int kWarpTma = 8, kWarpMma = 9, kWarpList = 10;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S (the scores of one query tile at a time, fp32), P_0, P_1 (bf16 pairs), O_0, O_1 (fp32)
constexpr uint32_t COL_S = 0;
__host__ __device__ constexpr uint32_t col_p(int x) { return 128u + static_cast<uint32_t>(x) * 64u; }
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u + static_cast<uint32_t>(x) * 128u; }
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the running max grows by more than 2^8

constexpr uint32_t OFF_Q = 0;                         // Q_0, Q_1
constexpr uint32_t OFF_K = OFF_Q + 2 * TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + NK * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + NV * TILE_BYTES;
constexpr uint32_t OFF_MISC = OFF_BAR + 256;
constexpr uint32_t OFF_TILES = OFF_MISC + 64;
constexpr uint32_t OFF_GMASK = OFF_TILES + 2 * MAX_TILES * 12;  // two tile lists (current / next item)
constexpr uint32_t SMEM_USED = OFF_GMASK + 2 * MAX_TILES * 16;     // and their global-key columns (block-sparse)
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024 bytes
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false, false);  // Q, K both K-major
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 128, false, true);   // P K-major, V MN-major

struct Tile {
    int row0;     // first source row (TMA row coordinate)
    int pbase;    // absolute position of column 0
    short chi;    // last valid column (columns past it belong to another tile or to nothing)
    short flags;  // bit 0: source (0 = this call's k/v rows, 1 = rolling cache); bit 1 + x: needed by query tile x
};
static_assert(sizeof(Tile) == 12, "tile record");

// Block-sparse mode: per column of a key tile, whether it holds a global key (bit c of word c / 32).
struct TileMask {
    uint32_t w[4];
};

struct Params {
    CUtensorMap tm_q, tm_k, tm_v, tm_kc, tm_vc;
    // block-sparse mode: the host-built key-tile lists of every 256-row query pair (MAX_TILES entries per pair,
    // bs_count[pair] used), their global-key columns, and the random key blocks of each query block
    const Tile *bs_tiles;
    const TileMask *bs_gmask;
    const int *bs_count;
    const int *bs_rand;  // [ceil(L / bs_block)][bs_r]; -1 = no block
    int bs_block, bs_r;
    void *o;
    float *lse;
    DeviceStatus *status;
    int64_t seq_stride;  // rows between (b, h) blocks of q/k/v/o/lse
    int L, pos0, w, s, m, BH;
    int n_qpairs, n_items;  // 256-row query pairs per (b, h); work items = n_qpairs * BH
    float scale_log2;
    uint32_t timeout_us;
};

// Build the key-tile list of the query tile [q0, q1] (absolute positions).  Returns the tile count
// (entries past MAX_TILES are not stored; the caller treats a larger count as an error).  In RoPE mode
// (pos0 = 0 or pos0 >= s, s <= BN) the sinks [0, min(s, q1 + 1)) always form the first tile, on their own
// (from the cache when pos0 >= s), and the band starts at position s: the sink scores use another query
// rotation than the band's.
__host__ __device__ int build_tiles(Tile *tl, int q0, int q1, int pos0, int s, int m, int w, bool rope) {
    int n = 0;
    auto add_range = [&](int src, int pa, int pb, int rowbase) {  // positions [pa, pb]; row = p - rowbase
        for (int p = pa; p <= pb; p += BN) {
            if (n < MAX_TILES) {
                tl[n].row0 = p - rowbase;
                tl[n].pbase = p;
                tl[n].chi = static_cast<short>((pb - p < BN - 1) ? pb - p : BN - 1);
                tl[n].flags = static_cast<short>(src);
            }
            ++n;
        }
    };
    int blo = q0 - m + 1 > 0 ? q0 - m + 1 : 0;
    int sink_hi = s < blo ? s : blo;  // sinks [0, sink_hi) are not inside the band range
    if (rope) {
        sink_hi = s < q1 + 1 ? s : q1 + 1;
        blo = blo > s ? blo : s;
    }
    const int sink_cache = sink_hi < pos0 ? sink_hi : pos0;
    // sinks first: their scores tend to be the largest, which keeps later rescales rare
    if (sink_cache > 0) add_range(1, 0, sink_cache - 1, 0);
    if (sink_hi > pos0) add_range(0, pos0, sink_hi - 1, pos0);
    // band positions below pos0: in the cache
    const int ce = q1 < pos0 - 1 ? q1 : pos0 - 1;
    if (ce >= blo) {
        const int ie = ce < s - 1 ? ce : s - 1;  // still in the sink block (slot = position)
        if (ie >= blo) add_range(1, blo, ie, 0);
        const int ra = blo > s ? blo : s;
        if (ce >= ra) {  // ring positions [ra, ce]: one or two contiguous slot runs
            const int sa = s + (ra - s) % m;
            const int run1_end = ra + (w - 1 - sa);
            if (ce <= run1_end) {
                add_range(1, ra, ce, ra - sa);
            } else {
                add_range(1, ra, run1_end, ra - sa);
                add_range(1, run1_end + 1, ce, run1_end + 1 - s);
            }
        }
    }
    // band positions from pos0 on: rows of this call's k/v
    const int ca = blo > pos0 ? blo : pos0;
    if (q1 >= ca) add_range(0, ca, q1, pos0);
    return n;
}

// Which query tiles of the pair [q0, qlast] need each key tile: rows [ra, rb] need a tile holding
// positions [pb, pb + chi] iff some position p <= rb in it is a sink (p < s) or lies in the window of
// some row (p >= ra - m + 1).
__host__ __device__ void mark_tiles(Tile *tl, int n, int q0, int qlast, int s, int m) {
    for (int i = 0; i < n && i < MAX_TILES; ++i) {
        const int pb = tl[i].pbase, pe = tl[i].pbase + tl[i].chi;
        for (int x = 0; x < 2; ++x) {
            const int ra = q0 + x * BH_ROWS;
            const int rb = (q0 + x * BH_ROWS + BH_ROWS - 1 < qlast) ? q0 + x * BH_ROWS + BH_ROWS - 1 : qlast;
            if (ra > rb) continue;
            if (pb <= rb && (pb < s || pe >= ra - m + 1)) tl[i].flags = static_cast<short>(tl[i].flags | (2 << x));
        }
    }
}

// Bits [lo, hi] of a 32-bit word (clipped to [0, 31]; 0 when the range is empty).
__device__ __forceinline__ uint32_t range_bits(int lo, int hi) {
    lo = lo < 0 ? 0 : lo;
    hi = hi > 31 ? 31 : hi;
    if (hi < lo) return 0u;
    return (0xFFFFFFFFu >> (31 - hi)) & (0xFFFFFFFFu << lo);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Maximum of three floats in one instruction (a NaN operand is ignored, as in fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed fp32 pairs (one instruction for two lanes of work): d = a * b + c and d = a + b, each lane
// rounded like the scalar fmaf / add.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void fadd2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}


// Both issued by a whole converged warp (one elected lane issues each MMA).  Shared-memory addresses stay
// below 2^18, so a K step only adds its offset / 16 to the low descriptor word.
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr) {
    const uint32_t qlo = sdesc_sw128_lo(q_addr, 16), klo = sdesc_sw128_lo(k_addr, 16);
    constexpr uint32_t hi = sdesc_sw128_hi(1024);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4;
        umma_ss_warp_lo(d_tmem, qlo + off, klo + off, hi, IDESC_QK, kk > 0 ? 1u : 0u);
    }
}

__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr, bool accumulate) {
    const uint32_t vlo = sdesc_sw128_lo(v_addr, HALF_BYTES);
    constexpr uint32_t hi = sdesc_sw128_hi(1024);
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
        // P from TMEM: 16 keys = 8 columns of packed bf16 pairs; V: 16 key rows of 128 bytes (MN-major)
        umma_ts_warp_lo(d_tmem, p_tmem + kk * 8, vlo + ((kk * 16 * 128) >> 4), hi, IDESC_PV,
                        (accumulate || kk > 0) ? 1u : 0u);
    }
}

// BS: the block-sparse mode (host-built tile lists with global keys and random key blocks; compiled apart, so
// that the plain kernel carries none of its checks)
template <bool BS>
__global__ void __launch_bounds__(kThreads, 1) swa_prefill_tc_kernel(const __grid_constant__ Params P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *qfull = bars;           // [2]: Q_x of the current item landed
    uint64_t *qempty = qfull + 2;     // [2]: the item's last QK_x product is done: Q_x may be reloaded
    uint64_t *kfull = qempty + 2;     // [NK]
    uint64_t *kempty = kfull + NK;    // [NK]
    uint64_t *vfull = kempty + NK;    // [NV]
    uint64_t *vempty = vfull + NV;    // [NV]
    uint64_t *sfull = vempty + NV;    // [2]: S = Q_x K_j^T ready (the S buffer holds query tile x's scores)
    uint64_t *pfull = sfull + 2;      // [2]: P_x ready in TMEM (128 arrivals)
    uint64_t *ofull = pfull + 2;      // [2]: the last PV_x product of an item is done
    uint64_t *oempty = ofull + 2;     // [2]: O_x has been read by the epilogue (128 arrivals)
    uint64_t *lready = oempty + 2;    // [2]: tile list buffer b written (1 arrival)
    uint64_t *lfree = lready + 2;     // [2]: tile list buffer b no longer read (8 softmax warps, MMA, 2 loaders)
    uint64_t *drain = lfree + 2;
    uint64_t *sfree = drain + 1;      // the S buffer has been read by the softmax warps of its last user (4 warps)
    uint64_t *pempty = sfree + 1;     // [2]: PV_x products issued so far are done (P_x and O_x free)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);
    int *ntiles_s = reinterpret_cast<int *>(sm + OFF_MISC + 8);  // [2]
    Tile *tiles_s = reinterpret_cast<Tile *>(sm + OFF_TILES);     // [2][MAX_TILES]
    TileMask *gmask_s = reinterpret_cast<TileMask *>(sm + OFF_GMASK);  // [2][MAX_TILES] (block-sparse)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < NK; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&qfull[x], 1);
            mbar_init(&qempty[x], 1);
            mbar_init(&sfull[x], 1);
            mbar_init(&pfull[x], BH_ROWS);
            mbar_init(&ofull[x], 1);
            mbar_init(&oempty[x], BH_ROWS);
            mbar_init(&lready[x], 1);
            mbar_init(&lfree[x], 11);
        }
        mbar_init(drain, 1);
        mbar_init(sfree, 4);
        mbar_init(&pempty[0], 1);
        mbar_init(&pempty[1], 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{smem_u32(const_cast<int *>(abort_flag)), P.timeout_us, P.status};

    if (warp == kWarpTma) {
        // ------------------------------------------------------------------ TMA producers (K, V)
        // Lane 0 streams the K tiles, lane 1 the V tiles, each in its own ring over all items of this CTA in
        // order, so neither waits for the other: a K slot frees when the QK products that read it are done,
        // a V slot after its PV products, and the K loads run ahead into the next item on their own.
        if (lane < 2) {
            const bool isk = lane == 0;
            const int ns = isk ? NK : NV;
            uint64_t *full = isk ? kfull : vfull;
            uint64_t *empty = isk ? kempty : vempty;
            uint8_t *ring = sm + (isk ? OFF_K : OFF_V);
            const CUtensorMap *m_seq = isk ? &P.tm_k : &P.tm_v;
            const CUtensorMap *m_cache = isk ? &P.tm_kc : &P.tm_vc;
            tma_prefetch_desc(m_seq);
            int g = 0;  // tiles issued so far
            for (int it = 0;; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * G;
                if (item >= P.n_items) break;
                const int b = it & 1;
                if (!mbar_wait(&lready[b], (it >> 1) & 1, wc, 15, it)) break;
                const int n = ntiles_s[b];
                const int bh = item % P.BH;
                bool fine = true;
                for (int j = 0; j < n; ++j) {
                    const int st = g % ns;
                    if (!mbar_wait(&empty[st], ((g / ns) & 1) ^ 1, wc, isk ? 1 : 9, j)) {
                        fine = false;
                        break;
                    }
                    const Tile T = tiles_s[b * MAX_TILES + j];
                    const CUtensorMap *mp = (T.flags & 1) ? m_cache : m_seq;
                    uint8_t *dst = ring + st * TILE_BYTES;
                    mbar_arrive_expect_tx(&full[st], TILE_BYTES);
                    tma_load_3d(dst, mp, &full[st], 0, T.row0, bh);
                    tma_load_3d(dst + HALF_BYTES, mp, &full[st], 64, T.row0, bh);
                    ++g;
                }
                if (!fine) break;
                mbar_arrive(&lfree[b]);  // this lane no longer reads the item's list
            }
            if (*abort_flag) {  // make sure no copy is still landing in shared memory
                for (int gg = (g > ns ? g - ns : 0); gg < g; ++gg) mbar_wait_drain(&full[gg % ns], (gg / ns) & 1);
            }
        }
    } else if (warp == kWarpList) {
        // ------------------------------------------------------------------ tile lists
        if (lane == 0) {
            // Per item: the key-tile list goes to buffer it & 1 as soon as the buffer's previous item
            // (it - 2) has been released by every reader; then Q_0, Q_1 of the item, as soon as the previous
            // item's last QK product is done (about two key tiles before that item ends), and the next
            // item's Q into L2, so that its load does not wait for DRAM.
            int nq = 0;              // items whose Q loads were issued
            int nqx[2] = {0, 0};     // Q_x loads issued
            for (int it = 0;; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * G;
                if (item >= P.n_items) break;
                const int bh = item % P.BH;
                const int row_start = (P.n_qpairs - 1 - item / P.BH) * BM;
                const int q0 = P.pos0 + row_start;
                const int qlast = P.pos0 + min(row_start + BM, P.L) - 1;
                const int b = it & 1;
                if (it >= 2 && !mbar_wait(&lfree[b], ((it - 2) >> 1) & 1, wc, 12, it)) break;
                Tile *tl = tiles_s + b * MAX_TILES;
                int n;
                if (BS) {  // the pair's list, built on the host
                    const int qp = row_start / BM;
                    n = P.bs_count[qp];
                    if (n >= 1 && n <= MAX_TILES) {
                        const Tile *src = P.bs_tiles + static_cast<int64_t>(qp) * MAX_TILES;
                        const TileMask *gsrc = P.bs_gmask + static_cast<int64_t>(qp) * MAX_TILES;
                        for (int i = 0; i < n; ++i) {
                            tl[i] = src[i];
                            gmask_s[b * MAX_TILES + i] = gsrc[i];
                        }
                    }
                } else {
                    n = build_tiles(tl, q0, qlast, P.pos0, P.s, P.m, P.w, false);
                }
                if (n < 1 || n > MAX_TILES) {
                    atomicOr(&P.status->word, kDevBadArg);
                    *abort_flag = 1;
                    break;
                }
                if (!BS) mark_tiles(tl, n, q0, qlast, P.s, P.m);
                ntiles_s[b] = n;
                mbar_arrive(&lready[b]);  // release: the list is visible to whoever sees the phase complete
                // Q_x of the item, each as soon as the previous item's last QK_x product is done (query tile 0
                // usually finishes a key tile before query tile 1)
                bool qfine = true;
                for (int x = 0; x < 2 && qfine; ++x) {
                    if (nq >= 1 && !mbar_wait(&qempty[x], (nq - 1) & 1, wc, 13, it)) {
                        qfine = false;
                        break;
                    }
                    uint8_t *qs = sm + OFF_Q + x * TILE_BYTES;
                    mbar_arrive_expect_tx(&qfull[x], TILE_BYTES);
                    tma_load_3d(qs, &P.tm_q, &qfull[x], 0, row_start + x * BH_ROWS, bh);
                    tma_load_3d(qs + HALF_BYTES, &P.tm_q, &qfull[x], 64, row_start + x * BH_ROWS, bh);
                    nqx[x] = nq + 1;
                }
                if (!qfine) break;
                ++nq;
                // into L2 meanwhile: the next item's Q rows
                const int nitem = item + G;
                if (nitem < P.n_items) {
                    const int nrow = (P.n_qpairs - 1 - nitem / P.BH) * BM;
                    for (int x = 0; x < 2; ++x) {
                        tma_prefetch_3d(&P.tm_q, 0, nrow + x * BH_ROWS, nitem % P.BH);
                        tma_prefetch_3d(&P.tm_q, 64, nrow + x * BH_ROWS, nitem % P.BH);
                    }
                }
            }
            if (*abort_flag) {  // no copy may still be landing
                for (int x = 0; x < 2; ++x)
                    if (nqx[x] > 0) mbar_wait_drain(&qfull[x], (nqx[x] - 1) & 1);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ MMA issuer
        // One S buffer serves the two query tiles in turn, and P_x has TMEM columns of its own, so a QK
        // product needs only the S buffer to have been read by the softmax warps of its previous user, not
        // their whole softmax.  Per key tile j of an item: QK_0(j), PV_0(j-1), QK_1(j), PV_1(j-1): the tensor
        // cores take the next QK products while the softmax warps still compute the previous tile's
        // exponentials.  The whole warp runs the loop (uniform operands); one elected lane issues each
        // instruction.
        {
            auto wwait = [&](uint64_t *bar, int parity, unsigned site, unsigned tag) -> bool {
                return __all_sync(0xFFFFFFFFu, mbar_wait(bar, static_cast<uint32_t>(parity), wc, site, tag));
            };
            const uint32_t q_addr = smem_u32(sm + OFF_Q);
            const uint32_t k_addr0 = smem_u32(sm + OFF_K), v_addr0 = smem_u32(sm + OFF_V);
            bool issued_any = false, fine = true;
            int gk = 0, gv = 0;                // K, V tiles consumed
            int cp[2] = {0, 0};                // PV_x products issued (pfull parity)
            int ce[2] = {0, 0};                // items in which query tile x had PV products (oempty)
            int qf[2] = {0, 0};                // Q_x loads consumed (qfull parity)
            int u = 0;                         // QK products issued into the S buffer (sfree parity)
            for (int it = 0; fine; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * G;
                if (item >= P.n_items) break;
                const int b = it & 1;
                if (!wwait(&lready[b], (it >> 1) & 1, 14, it)) break;  // the item's tile list
                bool qready[2] = {false, false};
                // Q_x of this item, waited for before its first QK_x product
                auto need_q = [&](int x) -> bool {
                    if (qready[x]) return true;
                    if (!wwait(&qfull[x], qf[x] & 1, 2, it)) return false;
                    ++qf[x];
                    qready[x] = true;
                    tc_fence_after();
                    return true;
                };
                const Tile *tl = tiles_s + b * MAX_TILES;
                const int n = ntiles_s[b];
                int last_used[2] = {-1, -1};
                for (int j = 0; j < n; ++j)
                    for (int x = 0; x < 2; ++x)
                        if (tl[j].flags & (2 << x)) last_used[x] = j;
                bool first_pv[2] = {true, true};
                for (int j = 0; fine && j <= n; ++j) {
                    const int fq = (j < n) ? tl[j].flags : 0;       // QK products of tile j
                    const int fp = (j >= 1) ? tl[j - 1].flags : 0;  // PV products of tile j - 1
                    const int sk = gk % NK, sv = gv % NV;
                    bool k_ready = false, v_ready = false;
                    for (int x = 0; x < 2 && fine; ++x) {
                        if (fq & (2 << x)) {
                            if (u >= 1 && !wwait(sfree, (u - 1) & 1, 16, j)) { fine = false; break; }
                            if (!k_ready) {
                                if (!wwait(&kfull[sk], (gk / NK) & 1, 3, j)) { fine = false; break; }
                                k_ready = true;
                            }
                            if (!need_q(x)) { fine = false; break; }
                            tc_fence_after();
                            issue_qk(tmem + COL_S, q_addr + x * TILE_BYTES, k_addr0 + sk * TILE_BYTES);
                            umma_commit_warp(&sfull[x]);
                            ++u;
                            issued_any = true;
                            if (j == last_used[x]) umma_commit_warp(&qempty[x]);  // the item's last QK_x product
                        }
                        if (fp & (2 << x)) {
                            if (!wwait(&pfull[x], cp[x] & 1, 4, j)) { fine = false; break; }
                            if (first_pv[x]) {  // O_x must have been read by the previous item's epilogue
                                if (!wwait(&oempty[x], (ce[x] & 1) ^ 1, 11, j)) { fine = false; break; }
                                ++ce[x];
                            }
                            if (!v_ready) {
                                if (!wwait(&vfull[sv], (gv / NV) & 1, 5, j)) { fine = false; break; }
                                v_ready = true;
                            }
                            tc_fence_after();
                            issue_pv(tmem + col_o(x), tmem + col_p(x), v_addr0 + sv * TILE_BYTES, !first_pv[x]);
                            first_pv[x] = false;
                            ++cp[x];
                            umma_commit_warp(&pempty[x]);
                            if (j - 1 == last_used[x]) umma_commit_warp(&ofull[x]);
                        }
                    }
                    if (!fine) break;
                    if (fq) {
                        umma_commit_warp(&kempty[sk]);
                        ++gk;
                    }
                    if (fp) {
                        umma_commit_warp(&vempty[sv]);
                        ++gv;
                    }
                }
                if (!fine) break;
                // a query tile with no key tile in this item still takes its Q load and releases it
                for (int x = 0; x < 2 && fine; ++x) {
                    if (last_used[x] < 0) {
                        if (!need_q(x)) {
                            fine = false;
                            break;
                        }
                        umma_commit_warp(&qempty[x]);
                    }
                }
                if (!fine) break;
                if (lane == 0) mbar_arrive(&lfree[b]);
            }
            if (issued_any) {  // no MMA may still be running when TMEM is freed
                umma_commit_warp(drain);
                mbar_wait_drain(drain, 0);
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------------ softmax + epilogue
        const int x = warp >> 2;                    // query tile of this warpgroup
        const int r = threadIdx.x & (BH_ROWS - 1);  // its row == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + COL_S;
        const uint32_t p_addr = tmem + lane_base + col_p(x);
        const uint32_t o_addr = tmem + lane_base + col_o(x);
        const float sl2 = P.scale_log2;
        const int bit = 2 << x;
        int cs = 0;  // tiles processed by this warpgroup (sfull / pfull / pempty parity)
        int ne = 0;  // epilogues done (ofull parity)
        bool fine = true;
        for (int it = 0; fine; ++it) {
            const int item = static_cast<int>(blockIdx.x) + it * G;
            if (item >= P.n_items) break;
            const int bh = item % P.BH;
            const int row_start = (P.n_qpairs - 1 - item / P.BH) * BM;
            const int q0 = P.pos0 + row_start;
            const int qlast = P.pos0 + min(row_start + BM, P.L) - 1;
            const int t = q0 + x * BH_ROWS + r;  // absolute position of this thread's row
            const int b = it & 1;
            fine = __all_sync(0xFFFFFFFFu, mbar_wait(&lready[b], (it >> 1) & 1, wc, 14, it));
            if (!fine) break;
            const Tile *tl = tiles_s + b * MAX_TILES;
            const int n = ntiles_s[b];
            float mrun = -INFINITY, lrun = 0.f;  // running max (log2 units) and sum
            int cnt = 0;
            for (int j = 0; j < n; ++j) {
                const Tile T = tl[j];
                if (!(T.flags & bit)) continue;
                fine = __all_sync(0xFFFFFFFFu, mbar_wait(&sfull[x], cs & 1, wc, 6, j));
                if (!fine) break;
                tc_fence_after();
                // valid columns of this row: [0, b1] (sinks) and [a2, hc] (window), hc = last causal
                // column, as four 32-bit column masks; interior tiles need none
                const int hc = min(static_cast<int>(T.chi), t - T.pbase);
                const int b1 = min(hc, P.s - 1 - T.pbase);
                const int a2 = max(0, t - P.m + 1 - T.pbase);
                bool full = (b1 >= BN - 1) || (hc >= BN - 1 && (a2 <= 0 || b1 >= a2 - 1));
                uint32_t mw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mw[k] = full ? 0xFFFFFFFFu : (range_bits(-32 * k, b1 - 32 * k) | range_bits(a2 - 32 * k, hc - 32 * k));
                if (BS && !full && t <= qlast) {
                    // block-sparse: also the global keys of the tile and the row's random key blocks, up to hc
                    const TileMask gm = gmask_s[b * MAX_TILES + j];
                    const int* rb = P.bs_rand + static_cast<int64_t>(t / P.bs_block) * P.bs_r;
                    for (int i = 0; i < P.bs_r; ++i) {
                        const int kb = rb[i];
                        if (kb < 0) continue;
                        const int lo = kb * P.bs_block - T.pbase;
                        const int hi = min(lo + P.bs_block - 1, hc);
#pragma unroll
                        for (int k = 0; k < 4; ++k) mw[k] |= range_bits(lo - 32 * k, hi - 32 * k);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) mw[k] |= gm.w[k] & range_bits(-32 * k, hc - 32 * k);
                    full = (mw[0] & mw[1] & mw[2] & mw[3]) == 0xFFFFFFFFu;
                }
                const bool any_masked = __any_sync(0xFFFFFFFFu, !full);  // warp-uniform: no divergent paths
                // the whole row of S in registers (one TMEM load); then the S buffer is free for the next QK
                float sv[BN];
                __syncwarp();
                tmem_ld128(s_addr, sv);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfree);
                if (any_masked) {
#pragma unroll
                    for (int c = 0; c < BN; ++c) sv[c] = (mw[c >> 5] & (1u << (c & 31))) ? sv[c] : -INFINITY;
                }
                float mx4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) mx4[i] = fmax3(sv[i], sv[4 + i], sv[8 + i]);
#pragma unroll
                for (int c = 12; c < BN - 4; c += 8)
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx4[i] = fmax3(mx4[i], sv[c + i], sv[c + 4 + i]);
                const float mx = fmax3(fmax3(mx4[0], mx4[1], sv[BN - 4]), fmax3(mx4[2], mx4[3], sv[BN - 3]),
                                       fmaxf(sv[BN - 2], sv[BN - 1])) * sl2;
                float alpha = 1.f;
                bool resc = false;
                const float mnew = fmaxf(mrun, mx);
                if (mnew > mrun + kRescaleLog2) {  // also taken when mrun is still -inf
                    if (mrun != -INFINITY) {
                        alpha = ex2(mrun - mnew);
                        resc = true;
                    }
                    mrun = mnew;
                }
                // P_x and O_x are free once the PV_x products issued so far are done
                if (cs >= 1) {
                    fine = __all_sync(0xFFFFFFFFu, mbar_wait(&pempty[x], (cs - 1) & 1, wc, 7, j));
                    if (!fine) break;
                    tc_fence_after();
                }
                if (__any_sync(0xFFFFFFFFu, resc)) {
                    // O_x holds the PV products of this item's earlier tiles, all complete (pempty above)
                    __syncwarp();
#pragma unroll 1
                    for (int c = 0; c < HD; c += 32) {
                        float ov[32];
                        tmem_ld32(o_addr + c, ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] *= alpha;
                        tmem_st32(o_addr + c, ov);
                    }
                }
                // p = 2^(scale*log2(e)*s - m); bf16 pairs of keys 0..63 / 64..127 go to columns [0, 32) /
                // [32, 64) of P_x: the A operand of PV_x
                const float nmu = (mrun == -INFINITY) ? 0.f : -mrun;
                float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int c = 64 * h + 2 * i;
                        float a0, a1;
                        ffma2(a0, a1, sv[c], sv[c + 1], sl2, sl2, nmu, nmu);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        const int k = (i & 1) * 2;
                        fadd2(rs4[k], rs4[k + 1], rs4[k], rs4[k + 1], p0, p1);
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    __syncwarp();
                    tmem_st32u_nowait(p_addr + 32 * h, pk);
                }
                tmem_wait_st();
                lrun = lrun * alpha + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
                tc_fence_before();
                mbar_arrive(&pfull[x]);
                ++cnt;
                ++cs;
            }
            if (!fine) break;
            if (lane == 0) mbar_arrive(&lfree[b]);  // this warp no longer reads the tile list
            if (cnt == 0) continue;                // no row of this query tile in the sequence
            // epilogue: O_x / l -> bf16 in registers, O_x handed back to the MMA, then the rows are
            // written to global memory (and lse)
            fine = __all_sync(0xFFFFFFFFu, mbar_wait(&ofull[x], ne & 1, wc, 8, it));
            if (!fine) break;
            ++ne;
            tc_fence_after();
            const float inv = (lrun > 0.f) ? 1.f / lrun : 0.f;
            uint32_t ob[HD / 2];
            __syncwarp();
#pragma unroll
            for (int c = 0; c < HD; c += 32) {
                float ov[32];
                tmem_ld32(o_addr + c, ov);
#pragma unroll
                for (int i = 0; i < 16; ++i) ob[c / 2 + i] = pack_bf16x2(ov[2 * i] * inv, ov[2 * i + 1] * inv);
            }
            tc_fence_before();
            mbar_arrive(&oempty[x]);
            if (t <= qlast) {
                const int64_t row = static_cast<int64_t>(bh) * P.seq_stride + row_start + x * BH_ROWS + r;
                uint8_t *dst = reinterpret_cast<uint8_t *>(static_cast<__nv_bfloat16 *>(P.o) + row * HD);
#pragma unroll
                for (int i = 0; i < HD / 16; ++i)
                    st_global_v8(dst + 32 * i, ob[8 * i], ob[8 * i + 1], ob[8 * i + 2], ob[8 * i + 3], ob[8 * i + 4],
                                 ob[8 * i + 5], ob[8 * i + 6], ob[8 * i + 7]);
                if (P.lse) P.lse[row] = (mrun + log2f(lrun)) * 0.69314718055994531f;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------------------- diagnostics
__global__ void selftest_wait_kernel(DeviceStatus *status, uint32_t timeout_us) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing ever arrives on `bar`: the wait runs out, records the timeout and returns
        const WaitCtl wc{smem_u32(&abort_flag), timeout_us, status};
        mbar_wait(&bar, 0, wc, 99);
    }
}

__global__ void __launch_bounds__(128, 1) selftest_umma_kernel(const __grid_constant__ CUtensorMap ma,
                                                             const __grid_constant__ CUtensorMap mb,
                                                             const __nv_bfloat16 *__restrict__ a_glob,
                                                             float *__restrict__ c, int mode, DeviceStatus *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *As = sm, *Bs = sm + TILE_BYTES;
    uint64_t *load_bar = reinterpret_cast<uint64_t *>(sm + 2 * TILE_BYTES);
    uint64_t *mma_bar = load_bar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(load_bar + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = threadIdx.x;
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(load_bar, 1);
        mbar_init(mma_bar, 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (mode == 2) {  // stage A by threads in the 128-byte-swizzled K-major layout
        const uint4 *src = reinterpret_cast<const uint4 *>(a_glob + r * 128);
        for (int ch = 0; ch < 16; ++ch) {
            const uint4 u = src[ch];
            st_shared_v4(smem_u32(As) + (ch >> 3) * HALF_BYTES + sw128_offset(r, (ch & 7) * 8), u.x, u.y, u.z, u.w);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (mode == 3) {  // stage A into TMEM columns [128, 192): lane = row, two bf16 per 32-bit column
        const uint32_t *src = reinterpret_cast<const uint32_t *>(a_glob + r * 128);
        uint32_t u[32];
        __syncwarp();
        for (int h = 0; h < 2; ++h) {
            for (int i = 0; i < 32; ++i) u[i] = src[h * 32 + i];
            tmem_st32u(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 128 + h * 32, u);
        }
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const WaitCtl wc{smem_u32(const_cast<int *>(abort_flag)), kWaitTimeoutUs, status};
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(load_bar, mode >= 2 ? TILE_BYTES : 2 * TILE_BYTES);
        if (mode < 2) {
            tma_load_3d(As, &ma, load_bar, 0, 0, 0);
            tma_load_3d(As + HALF_BYTES, &ma, load_bar, 64, 0, 0);
        }
        tma_load_3d(Bs, &mb, load_bar, 0, 0, 0);
        tma_load_3d(Bs + HALF_BYTES, &mb, load_bar, 64, 0, 0);
        if (mbar_wait(load_bar, 0, wc, 10)) {
            tc_fence_after();
            const uint32_t a_addr = smem_u32(As), b_addr = smem_u32(Bs);
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a_off = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
                if (mode == 0)
                    umma_ss(tmem, sdesc_sw128(a_addr + a_off, 16, 1024), sdesc_sw128(b_addr + a_off, 16, 1024),
                            IDESC_QK, kk > 0 ? 1u : 0u);
                else if (mode == 3)
                    umma_ts(tmem, tmem + 128 + kk * 8, sdesc_sw128(b_addr + kk * 2048, HALF_BYTES, 1024), IDESC_PV,
                            kk > 0 ? 1u : 0u);
                else
                    umma_ss(tmem, sdesc_sw128(a_addr + a_off, 16, 1024),
                            sdesc_sw128(b_addr + kk * 2048, HALF_BYTES, 1024), IDESC_PV, kk > 0 ? 1u : 0u);
            }
            umma_commit(mma_bar);
            mbar_wait_drain(mma_bar, 0);
        } else {
            mbar_wait_drain(load_bar, 0);
        }
    }
    const bool fine = __all_sync(0xFFFFFFFFu, mbar_wait(mma_bar, 0, wc, 11));
    tc_fence_after();
    if (fine) {
        __syncwarp();
        for (int cc = 0; cc < 128; cc += 32) {
            float v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc, v);
            for (int i = 0; i < 32; ++i) c[(warp * 32 + lane) * 128 + cc + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace tc

// ---------------------------------------------------------------------------------------- host side
static bool encode_rows_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t nbh, uint64_t bh_stride_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(tc::HD), rows, nbh};
    const cuuint64_t strides[2] = {tc::HD * 2, bh_stride_rows * tc::HD * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Upper bound of the key tiles of one query tile (sink ranges, band ranges split at pos0 and at the
// ring wrap).
static int max_tiles_bound(int w, int s) {
    const int m = w - s;
    return (s + tc::BN - 1) / tc::BN + 1 + (m + tc::BM - 1 + tc::BN - 1) / tc::BN + 3;
}

static int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        cached[dev] = n;
    }
    return cached[dev];
}

static int launch_impl(const PrefillArgs &a, const BlockSparseDev *bs) {
    using namespace tc;
    if (a.d != HD) return fail(SWA_ERR_UNSUPPORTED, "tensor-core prefill needs d = %d", HD);
    if (a.q_sink) return fail(SWA_ERR_INVALID, "the RoPE prefill runs on the sub-tile kernel");
    if (!bs && max_tiles_bound(a.w, a.s) > MAX_TILES)
        return fail(SWA_ERR_UNSUPPORTED, "window w=%d needs more than %d key tiles per query tile", a.w, MAX_TILES);
    if ((a.L + BM - 1) / BM * a.BH > 0x7FFFFFFF) return fail(SWA_ERR_UNSUPPORTED, "too many work items");
    if (!encode_tiled_fn()) return fail(SWA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    unsigned *status = device_status_word();
    if (!status) return SWA_ERR_CUDA;
    Params p;
    memset(&p, 0, sizeof(p));
    const uint64_t L = static_cast<uint64_t>(a.L), st = static_cast<uint64_t>(a.seq_stride);
    bool okm = encode_rows_map(&p.tm_q, a.q, L, a.BH, st) && encode_rows_map(&p.tm_k, a.k, L, a.BH, st) &&
               encode_rows_map(&p.tm_v, a.v, L, a.BH, st);
    if (a.pos0 > 0) {
        // Only slots 0..min(pos0, w)-1 have been written; the map stops there so that TMA zero-fills the
        // rest of a tile instead of loading stale bytes (a masked column still multiplies its V row by 0,
        // and 0 * NaN would poison the accumulator).
        const uint64_t written = static_cast<uint64_t>(a.pos0 < a.w ? a.pos0 : a.w);
        okm = okm && encode_rows_map(&p.tm_kc, a.k_cache, written, a.BH, a.w) &&
              encode_rows_map(&p.tm_vc, a.v_cache, written, a.BH, a.w);
    }
    else
        okm = okm && encode_rows_map(&p.tm_kc, a.k, L, a.BH, st) && encode_rows_map(&p.tm_vc, a.v, L, a.BH, st);
    if (!okm) return fail(SWA_ERR_INVALID, "cuTensorMapEncodeTiled rejected a tensor (alignment or size)");
    p.o = a.o;
    p.lse = a.lse;
    p.status = reinterpret_cast<DeviceStatus *>(status);
    p.seq_stride = a.seq_stride;
    p.L = static_cast<int>(a.L);
    p.pos0 = static_cast<int>(a.pos0);
    p.w = a.w;
    p.s = a.s;
    p.m = a.w - a.s;
    p.BH = a.BH;
    p.n_qpairs = static_cast<int>((a.L + BM - 1) / BM);
    p.n_items = p.n_qpairs * a.BH;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.timeout_us = kWaitTimeoutUs;
    if (bs) {
        p.bs_tiles = static_cast<const Tile *>(bs->tiles);
        p.bs_gmask = static_cast<const TileMask *>(bs->gmask);
        p.bs_count = bs->count;
        p.bs_rand = bs->rand;
        p.bs_block = bs->block;
        p.bs_r = bs->r;
    }
    auto *kern = bs ? swa_prefill_tc_kernel<true> : swa_prefill_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "prefill smem attribute: %s", cudaGetErrorString(e));
    // persistent: one CTA per SM, each walking work items blockIdx.x, blockIdx.x + gridDim.x, ...
    const int sms = sm_count();
    if (sms <= 0) return fail(SWA_ERR_CUDA, "cannot read the multiprocessor count");
    const dim3 grid(p.n_items < sms ? p.n_items : sms), block(kThreads);
    kern<<<grid, block, SMEM_BYTES, a.stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

int launch_prefill_bf16_tc_plain(const PrefillArgs &a) { return launch_impl(a, nullptr); }

int launch_prefill_bf16_tc_blocksparse(const PrefillArgs &a, const BlockSparseDev &bs) { return launch_impl(a, &bs); }

// Host: the key-tile lists of the block-sparse prefill, one per 256-row query pair, in the kernel's layout.  A
// pair [q0, qlast] needs the sinks, its band [q0 - m + 1, qlast], every global position <= qlast, and the
// random key blocks (<= qlast) of every query block it overlaps: these ranges are merged into disjoint runs,
// so that each key position appears in exactly one tile, and cut into tiles of up to 128 keys.  Per tile the
// columns holding a global key are listed (the per-row masks of the kernel add them to the band and sinks),
// and the tile is marked for the query tiles that have some row it can serve.  Returns SWA_OK or an error.
size_t blocksparse_tile_list_bytes(int64_t L) {
    const size_t pairs = static_cast<size_t>((L + tc::BM - 1) / tc::BM);
    return pairs * tc::MAX_TILES * (sizeof(tc::Tile) + sizeof(tc::TileMask));
}

int blocksparse_build_lists(int64_t L, int w, int s, const int32_t *globals, int n_globals, int block,
                            const int32_t *rand, int r, void *tiles_out, void *gmask_out, int *count_out) {
    using namespace tc;
    const int m = w - s;
    const int pairs = static_cast<int>((L + BM - 1) / BM);
    Tile *tiles = static_cast<Tile *>(tiles_out);
    TileMask *gmask = static_cast<TileMask *>(gmask_out);
    std::vector<std::pair<int, int>> iv;
    for (int qp = 0; qp < pairs; ++qp) {
        const int q0 = qp * BM;
        const int qlast = static_cast<int>(std::min<int64_t>(q0 + BM, L)) - 1;
        const int blo = std::max(0, q0 - m + 1);
        iv.clear();
        if (s > 0) iv.emplace_back(0, std::min(s, qlast + 1) - 1);
        iv.emplace_back(blo, qlast);
        for (int i = 0; i < n_globals && globals[i] <= qlast; ++i) iv.emplace_back(globals[i], globals[i]);
        for (int qb = q0 / block; qb <= qlast / block; ++qb)
            for (int i = 0; i < r; ++i) {
                const int kb = rand[static_cast<int64_t>(qb) * r + i];
                if (kb < 0 || static_cast<int64_t>(kb) * block > qlast) continue;
                iv.emplace_back(kb * block, static_cast<int>(std::min<int64_t>(static_cast<int64_t>(kb) * block + block - 1, qlast)));
            }
        std::sort(iv.begin(), iv.end());
        int n = 0;
        Tile *tl = tiles + static_cast<int64_t>(qp) * MAX_TILES;
        TileMask *gm = gmask + static_cast<int64_t>(qp) * MAX_TILES;
        size_t k = 0;
        while (k < iv.size()) {
            int a = iv[k].first, b = iv[k].second;
            for (++k; k < iv.size() && iv[k].first <= b + 1; ++k) b = std::max(b, iv[k].second);
            for (int p = a; p <= b; p += BN) {
                if (n >= MAX_TILES)
                    return fail(SWA_ERR_UNSUPPORTED, "query rows %d..%d need more than %d key tiles", q0, qlast, MAX_TILES);
                Tile &T = tl[n];
                T.row0 = p;
                T.pbase = p;
                T.chi = static_cast<short>(std::min(b - p, BN - 1));
                TileMask &G = gm[n];
                G.w[0] = G.w[1] = G.w[2] = G.w[3] = 0;
                const int32_t *g0 = std::lower_bound(globals, globals + n_globals, p);
                for (const int32_t *gp = g0; gp < globals + n_globals && *gp <= p + T.chi; ++gp)
                    G.w[(*gp - p) >> 5] |= 1u << ((*gp - p) & 31);
                // query tiles served: band / sink criterion, a global key at or before the tile's last row, or a
                // random key block of one of its query blocks
                int f = 0;
                const int pe = p + T.chi;
                for (int x = 0; x < 2; ++x) {
                    const int ra = q0 + x * BH_ROWS, rb = std::min(q0 + x * BH_ROWS + BH_ROWS - 1, qlast);
                    if (ra > rb || p > rb) continue;
                    bool need = p < s || pe >= ra - m + 1;
                    for (const int32_t *gp = g0; !need && gp < globals + n_globals && *gp <= std::min(pe, rb); ++gp) need = true;
                    for (int qb = ra / block; !need && qb <= rb / block; ++qb)
                        for (int i = 0; i < r && !need; ++i) {
                            const int64_t kb = rand[static_cast<int64_t>(qb) * r + i];
                            need = kb >= 0 && kb * block <= pe && kb * block + block - 1 >= p;
                        }
                    if (need) f |= 2 << x;
                }
                T.flags = static_cast<short>(f);
                if (f) ++n;  // a tile no query tile needs is dropped
            }
        }
        count_out[qp] = n;
    }
    return SWA_OK;
}

int prefill_tile_plan(int q0, int q1, int pos0, int w, int s, int rope, int *out, int max_tiles) {
    if (rope) return prefill_tile_plan_sub(q0, q1, pos0, w, s, rope, out, max_tiles);
    tc::Tile tl[tc::MAX_TILES];
    const int n = tc::build_tiles(tl, q0, q1, pos0, s, w - s, w, rope != 0);
    tc::mark_tiles(tl, n, q0, q1, s, w - s);
    for (int i = 0; i < n && i < max_tiles && i < tc::MAX_TILES; ++i) {
        out[5 * i + 0] = tl[i].flags & 1;
        out[5 * i + 1] = tl[i].row0;
        out[5 * i + 2] = tl[i].pbase;
        out[5 * i + 3] = tl[i].chi;
        out[5 * i + 4] = tl[i].flags >> 1;
    }
    return n;
}

int launch_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
    unsigned *status = device_status_word();
    if (!status) return SWA_ERR_CUDA;
    const uint32_t us = static_cast<uint32_t>((timeout_ns + 999) / 1000);
    tc::selftest_wait_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<DeviceStatus *>(status), us);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

int launch_selftest_umma(const void *a, const void *b, float *c, int mode, cudaStream_t stream) {
    unsigned *status = device_status_word();
    if (!status) return SWA_ERR_CUDA;
    if (!encode_tiled_fn()) return fail(SWA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    CUtensorMap ma, mb;
    if (!encode_rows_map(&ma, a, 128, 1, 128) || !encode_rows_map(&mb, b, 128, 1, 128))
        return fail(SWA_ERR_INVALID, "cuTensorMapEncodeTiled rejected a selftest operand");
    const uint32_t smem = 2 * tc::TILE_BYTES + 64 + 1024;
    cudaError_t e = cudaFuncSetAttribute(tc::selftest_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "selftest smem attribute: %s", cudaGetErrorString(e));
    tc::selftest_umma_kernel<<<1, 128, smem, stream>>>(ma, mb, static_cast<const __nv_bfloat16 *>(a), c, mode,
                                                       reinterpret_cast<DeviceStatus *>(status));
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

}  // namespace swa
