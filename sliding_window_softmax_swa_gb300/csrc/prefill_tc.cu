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
// Work item = one query tile of 128 rows of one (b, h).  The kernel is persistent: one CTA per SM walks the
// items blockIdx.x, blockIdx.x + gridDim.x, ..., ordered longest-first (the last query tiles of every head,
// whose windows are full, come first), so the short items fall in the last rounds and the CTAs finish
// together.  The key tiles of an item are split into two streams, the even and the odd tiles, each with its
// own S buffer, O accumulator, running max and sum: while one stream's softmax works on its tile, the tensor
// cores run the other stream's products, and no thread exchanges anything with another during the tile walk.
// The epilogue merges the two streams of each row by their maxima.  352 threads in four roles:
//   warps 0-7  softmax + epilogue: stream g = w / 4; warp w owns TMEM lanes 32 (w mod 4) .. +31 (rows of the
//              tile), one thread per row with all 128 columns of its score row.  At the end of an item the two
//              threads of a row (warps w and w + 4) exchange (max, sum) through shared memory at a named
//              barrier of the two warps, each merges half of the row's columns of both O buffers, and the
//              bf16 rows are staged in the item's Q buffer (free once its QK products are done);
//   warp 8     TMA producers: lane 0 streams K tiles, lane 1 V tiles (128 rows x 128 bf16, two 64-column boxes
//              with the 128-byte swizzle), each through its own 2-stage ring over all items of the CTA;
//   warp 9     MMA issuer, the whole warp converged, one elected lane issuing: per item QK(0), QK(1), then per
//              key tile j PV(j), QK(j+2), where QK(j) is S = Q K_j^T into S buffer j mod 2 and PV(j) is
//              O_{j mod 2} += P_j V_j with P_j (bf16 pairs written over the first 64 columns of its S buffer)
//              read by the MMA straight from tensor memory; S buffer j mod 2 is reused by QK(j+2) after PV(j) in
//              issue order (tcgen05 MMAs of a thread complete in order).  In block-sparse mode PV(j) runs in two
//              parts: keys 0..63 once that half of P_j is written (and O rescaled), the rest once all of it is.
//              The single issue order keeps the two streams out of phase.  A narrow tile (all keys in its first 16 columns, such as the sink tile)
//              takes an N = 16 QK product and one 16-key PV product;
//   warp 10    per item: builds the key-tile list into one of two buffers, one item ahead; stores the O rows
//              that the epilogue of the item two back staged in the item's Q buffer (TMA, so that the softmax
//              threads never wait on global stores), then loads the item's Q there and prefetches the next
//              item's Q into L2.
// TMEM (512 columns): S buffers [0,128), [128,256) and O buffers [256,384), [384,512) of the two streams (fp32,
// lane = row).  The online softmax keeps a running max in log2 units and only rescales O (TMEM load,
// multiply, store) when the max grows by more than 8 (a factor 256), so p <= 256 always fits bf16/fp32 and
// the rescale is rare; O and l of a stream always share the same reference max.  S_j complete implies every
// MMA issued before QK(j), in particular the stream's PV(j-2), is complete, so a rescale needs no wait.
//
// Key tiles.  For the query rows [q0, q1] of an item the key positions needed are the sinks [0, min(s, blo)) and
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

constexpr int BQ = 128;                    // query rows per work item (= TMEM lanes)
constexpr int BH_ROWS = BQ;                // rows per query tile in the tile-list marks
constexpr int BM = 2 * BQ;                 // rows of a query pair (the block-sparse lists are built per pair)
constexpr int BN = 128;                    // keys per key tile
constexpr int HD = 128;                    // head dimension
constexpr int NK = 2;                      // K tile slots: slot j mod 2 holds key tile j of an item
constexpr int NV = 2;                      // V tile stages (a slot frees after its PV products)
constexpr uint32_t HALF_BYTES = 128 * 128;  // one 64-column half of a 128-row bf16 tile (16 KB)
constexpr uint32_t TILE_BYTES = 2 * HALF_BYTES;
constexpr int MAX_TILES = 64;
constexpr int kSmWarps = 8;                    // softmax warps: four per stream
constexpr int kSmThreads = kSmWarps * 32;
constexpr int kWarpTma = kSmWarps, kWarpMma = kSmWarps + 1, kWarpList = kSmWarps + 2;
constexpr int kThreads = (kSmWarps + 3) * 32;  // softmax warps, TMA producers, MMA issuer, tile lists
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S buffers 0, 1 of the two streams (scores fp32, then P as bf16 pairs in their first 64
// columns) and their O buffers 0, 1 (fp32 accumulators)
__host__ __device__ constexpr uint32_t col_s(int b) { return static_cast<uint32_t>(b) * 128u; }
__host__ __device__ constexpr uint32_t col_o(int b) { return 256u + static_cast<uint32_t>(b) * 128u; }
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the running max grows by more than 2^8

constexpr uint32_t OFF_Q = 0;                         // Q buffers 0, 1 (alternate items; the O staging)
constexpr uint32_t OFF_K = OFF_Q + 2 * TILE_BYTES;
constexpr uint32_t OFF_V = OFF_K + NK * TILE_BYTES;
constexpr uint32_t OFF_BAR = OFF_V + NV * TILE_BYTES;
constexpr uint32_t OFF_MISC = OFF_BAR + 256;
constexpr uint32_t OFF_TILES = OFF_MISC + 64;
constexpr uint32_t TILE_RECORD = 16;                              // bytes of one tile record (struct Tile)
constexpr uint32_t OFF_GMASK = OFF_TILES + 2 * MAX_TILES * TILE_RECORD;  // two tile lists (current / next item)
constexpr uint32_t OFF_XCH = OFF_GMASK + 2 * MAX_TILES * 16;       // and their global-key columns (block-sparse)
constexpr uint32_t OFF_RKS = OFF_XCH + 2 * 4 * BQ * 4;               // (max, sum) exchange of the two streams
constexpr uint32_t SMEM_USED = OFF_RKS + 2 * BQ * 8;                // per softmax thread: its row's random blocks
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024 bytes
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false, false);  // Q, K both K-major
constexpr uint32_t IDESC_QK16 = idesc_bf16_f32(128, 16, false, false);  // a narrow tile: its first 16 keys
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 128, false, true);   // P K-major, V MN-major

struct Tile {
    int row0;     // first source row (TMA row coordinate)
    int pbase;    // absolute position of column 0
    short chi;    // last valid column (columns past it belong to another tile or to nothing)
    short flags;  // bit 0: source (0 = this call's k/v rows, 1 = rolling cache); bit 1 + x: needed by query tile x;
                  // bit 3: a packed tile of two 64-key blocks (block-sparse mode, rows = positions)
    int row1;     // packed tile: first row (= position) of columns 64..127 (rows row0 .. row0 + 63 fill 0..63)
};
static_assert(sizeof(Tile) == TILE_RECORD, "tile record");
constexpr short kTilePacked = 8;

// Block-sparse mode: per column of a key tile, whether it holds a global key (bit c of word c / 32).
struct TileMask {
    uint32_t w[4];
};

struct Params {
    CUtensorMap tm_q, tm_k, tm_v, tm_kc, tm_vc, tm_o;  // tm_o: the rows of o, laid out as tm_q
    CUtensorMap tm_k64, tm_v64;  // block-sparse mode: 64-row boxes of k / v, the halves of a packed tile
    // block-sparse mode: the host-built key-tile lists of every 256-row query pair (MAX_TILES entries per pair,
    // bs_count[pair] used), their global-key columns, and the random key blocks of each query block
    const Tile *bs_tiles;
    const TileMask *bs_gmask;
    const int *bs_count;
    const int *bs_rand;  // [ceil(L / bs_block)][bs_r]; -1 = no block
    int bs_block, bs_r;
    int bs_kblocks;  // key blocks of the sequence: ceil(L / bs_block)
    void *o;
    float *lse;
    DeviceStatus *status;
    int64_t seq_stride;  // rows between (b, h) blocks of q/k/v/o/lse
    int L, pos0, w, s, m, BH;
    int qoff;               // position of query row 0 of an item's sequence: pos0, or s in dilated mode
    int n_qtiles, n_items;  // 128-row query tiles per (b, h) (per class in dilated mode); work items
    // dilated mode: dil_r residue classes per (b, h); tm_q / tm_k / tm_v are 4-D maps (d, class, group, (b, h))
    // over position = group * dil_r + class for the groups [0, dil_G); tm_kc / tm_vc the plain rows (sinks)
    int dil_r, dil_G;
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
                tl[n].row1 = 0;
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

// Dilated mode.  Residue class c of the positions mod r starts (after the sinks) at position p0(c) =
// s + ((c - s) mod r), in group g0(c) = (p0(c) - c) / r of the 4-D map (position = group * r + class).
__host__ __device__ inline int dil_p0(int c, int s, int r) { return s + ((c - s) % r + r) % r; }
__host__ __device__ inline int dil_g0(int c, int s, int r) { return (dil_p0(c, s, r) - c) / r; }

// The key tiles of the dilated-mode work item over the class-c virtual rows [s + row_start, s + row_start + 127]
// (clipped to s + nrows - 1), in virtual positions (the sinks, then the class's positions >= s one per row):
// the sinks on their own (source bit set: plain rows of k / v), then the band from s, whose tiles start at group
// g0 + (position - s) of the class.  Returns the tile count as build_tiles does.
__host__ __device__ int build_tiles_dilated(Tile *tl, int row_start, int c, int s, int m, int w, int r, int nrows) {
    const int q0 = s + row_start;
    const int qlast = s + (row_start + BQ < nrows ? row_start + BQ : nrows) - 1;
    const int n = build_tiles(tl, q0, qlast, 0, s, m, w, true);
    if (n >= 1 && n <= MAX_TILES) {
        mark_tiles(tl, n, q0, qlast, s, m);
        const int g0 = dil_g0(c, s, r);
        for (int i = 0; i < n; ++i) {
            if (tl[i].pbase < s)
                tl[i].flags = static_cast<short>(tl[i].flags | 1);
            else
                tl[i].row0 = g0 + (tl[i].pbase - s);
        }
    }
    return n;
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
// A narrow tile (every key in its first 16 columns, as the sink tile with s <= 16) takes a 16-column QK
// product and one 16-key PV product.
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr, bool narrow) {
    const uint32_t qlo = sdesc_sw128_lo(q_addr, 16), klo = sdesc_sw128_lo(k_addr, 16);
    constexpr uint32_t hi = sdesc_sw128_hi(1024);
    const uint32_t idesc = narrow ? IDESC_QK16 : IDESC_QK;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4;
        umma_ss_warp_lo(d_tmem, qlo + off, klo + off, hi, idesc, kk > 0 ? 1u : 0u);
    }
}

// Key steps [k0, k1) of 16 keys each (block-sparse mode runs PV in two parts, keys 0..63 as soon as their half
// of P is written).
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr, bool accumulate,
                                         int k0, int k1) {
    const uint32_t vlo = sdesc_sw128_lo(v_addr, HALF_BYTES);
    constexpr uint32_t hi = sdesc_sw128_hi(1024);
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
        if (kk < k0 || kk >= k1) continue;
        // P from TMEM: 16 keys = 8 columns of packed bf16 pairs; V: 16 key rows of 128 bytes (MN-major)
        umma_ts_warp_lo(d_tmem, p_tmem + kk * 8, vlo + ((kk * 16 * 128) >> 4), hi, IDESC_PV,
                        (accumulate || kk > 0) ? 1u : 0u);
    }
}

// MODE 0: plain.  MODE 1: block-sparse (host-built tile lists with global keys and random key blocks).  MODE 2:
// dilated window (a work item is one query tile of one residue class of one (b, h), in the class's virtual
// rows: the sinks, then the class's positions >= s; the band tiles and Q come through 4-D maps that step r
// positions per row, and the epilogue writes each row back at its own position).  The modes are compiled apart,
// so that the plain kernel carries none of the others' work.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) swa_prefill_tc_kernel(const __grid_constant__ Params P) {
    constexpr bool BS = MODE == 1, DIL = MODE == 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *qfull = bars;           // [2]: Q buffer b landed
    uint64_t *ostage = qfull + 2;     // [2]: the item's O rows staged in Q buffer b (all softmax threads)
    uint64_t *kfull = ostage + 2;     // [NK] (K slot g is free again once sfull[g] completes)
    uint64_t *vfull = kfull + NK;     // [NV]
    uint64_t *vempty = vfull + NV;    // [NV]
    uint64_t *sfull = vempty + NV;    // [2]: S buffer g holds Q K_j^T of stream g
    uint64_t *pfull = sfull + 2;      // [2]: P_j written over S buffer g (the stream's 128 softmax threads)
    uint64_t *ofull = pfull + 2;      // the last PV product of an item is done
    uint64_t *oempty = ofull + 1;     // both O buffers have been read by the item's epilogue (all softmax threads)
    uint64_t *lready = oempty + 1;    // [2]: tile list buffer b written (1 arrival)
    uint64_t *lfree = lready + 2;     // [2]: tile list buffer b no longer read (softmax warps, MMA, 2 loaders)
    uint64_t *drain = lfree + 2;
    uint64_t *phalf = drain + 1;      // [2] (block-sparse mode): keys 0..63 of P_j written and O rescaled
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);
    int *ntiles_s = reinterpret_cast<int *>(sm + OFF_MISC + 8);  // [2]
    Tile *tiles_s = reinterpret_cast<Tile *>(sm + OFF_TILES);     // [2][MAX_TILES]
    TileMask *gmask_s = reinterpret_cast<TileMask *>(sm + OFF_GMASK);  // [2][MAX_TILES] (block-sparse)
    float *xch = reinterpret_cast<float *>(sm + OFF_XCH);  // [2 slots][2 streams][max, sum][128 rows]
    uint2 *rks_s = reinterpret_cast<uint2 *>(sm + OFF_RKS);  // [2 streams][128 rows] (block-sparse)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&ostage[i], kSmThreads);
            mbar_init(&kfull[i], 1);
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], 1);
            mbar_init(&sfull[i], 1);
            mbar_init(&pfull[i], kSmThreads / 2);
            mbar_init(&phalf[i], kSmThreads / 2);
            mbar_init(&lready[i], 1);
            mbar_init(&lfree[i], kSmWarps + 3);
        }
        mbar_init(ofull, 1);
        mbar_init(oempty, kSmThreads);
        mbar_init(drain, 1);
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
    // work item -> (b, h), residue class (dilated mode) and first row of its query tile (longest-first order:
    // the last query tiles of every head, whose windows are full, come first)
    auto item_rows = [&](int item, int &bh, int &row_start, int &cls) {
        const int grp = DIL ? P.BH * P.dil_r : P.BH;
        const int rem = item % grp;
        bh = rem % P.BH;
        cls = DIL ? rem / P.BH : 0;
        row_start = (P.n_qtiles - 1 - item / grp) * BQ;
    };
    // dilated mode: the first position >= s of class c, and its group
    auto class_p0 = [&](int c) { return dil_p0(c, P.s, P.dil_r); };
    auto class_g0 = [&](int c) { return dil_g0(c, P.s, P.dil_r); };

    if (warp == kWarpTma) {
        // ------------------------------------------------------------------ TMA producers (K, V)
        // Lane 0 streams the K tiles, lane 1 the V tiles, each over all items of this CTA in order, so neither
        // waits for the other, and the K loads run ahead into the next item on their own.  Key tile j of an
        // item goes to K slot j mod 2, the index of the S buffer its QK product writes, so the slot is free
        // again when the previous QK product into that S buffer is done: the sfull phase the softmax waits for
        // (no commit of its own).  The V tiles run through a 2-stage ring whose slots free after their PV
        // products.
        if (lane < 2) {
            const bool isk = lane == 0;
            uint64_t *full = isk ? kfull : vfull;
            uint8_t *ring = sm + (isk ? OFF_K : OFF_V);
            const CUtensorMap *m_seq = isk ? &P.tm_k : &P.tm_v;
            const CUtensorMap *m_cache = isk ? &P.tm_kc : &P.tm_vc;
            tma_prefetch_desc(m_seq);
            int g = 0;           // tiles issued so far
            int nk0 = 0, nk1 = 0;  // K lane: tiles loaded into slot 0 / 1
            for (int it = 0;; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * G;
                if (item >= P.n_items) break;
                const int b = it & 1;
                if (!mbar_wait(&lready[b], (it >> 1) & 1, wc, 15, it)) break;
                const int n = ntiles_s[b];
                int bh, row_start, cls;
                item_rows(item, bh, row_start, cls);
                bool fine = true;
                for (int j = 0; j < n; ++j) {
                    const int st = isk ? (j & 1) : g % NV;
                    const int nst = st ? nk1 : nk0;  // K: earlier loads into this slot
                    const bool ready = isk ? (nst == 0 || mbar_wait(&sfull[st], (nst - 1) & 1, wc, 1, j))
                                           : mbar_wait(&vempty[st], ((g / NV) & 1) ^ 1, wc, 9, j);
                    if (!ready) {
                        fine = false;
                        break;
                    }
                    const Tile T = tiles_s[b * MAX_TILES + j];
                    const CUtensorMap *mp = (T.flags & 1) ? m_cache : m_seq;
                    uint8_t *dst = ring + st * TILE_BYTES;
                    mbar_arrive_expect_tx(&full[st], TILE_BYTES);
                    if (DIL && !(T.flags & 1)) {  // band rows of the class: row0 is the group index
                        tma_load_4d(dst, mp, &full[st], 0, cls, T.row0, bh);
                        tma_load_4d(dst + HALF_BYTES, mp, &full[st], 64, cls, T.row0, bh);
                    } else if (BS && (T.flags & kTilePacked)) {  // two 64-row blocks: rows 0..63 and 64..127
                        const CUtensorMap *m64 = isk ? &P.tm_k64 : &P.tm_v64;
                        tma_load_3d(dst, m64, &full[st], 0, T.row0, bh);
                        tma_load_3d(dst + HALF_BYTES, m64, &full[st], 64, T.row0, bh);
                        tma_load_3d(dst + 64 * 128, m64, &full[st], 0, T.row1, bh);
                        tma_load_3d(dst + HALF_BYTES + 64 * 128, m64, &full[st], 64, T.row1, bh);
                    } else {
                        tma_load_3d(dst, mp, &full[st], 0, T.row0, bh);
                        tma_load_3d(dst + HALF_BYTES, mp, &full[st], 64, T.row0, bh);
                    }
                    if (isk) {
                        nk0 += st ^ 1;
                        nk1 += st;
                    }
                    ++g;
                }
                if (!fine) break;
                mbar_arrive(&lfree[b]);  // this lane no longer reads the item's list
            }
            if (*abort_flag) {  // make sure no copy is still landing in shared memory
                if (isk) {
                    if (nk0 > 0) mbar_wait_drain(&full[0], (nk0 - 1) & 1);
                    if (nk1 > 0) mbar_wait_drain(&full[1], (nk1 - 1) & 1);
                } else {
                    for (int gg = (g > NV ? g - NV : 0); gg < g; ++gg) mbar_wait_drain(&full[gg % NV], (gg / NV) & 1);
                }
            }
        }
    } else if (warp == kWarpList) {
        // ------------------------------------------------------------------ tile lists and Q
        // Per item: the key-tile list goes to buffer it & 1 as soon as the buffer's previous item (it - 2) has
        // been released by every reader.  Q buffer it & 1 then holds item it - 2's O rows, staged there by its
        // epilogue: they go to global memory by TMA (the epilogue's own threads never wait for global stores),
        // and once the store has read them the item's Q tile is loaded there, and the next item's Q into L2.
        if (lane == 0) {
            // the O tile of an item, staged in a Q buffer, to global memory (rows outside o are not written)
            auto store_o = [&](int oitem, const uint8_t *src) {
                int obh, orow, ocls;
                item_rows(oitem, obh, orow, ocls);
                if (DIL) {
                    const int gq = class_g0(ocls) + orow;
                    tma_store_4d(&P.tm_o, src, 0, ocls, gq, obh);
                    tma_store_4d(&P.tm_o, src + HALF_BYTES, 64, ocls, gq, obh);
                } else {
                    tma_store_3d(&P.tm_o, src, 0, orow, obh);
                    tma_store_3d(&P.tm_o, src + HALF_BYTES, 64, orow, obh);
                }
                bulk_commit_group();
            };
            int nq = 0;  // Q loads issued
            for (int it = 0;; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * G;
                if (item >= P.n_items) break;
                int bh, row_start, cls;
                item_rows(item, bh, row_start, cls);
                const int q0 = P.qoff + row_start;
                const int qlast = P.qoff + min(row_start + BQ, P.L) - 1;
                const int b = it & 1;
                if (it >= 2 && !mbar_wait(&lfree[b], ((it - 2) >> 1) & 1, wc, 12, it)) break;
                Tile *tl = tiles_s + b * MAX_TILES;
                int n = 0;
                if (BS) {  // the tiles of the 256-row pair's host-built list that this query tile uses
                    const int qp = row_start / (2 * BQ), bit = 2 << ((row_start / BQ) & 1);
                    const int cnt = P.bs_count[qp];
                    if (cnt >= 1 && cnt <= MAX_TILES) {
                        const Tile *src = P.bs_tiles + static_cast<int64_t>(qp) * MAX_TILES;
                        const TileMask *gsrc = P.bs_gmask + static_cast<int64_t>(qp) * MAX_TILES;
                        for (int i = 0; i < cnt; ++i) {
                            if (!(src[i].flags & bit)) continue;
                            tl[n] = src[i];
                            tl[n].flags = static_cast<short>((src[i].flags & (1 | kTilePacked)) | 2);
                            gmask_s[b * MAX_TILES + n] = gsrc[i];
                            ++n;
                        }
                    }
                } else if (DIL) {
                    n = build_tiles_dilated(tl, row_start, cls, P.s, P.m, P.w, P.dil_r, P.L);
                } else {
                    n = build_tiles(tl, q0, qlast, P.pos0, P.s, P.m, P.w, false);
                    if (n >= 1 && n <= MAX_TILES) mark_tiles(tl, n, q0, qlast, P.s, P.m);
                }
                if (n < 1 || n > MAX_TILES) {
                    atomicOr(&P.status->word, kDevBadArg);
                    *abort_flag = 1;
                    break;
                }
                ntiles_s[b] = n;
                mbar_arrive(&lready[b]);  // release: the list is visible to whoever sees the phase complete
                // Q buffer b: item it - 2's O rows, staged there by its epilogue, go out first; then the item's Q
                uint8_t *qs = sm + OFF_Q + b * TILE_BYTES;
                if (it >= 2) {
                    if (!mbar_wait(&ostage[b], ((it - 2) >> 1) & 1, wc, 13, it)) break;
                    store_o(item - 2 * G, qs);
                    bulk_wait_read_all();
                }
                mbar_arrive_expect_tx(&qfull[b], TILE_BYTES);
                if (DIL) {
                    const int gq = class_g0(cls) + row_start;
                    tma_load_4d(qs, &P.tm_q, &qfull[b], 0, cls, gq, bh);
                    tma_load_4d(qs + HALF_BYTES, &P.tm_q, &qfull[b], 64, cls, gq, bh);
                } else {
                    tma_load_3d(qs, &P.tm_q, &qfull[b], 0, row_start, bh);
                    tma_load_3d(qs + HALF_BYTES, &P.tm_q, &qfull[b], 64, row_start, bh);
                }
                ++nq;
                // into L2 meanwhile: the next item's Q rows
                const int nitem = item + G;
                if (nitem < P.n_items) {
                    int nbh, nrow, ncls;
                    item_rows(nitem, nbh, nrow, ncls);
                    if (DIL) {
                        const int gq = class_g0(ncls) + nrow;
                        tma_prefetch_4d(&P.tm_q, 0, ncls, gq, nbh);
                        tma_prefetch_4d(&P.tm_q, 64, ncls, gq, nbh);
                    } else {
                        tma_prefetch_3d(&P.tm_q, 0, nrow, nbh);
                        tma_prefetch_3d(&P.tm_q, 64, nrow, nbh);
                    }
                }
            }
            // the O rows of the last two items
            const int it_end = (P.n_items - static_cast<int>(blockIdx.x) + G - 1) / G;  // items of this CTA
            for (int it = (it_end > 2 ? it_end - 2 : 0); it < it_end && !*abort_flag; ++it) {
                if (!mbar_wait(&ostage[it & 1], (it >> 1) & 1, wc, 13, it)) break;
                store_o(static_cast<int>(blockIdx.x) + it * G, sm + OFF_Q + (it & 1) * TILE_BYTES);
            }
            bulk_wait_all();
            if (*abort_flag) {  // no copy may still be landing
                for (int i = (nq > 2 ? nq - 2 : 0); i < nq; ++i) mbar_wait_drain(&qfull[i & 1], (i >> 1) & 1);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------------ MMA issuer
        // Two streams per item: key tile j belongs to stream j mod 2, which owns S buffer and O buffer j mod 2.
        // Per item with key tiles 0..n-1: QK(0), QK(1), then per j: PV(j) into O buffer j mod 2 once P_j is in
        // S buffer j mod 2, followed by QK(j + 2) into that S buffer (tcgen05 MMAs of a thread run in order, so
        // QK(j + 2) overwrites P_j only after PV(j) has read it).  While one stream's softmax works on its tile,
        // the tensor cores run the other stream's products; the single issue order keeps the two streams out
        // of phase.  An item's first PV product waits until the previous item's epilogue has read both O
        // buffers.  The whole warp runs the loop (uniform operands); one elected lane issues each instruction.
        {
            auto wwait = [&](uint64_t *bar, int parity, unsigned site, unsigned tag) -> bool {
                return __all_sync(0xFFFFFFFFu, mbar_wait(bar, static_cast<uint32_t>(parity), wc, site, tag));
            };
            const uint32_t q_addr0 = smem_u32(sm + OFF_Q);
            const uint32_t k_addr0 = smem_u32(sm + OFF_K), v_addr0 = smem_u32(sm + OFF_V);
            bool issued_any = false, fine = true;
            int nk0 = 0, nk1 = 0;  // K tiles consumed from slot 0 / 1
            int gv = 0;            // V tiles consumed
            int np0 = 0, np1 = 0;  // P tiles consumed per stream (pfull parity)
            for (int it = 0; fine; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * G;
                if (item >= P.n_items) break;
                const int b = it & 1;  // tile list and Q buffer of this item
                if (!wwait(&lready[b], (it >> 1) & 1, 14, it)) break;
                if (!wwait(&qfull[b], (it >> 1) & 1, 2, it)) break;
                tc_fence_after();
                const int n = ntiles_s[b];
                const uint32_t q_addr = q_addr0 + b * TILE_BYTES;
                const Tile *tl = tiles_s + b * MAX_TILES;
                auto qk = [&](int j) -> bool {  // QK(j) into S buffer j mod 2, K from slot j mod 2
                    const int sk = j & 1;
                    if (!wwait(&kfull[sk], (sk ? nk1 : nk0) & 1, 3, j)) return false;
                    tc_fence_after();
                    issue_qk(tmem + col_s(sk), q_addr, k_addr0 + sk * TILE_BYTES, tl[j].chi < 16);
                    umma_commit_warp(&sfull[sk]);  // S ready, and K slot sk free
                    nk0 += sk ^ 1;
                    nk1 += sk;
                    issued_any = true;
                    return true;
                };
                fine = qk(0) && (n < 2 || qk(1));
                for (int j = 0; fine && j < n; ++j) {
                    const int st = j & 1;
                    // block-sparse mode: PV(j) in two parts, keys 0..63 once their half of P is written (the
                    // softmax threads write the other half meanwhile), keys 64..127 once all of P is
                    const int pp = (st ? np1 : np0) & 1;
                    if (!wwait(BS ? &phalf[st] : &pfull[st], pp, BS ? 16 : 4, j)) { fine = false; break; }
                    np1 += st;
                    np0 += st ^ 1;
                    if (j == 0 && it >= 1 && !wwait(oempty, (it - 1) & 1, 11, j)) { fine = false; break; }
                    const int sv = gv % NV;
                    if (!wwait(&vfull[sv], (gv / NV) & 1, 5, j)) { fine = false; break; }
                    tc_fence_after();
                    const bool nar = tl[j].chi < 16;
                    const uint32_t o_t = tmem + col_o(st), p_t = tmem + col_s(st), v_a = v_addr0 + sv * TILE_BYTES;
                    if (BS) {
                        issue_pv(o_t, p_t, v_a, j >= 2, 0, nar ? 1 : BN / 32);
                        if (!wwait(&pfull[st], pp, 4, j)) { fine = false; break; }
                        tc_fence_after();
                        if (!nar) issue_pv(o_t, p_t, v_a, true, BN / 32, BN / 16);
                    } else {
                        issue_pv(o_t, p_t, v_a, j >= 2, 0, nar ? 1 : BN / 16);
                    }
                    umma_commit_warp(&vempty[sv]);
                    if (j == n - 1) umma_commit_warp(ofull);  // the item's last product
                    ++gv;
                    if (j + 2 < n && !qk(j + 2)) { fine = false; break; }
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
        // Stream g = warp / 4: the warps 4 g .. 4 g + 3 take the key tiles j = g, g + 2, ... of every item, with
        // S buffer g, O buffer g and their own running max and sum.  Thread = row of the query tile = TMEM lane
        // 32 (w mod 4) + lane, all 128 columns of its score row, so the softmax needs no exchange per tile.  At
        // the end of an item the two threads of a row (warps w and w + 4) exchange (max, sum) through shared
        // memory and merge the two O buffers, each writing half of the row's columns.
        const int g = warp >> 2;
        // the two warps that share rows (w and w + 4) meet once per item: named barrier 1 + w mod 4
        const uint32_t pair_bar = 1u + static_cast<uint32_t>(warp & 3);
        const int r = threadIdx.x & (BQ - 1);  // row within the query tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + col_s(g);
        const uint32_t o_addr = tmem + lane_base + col_o(g);
        const float sl2 = P.scale_log2;
        const uint32_t abort_a = smem_u32(const_cast<int *>(abort_flag));
        int v = 0;   // S tiles of this stream processed (sfull / pfull parity)
        int nx = 0;  // exchanges done (slot parity)
        for (int it = 0;; ++it) {
            const int item = static_cast<int>(blockIdx.x) + it * G;
            if (item >= P.n_items) break;
            int bh, row_start, cls;
            item_rows(item, bh, row_start, cls);
            const int q0 = P.qoff + row_start;
            const int qlast = P.qoff + min(row_start + BQ, P.L) - 1;
            const int t = q0 + r;  // absolute (dilated mode: virtual) position of this thread's row
            const int b = it & 1;
            // a failed wait ends this stream's tiles; the exchange below then stops both warps of the pair
            bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&lready[b], (it >> 1) & 1, wc, 14, it));
            const Tile *tl = tiles_s + b * MAX_TILES;
            const int n = ok ? ntiles_s[b] : 0;
            // block-sparse: the row's random key blocks (its query block's), the first four kept in this thread's
            // shared slot for the item as 16-bit block indices (0xFFFF = none) when every index fits, the rest read
            // per tile; rows past the end have none
            if (BS) {
                const int nr_slot = P.bs_kblocks < 0xFFFF ? min(P.bs_r, 4) : 0;
                uint32_t rkp[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};
                if (t <= qlast) {
                    const int *rb = P.bs_rand + static_cast<int64_t>(t / P.bs_block) * P.bs_r;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int kb = i < nr_slot ? rb[i] : -1;
                        const uint32_t v16 = kb >= 0 ? static_cast<uint32_t>(kb) : 0xFFFFu;
                        rkp[i >> 1] = (rkp[i >> 1] & ~(0xFFFFu << (16 * (i & 1)))) | (v16 << (16 * (i & 1)));
                    }
                }
                rks_s[g * BQ + r] = make_uint2(rkp[0], rkp[1]);
            }
            float mrun = -INFINITY, lrun = 0.f;  // running max (log2 units) and sum of this stream
            for (int j = g; j < n; j += 2) {
                const Tile T = tl[j];
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(&sfull[g], v & 1, wc, 6, j));
                if (!ok) break;
                tc_fence_after();
                // valid columns of this row: [0, b1] (sinks) and [a2, hc] (window), hc = last causal column, as
                // 32-bit column masks, built only where some row of the warp needs one (interior tiles need none)
                const int hc = min(static_cast<int>(T.chi), t - T.pbase);
                const int b1 = min(hc, P.s - 1 - T.pbase);
                const int a2 = max(0, t - P.m + 1 - T.pbase);
                // a packed tile (block-sparse) holds two lone 64-key blocks, outside every window and the sinks
                const bool packed = BS && (T.flags & kTilePacked);
                const bool full = !packed && ((b1 >= BN - 1) || (hc >= BN - 1 && (a2 <= 0 || b1 >= a2 - 1)));
                const bool narrow = T.chi < 16;
                const bool masked = __any_sync(0xFFFFFFFFu, !full) || narrow;
                uint32_t mw[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
                if (masked) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mw[k] = (full || packed) ? (full ? 0xFFFFFFFFu : 0u)
                                                 : (range_bits(-32 * k, b1 - 32 * k) | range_bits(a2 - 32 * k, hc - 32 * k));
                }
                if (BS && (packed || !full) && t <= qlast) {
                    // block-sparse: also the global keys of the tile and the row's random key blocks, up to the
                    // row's own position.  Columns [c0, c1] of the tile hold positions base + c0 .. base + c1: the
                    // whole tile (hc = its last causal column), or for a packed tile each 64-column half (h) with
                    // its own base.
                    const TileMask gm = gmask_s[b * MAX_TILES + j];
                    const uint2 rk = rks_s[g * BQ + r];
                    auto add_cols = [&](int base, int c0, int c1, int kw0, int kw1) {
                        auto add_block = [&](int start) {
                            const int lo = max(start - base, c0), hi = min(start - base + P.bs_block - 1, c1);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                if (k >= kw0 && k < kw1) mw[k] |= range_bits(lo - 32 * k, hi - 32 * k);
                        };
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t kb = ((i < 2 ? rk.x : rk.y) >> (16 * (i & 1))) & 0xFFFFu;
                            if (kb != 0xFFFFu) add_block(static_cast<int>(kb) * P.bs_block);
                        }
                        const int nr_slot = P.bs_kblocks < 0xFFFF ? min(P.bs_r, 4) : 0;
                        if (P.bs_r > nr_slot) {
                            const int *rb = P.bs_rand + static_cast<int64_t>(t / P.bs_block) * P.bs_r;
                            for (int i = nr_slot; i < P.bs_r; ++i) {
                                const int kb = rb[i];
                                if (kb >= 0) add_block(kb * P.bs_block);
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (k >= kw0 && k < kw1) mw[k] |= gm.w[k] & range_bits(c0 - 32 * k, c1 - 32 * k);
                    };
                    if (packed) {
                        add_cols(T.pbase, 0, min(63, t - T.pbase), 0, 2);
                        add_cols(T.row1 - 64, 64, min(127, t - (T.row1 - 64)), 2, 4);
                    } else {
                        add_cols(T.pbase, 0, hc, 0, 4);
                    }
                }
                // the running max: O is rescaled only when it grows by more than 2^8 (also taken when mrun is
                // still -inf); returns -m for the exponent
                float alpha = 1.f;
                bool resc = false;
                auto new_max = [&](float mx) -> float {
                    const float mnew = fmaxf(mrun, mx);
                    if (mnew > mrun + kRescaleLog2) {
                        if (mrun != -INFINITY) {
                            alpha = ex2(mrun - mnew);
                            resc = true;
                        }
                        mrun = mnew;
                    }
                    return (mrun == -INFINITY) ? 0.f : -mrun;
                };
                // block-sparse mode: O rescaled before the first half of P_j is announced (PV(j) starts on it),
                // 16 columns at a time while half of the scores are still live
                auto rescale_o16 = [&]() {
                    if (__any_sync(0xFFFFFFFFu, resc)) {
                        __syncwarp();
#pragma unroll 1
                        for (int c = 0; c < 128; c += 16) {
                            float ov[16];
                            tmem_ld16(o_addr + c, ov);
                            uint32_t ou[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) ou[i] = __float_as_uint(ov[i] * alpha);
                            tmem_st16u_nowait(o_addr + c, ou);
                        }
                    }
                };
                // p = 2^(scale*log2(e)*s - m); bf16 pairs go to columns [0, 64) of the S buffer: the A operand
                // of PV(j)
                float rs4[4] = {0.f, 0.f, 0.f, 0.f};
                if (narrow) {
                    // a narrow tile (every key in columns 0..15, as the sink tile): its QK product had N = 16, and
                    // PV reads 16 keys, 8 packed columns
                    float sv[16];
                    __syncwarp();
                    tmem_ld16(s_addr, sv);
#pragma unroll
                    for (int c = 0; c < 16; ++c) sv[c] = (mw[0] & (1u << c)) ? sv[c] : -INFINITY;
                    float m4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) m4[i] = fmax3(sv[i], sv[4 + i], fmaxf(sv[8 + i], sv[12 + i]));
                    const float nmu = new_max(fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2);
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float a0, a1;
                        ffma2(a0, a1, sv[2 * i], sv[2 * i + 1], sl2, sl2, nmu, nmu);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        const int k = (i & 1) * 2;
                        fadd2(rs4[k], rs4[k + 1], rs4[k], rs4[k + 1], p0, p1);
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    __syncwarp();
                    tmem_st8u_nowait(s_addr, pk);
                    if (BS) {
                        rescale_o16();
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(&phalf[g]);
                    }
                } else {
                    float sv[128];
                    __syncwarp();
                    tmem_ld128(s_addr, sv);
                    if (masked) {
#pragma unroll
                        for (int c = 0; c < 128; ++c) sv[c] = (mw[c >> 5] & (1u << (c & 31))) ? sv[c] : -INFINITY;
                    }
                    float mx8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmax3(sv[i], sv[8 + i], sv[16 + i]);
#pragma unroll
                    for (int c = 24; c < 120; c += 16)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], sv[c + i], sv[c + 8 + i]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], sv[120 + i]);
                    const float nmu = new_max(
                        fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])) *
                        sl2);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float a0, a1;
                            ffma2(a0, a1, sv[64 * h + 2 * i], sv[64 * h + 2 * i + 1], sl2, sl2, nmu, nmu);
                            const float p0 = ex2(a0), p1 = ex2(a1);
                            const int k = (i & 1) * 2;
                            fadd2(rs4[k], rs4[k + 1], rs4[k], rs4[k + 1], p0, p1);
                            pk[i] = pack_bf16x2(p0, p1);
                        }
                        __syncwarp();
                        tmem_st32u_nowait(s_addr + 32 * h, pk);
                        if (BS && h == 0) {
                            rescale_o16();
                            tmem_wait_st();
                            tc_fence_before();
                            mbar_arrive(&phalf[g]);
                        }
                    }
                }
                lrun = lrun * alpha + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
                if (!BS && __any_sync(0xFFFFFFFFu, resc)) {
                    // O holds this stream's earlier PV products, all complete: S_j complete implies every MMA
                    // issued before QK(j) is, and PV(j) comes only after P_j
                    __syncwarp();
#pragma unroll 1
                    for (int c = 0; c < 128; c += 32) {
                        float ov[32];
                        tmem_ld32(o_addr + c, ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] *= alpha;
                        tmem_st32(o_addr + c, ov);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&pfull[g]);
                ++v;
            }
            if (lane == 0) mbar_arrive(&lfree[b]);  // this warp no longer reads the tile list
            // ---- epilogue: merge the two streams of each row, O / l -> bf16 rows (and lse)
            ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait(ofull, it & 1, wc, 8, it));
            float *slot = xch + (nx & 1) * 512;
            slot[g * 256 + r] = mrun;
            slot[g * 256 + 128 + r] = lrun;
            if (named_barrier_or(pair_bar, 64, !ok || ld_abort(abort_a) != 0)) break;  // both warps or none go on
            ++nx;
            const float mo = slot[(g ^ 1) * 256 + r], lo = slot[(g ^ 1) * 256 + 128 + r];
            tc_fence_after();
            const float mtot = fmaxf(mrun, mo);   // finite for every row that has a key
            const float wme = ex2(mrun - mtot);   // 0 for a stream that saw no key of the row
            const float wot = ex2(mo - mtot);
            const float lsum = lrun * wme + lo * wot;
            const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
            const float c0 = (g == 0 ? wme : wot) * inv, c1 = (g == 0 ? wot : wme) * inv;
            uint32_t ob[32];
            __syncwarp();
            const uint32_t oa = tmem + lane_base + col_o(0) + 64 * g;  // this thread's half of both O buffers
            // both buffers' columns in flight before one wait; O buffer 1 holds stream 1's products only when
            // n >= 2 (otherwise its contents are selected away, never multiplied)
            const bool two = n >= 2;
#pragma unroll
            for (int c = 0; c < 64; c += 32) {
                uint32_t x0[32], x1[32];
                tmem_ld32_nowait(oa + c, x0);
                tmem_ld32_nowait(oa + 128 + c, x1);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float a0 = __uint_as_float(x0[2 * i]) * c0, a1 = __uint_as_float(x0[2 * i + 1]) * c0;
                    const float b0 = two ? __uint_as_float(x1[2 * i]) * c1 : 0.f;
                    const float b1 = two ? __uint_as_float(x1[2 * i + 1]) * c1 : 0.f;
                    ob[c / 2 + i] = pack_bf16x2(a0 + b0, a1 + b1);
                }
            }
            tc_fence_before();
            mbar_arrive(oempty);
            // the row's half g into Q buffer b (free: every QK product of the item is done) in the 128-byte
            // swizzled layout of the tensor map; the tile-list warp stores the tile with TMA
            const uint32_t stage = smem_u32(sm + OFF_Q + b * TILE_BYTES + g * HALF_BYTES);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                st_shared_v4(stage + sw128_offset(r, 8 * k), ob[4 * k], ob[4 * k + 1], ob[4 * k + 2], ob[4 * k + 3]);
            fence_proxy_async_smem();
            mbar_arrive(&ostage[b]);
            if (P.lse && g == 0) {
                // row i < nvalid of the tile is row rbase + i * rstep of its (b, h)
                int rbase = row_start, rstep = 1, nvalid = qlast - q0 + 1;
                if (DIL) {  // virtual row q0 + i is position p0 + (row_start + i) r; whole groups only (g < dil_G)
                    rbase = class_p0(cls) + row_start * P.dil_r;
                    rstep = P.dil_r;
                    nvalid = min(nvalid, P.dil_G - class_g0(cls) - row_start);
                }
                if (r < nvalid)
                    P.lse[static_cast<int64_t>(bh) * P.seq_stride + rbase + r * rstep] =
                        (mtot + log2f(lsum)) * 0.69314718055994531f;
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
static bool encode_rows_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t nbh, uint64_t bh_stride_rows,
                            uint32_t box_rows = 128) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(tc::HD), rows, nbh};
    const cuuint64_t strides[2] = {tc::HD * 2, bh_stride_rows * tc::HD * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 4-D map over the rows of a residue class: (d, class, group, (b, h)) with position = group * r + class, for the
// groups [0, groups) (whole groups of r positions only, so that no load leaves the (b, h) block).  The box is one
// class, 128 consecutive groups, 64 columns: the same 128-byte-swizzled tile as a box of encode_rows_map.
static bool encode_class_map(CUtensorMap *m, const void *base, uint64_t r, uint64_t groups, uint64_t nbh,
                             uint64_t bh_stride_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(tc::HD), r, groups, nbh};
    const cuuint64_t strides[3] = {tc::HD * 2, r * tc::HD * 2, bh_stride_rows * tc::HD * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
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

// dil_r > 0: the dilated mode (pos0 = 0), over the rows [s, G r) with G = L / dil_r; a call with no such row
// launches nothing.
static int launch_impl(const PrefillArgs &a, const BlockSparseDev *bs, int dil_r = 0) {
    using namespace tc;
    if (a.d != HD) return fail(SWA_ERR_UNSUPPORTED, "tensor-core prefill needs d = %d", HD);
    if (a.rope) return fail(SWA_ERR_INVALID, "the RoPE prefill runs on the sub-tile kernel");
    if (!bs && max_tiles_bound(a.w, a.s) > MAX_TILES)
        return fail(SWA_ERR_UNSUPPORTED, "window w=%d needs more than %d key tiles per query tile", a.w, MAX_TILES);
    // dilated mode: every class runs over the virtual rows [s, s + nrows), nrows = the rows of the longest
    // class among the positions [s, G r); a shorter class's last virtual row reads zeros and is not written
    DilatedSplit dsp{};
    if (dil_r > 0) dsp = dilated_split(a.L, a.s, dil_r);
    const int64_t dil_G = dsp.G;
    const int64_t nrows = dil_r > 0 ? dsp.nrows : a.L;
    if (dil_r > 0 && a.pos0 != 0) return fail(SWA_ERR_INVALID, "dilated mode needs pos0 = 0");
    if (nrows == 0) return SWA_OK;
    if ((nrows + BQ - 1) / BQ * a.BH * (dil_r > 0 ? dil_r : 1) > 0x7FFFFFFF)
        return fail(SWA_ERR_UNSUPPORTED, "too many work items");
    if (!encode_tiled_fn()) return fail(SWA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    unsigned *status = device_status_word();
    if (!status) return SWA_ERR_CUDA;
    Params p;
    memset(&p, 0, sizeof(p));
    const uint64_t L = static_cast<uint64_t>(a.L), st = static_cast<uint64_t>(a.seq_stride);
    bool okm;
    if (dil_r > 0) {
        const uint64_t r = static_cast<uint64_t>(dil_r), G = static_cast<uint64_t>(dil_G);
        okm = encode_class_map(&p.tm_q, a.q, r, G, a.BH, st) && encode_class_map(&p.tm_k, a.k, r, G, a.BH, st) &&
              encode_class_map(&p.tm_v, a.v, r, G, a.BH, st) && encode_class_map(&p.tm_o, a.o, r, G, a.BH, st);
    } else {
        okm = encode_rows_map(&p.tm_q, a.q, L, a.BH, st) && encode_rows_map(&p.tm_k, a.k, L, a.BH, st) &&
              encode_rows_map(&p.tm_v, a.v, L, a.BH, st) && encode_rows_map(&p.tm_o, a.o, L, a.BH, st);
    }
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
    if (bs)  // the 64-row halves of packed tiles
        okm = okm && encode_rows_map(&p.tm_k64, a.k, L, a.BH, st, 64) && encode_rows_map(&p.tm_v64, a.v, L, a.BH, st, 64);
    if (!okm) return fail(SWA_ERR_INVALID, "cuTensorMapEncodeTiled rejected a tensor (alignment or size)");
    p.o = a.o;
    p.lse = a.lse;
    p.status = reinterpret_cast<DeviceStatus *>(status);
    p.seq_stride = a.seq_stride;
    p.L = static_cast<int>(nrows);
    p.pos0 = static_cast<int>(a.pos0);
    p.qoff = dil_r > 0 ? a.s : p.pos0;
    p.w = a.w;
    p.s = a.s;
    p.m = a.w - a.s;
    p.BH = a.BH;
    p.dil_r = dil_r > 0 ? dil_r : 1;
    p.dil_G = static_cast<int>(dil_G);
    p.n_qtiles = static_cast<int>((nrows + BQ - 1) / BQ);
    p.n_items = p.n_qtiles * a.BH * p.dil_r;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.timeout_us = kWaitTimeoutUs;
    if (bs) {
        p.bs_tiles = static_cast<const Tile *>(bs->tiles);
        p.bs_gmask = static_cast<const TileMask *>(bs->gmask);
        p.bs_count = bs->count;
        p.bs_rand = bs->rand;
        p.bs_block = bs->block;
        p.bs_r = bs->r;
        p.bs_kblocks = static_cast<int>((a.L + bs->block - 1) / bs->block);
    }
    auto *kern = bs ? swa_prefill_tc_kernel<1> : dil_r > 0 ? swa_prefill_tc_kernel<2> : swa_prefill_tc_kernel<0>;
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

int launch_prefill_bf16_tc_dilated(const PrefillArgs &a, int r) { return launch_impl(a, nullptr, r); }

// Host: the key-tile lists of the block-sparse prefill, one per 256-row query pair, in the kernel's layout.  A
// pair [q0, qlast] needs the sinks, its band [q0 - m + 1, qlast], every global position <= qlast, and the
// random key blocks (<= qlast) of every query block it overlaps: these ranges are merged into disjoint runs,
// so that each key position appears in exactly one tile, and cut into tiles of up to 128 keys.  Per tile the
// columns holding a global key are listed (the per-row masks of the kernel add them to the band and sinks),
// and the tile is marked for the query tiles that have some row it can serve.  Two 64-key tiles outside the sinks
// and the band that serve the same query tiles are packed into one (one QK and one PV product for both).  Returns
// SWA_OK or an error.
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
    std::vector<Tile> tv;
    std::vector<TileMask> mv;
    std::vector<int> mate;  // per tile of tv: the tile it is packed with, or -1
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
        tv.clear();
        mv.clear();
        size_t k = 0;
        while (k < iv.size()) {
            int a = iv[k].first, b = iv[k].second;
            for (++k; k < iv.size() && iv[k].first <= b + 1; ++k) b = std::max(b, iv[k].second);
            for (int p = a; p <= b; p += BN) {
                Tile T{};
                T.row0 = p;
                T.pbase = p;
                T.chi = static_cast<short>(std::min(b - p, BN - 1));
                TileMask G{};
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
                if (!f) continue;  // a tile no query tile needs is dropped
                tv.push_back(T);
                mv.push_back(G);
            }
        }
        // Packing: a tile of exactly 64 keys that holds no sink and no band position of the pair (only random
        // blocks and global tokens) shares a 128-key tile with another such tile: first with one used by the same
        // query tiles, then a tile used by both query tiles with one used by a single query tile (each pairing
        // saves a walk of some query tile).  Columns 0..63 hold the earlier, 64..127 the later, each loaded as
        // a 64-row box.
        auto lone = [&](const Tile &T) { return T.chi == 63 && T.pbase >= s && T.pbase + 63 < blo; };
        mate.assign(tv.size(), -1);
        for (int pass = 0; pass < 2; ++pass)
            for (size_t i = 0; i < tv.size(); ++i) {
                if (mate[i] >= 0 || !lone(tv[i])) continue;
                for (size_t j = i + 1; j < tv.size(); ++j) {
                    const int fi = tv[i].flags, fj = tv[j].flags;
                    if (mate[j] >= 0 || !lone(tv[j])) continue;
                    if (pass == 0 ? fi != fj : (fi | fj) != (fi > fj ? fi : fj)) continue;
                    mate[i] = static_cast<int>(j);
                    mate[j] = static_cast<int>(i);
                    break;
                }
            }
        int n = 0;
        Tile *tl = tiles + static_cast<int64_t>(qp) * MAX_TILES;
        TileMask *gm = gmask + static_cast<int64_t>(qp) * MAX_TILES;
        for (size_t i = 0; i < tv.size(); ++i) {
            if (mate[i] >= 0 && static_cast<size_t>(mate[i]) < i) continue;  // the upper half of a packed tile
            if (n >= MAX_TILES)
                return fail(SWA_ERR_UNSUPPORTED, "query rows %d..%d need more than %d key tiles", q0, qlast, MAX_TILES);
            tl[n] = tv[i];
            gm[n] = mv[i];
            if (mate[i] >= 0) {
                const size_t j = static_cast<size_t>(mate[i]);
                tl[n].chi = BN - 1;
                tl[n].row1 = tv[j].pbase;
                tl[n].flags = static_cast<short>(tv[i].flags | tv[j].flags | kTilePacked);
                gm[n].w[2] = mv[j].w[0];
                gm[n].w[3] = mv[j].w[1];
            }
            ++n;
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

int prefill_tile_plan_dilated(int64_t L, int w, int s, int r, int cls, int row_start, int *out, int max_tiles) {
    const DilatedSplit sp = dilated_split(L, s, r);
    if (row_start < 0 || row_start % tc::BQ != 0 || row_start >= sp.nrows)
        return fail(SWA_ERR_INVALID, "row_start=%d is not the first row of a query tile of the %lld rows of a class",
                    row_start, (long long)sp.nrows);
    tc::Tile tl[tc::MAX_TILES];
    const int n = tc::build_tiles_dilated(tl, row_start, cls, s, w - s, w, r, static_cast<int>(sp.nrows));
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
