// prefill_tc_sub.cu -- bf16 prefill of causal sliding-window attention with sinks on the sm_103a tensor
// cores (TMA + tcgen05.mma + TMEM), walking the keys in sub-tiles of 64: the kernel of the RoPE prefills
// (rotated q and k as bf16 hi/lo pairs, three products per score) and of head dimension 64.
//
// The computation (hyper.ai summary of arXiv 2608.28444, section "带 Sink 的滑动窗口注意力"; causal
// softmax attention of "模糊窗口注意力" section 2.1, eq (1)): query t attends
//     K(t) = { i <= t : i < s  or  i >= t - m + 1 },  m = w - s,
// with softmax over scale * q.k.  A fixed sparsity pattern known from positions alone ("滑窗与固定稀疏":
// O(n^2) -> O(n k), banded patterns are hardware friendly), so each CTA walks only the keys that
// intersect the band or the sink block of its query rows; no skipped key block is ever loaded.
//
// Work item = two query tiles of 128 rows (256 consecutive rows) of one (b, h).  The kernel is
// persistent: one CTA per SM walks the items blockIdx.x, blockIdx.x + gridDim.x, ..., ordered
// longest-first (the last query pairs of every head, whose windows are full, come first), so the short
// items fall in the last rounds and the CTAs finish together.
//
// The keys of an item are listed as tiles of up to 128 positions (build_tiles); each tile is walked as
// two sub-tiles of 64 keys, and the sub-tile is the unit of everything below: a TMA load of K and of V,
// one S = Q K^T product per query tile (N = 64), one softmax pass, one O += P V product (K = 64).  A
// sub-tile no row of the item needs is neither loaded nor computed, and a query tile skips the
// sub-tiles none of its own rows needs.  384 threads (12 warps) in these roles:
//   warps 0-3 / 4-7  softmax + epilogue of query tile 0 / 1: thread r owns row r of its tile (= TMEM lane r);
//   warp 8     loads, lane 0 K and lane 1 V: one stream of sub-tiles over all items of the CTA into a K ring
//              of NK slots and a V ring of NV slots;
//   warps 9 / 11  MMA issuers of query tile 0 / 1 (one thread each: a thread can issue a tcgen05.mma only
//              about every 100 cycles, so one issuer alone keeps the tensor pipe at most ~2/3 busy);
//   warp 10    per item: builds the key-tile list into one of two buffers, one item ahead, loads Q_0 and
//              Q_1 as soon as the previous item's last QK product is done, and prefetches the next
//              item's Q into L2.
// TMEM (512 columns): S_0 = [0, 128), S_1 = [128, 256), O_0 = [256, 256 + d), O_1 = [384, 384 + d).  Each
// S_x is two halves of 64 columns, used by query tile x's sub-tiles in turn, so QK_x of the next
// sub-tile runs into one half while the softmax warpgroup reads the other: the softmax never waits for
// a hand-off and a QK product.  The softmax writes P (bf16 pairs, 32 columns) over the first columns
// of the half it has read, and PV_x reads P straight from TMEM.  The issuer of query tile x keeps two QK
// products in flight: after PV_x of a sub-tile it issues QK_x of the sub-tile two ahead into the half
// that PV has just released (tcgen05 MMAs of one thread run in issue order, so the QK cannot overwrite
// P before the PV has read it).  The online softmax keeps a running max in log2 units and only rescales
// O (TMEM load, multiply, store) when the max grows by more than 8 (a factor 256), so p <= 256 always
// fits bf16/fp32 and the rescale is rare; before a rescale the warpgroup waits for its previous PV
// product (the only one that can still be in flight).
//
// Precision mode (HILO, used by the RoPE prefill): q and k arrive as a bf16 pair (hi, lo) with
// hi + lo the rotated fp32 value, and every window score S = hi_q hi_k + hi_q lo_k + lo_q hi_k (three
// products accumulated in fp32), so the scores carry the error of fp32 operands, not of bf16 ones.  The
// sink scores, whose query rotation differs, come ready-made from the rotation pass (fp32): the sink
// sub-tiles take no K load and no QK product, only their PV product, and Q is loaded once per item.
//
// Key tiles.  For the query rows [q0, q1] of a CTA the key positions needed are the sinks [0, min(s, blo)) and
// the band [blo, q1] with blo = max(0, q0 - m + 1).  Positions >= pos0 are rows of this call's k/v;
// positions < pos0 (chunked prefill) live in the rolling cache: slot p for p < s, slot
// s + ((p - s) mod m) for the rest ("滑窗与固定稀疏", eq attn-fixed-rolling and eq attn-fixed-streaming).
// A contiguous position range maps to at most two contiguous slot runs (the ring wraps once), so every
// range becomes a list of 128-row tiles, each with: source, first row, position of its column 0, and
// the last valid column.  Columns past the range end, positions past t and positions outside the
// window are masked per row; interior sub-tiles need no mask at all.  Every key position appears in
// exactly one tile.  TMA zero-fills rows outside the source tensor.
//
// Every mbarrier wait is bounded (1 s).  A wait that runs out records the timeout in the device error
// word and sets a CTA-wide abort flag; all roles leave their loops, the loaders wait (bounded) for their
// copies in flight, each MMA issuer waits for its MMAs, and TMEM is freed before the CTA exits.
#include <math.h>

#include "../../include/swa_sink.h"
#include "swa_device.cuh"
#include "swa_internal.h"

namespace swa {
namespace tcs {

constexpr int BH_ROWS = 128;    // query rows per query tile (= TMEM lanes)
constexpr int BM = 2 * BH_ROWS; // query rows per CTA: two query tiles
constexpr int BN = 128;         // keys per tile of the key-tile list
constexpr int SUB = 64;         // keys per sub-tile: the unit of loads, MMAs and softmax passes
constexpr int MAX_TILES = 64;
constexpr int kThreads = 384;   // warps 0-3 / 4-7: softmax of query tile 0 / 1; 8: loads (lane 0 K, lane 1 V);
                                // 9 / 11: MMA of query tile 0 / 1; 10: lists.  12 warps: 3 per SMSP, 168 registers
constexpr int kWarpLoad = 8, kWarpMma0 = 9, kWarpList = 10, kWarpMma1 = 11;
constexpr int kListUsers = 12;  // threads that read a tile list: 8 softmax warps, 2 MMA issuers, K and V loaders
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S_0, S_1 (two halves of 64 each; P over the first 32 columns of a half), O_0, O_1
__host__ __device__ constexpr uint32_t col_s(int x) { return static_cast<uint32_t>(x) * 128u; }
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u + static_cast<uint32_t>(x) * 128u; }
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the running max grows by more than 2^8
constexpr uint32_t QBOX = 128 * 128;  // one 64-column box of a 128-row Q tile (128 rows x 128 bytes)
constexpr uint32_t KBOX = 64 * 128;   // one 64-column box of a 64-row K or V sub-tile

// Shared-memory layout per head dimension HD (64 or 128) and precision mode.
template <int HD, bool HILO>
struct Layout {
    static constexpr int NB = HD / 64;                         // 64-column boxes per row
    static constexpr uint32_t QPART = NB * QBOX;               // one Q operand (hi or lo) of a query tile
    static constexpr uint32_t QTILE = (HILO ? 2 : 1) * QPART;  // Q of a query tile
    static constexpr uint32_t KPART = NB * KBOX;               // one K operand of a sub-tile
    static constexpr uint32_t KSLOT = (HILO ? 2 : 1) * KPART;  // K ring slot (hi, then lo)
    static constexpr uint32_t VSLOT = KPART;                   // V ring slot
    static constexpr int NK = HILO ? 2 : (HD == 64 ? 8 : 4);   // K sub-tile slots
    static constexpr int NV = HILO ? 2 : (HD == 64 ? 8 : 4);   // V sub-tile slots
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + 2 * QTILE;
    static constexpr uint32_t OFF_V = OFF_K + NK * KSLOT;
    static constexpr uint32_t OFF_BAR = OFF_V + NV * VSLOT;
    static constexpr int NBARS = 22 + 2 * (NK + NV);
    static constexpr uint32_t OFF_MISC = OFF_BAR + ((NBARS * 8 + 63) / 64) * 64;
    static constexpr uint32_t OFF_TILES = OFF_MISC + 128;  // misc: TMEM slot, abort flag, list sizes, slot owners
    static constexpr uint32_t SMEM_USED = OFF_TILES + 2 * MAX_TILES * 12;  // two tile lists (current / next item)
    static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;               // slack to align the base to 1024 bytes
    static_assert(SMEM_BYTES <= 232448, "shared memory budget of one CTA");
    static_assert(NK <= 8 && NV <= 8, "slot owner words");
    static_assert(QBOX % 1024 == 0 && KBOX % 1024 == 0 && OFF_K % 1024 == 0 && OFF_V % 1024 == 0,
                  "128-byte-swizzled operands start on 1024-byte boundaries");
};

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, SUB, false, false);  // Q, K both K-major; N = 64 keys
template <int HD>
__host__ __device__ constexpr uint32_t idesc_pv() { return idesc_bf16_f32(128, HD, false, true); }  // V MN-major

struct Tile {
    int row0;     // first source row (TMA row coordinate)
    int pbase;    // absolute position of column 0
    short chi;    // last valid column (columns past it belong to another tile or to nothing)
    short flags;  // bit 0: source (0 = this call's k/v rows, 1 = rolling cache); bit 1 + x: needed by query
                  // tile x; bit 3 + 2 h + x: sub-tile h (columns 64 h .. 64 h + 63) needed by query tile x
};
static_assert(sizeof(Tile) == 12, "tile record");

struct Params {
    CUtensorMap tm_q, tm_k, tm_v, tm_kc, tm_vc;
    CUtensorMap tm_ql, tm_kl, tm_kcl;  // HILO: the lo parts of q, k and the cached keys
    // RoPE mode: the sink tile's scores (the query rotated at min(t, w - 1) against the rotated sinks), fp32,
    // row (b, h) * seq_stride + local row, sstride floats per row
    const float *ssink;
    int sstride;
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

// Which query tiles of the pair [q0, qlast] need each key tile and each of its two sub-tiles: rows
// [ra, rb] need positions [pb, pe] iff some position p <= rb in it is a sink (p < s) or lies in the
// window of some row (p >= ra - m + 1).
__host__ __device__ void mark_tiles(Tile *tl, int n, int q0, int qlast, int s, int m) {
    for (int i = 0; i < n && i < MAX_TILES; ++i) {
        const int pb = tl[i].pbase, pe = tl[i].pbase + tl[i].chi;
        int f = tl[i].flags & 1;
        for (int x = 0; x < 2; ++x) {
            const int ra = q0 + x * BH_ROWS;
            const int rb = (q0 + x * BH_ROWS + BH_ROWS - 1 < qlast) ? q0 + x * BH_ROWS + BH_ROWS - 1 : qlast;
            if (ra > rb) continue;
            if (pb <= rb && (pb < s || pe >= ra - m + 1)) f |= 2 << x;
            for (int h = 0; h < 2; ++h) {
                if (SUB * h > tl[i].chi) continue;  // no columns in this half
                const int hb = pb + SUB * h;
                const int he = pb + (tl[i].chi < SUB * h + SUB - 1 ? tl[i].chi : SUB * h + SUB - 1);
                if (hb <= rb && (hb < s || he >= ra - m + 1)) f |= 1 << (3 + 2 * h + x);
            }
        }
        tl[i].flags = static_cast<short>(f);
    }
}

__host__ __device__ __forceinline__ int half_users(const Tile &T, int h) { return (T.flags >> (3 + 2 * h)) & 3; }
__host__ __device__ __forceinline__ void walk_step(int &j, int &h) {
    if (++h == 2) {
        h = 0;
        ++j;
    }
}
// Move (j, h) forward, starting at the current position, to the first sub-tile some query tile in `mask`
// needs.  Returns false at the end of the list.
__host__ __device__ __forceinline__ bool walk_seek(const Tile *tl, int n, int &j, int &h, int mask) {
    while (j < n) {
        if (half_users(tl[j], h) & mask) return true;
        walk_step(j, h);
    }
    return false;
}

// Move (j, h) forward, starting at the current position, to the next walked sub-tile (one some query tile
// needs) that the query tiles in `bit` need, counting in g the walked sub-tiles passed on the way.
__device__ __forceinline__ bool seek_mine(const Tile *tl, int n, int &j, int &h, int &g, int bit) {
    while (walk_seek(tl, n, j, h, 3)) {
        if (half_users(tl[j], h) & bit) return true;
        walk_step(j, h);
        ++g;
    }
    return false;
}

// Wait (bounded) until a ring slot's owner word holds `want` (the stream index of the sub-tile loaded into it).
__device__ __noinline__ bool slot_wait_slow(const volatile int *seq, int want, const WaitCtl c, unsigned where) {
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = static_cast<uint64_t>(c.timeout_us) * 1000ull;
    for (uint32_t it = 1;; ++it) {
        if (*seq == want) return true;
        if ((it & 31u) == 0) {
            if (ld_abort(c.abort_smem)) return false;
            if (globaltimer_ns() - t0 > limit) {
                wait_gave_up(c, where, static_cast<unsigned>(want));
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool slot_wait(const volatile int *seq, int want, const WaitCtl c, unsigned where) {
    return *seq == want || slot_wait_slow(seq, want, c, where);
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


// S (128 x 64, fp32 in TMEM) (+)= Q (128 x HD) K_sub^T: Q and the 64-row K sub-tile K-major, 128-byte
// swizzled, one 64-column box after the other.
template <int HD>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        umma_ss(d_tmem, sdesc_sw128(q_addr + (kk >> 2) * QBOX + (kk & 3) * 32, 16, 1024),
                sdesc_sw128(k_addr + (kk >> 2) * KBOX + (kk & 3) * 32, 16, 1024), IDESC_QK,
                (accumulate || kk > 0) ? 1u : 0u);
    }
}

// O (128 x HD) (+)= P (128 x 64, bf16 pairs in TMEM) V_sub (64 x HD, MN-major: 16 key rows of 128 bytes
// per instruction; the two 64-column boxes KBOX apart).
template <int HD>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < SUB / 16; ++kk) {
        umma_ts(d_tmem, p_tmem + kk * 8, sdesc_sw128(v_addr + kk * 16 * 128, KBOX, 1024), idesc_pv<HD>(),
                (accumulate || kk > 0) ? 1u : 0u);
    }
}

// ROPE: the RoPE mode (the sink tile scored with its own query rotation) with hi/lo operands; compiled
// apart, so that the plain kernel carries none of its checks.
template <int HD, bool ROPE>
__global__ void __launch_bounds__(kThreads, 1) swa_prefill_tc_kernel(const __grid_constant__ Params P) {
    using LY = Layout<HD, ROPE>;
    constexpr int NK = LY::NK, NV = LY::NV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + LY::OFF_BAR);
    uint64_t *qfull = bars;           // Q_0, Q_1 of the current item landed
    uint64_t *qempty = qfull + 1;     // the QK products reading the Q buffer are done: Q may be reloaded (2 issuers)
    uint64_t *kfull = qempty + 1;     // [NK]
    uint64_t *kempty = kfull + NK;    // [NK] 2 arrivals: the softmax warpgroups that used the slot (x2 if one did)
    uint64_t *vfull = kempty + NK;    // [NV]
    uint64_t *vempty = vfull + NV;    // [NV] 2 arrivals: the MMA issuers that used the slot (x2 if one did)
    uint64_t *sfull = vempty + NV;    // [2][2]: half h of S_x holds Q_x K^T of a sub-tile (x * 2 + h)
    uint64_t *pfull = sfull + 4;      // [2][2]: P_x written over half h (128 arrivals)
    uint64_t *ofull = pfull + 4;      // [2]: the last PV_x product of an item is done
    uint64_t *oempty = ofull + 2;     // [2]: O_x has been read by the epilogue (128 arrivals)
    uint64_t *pvdone = oempty + 2;    // [2]: the second-to-last PV_x product of an item is done
    uint64_t *lready = pvdone + 2;    // [2]: tile list buffer b written (1 arrival)
    uint64_t *lfree = lready + 2;     // [2]: tile list buffer b no longer read (kListUsers warps)
    uint64_t *drain = lfree + 2;      // [2]: each MMA issuer's last products are done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + LY::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + LY::OFF_MISC + 4);
    int *ntiles_s = reinterpret_cast<int *>(sm + LY::OFF_MISC + 8);  // [2]
    Tile *tiles_s = reinterpret_cast<Tile *>(sm + LY::OFF_TILES);     // [2][MAX_TILES]
    // stream index of the sub-tile last loaded into each K / V slot (written by the loaders before the load)
    volatile int *kseq = reinterpret_cast<volatile int *>(sm + LY::OFF_MISC + 16);  // [NK] (NK <= 8)
    volatile int *vseq = kseq + 8;                                                  // [NV] (NV <= 8)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 16; ++i) kseq[i] = -1;
        mbar_init(qfull, 1);
        mbar_init(qempty, 2);
        for (int i = 0; i < NK; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], 2);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], 2);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&pfull[i], BH_ROWS);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&ofull[x], 1);
            mbar_init(&oempty[x], BH_ROWS);
            mbar_init(&pvdone[x], 1);
            mbar_init(&lready[x], 1);
            mbar_init(&lfree[x], kListUsers);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
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

    if (warp == kWarpLoad) {
        // ------------------------------------------------------------------ loaders (lane 0: K, lane 1: V)
        // One stream of walked sub-tiles over all items of the CTA; K and V each have their own ring and
        // their own thread, so neither waits for the other.  A slot frees when the MMAs reading it are done.
        if (lane < 2) {
            const bool isk = lane == 0;
            const int NS = isk ? NK : NV;
            const uint32_t slot_bytes = isk ? LY::KSLOT : LY::VSLOT;
            uint8_t *ring = sm + (isk ? LY::OFF_K : LY::OFF_V);
            uint64_t *full = isk ? kfull : vfull;
            uint64_t *empty = isk ? kempty : vempty;
            tma_prefetch_desc(isk ? &P.tm_k : &P.tm_v);
            int g = 0;  // sub-tiles issued so far
            bool fine = true;
            for (int it = 0; fine; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * G;
                if (item >= P.n_items) break;
                const int b = it & 1;
                if (!mbar_wait(&lready[b], (it >> 1) & 1, wc, 15, it)) {
                    fine = false;
                    break;
                }
                const int n = ntiles_s[b];
                const Tile *tl = tiles_s + b * MAX_TILES;
                const int bh = item % P.BH;
                int j = 0, h = 0;
                while (walk_seek(tl, n, j, h, 3)) {
                    const int st = g % NS;
                    if (!mbar_wait(&empty[st], ((g / NS) & 1) ^ 1, wc, isk ? 1 : 9, g)) {
                        fine = false;
                        break;
                    }
                    const Tile T = tl[j];
                    const int row = T.row0 + SUB * h;
                    uint8_t *dst = ring + st * slot_bytes;
                    (isk ? kseq : vseq)[st] = g;
                    if (ROPE && isk && T.pbase < P.s) {  // the sink scores are ready-made: no K rows
                        mbar_arrive(&full[st]);
                        ++g;
                        walk_step(j, h);
                        continue;
                    }
                    mbar_arrive_expect_tx(&full[st], slot_bytes);
                    if (isk) {
                        const CUtensorMap *mk = (T.flags & 1) ? &P.tm_kc : &P.tm_k;
#pragma unroll
                        for (int c = 0; c < LY::NB; ++c) tma_load_3d(dst + c * KBOX, mk, &full[st], 64 * c, row, bh);
                        if (ROPE) {
                            const CUtensorMap *ml = (T.flags & 1) ? &P.tm_kcl : &P.tm_kl;
#pragma unroll
                            for (int c = 0; c < LY::NB; ++c)
                                tma_load_3d(dst + LY::KPART + c * KBOX, ml, &full[st], 64 * c, row, bh);
                        }
                    } else {
                        const CUtensorMap *mv = (T.flags & 1) ? &P.tm_vc : &P.tm_v;
#pragma unroll
                        for (int c = 0; c < LY::NB; ++c) tma_load_3d(dst + c * KBOX, mv, &full[st], 64 * c, row, bh);
                    }
                    ++g;
                    walk_step(j, h);
                }
                if (!fine) break;
                mbar_arrive(&lfree[b]);  // this loader no longer reads the item's list
            }
            if (*abort_flag) {  // make sure no copy is still landing in shared memory
                for (int q = (g > NS ? g - NS : 0); q < g; ++q) mbar_wait_drain(&full[q % NS], (q / NS) & 1);
            }
        }
    } else if (warp == kWarpList) {
        // ------------------------------------------------------------------ tile lists
        if (lane == 0) {
            // Per item: the key-tile list goes to buffer it & 1 as soon as the buffer's previous item
            // (it - 2) has been released by every reader; then Q_0, Q_1 of the item, as soon as the previous
            // item's last QK product is done, and the next item's Q into L2, so that its load does not wait
            // for DRAM.
            using LYQ = Layout<HD, ROPE>;
            int nq = 0;
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
                const int n = build_tiles(tl, q0, qlast, P.pos0, P.s, P.m, P.w, ROPE);
                if (n < 1 || n > MAX_TILES) {
                    atomicOr(&P.status->word, kDevBadArg);
                    *abort_flag = 1;
                    break;
                }
                mark_tiles(tl, n, q0, qlast, P.s, P.m);
                ntiles_s[b] = n;
                mbar_arrive(&lready[b]);  // release: the list is visible to whoever sees the phase complete
                // Q_0, Q_1 of the item (in HILO mode hi and lo parts), once the previous item's QK products are
                // done; then the next item's Q into L2, so that its load does not wait for DRAM
                bool ok = true;
                if (nq >= 1 && !mbar_wait(qempty, (nq - 1) & 1, wc, 13, it)) {
                    ok = false;
                } else {
                    uint8_t *qs = sm + LYQ::OFF_Q;
                    mbar_arrive_expect_tx(qfull, 2 * LYQ::QTILE);
                    for (int x = 0; x < 2; ++x) {
#pragma unroll
                        for (int c = 0; c < LYQ::NB; ++c) {
                            tma_load_3d(qs + x * LYQ::QTILE + c * QBOX, &P.tm_q, qfull, 64 * c, row_start + x * BH_ROWS, bh);
                            if (ROPE)
                                tma_load_3d(qs + x * LYQ::QTILE + LYQ::QPART + c * QBOX, &P.tm_ql, qfull, 64 * c,
                                            row_start + x * BH_ROWS, bh);
                        }
                    }
                    ++nq;
                    const int nitem = item + G;
                    if (nitem < P.n_items) {
                        const int nrow = (P.n_qpairs - 1 - nitem / P.BH) * BM;
                        for (int x = 0; x < 2; ++x)
                            for (int c = 0; c < LYQ::NB; ++c) tma_prefetch_3d(&P.tm_q, 64 * c, nrow + x * BH_ROWS, nitem % P.BH);
                    }
                }
                if (!ok) break;
            }
            if (*abort_flag && nq > 0) mbar_wait_drain(qfull, (nq - 1) & 1);  // no copy may still be landing
        }
    } else if (warp == kWarpMma0 || warp == kWarpMma1) {
        // ------------------------------------------------------------------ MMA issuers (one per query tile)
        // A thread can issue a tcgen05 instruction (an MMA or a commit) only about every 100 cycles, so one
        // issuer per query tile keeps the tensor pipe fed, and the issuers commit as little as they can: per
        // sub-tile one commit for S ready and one for the V slot; the K slots are released by the softmax warps,
        // which see the QK products complete.  Issuer x walks only the sub-tiles x needs, twice over: a QK walk
        // and a PV walk.  Per sub-tile of the PV walk: PV_x, then QK_x of x's sub-tile two ahead into the half of
        // S_x that PV_x has just released (tcgen05 MMAs of one thread run in issue order).  A parity wait tells
        // only adjacent phases of a barrier apart, and an issuer that skips some uses of a ring slot could take the
        // slot's earlier, still pending phase for the one it wants; so before the parity wait it waits until the
        // loader has put its sub-tile in the slot (kseq / vseq), after which the phase it wants is the slot's
        // current or last one (the slot cannot move on before this issuer's own release).  K and V slots take two
        // arrivals per use, one per query tile that used them (both from the one that did, if only one did; the
        // second as a plain arrival, which lands no earlier than the load and no later than the products).  The Q
        // buffer takes one committed arrival per issuer after its last QK product that reads it.
        if (lane == 0) {
            using LYM = Layout<HD, ROPE>;
            const int x = warp == kWarpMma0 ? 0 : 1;
            const int mybit = 1 << x;
            const uint32_t qa = smem_u32(sm + LYM::OFF_Q) + x * LYM::QTILE;
            const uint32_t k_addr0 = smem_u32(sm + LYM::OFF_K), v_addr0 = smem_u32(sm + LYM::OFF_V);
            const uint32_t s_tm = tmem + col_s(x), o_tm = tmem + col_o(x);
            bool issued_any = false, fine = true;
            int gbase = 0;  // stream index of the item's first walked sub-tile
            int cnt = 0;    // PV_x products issued, kernel-wide (S half / pfull parity clock)
            int qi = 0;     // QK_x products issued, kernel-wide
            int ce = 0;     // items with PV_x products (oempty parity)
            int nqf = 0;    // Q loads consumed (qfull parity)
            for (int it = 0; fine; ++it) {
                const int item = static_cast<int>(blockIdx.x) + it * G;
                if (item >= P.n_items) break;
                const int b = it & 1;
                if (!mbar_wait(&lready[b], (it >> 1) & 1, wc, 14, it)) break;  // the item's tile list
                if (!mbar_wait(qfull, nqf & 1, wc, 2, it)) break;                // Q of this item
                ++nqf;
                const Tile *tl = tiles_s + b * MAX_TILES;
                const int n = ntiles_s[b];
                int left_pv = 0, nwalk = 0;  // PV_x products of this item still to issue; walked sub-tiles
                for (int j = 0; j < n; ++j)
                    for (int h = 0; h < 2; ++h) {
                        const int u = half_users(tl[j], h);
                        left_pv += (u & mybit) ? 1 : 0;
                        nwalk += u ? 1 : 0;
                    }
                int left_qk = left_pv;  // QK_x products of this item still to issue
                int kj = 0, kh = 0, kg = gbase;  // QK walk position (stream index kg)
                // QK_x of the next sub-tile x needs: 1 if issued, 0 if there is none in this item, -1 on a failed
                // wait.  In RoPE mode the sink sub-tiles take no product (their scores are ready-made), only the
                // commit that tells the softmax its turn has come and the K slot's (empty) load has landed.
                auto qk_step = [&]() -> int {
                    if (!seek_mine(tl, n, kj, kh, kg, mybit)) return 0;
                    const int st = kg % NK;
                    if (!slot_wait(&kseq[st], kg, wc, 16) || !mbar_wait(&kfull[st], (kg / NK) & 1, wc, 3, kg)) return -1;
                    tc_fence_after();
                    const uint32_t ka = k_addr0 + st * LYM::KSLOT;
                    const uint32_t d = s_tm + SUB * (qi & 1);
                    if (!(ROPE && tl[kj].pbase < P.s)) {
                        issue_qk<HD>(d, qa, ka, false);
                        if (ROPE) {  // + hi_q lo_k + lo_q hi_k
                            issue_qk<HD>(d, qa, ka + LYM::KPART, true);
                            issue_qk<HD>(d, qa + LYM::QPART, ka, true);
                        }
                    }
                    umma_commit(&sfull[x * 2 + (qi & 1)]);  // the softmax releases the K slot once this is done
                    ++qi;
                    issued_any = true;
                    if (--left_qk == 0) umma_commit(qempty);  // the item's last QK_x product
                    walk_step(kj, kh);
                    ++kg;
                    return 1;
                };
                // keep up to two QK_x products in flight
                auto top_up = [&]() -> bool {
                    while (qi - cnt < 2 && left_qk > 0) {
                        const int r = qk_step();
                        if (r < 0) return false;
                        if (r == 0) break;
                    }
                    return true;
                };
                if (left_qk == 0) umma_commit(qempty);  // no (more) QK_x product in this item
                if (!top_up()) break;
                int pj = 0, ph = 0, pg = gbase;  // PV walk position
                bool first_pv = true;
                while (fine && seek_mine(tl, n, pj, ph, pg, mybit)) {
                    const int sv = pg % NV;
                    const int hs = cnt & 1;
                    if (!mbar_wait(&pfull[x * 2 + hs], (cnt >> 1) & 1, wc, 4, pg)) { fine = false; break; }
                    if (first_pv) {  // O_x must have been read by the previous item's epilogue
                        if (!mbar_wait(&oempty[x], (ce & 1) ^ 1, wc, 11, pg)) { fine = false; break; }
                        ++ce;
                    }
                    if (!slot_wait(&vseq[sv], pg, wc, 17) || !mbar_wait(&vfull[sv], (pg / NV) & 1, wc, 5, pg)) {
                        fine = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv<HD>(o_tm, s_tm + SUB * hs, v_addr0 + sv * LYM::VSLOT, !first_pv);
                    umma_commit(&vempty[sv]);
                    if (half_users(tl[pj], ph) == mybit) mbar_arrive(&vempty[sv]);  // the other query tile's share
                    first_pv = false;
                    ++cnt;
                    --left_pv;
                    if (left_pv == 1) umma_commit(&pvdone[x]);  // the item's second-to-last PV_x (rescale waits)
                    if (left_pv == 0) umma_commit(&ofull[x]);
                    if (!top_up()) { fine = false; break; }
                    walk_step(pj, ph);
                    ++pg;
                }
                if (!fine) break;
                gbase += nwalk;
                mbar_arrive(&lfree[b]);
            }
            if (issued_any) {  // no MMA may still be running when TMEM is freed
                umma_commit(&drain[x]);
                mbar_wait_drain(&drain[x], 0);
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------------ softmax + epilogue
        const int x = warp >> 2;                    // query tile of this warpgroup
        const int r = threadIdx.x & (BH_ROWS - 1);  // its row == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + col_s(x);
        const uint32_t o_addr = tmem + lane_base + col_o(x);
        const float sl2 = P.scale_log2;
        const int mybit = 1 << x;
        int cs = 0;  // sub-tiles processed by this warpgroup, kernel-wide (S half / sfull / pfull clock)
        int ne = 0;  // epilogues done (ofull parity)
        int kp = 0;  // items in which this query tile had two or more sub-tiles (pvdone parity)
        int gbase = 0;  // stream index of the item's first walked sub-tile (K/V ring position)
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
            int j = 0, h = 0, g = gbase;
            while (seek_mine(tl, n, j, h, g, mybit)) {
                const Tile T = tl[j];
                const int hs = cs & 1;
                fine = __all_sync(0xFFFFFFFFu, mbar_wait(&sfull[x * 2 + hs], (cs >> 1) & 1, wc, 6, j));
                if (!fine) break;
                tc_fence_after();
                // QK_x of this sub-tile is done: its K slot is free for this query tile (a slot only this query
                // tile used takes both arrivals)
                if (r == 0) mbar_arrive_n(&kempty[g % NK], (half_users(T, h) == mybit) ? 2u : 1u);
                // valid columns of this row in the sub-tile: [0, b1] (sinks) and [a2, hc] (window), hc = last
                // causal column, as two 32-bit column masks; interior sub-tiles need none
                const int pb = T.pbase + SUB * h;
                const int chi = min(static_cast<int>(T.chi) - SUB * h, SUB - 1);
                const int hc = min(chi, t - pb);
                const int b1 = min(hc, P.s - 1 - pb);
                const int a2 = max(0, t - P.m + 1 - pb);
                const bool full = (b1 >= SUB - 1) || (hc >= SUB - 1 && (a2 <= 0 || b1 >= a2 - 1));
                const bool any_masked = __any_sync(0xFFFFFFFFu, !full);  // warp-uniform: no divergent paths
                uint32_t mw[2];
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    mw[k] = full ? 0xFFFFFFFFu : (range_bits(-32 * k, b1 - 32 * k) | range_bits(a2 - 32 * k, hc - 32 * k));
                // the row's 64 scores of this half of S_x in registers (one TMEM load)
                float sv[SUB];
                __syncwarp();
                if (ROPE && T.pbase < P.s) {
                    // a sink sub-tile of RoPE mode: the rotation pass's fp32 scores (rows of this call only)
                    const int lrow = row_start + x * BH_ROWS + r;
                    const bool rowok = lrow < P.L;
                    const float *sr = P.ssink + (static_cast<int64_t>(bh) * P.seq_stride + lrow) * P.sstride + pb;
#pragma unroll
                    for (int c = 0; c < SUB; ++c) sv[c] = (rowok && c <= chi) ? sr[c] : -INFINITY;
                } else {
                    tmem_ld64(s_addr + SUB * hs, sv);
                }
                if (any_masked) {
#pragma unroll
                    for (int c = 0; c < SUB; ++c) sv[c] = (mw[c >> 5] & (1u << (c & 31))) ? sv[c] : -INFINITY;
                }
                float mx4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) mx4[i] = fmax3(sv[i], sv[4 + i], sv[8 + i]);
#pragma unroll
                for (int c = 12; c < SUB - 4; c += 8)
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx4[i] = fmax3(mx4[i], sv[c + i], sv[c + 4 + i]);
                const float mx = fmax3(fmax3(mx4[0], mx4[1], sv[SUB - 4]), fmax3(mx4[2], mx4[3], sv[SUB - 3]),
                                       fmaxf(sv[SUB - 2], sv[SUB - 1])) * sl2;
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
                if (__any_sync(0xFFFFFFFFu, resc)) {
                    // O_x holds the PV products of this item's earlier sub-tiles.  All but the last are complete
                    // (the QK product of this sub-tile was issued after them and is complete; tcgen05 MMAs of
                    // one thread complete in order).  The last, PV_x of the previous sub-tile, is complete once the
                    // QK product of the next sub-tile is (issued after it), or, at the item's last sub-tile, once
                    // the item's second-to-last PV_x product is (pvdone).
                    int jn = j, hn = h;
                    walk_step(jn, hn);
                    if (walk_seek(tl, n, jn, hn, mybit))  // not the item's last sub-tile of this query tile
                        fine = __all_sync(0xFFFFFFFFu, mbar_wait(&sfull[x * 2 + (hs ^ 1)], ((cs + 1) >> 1) & 1, wc, 7, j));
                    else
                        fine = __all_sync(0xFFFFFFFFu, mbar_wait(&pvdone[x], kp & 1, wc, 7, j));
                    if (!fine) break;
                    tc_fence_after();
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
                // p = 2^(scale*log2(e)*s - m); bf16 pairs of the 64 keys go to the first 32 columns of the half
                // (already read): the A operand of PV_x
                const float nmu = (mrun == -INFINITY) ? 0.f : -mrun;
                float rs4[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float a0, a1;
                    ffma2(a0, a1, sv[2 * i], sv[2 * i + 1], sl2, sl2, nmu, nmu);
                    const float p0 = ex2(a0), p1 = ex2(a1);
                    const int k = (i & 1) * 2;
                    fadd2(rs4[k], rs4[k + 1], rs4[k], rs4[k + 1], p0, p1);
                    pk[i] = pack_bf16x2(p0, p1);
                }
                __syncwarp();
                tmem_st32u(s_addr + SUB * hs, pk);
                lrun = lrun * alpha + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
                tc_fence_before();
                mbar_arrive(&pfull[x * 2 + hs]);
                ++cnt;
                ++cs;
                walk_step(j, h);
                ++g;
            }
            if (!fine) break;
            if (lane == 0) mbar_arrive(&lfree[b]);  // this warp no longer reads the tile list
            gbase = g;  // seek_mine counted every walked sub-tile of the item
            if (cnt >= 2) ++kp;
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

}  // namespace tcs

// ---------------------------------------------------------------------------------------- host side
// Tensor map over rows of [nbh, rows, d] bf16 (row stride d * 2 bytes, (b, h) stride bh_stride_rows rows),
// loaded as boxes of 64 columns x box_rows rows with the 128-byte swizzle.
static bool encode_rows_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t nbh, uint64_t bh_stride_rows,
                            int d, uint32_t box_rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), rows, nbh};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, bh_stride_rows * static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Upper bound of the key tiles of one query tile (sink ranges, band ranges split at pos0 and at the
// ring wrap).
static int max_tiles_bound(int w, int s) {
    const int m = w - s;
    return (s + tcs::BN - 1) / tcs::BN + 1 + (m + tcs::BM - 1 + tcs::BN - 1) / tcs::BN + 3;
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

template <int HD, bool ROPE>
static int launch_typed(const tcs::Params &p, int n_ctas, cudaStream_t stream) {
    using LY = tcs::Layout<HD, ROPE>;
    auto *kern = tcs::swa_prefill_tc_kernel<HD, ROPE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(LY::SMEM_BYTES));
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "prefill smem attribute: %s", cudaGetErrorString(e));
    kern<<<n_ctas, tcs::kThreads, LY::SMEM_BYTES, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SWA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return SWA_OK;
}

int launch_prefill_bf16_tc_sub(const PrefillArgs &a) {
    using namespace tcs;
    if (a.d != 64 && a.d != 128) return fail(SWA_ERR_UNSUPPORTED, "tensor-core prefill needs d = 64 or 128");
    const bool rope = a.rope;
    if (rope && (a.d != 128 || !a.q_lo || !a.k_lo || (a.pos0 > 0 && !a.k_cache_lo) || (a.s > 0 && !a.rope_ssink) ||
                 a.rope_sstride < a.s))
        return fail(SWA_ERR_INVALID, "RoPE prefill needs d = 128, the lo parts of q and k and the sink scores");
    if (rope && ((a.pos0 > 0 && a.pos0 < a.s) || a.s > BN))
        return fail(SWA_ERR_UNSUPPORTED, "RoPE prefill needs pos0 = 0 or pos0 >= s, and s <= %d", BN);
    if (max_tiles_bound(a.w, a.s) + (rope ? 1 : 0) > MAX_TILES)
        return fail(SWA_ERR_UNSUPPORTED, "window w=%d needs more than %d key tiles per query tile", a.w, MAX_TILES);
    if ((a.L + BM - 1) / BM * a.BH > 0x7FFFFFFF) return fail(SWA_ERR_UNSUPPORTED, "too many work items");
    if (!encode_tiled_fn()) return fail(SWA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    unsigned *status = device_status_word();
    if (!status) return SWA_ERR_CUDA;
    Params p;
    memset(&p, 0, sizeof(p));
    const uint64_t L = static_cast<uint64_t>(a.L), st = static_cast<uint64_t>(a.seq_stride);
    const int d = a.d;
    bool okm = encode_rows_map(&p.tm_q, a.q, L, a.BH, st, d, 128) && encode_rows_map(&p.tm_k, a.k, L, a.BH, st, d, 64) &&
               encode_rows_map(&p.tm_v, a.v, L, a.BH, st, d, 64);
    // Only slots 0..min(pos0, w)-1 of the cache have been written; the map stops there so that TMA
    // zero-fills the rest of a sub-tile instead of loading stale bytes (a masked column still multiplies its
    // V row by 0, and 0 * NaN would poison the accumulator).  Without a cache the maps alias k and v.
    const uint64_t written = static_cast<uint64_t>(a.pos0 < a.w ? a.pos0 : a.w);
    if (a.pos0 > 0)
        okm = okm && encode_rows_map(&p.tm_kc, a.k_cache, written, a.BH, a.w, d, 64) &&
              encode_rows_map(&p.tm_vc, a.v_cache, written, a.BH, a.w, d, 64);
    else
        okm = okm && encode_rows_map(&p.tm_kc, a.k, L, a.BH, st, d, 64) && encode_rows_map(&p.tm_vc, a.v, L, a.BH, st, d, 64);
    if (rope) {
        okm = okm && encode_rows_map(&p.tm_ql, a.q_lo, L, a.BH, st, d, 128) &&
              encode_rows_map(&p.tm_kl, a.k_lo, L, a.BH, st, d, 64);
        if (a.pos0 > 0)
            okm = okm && encode_rows_map(&p.tm_kcl, a.k_cache_lo, written, a.BH, a.w, d, 64);
        else
            okm = okm && encode_rows_map(&p.tm_kcl, a.k_lo, L, a.BH, st, d, 64);
    } else {
        p.tm_ql = p.tm_q;
        p.tm_kl = p.tm_k;
        p.tm_kcl = p.tm_kc;
    }
    p.ssink = a.rope_ssink;
    p.sstride = a.rope_sstride;
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
    // persistent: one CTA per SM, each walking work items blockIdx.x, blockIdx.x + gridDim.x, ...
    const int sms = sm_count();
    if (sms <= 0) return fail(SWA_ERR_CUDA, "cannot read the multiprocessor count");
    const int n_ctas = p.n_items < sms ? p.n_items : sms;
    if (rope) return launch_typed<128, true>(p, n_ctas, a.stream);
    if (d != 64) return fail(SWA_ERR_UNSUPPORTED, "the sub-tile prefill runs RoPE (d = 128) and d = 64");
    return launch_typed<64, false>(p, n_ctas, a.stream);
}

// The walked sub-tiles of one CTA (query rows q0..q1), in the kernel's order: {source, first row, position of
// column 0, last valid column (< 64), mask of the query tiles that use it}.
int prefill_tile_plan_sub(int q0, int q1, int pos0, int w, int s, int rope, int *out, int max_tiles) {
    tcs::Tile tl[tcs::MAX_TILES];
    const int n = tcs::build_tiles(tl, q0, q1, pos0, s, w - s, w, rope != 0);
    if (n > tcs::MAX_TILES) return fail(SWA_ERR_UNSUPPORTED, "more than %d key tiles", tcs::MAX_TILES);
    tcs::mark_tiles(tl, n, q0, q1, s, w - s);
    int k = 0, j = 0, h = 0;
    while (tcs::walk_seek(tl, n, j, h, 3)) {
        if (k < max_tiles) {
            const int chi = tl[j].chi - tcs::SUB * h;
            out[5 * k + 0] = tl[j].flags & 1;
            out[5 * k + 1] = tl[j].row0 + tcs::SUB * h;
            out[5 * k + 2] = tl[j].pbase + tcs::SUB * h;
            out[5 * k + 3] = chi < tcs::SUB - 1 ? chi : tcs::SUB - 1;
            out[5 * k + 4] = tcs::half_users(tl[j], h);
        }
        ++k;
        tcs::walk_step(j, h);
    }
    return k;
}

}  // namespace swa
