// k_attend_tc.cu -- CSA / HCA core attention on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), bf16 rows of 512 dims, 64 query heads.
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2: CSA Step 3 (multi-query attention
// over the top-k compressed blocks), HCA (dense attention over every block),
// and 四项关键 Trick: RMSNorm and partial RoPE on q, a sliding window of the
// last W raw tokens, a learnable sink in the softmax denominator, RoPE at -i
// on the output.
//
// One query's row list is cut into tiles of 64 rows: ceil(k/64) tiles of
// selected blocks (CSA) or ceil(n_cap/64) tiles of consecutive blocks (HCA),
// then ceil(W/64) window tiles.  The (query, tile) pairs are dealt out in
// contiguous, balanced ranges to one persistent CTA per SM; the run of one
// query's tiles inside a CTA is a segment.  A segment that is the whole query
// is finished in place (sink, normalisation, rotation, bf16 store); the others
// leave an unnormalised partial (m, l, o) for attend_combine_kernel.  In the
// batch-invariant mode [gitcode §5.3 "批次不变且确定性内核"] every query's tiles
// are cut into fixed splits of `seg` tiles (a function of the list length),
// CTAs take whole splits, every split leaves a partial and the combine merges
// them in split order, so the rounding of a query's result never depends on
// the rest of the batch.
//
// Per tile (one shared KV head, so key = value = row e_j):
//   S^T[64 rows, 64 heads] = E[64, 512] . Q'^T          (swap-AB: rows are M)
//   P = 2^(S^T * scale * log2 e - m)  (bf16, per head running reference m)
//   O^T[512, 64] += E^T[512, 64] . P^T                   (4 MMAs of M = 128)
// The tile (8 boxes of 64 rows x 64 dims, 128-byte swizzle) is the K-major A
// operand of the first product and, read along its rows, the MN-major A
// operand of the second.  Two tile stages alternate; S^T and P are double
// buffered, so the QK product of the next tile runs while the softmax of this
// one does.  The running reference m is raised only when a logit exceeds it
// by more than 2^8; O^T (in TMEM) and the partial sums are then rescaled in
// place.
//
// Warp roles (at most 20 warps, five per scheduler, so that each thread
// keeps 96 registers): warp 0 orders every use of a stage and loads TMA
// tiles (consecutive rows); warps 2..17 prepare q', run the softmax and the
// epilogue.  Where every tile is a TMA tile (dense lists, pre-gathered rows)
// warp 1 issues the QK products (a tile's as soon as its stage has landed
// and its S^T buffer is free) and warp 18 the PV products (a tile's as soon
// as its P is written), so that neither waits behind the other's issue.
// Where selected rows are gathered, warp 1 issues both products and warps
// 18..19 fetch the rows with TMA gather4 (gather issue, not MMA issue,
// bounds those tiles).  FP8 rows are first
// dequantised to bf16 in the workspace (dequant_gather_kernel or
// dequant_rows_kernel).  Every wait is bounded; on a timeout the kernel sets
// CSA_DEV_TIMEOUT, every role leaves its loop, outstanding copies and MMAs are
// waited for and TMEM is freed.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa {

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

namespace {

constexpr int kD = 512;
constexpr int kH = 64;
constexpr int kRows = 64;                           // rows per tile (QK MMA M)
constexpr int kStages = 2;
// A CTA's start of a query (preparing its q' and writing its partial) costs
// about as much as this many tiles (HCA decode timelines: a CTA meeting two
// queries ended 10-30 us after one meeting one, at ~3.3 us a tile; attention
// at batch 32, 1M context: 124.9 us with 3, 122.9 us with 5, 7 or 9)
constexpr int kQueryCostTiles = 5;
constexpr uint32_t kBoxBytes = kRows * 128;         // 64 rows x 64 dims (bf16)
constexpr uint32_t kStageBytes = 8 * kBoxBytes;     // 64 rows x 512 dims
constexpr uint32_t kQBoxBytes = kH * 128;           // 64 heads x 64 dims
constexpr uint32_t kQBytes = 8 * kQBoxBytes;        // 64 heads x 512 dims
constexpr uint32_t kPBytes = kRows * kH * 2;        // 64 rows x 64 heads
constexpr size_t kSmem = 1024 + kStages * kStageBytes + kQBytes + 2 * kPBytes;
constexpr int kSoftWarps = 16;                      // 4 TMEM lane quarters x 4 head quarters
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kHW = kH / 4;                         // heads per softmax warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S^T buffers: 2 x 64 columns
constexpr uint32_t kColO = 256;  // O^T: 4 x 64 columns
constexpr float kRescaleLog2 = 8.f;
constexpr float kNoRef = -1e30f; // running reference before any valid logit
constexpr int kBarSoftmax = 1;   // named barrier of the softmax warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttTcArgs {
    const uint16_t* q;        // [Q, 64, 512] bf16
    const int64_t* q_pos;     // [Q]
    const int32_t* topk_idx;  // [Q, k]; nullptr: dense (HCA)
    int k;
    int pre;                  // tm_sel maps [Q, T * 64, 512]: each query's rows in tile order
    const uint8_t* cache;     // [B, n_cap, 512] bf16 rows the gather warps copy
    int64_t n_cap, n_win;
    const int64_t* win_pos0;  // [B]; nullptr: ring window (position p at row p mod n_win)
    int W, m, qps;
    float eps, scale_log2;
    int T_sel, T;             // tiles per query: selected / cache part, all
    int64_t total;            // Q * T
    int grid;
    int seg, nseg;            // batch-invariant splits of seg tiles, nseg per query (seg 0: off)
    int qcta, qrem, qc;       // the ranges' TileDeal (qcta 0: balanced, a query counted as qc + T tiles)
    int S;                    // partial slots per query
    float* part_o;            // [Q, S, 64, 512]
    float* part_ml;           // [Q, S, 64, 2]
    int32_t* nslots;          // [Q]: partials of each query, 0 if finished in one CTA (ranges; else nullptr)
    const float* sink;        // [64]
    uint16_t* out;            // [Q, 64, 512] bf16 (queries finished in one CTA)
    float* lse;               // [Q, 64] or nullptr
    int derotate;
    uint32_t* status;
    RopeTheta theta;
};

// Tile, query and split indices stay below 2^31 (the host plans no more
// tiles, or query-start units, than that), so their divisions run in 32 bits:
// a 64-bit division is a long inlined sequence, and the kernel's code
// outgrew the instruction cache (ncu: 57% hits at CSA decode).
__device__ __forceinline__ int64_t idiv(int64_t x, int64_t y) { return (int64_t)((uint32_t)x / (uint32_t)y); }
// Positions may exceed 32 bits: their divisions take the 64-bit sequence out
// of line, where it is never reached below 2^32.
__device__ __noinline__ int64_t div_wide(int64_t x, int64_t y) { return x / y; }
__device__ __noinline__ int64_t mod_wide(int64_t x, int64_t y) {  // in [0, y)
    const int64_t m = x % y;
    return m < 0 ? m + y : m;
}
// floor((i + 1) / m) for a position i
__device__ __forceinline__ int64_t blocks_of(int64_t i, int m) {
    const int64_t x = i + 1;
    return (x >= 0 && x <= 0xffffffffLL) ? (int64_t)((uint32_t)x / (uint32_t)m) : div_wide(x, m);
}

__device__ __forceinline__ TileDeal deal_of(const AttTcArgs& a) {
    return TileDeal{a.total, (int64_t)a.T, a.grid, a.qcta, a.qrem, a.qc};
}

// CTA that owns global tile g (ranges without fixed splits).
__device__ __forceinline__ int64_t cta_of(const AttTcArgs& a, int64_t g) { return deal_of(a).cta_of(g); }

// First global tile of CTA c's range: balanced over tiles or query-aligned
// (TileDeal), or, with fixed splits, over whole splits (CTA c takes splits
// [c*n/grid, (c+1)*n/grid) of the n = Q * nseg in query order).
template <bool L>
__device__ __forceinline__ int64_t range_begin(const AttTcArgs& a, int64_t c) {
    if (L || a.seg == 0) return deal_of(a).begin(c);
    const int64_t sp = TileDeal::share(c, idiv(a.total, a.T) * a.nseg, a.grid);
    const int64_t qi = idiv(sp, a.nseg);
    return qi * a.T + min((int64_t)a.T, (sp - qi * a.nseg) * a.seg);
}

// End of the segment that starts at global tile g: the end of the query's
// tiles, of the fixed split holding g, or of the CTA's range.
template <bool L>
__device__ __forceinline__ int64_t seg_end_of(const AttTcArgs& a, int64_t g, int64_t g_end) {
    const int64_t qi = idiv(g, a.T);
    int64_t e = (qi + 1) * a.T;
    if (!L && a.seg > 0) e = min(e, qi * a.T + (idiv(g - qi * a.T, a.seg) + 1) * a.seg);
    return min(g_end, e);
}

struct QueryInfo {
    int64_t i, n_av;
    int seq;
};

__device__ __forceinline__ QueryInfo query_info(const AttTcArgs& a, int64_t qi) {
    QueryInfo r;
    r.i = a.q_pos[qi];
    r.seq = (int)idiv(qi, a.qps);
    int64_t n = blocks_of(r.i, a.m);
    if (n < 0) n = 0;
    r.n_av = n < a.n_cap ? n : a.n_cap;  // an overflow is flagged by the softmax warps
    return r;
}

// Whether tile lt of a query has any row that can be valid.  Every role
// evaluates the same predicate, so skipped tiles cost nothing anywhere.
template <bool L>
__device__ __forceinline__ bool tile_live(const AttTcArgs& a, const QueryInfo& qi, int lt) {
    if (lt < a.T_sel) {
        if (a.topk_idx) return qi.n_av > 0;
        return (int64_t)lt * kRows < qi.n_av;
    }
    const int r0 = (lt - a.T_sel) * kRows;
    if (L || a.win_pos0 == nullptr) return r0 < a.n_win && r0 <= qi.i;  // ring rows r0 ..: some hold positions <= i
    if (r0 >= a.W) return false;
    const int rlast = min(a.W, r0 + kRows) - 1;
    return qi.i - a.W + 1 + rlast >= 0;
}

// Ring window: the position row r holds for a query at position i, the
// latest p <= i with p = r mod n_win (negative: not written yet).
__device__ __forceinline__ int64_t ring_pos(int64_t i, int64_t r, int64_t n_win) {
    const int64_t d = i - r;
    return i - ((d >= 0 && d <= 0xffffffffLL) ? (int64_t)((uint32_t)d % (uint32_t)n_win) : mod_wide(d, n_win));
}

// Warp roles of the two layouts.  Split (tiles loaded by TMA only): warp 1
// issues the QK products and warp 18 the PV products.  Otherwise (gathered
// tiles): warp 1 issues both and warps 18..19 fetch the selected rows with
// TMA gather4, each four of the eight 64-dim boxes of every row (TMA gathers
// issued from several warps proceed in parallel; two warps issue them twice
// as fast as one).
template <bool kSplit>
struct Roles {
    static constexpr int kLoadWarps = kSplit ? 0 : 2;
    static constexpr int kPvWarp = kSplit ? 2 + kSoftWarps : 1;
    static constexpr int kThreads = 32 * (2 + kSoftWarps + kLoadWarps + (kSplit ? 1 : 0));
    static constexpr int kLoaderBoxes = kLoadWarps > 0 ? 8 / kLoadWarps : 0;
};

// Whether tile lt is copied row by row from the selected cache rows (by
// gather4) rather than loaded as a TMA tile.
template <bool L>
__device__ __forceinline__ bool is_gathered(const AttTcArgs& a, int lt) {
    return (L || !a.pre) && a.topk_idx != nullptr && lt < a.T_sel;
}

// Cache rows of the selected blocks of gathered tile lt of query qi that
// lane l gathers: tile rows 4*(l%16) .. +3 (a masked row fetches the
// sequence's row 0; the softmax warps mask it).
__device__ __forceinline__ void gather_rows(const AttTcArgs& a, int64_t qi, const QueryInfo& inf, int lt,
                                            int lane, int (&rows)[4]) {
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int p = lt * kRows + 4 * (lane & 15) + j;
        int64_t e = p < a.k ? (int64_t)a.topk_idx[qi * a.k + p] : -1;
        if (e < 0 || e >= inf.n_av) e = 0;
        rows[j] = (int)((int64_t)inf.seq * a.n_cap + e);
    }
}

// Boxes box0 .. box0+nbox-1 (64 dims each) of those rows into a stage, by
// one warp.
__device__ __forceinline__ void gather_boxes(const CUtensorMap* tm, uint64_t* bar, uint8_t* stage,
                                             const int (&rows)[4], int box0, int nbox, int lane) {
    const int rg = lane & 15;
    for (int pi = lane; pi < 16 * nbox; pi += 32) {  // pi % 16 == rg
        const int box = box0 + pi / 16;
        tc::tma_gather4(stage + box * kBoxBytes + rg * 512, tm, bar, box * 64, rows[0], rows[1], rows[2], rows[3]);
    }
}

// Last live tile of the segment [lt0, lt1) of a query, or -1.
template <bool L>
__device__ __forceinline__ int last_live(const AttTcArgs& a, const QueryInfo& qi, int lt0, int lt1) {
    for (int lt = lt1 - 1; lt >= lt0; --lt)
        if (tile_live<L>(a, qi, lt)) return lt;
    return -1;
}

// The first query from global tile g on (up to g_end) whose segment has a
// live tile, or -1.
template <bool L>
__device__ __forceinline__ int64_t next_live_query(const AttTcArgs& a, int64_t g, int64_t g_end) {
    while (g < g_end) {
        const int64_t qi = idiv(g, a.T);
        const int64_t seg_end = seg_end_of<L>(a, g, g_end);
        const QueryInfo inf = query_info(a, qi);
        if (last_live<L>(a, inf, (int)(g - qi * a.T), (int)(seg_end - qi * a.T)) >= 0) return qi;
        g = seg_end;
    }
    return -1;
}

// -------------------------------------------------------------- softmax helpers
// Reduce 16 per-lane values over the warp so that lanes l and l+16 end with
// the reduction of entry (l % 16) over all 32 lanes (31 shuffles).
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter16(const float (&v)[16], int lane) {
    auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
    float a[16], b[8], c[4], d[2];
#pragma unroll
    for (int j = 0; j < 16; j++) a[j] = op(v[j], __shfl_xor_sync(0xffffffffu, v[j], 16));
    {
        const bool up = lane & 8;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float keep = up ? a[j + 8] : a[j], send = up ? a[j] : a[j + 8];
            b[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
        }
    }
    {
        const bool up = lane & 4;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float keep = up ? b[j + 4] : b[j], send = up ? b[j] : b[j + 4];
            c[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
        }
    }
    {
        const bool up = lane & 2;
#pragma unroll
        for (int j = 0; j < 2; j++) {
            float keep = up ? c[j + 2] : c[j], send = up ? c[j] : c[j + 2];
            d[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
        }
    }
    const bool up = lane & 1;
    float keep = up ? d[1] : d[0], send = up ? d[0] : d[1];
    return op(keep, __shfl_xor_sync(0xffffffffu, send, 1));
}

__device__ __forceinline__ bool softmax_barrier_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(kBarSoftmax), "r"(kSoftThreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void softmax_barrier() { tc::named_barrier(kBarSoftmax, kSoftThreads); }

// Wait by lane 0, verdict shared with the warp (tcgen05.ld is warp-wide).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status, int lane) {
    int ok = 1;
    if (lane == 0) ok = tc::mbar_wait(bar, parity, abort_flag, status) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// 2^x with the hardware approximation (relative error ~2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)f32_to_bf16_rn(lo) | ((uint32_t)f32_to_bf16_rn(hi) << 16);
}


// ------------------------------------------------------------- FP8 rows -> bf16
// Stored FP8_MIXED row of 512 dims: 448 E4M3 codes, the 64 rotated dims as
// bf16, then one float32 scale per 64-dim group of codes.
constexpr int kNf = kD - kRopeDims;             // quantised dims
constexpr int kScaleOff = kNf + 2 * kRopeDims;  // byte offset of the scales

// One warp dequantises one row into 512 bf16 (code * group scale, rounded to
// nearest even; the rotated dims are copied).  A null row writes zeros: a
// masked row must hold finite values, as its weight P = 0 multiplies it.
__device__ __forceinline__ void warp_dequant_row(const uint8_t* row, uint16_t* out, int lane) {
    uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
    if (row != nullptr) {
        if (lane < kNf / 16) {  // 16 codes per lane, four lanes per group
            const uint4 c = __ldg(reinterpret_cast<const uint4*>(row) + lane);
            const float sc = __ldg(reinterpret_cast<const float*>(row + kScaleOff) + (lane >> 2));
            const uint32_t w[4] = {c.x, c.y, c.z, c.w};
            uint32_t r[8];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                r[2 * e] = pack_bf16x2(e4m3_to_f32((uint8_t)w[e]) * sc, e4m3_to_f32((uint8_t)(w[e] >> 8)) * sc);
                r[2 * e + 1] =
                    pack_bf16x2(e4m3_to_f32((uint8_t)(w[e] >> 16)) * sc, e4m3_to_f32((uint8_t)(w[e] >> 24)) * sc);
            }
            o0 = make_uint4(r[0], r[1], r[2], r[3]);
            o1 = make_uint4(r[4], r[5], r[6], r[7]);
        } else {  // lanes 28..31: 16 rotated dims each, already bf16
            const uint4* src = reinterpret_cast<const uint4*>(row + kNf) + 2 * (lane - kNf / 16);
            o0 = __ldg(src);
            o1 = __ldg(src + 1);
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(out) + 2 * lane;
    dst[0] = o0;
    dst[1] = o1;
}

constexpr int kDeqThreads = 256;  // one row per warp

// Every stored row of a buffer [n, rb bytes] -> [n, 512] bf16.
__global__ void __launch_bounds__(kDeqThreads) dequant_rows_kernel(const uint8_t* __restrict__ src, int64_t rb,
                                                                   int64_t n, uint16_t* __restrict__ out) {
    const int64_t r = (int64_t)blockIdx.x * (kDeqThreads / 32) + (threadIdx.x >> 5);
    if (r < n) warp_dequant_row(src + r * rb, out + r * kD, threadIdx.x & 31);
}

struct DeqGatherArgs {
    const uint8_t* cache;     // [B, n_cap, rb]
    const uint8_t* window;    // [B, n_win, rb]
    int64_t rb, n_cap, n_win;
    const int64_t* q_pos;     // [Q]
    const int64_t* win_pos0;  // [B]; nullptr: ring window
    const int32_t* topk_idx;  // [Q, k]; nullptr: every cache row in order
    int k, W, m, qps, T_sel, T;
    int64_t rows;             // Q * T * 64
    uint16_t* out;            // [Q, T * 64, 512]
};

// Row p of query qi's list in tile order: the p-th selected (or cache) row
// for p < T_sel * 64, then window row p - T_sel * 64.  Rows the attention
// masks (padding, index -1, out of range, before position 0) are zeros.
__global__ void __launch_bounds__(kDeqThreads) dequant_gather_kernel(const DeqGatherArgs a) {
    const int64_t r = (int64_t)blockIdx.x * (kDeqThreads / 32) + (threadIdx.x >> 5);
    if (r >= a.rows) return;
    const int64_t per = (int64_t)a.T * kRows;
    const int64_t qi = r / per;
    const int p = (int)(r - qi * per);
    const int64_t i = a.q_pos[qi];
    const int seq = (int)idiv(qi, a.qps);
    int64_t n_av = blocks_of(i, a.m);
    n_av = n_av < 0 ? 0 : (n_av < a.n_cap ? n_av : a.n_cap);
    const uint8_t* src = nullptr;
    if (p < a.T_sel * kRows) {
        const int64_t e = a.topk_idx ? (p < a.k ? (int64_t)a.topk_idx[qi * a.k + p] : -1) : p;
        if (e >= 0 && e < n_av) src = a.cache + ((int64_t)seq * a.n_cap + e) * a.rb;
    } else {
        const int rw = p - a.T_sel * kRows;
        if (a.win_pos0 == nullptr) {  // ring rows in buffer order
            const int64_t wpos = rw < a.n_win ? ring_pos(i, rw, a.n_win) : -1;
            if (wpos >= 0 && wpos >= i - a.W + 1) src = a.window + ((int64_t)seq * a.n_win + rw) * a.rb;
        } else {
            const int64_t wr = i - a.W + 1 + rw - a.win_pos0[seq];
            if (rw < a.W && i - a.W + 1 + rw >= 0 && wr >= 0 && wr < a.n_win)
                src = a.window + ((int64_t)seq * a.n_win + wr) * a.rb;
        }
    }
    warp_dequant_row(src, a.out + r * kD, threadIdx.x & 31);
}

}  // namespace

// kLean: no fixed splits, no pre-gathered rows and a ring window (the
// decode step's form); the instantiation leaves out the code of the others,
// which keeps the kernel's instruction footprint down.
template <bool kSplit, bool kLean>
__global__ void __launch_bounds__(Roles<kSplit>::kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tm_sel, const __grid_constant__ CUtensorMap tm_win,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ AttTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sE = sm;                              // kStages x (8 boxes of 64 rows x 64 dims)
    uint8_t* sQ = sE + kStages * kStageBytes;      // 8 boxes of 64 heads x 64 dims
    uint8_t* sP = sQ + kQBytes;                    // 2 x (64 rows x 64 heads)

    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], go[kStages];
    __shared__ __align__(8) uint64_t s_full[2], p_full[2];
    __shared__ __align__(8) uint64_t o_full, o_seg, q_full, q_raw, mma_done, pv_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_sh;
    __shared__ float red[4][kH];
    __shared__ float mref_s[kH], alph_s[kH], fac_s[kH];
    __shared__ float rot_cs[64];
    volatile int* abort_flag = &abort_sh;

    constexpr int kLoadWarps = Roles<kSplit>::kLoadWarps;
    constexpr int kPvWarp = Roles<kSplit>::kPvWarp;
    constexpr int kLoaderBoxes = Roles<kSplit>::kLoaderBoxes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
            tc::mbar_init(&go[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            tc::mbar_init(&s_full[b], 1);
            tc::mbar_init(&p_full[b], kSoftWarps);
        }
        tc::mbar_init(&o_full, 1);  // after every PV product
        tc::mbar_init(&o_seg, 1);   // after the last PV product of a segment
        tc::mbar_init(&q_full, 1);
        tc::mbar_init(&q_raw, 1);   // raw q of the CTA's first segment landed in sQ
        tc::mbar_init(&mma_done, 1);
        tc::mbar_init(&pv_done, 1);
        abort_sh = 0;
        tc::fence_barrier_init();
        tc::fence_proxy_async_smem();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    // Launched as a programmatic dependent: the setup above overlapped the
    // kernel before; every global read comes after it has completed.
    tc::grid_dep_wait();

    const int64_t g_begin = range_begin<kLean>(a, blockIdx.x);
    const int64_t g_end = range_begin<kLean>(a, blockIdx.x + 1);

    if (warp == 0) {
        // ------------------------------------------------------------ loads
        // The raw q rows of the first segment go into sQ ahead of any tile:
        // the softmax warps normalise and rotate them in place.
        const int64_t q_first = next_live_query<kLean>(a, g_begin, g_end);
        if (q_first >= 0) {
            if (lane == 0) tc::mbar_arrive_expect_tx(&q_raw, kQBytes);
            __syncwarp();
            if (lane < 8) tc::tma_load_3d(sQ + lane * kQBoxBytes, &tm_q, &q_raw, lane * 64, 0, (int)q_first);
        }
        if (lane == 0) {
            tc::tma_prefetch_map(&tm_sel);
            if (a.W > 0) tc::tma_prefetch_map(&tm_win);
        }
        uint32_t tcount = 0;
        uint32_t fills[kStages] = {0, 0};  // fills of each stage (by any warp)
        auto box_row0 = [&](const QueryInfo& inf, int lt) {
            if (lt < a.T_sel) return lt * kRows;
            if (kLean || a.win_pos0 == nullptr) return (lt - a.T_sel) * kRows;  // ring rows in buffer order
            return (int)(inf.i - a.W + 1 + (int64_t)(lt - a.T_sel) * kRows - a.win_pos0[inf.seq]);
        };
        // The next live TMA-tile (not gathered) after global tile g within this
        // CTA's range is prefetched into L2 while the current one is loaded.
        auto prefetch_after = [&](int64_t g) {
            for (++g; g < g_end; ++g) {
                const int64_t qi = idiv(g, a.T);
                const int lt = (int)(g - qi * a.T);
                const QueryInfo inf = query_info(a, qi);
                if (!tile_live<kLean>(a, inf, lt)) continue;
                if (!kLean && a.pre) {
                    if (lane < 8) tc::tma_prefetch_3d(&tm_sel, lane * 64, lt * kRows, (int)qi);
                } else if (!is_gathered<kLean>(a, lt) && lane < 8) {
                    const int r0 = box_row0(inf, lt);
                    if (r0 >= 0)  // a window box that starts before row 0 is not prefetched
                        tc::tma_prefetch_3d(lt < a.T_sel ? &tm_sel : &tm_win, lane * 64, r0, inf.seq);
                }
                return;
            }
        };
        for (int64_t g = g_begin; g < g_end; ++g) {
            const int64_t qi = idiv(g, a.T);
            const int lt = (int)(g - qi * a.T);
            const QueryInfo inf = query_info(a, qi);
            if (!tile_live<kLean>(a, inf, lt)) continue;
            const int st = tcount & 1;
            prefetch_after(g);
            // every use of a stage is waited for here, in order, whoever fills it
            if (!warp_wait(&empty[st], ((tcount >> 1) & 1u) ^ 1u, abort_flag, a.status, lane)) break;
            if (lane == 0) tc::mbar_arrive_expect_tx(&full[st], kStageBytes);
            if (is_gathered<kLean>(a, lt)) {
                if (lane == 0) tc::mbar_arrive(&go[st]);  // the gather warps join in
            } else {
                uint8_t* dst = sE + st * kStageBytes;
                __syncwarp();
                if (lane < 8) {
                    if (!kLean && a.pre)
                        tc::tma_load_3d(dst + lane * kBoxBytes, &tm_sel, &full[st], lane * 64, lt * kRows, (int)qi);
                    else
                        tc::tma_load_3d(dst + lane * kBoxBytes, lt < a.T_sel ? &tm_sel : &tm_win, &full[st],
                                        lane * 64, box_row0(inf, lt), inf.seq);
                }
            }
            ++fills[st];
            ++tcount;
        }
        // Leave no copy in flight: the newest load of every stage must have
        // landed (at most one phase of a stage is ever outstanding).
        if (lane == 0) {
            for (int st = 0; st < kStages; st++) {
                if (fills[st] == 0) continue;
                if (!tc::mbar_drain(&full[st], (fills[st] - 1u) & 1u)) atomicOr(a.status, CSA_DEV_TIMEOUT);
            }
        }
    } else if (warp == 1 || warp == kPvWarp) {
        if constexpr (kSplit) {
            // ------------------------------------------------------------ MMA issue
            // Two issuing threads, so that a PV product never waits behind the
            // issue of a QK product (one thread issues an MMA every ~85 cycles while
            // the softmax warps share its scheduler): warp 1 issues the QK product
            // of every tile as soon as its stage has landed and the S^T buffer it
            // reuses is free (the softmax of the tile two before has read it);
            // warp kPvWarp issues the PV product of every tile as soon as its P is
            // written.  The QK product of tile t+2 cannot start before the PV
            // product of tile t has freed its stage, so neither thread can see a
            // barrier phase of the other's overtaken.  Descriptors are built once
            // per operand and advanced by constant offsets of the 128-byte-swizzled
            // boxes (the start-address field never carries: shared addresses stay
            // below 2^18).
            if (lane == 0) {
                const bool qk_role = warp == 1;
                constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kRows, kH, 0, 0);
                constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, kH, 1, 1);
                const uint32_t sE0 = tc::smem_u32(sE), sQ0 = tc::smem_u32(sQ), sP0 = tc::smem_u32(sP);
                const uint64_t dq0 = tc::sdesc_sw128(sQ0, 16, 1024);
                uint32_t t = 0, nq = 0;
                // cursor over this CTA's live tiles
                int64_t g = g_begin;
                int64_t cur_q = -1, cur_end = g_begin, q_in = -1;  // q_in: query whose q' is in sQ
                QueryInfo inf{};
                int lt_last = -1;
                bool at_seg_start = true;
                auto advance = [&]() -> bool {  // move g to the next live tile; false at the end
                    for (; g < g_end; ++g) {
                        const int64_t qi = idiv(g, a.T);
                        if (g >= cur_end) {
                            cur_q = qi;
                            inf = query_info(a, qi);
                            cur_end = seg_end_of<kLean>(a, g, g_end);
                            lt_last = last_live<kLean>(a, inf, (int)(g - qi * a.T), (int)(cur_end - qi * a.T));
                            at_seg_start = true;
                        }
                        if (tile_live<kLean>(a, inf, (int)(g - qi * a.T))) return true;
                    }
                    return false;
                };
                while (advance()) {
                    const int b = t & 1;
                    const uint32_t stage = sE0 + b * kStageBytes;
                    if (qk_role) {
                        // the S^T buffer of tile t: the softmax of tile t - 2 has read it
                        if (t >= 2 && !tc::mbar_wait(&p_full[b], ((t - 2) >> 1) & 1u, abort_flag, a.status)) break;
                        // q' is prepared once per query: a later split of the same query in
                        // this CTA reuses it
                        const bool need_q = at_seg_start && cur_q != q_in;
                        if (need_q && !tc::mbar_wait(&q_full, nq & 1u, abort_flag, a.status)) break;
                        if (!tc::mbar_wait(&full[b], (t >> 1) & 1u, abort_flag, a.status)) break;
                        tc::fence_after_sync();
                        const uint64_t da0 = tc::sdesc_sw128(stage, 16, 1024);
    #pragma unroll
                        for (int kg = 0; kg < kD / 16; kg++) {
                            const uint32_t off = ((kg >> 2) * kBoxBytes + (kg & 3) * 32) >> 4;
                            const uint32_t offq = ((kg >> 2) * kQBoxBytes + (kg & 3) * 32) >> 4;
                            tc::mma_bf16_ss(tmem + kColS + 64 * b, da0 + off, dq0 + offq, idesc_qk, kg != 0 ? 1u : 0u);
                        }
                        tc::mma_commit(&s_full[b]);
                        if (need_q) {
                            ++nq;
                            q_in = cur_q;
                        }
                    } else {
                        const bool first = at_seg_start;
                        const bool last = (int)(g - cur_q * a.T) == lt_last;
                        if (!tc::mbar_wait(&p_full[b], (t >> 1) & 1u, abort_flag, a.status)) break;
                        tc::fence_after_sync();
                        const uint64_t da0 = tc::sdesc_sw128(stage, kBoxBytes, 1024);
                        const uint64_t db0 = tc::sdesc_sw128(sP0 + b * kPBytes, kBoxBytes, 1024);
    #pragma unroll
                        for (int c = 0; c < 4; c++) {
    #pragma unroll
                            for (int kk = 0; kk < kRows / 16; kk++) {
                                const uint32_t off = (2 * c * kBoxBytes + kk * 2048) >> 4;
                                tc::mma_bf16_ss(tmem + kColO + 64 * c, da0 + off, db0 + ((kk * 2048) >> 4), idesc_pv,
                                                (first && kk == 0) ? 0u : 1u);
                            }
                        }
                        tc::mma_commit(&empty[b]);
                        tc::mma_commit(&o_full);
                        if (last) tc::mma_commit(&o_seg);
                    }
                    at_seg_start = false;
                    ++t;
                    ++g;
                }
                // every MMA this thread issued must be complete before TMEM is freed
                uint64_t* done = qk_role ? &mma_done : &pv_done;
                tc::mma_commit(done);
                if (!tc::mbar_drain(done, 0)) atomicOr(a.status, CSA_DEV_TIMEOUT);
            }
        } else {
            // ------------------------------------------------------------ MMA issue
            // Issue order is dynamic: the PV product of tile t as soon as its P is
            // written, the QK product of tile t+1 as soon as its stage has landed
            // and the S^T buffer it reuses is free (PV of tile t-1 issued).
            if (lane == 0) {
                constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kRows, kH, 0, 0);
                constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, kH, 1, 1);
                const uint32_t sE0 = tc::smem_u32(sE), sQ0 = tc::smem_u32(sQ), sP0 = tc::smem_u32(sP);
                uint32_t t_qk = 0, t_pv = 0, nq = 0;
                bool first_of[4], last_of[4];  // segment flags of tiles t_pv .. t_qk-1 (at most 2)
                // QK cursor over this CTA's live tiles
                int64_t g = g_begin;
                int64_t cur_q = -1, cur_end = g_begin, q_in = -1;  // q_in: query whose q' is in sQ
                QueryInfo inf{};
                int lt_last = -1;
                bool at_seg_start = true;
                auto advance = [&]() -> bool {  // move g to the next live tile; false at the end
                    for (; g < g_end; ++g) {
                        const int64_t qi = idiv(g, a.T);
                        if (g >= cur_end) {
                            cur_q = qi;
                            inf = query_info(a, qi);
                            cur_end = seg_end_of<kLean>(a, g, g_end);
                            lt_last = last_live<kLean>(a, inf, (int)(g - qi * a.T), (int)(cur_end - qi * a.T));
                            at_seg_start = true;
                        }
                        if (tile_live<kLean>(a, inf, (int)(g - qi * a.T))) return true;
                    }
                    return false;
                };
                bool more = advance();
                uint64_t idle_since = 0;
                while (more || t_pv < t_qk) {
                    bool progress = false;
                    if (t_pv < t_qk) {
                        const int b = t_pv & 1;
                        if (tc::mbar_test_wait(&p_full[b], (t_pv >> 1) & 1u)) {
                            tc::fence_after_sync();
                            const uint32_t stage = sE0 + b * kStageBytes;
                            const uint32_t pb = sP0 + b * kPBytes;
                            const bool first = first_of[t_pv & 3];
    #pragma unroll
                            for (int c = 0; c < 4; c++) {
    #pragma unroll
                                for (int kk = 0; kk < kRows / 16; kk++) {
                                    const uint64_t ad = tc::sdesc_sw128(stage + 2 * c * kBoxBytes + kk * 2048, kBoxBytes, 1024);
                                    const uint64_t bd = tc::sdesc_sw128(pb + kk * 2048, kBoxBytes, 1024);
                                    tc::mma_bf16_ss(tmem + kColO + 64 * c, ad, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
                                }
                            }
                            tc::mma_commit(&empty[b]);
                            tc::mma_commit(&o_full);
                            if (last_of[t_pv & 3]) tc::mma_commit(&o_seg);
                            ++t_pv;
                            progress = true;
                        }
                    }
                    if (more && t_pv + 1 >= t_qk) {  // S^T buffer of tile t_qk is free
                        const int b = t_qk & 1;
                        // q' is prepared once per query: a later split of the same
                        // query in this CTA reuses it
                        const bool need_q = at_seg_start && cur_q != q_in;
                        bool ready = !need_q || tc::mbar_test_wait(&q_full, nq & 1u);
                        if (ready) ready = tc::mbar_test_wait(&full[b], (t_qk >> 1) & 1u);
                        if (ready) {
                            tc::fence_after_sync();
                            const uint32_t stage = sE0 + b * kStageBytes;
    #pragma unroll 8
                            for (int kg = 0; kg < kD / 16; kg++) {
                                const uint64_t ad = tc::sdesc_sw128(stage + (kg >> 2) * kBoxBytes + (kg & 3) * 32, 16, 1024);
                                const uint64_t bd = tc::sdesc_sw128(sQ0 + (kg >> 2) * kQBoxBytes + (kg & 3) * 32, 16, 1024);
                                tc::mma_bf16_ss(tmem + kColS + 64 * b, ad, bd, idesc_qk, kg != 0 ? 1u : 0u);
                            }
                            tc::mma_commit(&s_full[b]);
                            if (need_q) {
                                ++nq;
                                q_in = cur_q;
                            }
                            first_of[t_qk & 3] = at_seg_start;
                            last_of[t_qk & 3] = (int)(g - cur_q * a.T) == lt_last;
                            at_seg_start = false;
                            ++t_qk;
                            ++g;
                            more = advance();
                            progress = true;
                        }
                    }
                    if (progress) {
                        idle_since = 0;
                    } else {
                        if (*abort_flag) break;
                        const uint64_t now = tc::globaltimer_ns();
                        if (idle_since == 0) {
                            idle_since = now;
                        } else if (now - idle_since > tc::kWaitLimitNs) {
                            atomicOr(a.status, CSA_DEV_TIMEOUT);
                            *abort_flag = 1;
                            break;
                        }
                    }
                }
                // every MMA issued so far must be complete before TMEM is freed
                tc::mma_commit(&mma_done);
                if (!tc::mbar_drain(&mma_done, 0)) atomicOr(a.status, CSA_DEV_TIMEOUT);
            }
        }
    } else if (warp < 2 + kSoftWarps) {
        // ------------------------------------------------------------ softmax + epilogue
        // Warp w owns TMEM lane quarter (w % 4) and the 16 heads of head quarter
        // (w - 2) / 4.  S^T rows (M = 64) sit in lanes 0..15 of each quarter:
        // row = 16 * quarter + lane.  O^T rows (dims, M = 128) fill all lanes.
        const int sw = warp - 2;                 // 0..15
        const int tid = threadIdx.x - 64;        // 0..511
        const int quarter = warp & 3;
        const int h0 = (sw >> 2) * kHW;
        const bool row_lane = lane < 16;
        const int row = quarter * 16 + (lane & 15);  // tile row of this lane (lanes 0..15)
        const int dim = quarter * 32 + lane;         // O^T lane: dim within a 128-dim slice
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;

        // q' = RoPE(RMSNorm(q), i) of query qi into sQ (bf16, 128-byte
        // swizzle).  The raw rows are loaded into sQ by TMA (q_raw): by warp 0
        // for the CTA's first query, by this role for every later one as soon
        // as the QK products of the query before are done (its rows were
        // prefetched into L2 when that query's segment started); they are
        // normalised and rotated in place.  Lane l of a warp holds dims
        // 16l .. 16l+15 of a head: two 16-byte chunks of box l/4 of that
        // head's 128-byte row.
        uint32_t qraw_issued = next_live_query<kLean>(a, g_begin, g_end) >= 0 ? 1u : 0u, qraw_done = 0;
        auto load_q = [&](int64_t qi) {  // by one thread
            tc::mbar_arrive_expect_tx(&q_raw, kQBytes);
            for (int bx = 0; bx < 8; bx++)
                tc::tma_load_3d(sQ + bx * kQBoxBytes, &tm_q, &q_raw, bx * 64, 0, (int)qi);
        };
        auto prep_q = [&](int64_t qi) {
            constexpr int kHq = kH / kSoftWarps;  // heads of this warp
            const int64_t i = a.q_pos[qi];
            const int ch = (lane & 3) * 2;
            // this lane's chunk c (0, 1) of head h in sQ
            uint8_t* const qbase = sQ + (lane >> 2) * kQBoxBytes;
#define QCHUNK(h, c) reinterpret_cast<uint4*>(qbase + (h) * 128 + (((ch + (c)) ^ ((h) & 7)) << 4))
            if (tid < 32) {
                float c, s;
                rope_cs((double)i, a.theta.t[tid], &c, &s);
                rot_cs[2 * tid] = c;
                rot_cs[2 * tid + 1] = s;
            }
            const bool ok = warp_wait(&q_raw, qraw_done & 1u, abort_flag, a.status, lane);
            if (ok) ++qraw_done;
            softmax_barrier();
            if (ok) {
#pragma unroll 1
                for (int hh = 0; hh < kHq; hh++) {
                    const int h = sw * kHq + hh;
                    const uint4 u0 = *QCHUNK(h, 0), u1 = *QCHUNK(h, 1);
                    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                    float x[16];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        x[2 * e] = __uint_as_float(w[e] << 16);
                        x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
                    }
                    float ss = 0.f;
#pragma unroll
                    for (int e = 0; e < 16; e++) ss = fmaf(x[e], x[e], ss);
                    ss = warp_sum(ss);
                    const float r = 1.f / sqrtf(ss / (float)kD + a.eps);
#pragma unroll
                    for (int e = 0; e < 16; e++) x[e] *= r;
                    if (lane >= 28) {  // dims 448..511: the rotated ones
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            const int j = (lane - 28) * 8 + e;
                            const float c = rot_cs[2 * j], s = rot_cs[2 * j + 1];
                            const float x0 = x[2 * e], x1 = x[2 * e + 1];
                            x[2 * e] = x0 * c - x1 * s;
                            x[2 * e + 1] = x0 * s + x1 * c;
                        }
                    }
                    *QCHUNK(h, 0) = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                              pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
                    *QCHUNK(h, 1) = make_uint4(pack_bf16x2(x[8], x[9]), pack_bf16x2(x[10], x[11]),
                                              pack_bf16x2(x[12], x[13]), pack_bf16x2(x[14], x[15]));
                }
            }
#undef QCHUNK
            tc::fence_proxy_async_smem();
            softmax_barrier();
            if (tid == 0) tc::mbar_arrive(&q_full);
        };


        {
            const int64_t q0 = next_live_query<kLean>(a, g_begin, g_end);
            if (q0 >= 0) prep_q(q0);
        }
        uint32_t tcount = 0, nseg = 0;
        bool stop = false;
        float l_part[kHW];
        const float* mref = mref_s + h0;  // running reference of this warp's heads (valid once ref_set)
        for (int64_t g = g_begin; g < g_end && !stop;) {
            const int64_t qi = idiv(g, a.T);
            const int64_t seg_end = seg_end_of<kLean>(a, g, g_end);
            const QueryInfo inf = query_info(a, qi);
            const int lt0 = (int)(g - qi * a.T), lt1 = (int)(seg_end - qi * a.T);
            const int lt_last = last_live<kLean>(a, inf, lt0, lt1);
            if (tid == 0 && blocks_of(inf.i, a.m) > a.n_cap) atomicOr(a.status, CSA_DEV_BAD_POSITION);
            // the next query's q rows head for L2 while this segment runs
            const int64_t qn = next_live_query<kLean>(a, seg_end, g_end);
            const bool q_next = qn >= 0 && qn != qi;  // a further split of this query keeps q'
            if (q_next) prefetch_l2(a.q + (qn * kH + sw * (kH / kSoftWarps) + (lane >> 3)) * kD + (lane & 7) * 64);
#pragma unroll
            for (int h = 0; h < kHW; h++) l_part[h] = 0.f;
            int seg_tiles = 0;
            bool ref_set = false;  // mref_s holds this segment's reference
            for (int lt = lt0; lt <= lt_last; ++lt) {
                if (!tile_live<kLean>(a, inf, lt)) continue;
                const int b = tcount & 1;
                // row validity (and the device-side checks of the row list)
                bool valid = false;
                const bool report = row_lane && sw < 4;
                if (row_lane) {
                    if (lt < a.T_sel) {
                        const int p = lt * kRows + row;
                        if (a.topk_idx) {
                            if (p < a.k) {
                                const int64_t e = a.topk_idx[qi * a.k + p];
                                if (e >= 0) {
                                    if (e < inf.n_av) valid = true;
                                    else if (report) atomicOr(a.status, CSA_DEV_BAD_TOPK_INDEX);
                                }
                            }
                        } else {
                            valid = p < inf.n_av;
                        }
                    } else {
                        const int r = (lt - a.T_sel) * kRows + row;
                        if (kLean || a.win_pos0 == nullptr) {  // ring row r: valid when its position is in the window
                            const int64_t wpos = r < a.n_win ? ring_pos(inf.i, r, a.n_win) : -1;
                            valid = wpos >= 0 && wpos >= inf.i - a.W + 1;
                        } else {
                            const int64_t wpos = inf.i - a.W + 1 + r;
                            if (r < a.W && wpos >= 0) {
                                const int64_t wr = wpos - a.win_pos0[inf.seq];
                                if (wr >= 0 && wr < a.n_win) valid = true;
                                else if (report) atomicOr(a.status, CSA_DEV_BAD_WINDOW);
                            }
                        }
                    }
                }
                const float mask = valid ? 0.f : -INFINITY;  // x = s * scale + mask
                const bool ok = warp_wait(&s_full[b], (tcount >> 1) & 1u, abort_flag, a.status, lane);
                // the segment's QK products are all done: the next query's raw
                // rows may replace q' in sQ while this tile's softmax runs
                if (ok && lt == lt_last && q_next && tid == 0) {
                    load_q(qn);
                    ++qraw_issued;
                }
                float x[kHW];
                bool need = false;
                if (ok) {
                    tc::fence_after_sync();
                    tc::tmem_ld16(tmem + lane_off + kColS + 64 * b + h0, x);
                    tc::tmem_ld_wait();
                    need = !ref_set;  // the first tile of a segment sets the reference
#pragma unroll
                    for (int h = 0; h < kHW; h++) {
                        x[h] = fmaf(x[h], a.scale_log2, mask);
                        if (ref_set) need |= x[h] > mref[h] + kRescaleLog2;
                    }
                }
                // one barrier per tile: leave together on a failed wait, and
                // raise the running reference when any logit outgrew it
                if (softmax_barrier_or(!ok || need)) {
                    if (softmax_barrier_or(!ok)) { stop = true; break; }
                    // tile maximum per head (over this quarter's rows), then over quarters
                    const float mx = warp_reduce_scatter16<true>(x, lane);
                    if (row_lane) red[quarter][h0 + lane] = mx;
                    softmax_barrier();
                    bool mine = false;
                    if (tid < kH) {
                        const float tm = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
                        float mn = ref_set ? mref_s[tid] : kNoRef;
                        float al = 1.f;
                        if (tm > mn + kRescaleLog2) {
                            al = (mn == kNoRef) ? 0.f : ex2_approx(mn - tm);
                            mine = mn != kNoRef;
                            mn = tm;
                        }
                        mref_s[tid] = mn;
                        alph_s[tid] = al;
                    }
                    const bool resc = softmax_barrier_or(mine);
                    ref_set = true;
                    if (resc) {
#pragma unroll
                        for (int h = 0; h < kHW; h++) l_part[h] *= alph_s[h0 + h];
                        // O^T holds this segment's earlier tiles: once the previous
                        // PV product is done, rescale this warp's block of it
                        const bool okr = warp_wait(&o_full, (tcount - 1u) & 1u, abort_flag, a.status, lane);
                        if (softmax_barrier_or(!okr)) { stop = true; break; }
                        tc::fence_after_sync();
                        for (int c = 0; c < 4; c++) {
                            float r[kHW];
                            tc::tmem_ld16(tmem + lane_off + kColO + 64 * c + h0, r);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int h = 0; h < kHW; h++) r[h] *= alph_s[h0 + h];
                            tc::tmem_st16(tmem + lane_off + kColO + 64 * c + h0, r);
                        }
                        tc::tmem_st_wait();
                    }
                }
                // P row (bf16) into the MN-major B operand, 128-byte swizzle:
                // this warp writes bytes 32*(w-2)/4 .. +31 of its rows
                if (row_lane) {
                    uint8_t* prow = sP + b * kPBytes + row * 128;
#pragma unroll
                    for (int ch = 0; ch < 2; ch++) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int h = ch * 8 + 2 * e;
                            w[e] = pack_bf16x2(ex2_approx(x[h] - mref[h]), ex2_approx(x[h + 1] - mref[h + 1]));
                            l_part[h] += __uint_as_float(w[e] << 16);
                            l_part[h + 1] += __uint_as_float(w[e] & 0xffff0000u);
                        }
                        const int chunk = 2 * (sw >> 2) + ch;
                        *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&p_full[b]);
                ++seg_tiles;
                ++tcount;
                if (lt == lt_last && q_next) prep_q(qn);
            }
            if (stop) break;
            // ---------------------------------------------------- segment epilogue
            // partial slot: the split's index, or the CTA's rank among those
            // meeting the query; a query no other CTA meets is finished here
            // (never with fixed splits: their merge order is the same in any batch)
            const int seg = kLean ? 0 : a.seg;
            const int64_t c_first = seg ? 0 : cta_of(a, qi * a.T);
            const int64_t c_last = seg ? 0 : cta_of(a, (qi + 1) * a.T - 1);
            const int64_t slot = seg ? idiv(lt0, seg) : (int64_t)blockIdx.x - c_first;
            const bool whole = !seg && c_first == c_last;
            // the CTA holding the query's first tile tells the combine how many partials it has
            if (a.nslots && lt0 == 0 && tid == 0) a.nslots[qi] = whole ? 0 : (int32_t)(c_last - c_first + 1);
            {
                const float ls = warp_reduce_scatter16<false>(l_part, lane);
                if (row_lane) red[quarter][h0 + lane] = ls;
            }
            softmax_barrier();
            if (tid < kH) {
                const float l = (red[0][tid] + red[1][tid]) + (red[2][tid] + red[3][tid]);
                const float mr = ref_set ? mref_s[tid] : kNoRef;
                const float m = (mr == kNoRef || l == 0.f) ? -INFINITY : mr * kLn2;
                if (whole) {
                    // merge with the sink here: out = o / (l + e^(sink - m)), lse
                    const float sk = a.sink[tid];
                    const float ms = fmaxf(m, sk);
                    float L = 0.f, f = 0.f;
                    if (ms != -INFINITY) {
                        const float em = (m == -INFINITY) ? 0.f : expf(m - ms);
                        L = l * em + ((sk == -INFINITY) ? 0.f : expf(sk - ms));
                        f = L > 0.f ? em / L : 0.f;
                    }
                    fac_s[tid] = f;
                    if (a.lse) a.lse[qi * kH + tid] = L > 0.f ? ms + logf(L) : -INFINITY;
                } else {
                    const int64_t pb = (qi * a.S + slot) * kH + tid;
                    a.part_ml[pb * 2] = m;
                    a.part_ml[pb * 2 + 1] = l;
                }
            }
            if (whole && a.derotate && tid < 32) {
                float c, s;
                rope_cs((double)inf.i, a.theta.t[tid], &c, &s);
                rot_cs[2 * tid] = c;
                rot_cs[2 * tid + 1] = s;
            }
            bool okw = true;
            if (seg_tiles > 0) okw = warp_wait(&o_seg, (nseg++) & 1u, abort_flag, a.status, lane);
            if (softmax_barrier_or(!okw)) { stop = true; break; }  // also publishes fac_s, rot_cs
            tc::fence_after_sync();
            for (int c = 0; c < 4; c++) {
                const int d = c * 128 + dim;
                float v[kHW];
                if (seg_tiles > 0) {
                    tc::tmem_ld16(tmem + lane_off + kColO + 64 * c + h0, v);
                    tc::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int h = 0; h < kHW; h++) v[h] = 0.f;
                }
                if (whole) {
#pragma unroll
                    for (int h = 0; h < kHW; h++) v[h] *= fac_s[h0 + h];
                    if (a.derotate && c == 3 && dim >= 128 - kRopeDims) {  // uniform per warp
                        // RoPE at -i on dims 448..511: pairs (d, d+1) sit on adjacent lanes
                        const int j = (dim - (128 - kRopeDims)) >> 1;
                        const float cs = rot_cs[2 * j], sn = rot_cs[2 * j + 1];
                        const bool odd = dim & 1;
#pragma unroll
                        for (int h = 0; h < kHW; h++) {
                            const float other = __shfl_xor_sync(0xffffffffu, v[h], 1);
                            v[h] = odd ? (v[h] * cs - other * sn) : (v[h] * cs + other * sn);
                        }
                    }
                    uint16_t* dst = a.out + (qi * kH + h0) * kD + d;
#pragma unroll
                    for (int h = 0; h < kHW; h++) dst[(int64_t)h * kD] = f32_to_bf16_rn(v[h]);
                } else {
                    float* dst = a.part_o + ((qi * a.S + slot) * kH + h0) * kD + d;
#pragma unroll
                    for (int h = 0; h < kHW; h++) dst[(int64_t)h * kD] = v[h];
                }
            }
            tc::fence_before_sync();
            softmax_barrier();  // red[], fac_s[], rot_cs[] are free again
            g = seg_end;
        }
        // leave no copy of q rows in flight (a wait that gave up left one)
        if (tid == 0 && qraw_issued > qraw_done && !tc::mbar_drain(&q_raw, (qraw_issued - 1u) & 1u))
            atomicOr(a.status, CSA_DEV_TIMEOUT);
    } else if (warp < 2 + kSoftWarps + kLoadWarps) {
        // ------------------------------------------------------------ gathers
        // The gathered tiles (selected rows) are fetched with TMA gather4 by
        // the gather warps, each its own boxes of every row; the producer
        // warp, which waits for every use of a stage in order, arms the
        // stage's full barrier with the tile's bytes and hands it over
        // through go[stage].
        const int lw = warp - 2 - kSoftWarps;
        // Cursor over this CTA's gathered tiles; the indices of the next one
        // are read while the current one waits for its stage.
        uint32_t tcount = 0, ngo[kStages] = {0, 0};
        int64_t g = g_begin;
        auto next_gathered = [&](int64_t& qi, int& lt, int& st) -> bool {
            for (; g < g_end; ++g) {
                qi = idiv(g, a.T);
                lt = (int)(g - qi * a.T);
                const QueryInfo inf = query_info(a, qi);
                if (!tile_live<kLean>(a, inf, lt)) continue;
                st = tcount & 1;
                ++tcount;
                if (is_gathered<kLean>(a, lt)) {
                    ++g;
                    return true;
                }
            }
            return false;
        };
        int64_t qi = 0;
        int lt = 0, st = 0;
        int rows[4];
        bool have = next_gathered(qi, lt, st);
        if (have) gather_rows(a, qi, query_info(a, qi), lt, lane, rows);
        while (have) {
            int64_t qi_n = 0;
            int lt_n = 0, st_n = 0;
            int rows_n[4];
            const bool have_n = next_gathered(qi_n, lt_n, st_n);
            if (have_n) gather_rows(a, qi_n, query_info(a, qi_n), lt_n, lane, rows_n);
            if (!warp_wait(&go[st], (ngo[st]++) & 1u, abort_flag, a.status, lane)) break;
            gather_boxes(&tm_sel, &full[st], sE + st * kStageBytes, rows, lw * kLoaderBoxes, kLoaderBoxes, lane);
            have = have_n;
            qi = qi_n;
            lt = lt_n;
            st = st_n;
#pragma unroll
            for (int j = 0; j < 4; j++) rows[j] = rows_n[j];
        }
    }
    // ---------------------------------------------------------------- teardown
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
bool attend_tc_supported(const Geometry& g, bool sparse, int H, int64_t n_cap, int64_t n_win) {
    if (g.act != CSA_BF16 || (g.kv != CSA_BF16 && g.kv != CSA_FP8_MIXED)) return false;
    if (g.D != kD || g.R != 64 || H != kH) return false;
    if (!sparse && n_cap < kRows) return false;     // tile boxes of 64 rows
    if (sparse && (n_cap < 1 || g.k < 1)) return false;
    if (g.W > 0 && n_win < kRows) return false;
    return true;
}

bool plan_attend_tc(const Geometry& g, bool sparse, int Q, int64_t n_cap, int64_t n_win, bool ring, AttendPlan* pl) {
    pl->tc_T_sel = sparse ? (g.k + kRows - 1) / kRows : (int)((n_cap + (int64_t)kRows - 1) / kRows);
    const int64_t win_rows = g.W > 0 ? (ring ? n_win : (int64_t)g.W) : 0;
    const int64_t T = pl->tc_T_sel + (win_rows + kRows - 1) / kRows;
    // the kernel's tile, unit and split indices are 32-bit
    if ((int64_t)Q * (T + kQueryCostTiles) >= (1LL << 31)) return false;
    pl->tc_T = (int)T;
    pl->tc_total = (int64_t)Q * pl->tc_T;
    const int64_t sms = num_sms();
    if (g.inv) {  // fixed splits of tc_seg tiles, whole splits per CTA
        pl->tc_seg = inv_split_tiles(pl->tc_T);
        pl->tc_nseg = (pl->tc_T + pl->tc_seg - 1) / pl->tc_seg;
        const int64_t segs = (int64_t)Q * pl->tc_nseg;
        pl->tc_grid = (int)(segs < sms ? segs : sms);
        pl->splits = pl->tc_nseg;
        return true;
    }
    pl->tc_grid = (int)(pl->tc_total < sms ? pl->tc_total : sms);
    pl->tc_qcta = pl->tc_qrem = 0;
    // with no more queries than CTAs, a query's start counts as
    // kQueryCostTiles more tiles (where every CTA's share still holds a
    // tile); with more, every CTA starts about as many queries as another
    pl->tc_qc = 0;
    if (pl->tc_total > 0 && Q <= pl->tc_grid &&
        (int64_t)Q * (pl->tc_T + kQueryCostTiles) / pl->tc_grid >= kQueryCostTiles + 1)
        pl->tc_qc = kQueryCostTiles;
    int smax = 1;
    if (pl->tc_total > 0) {
        const TileDeal deal{pl->tc_total, (int64_t)pl->tc_T, pl->tc_grid, 0, 0, pl->tc_qc};
        for (int64_t q = 0; q < Q; q++) {
            int n = (int)(deal.cta_of((q + 1) * pl->tc_T - 1) - deal.cta_of(q * pl->tc_T) + 1);
            if (n > smax) smax = n;
        }
    }
    pl->splits = smax;
    return true;
}

// Query-aligned ranges (TileDeal) for gathered tiles when there are no more
// queries than SMs: a CTA that met two queries would load the second q
// behind the first one's gathers in its TMA queue (~8 us at 128K context),
// and the slowest CTA sets the kernel's time.  Lists of TMA tiles keep the
// balanced ranges (measured: HCA decode 120.8 -> 123.9 us aligned).
void plan_attend_tc_aligned(int Q, AttendPlan* pl) {
    const int64_t sms = num_sms();
    if (pl->tc_seg != 0 || Q < 1 || Q > sms || pl->tc_T < 2) return;
    const int64_t per = sms / Q;
    pl->tc_qcta = (int)(per < pl->tc_T ? per : pl->tc_T);
    pl->tc_qrem = pl->tc_qcta < pl->tc_T ? (int)(sms - (int64_t)Q * pl->tc_qcta) : 0;
    pl->tc_qc = 0;
    pl->tc_grid = Q * pl->tc_qcta + pl->tc_qrem;
    pl->splits = pl->tc_qcta + (pl->tc_qrem > 0 ? 1 : 0);
}

cudaError_t launch_attend_tc(const Geometry& g, const AttendPlan& pl, bool sparse, const void* q,
                             int H, int B, int Q, const int64_t* q_pos, const void* cache,
                             int64_t n_cap, const int32_t* topk_idx, const void* window,
                             int64_t n_win, const int64_t* win_pos0, const float* sink,
                             void* out, float* lse, float* part_o, float* part_ml, int32_t* nslots,
                             uint8_t* deq, uint32_t* status, cudaStream_t st) {
    (void)H;
    if (pl.tc_total == 0) return cudaSuccess;
    const int64_t rb = g.kv_row_bytes;
    CUtensorMap tm_sel, tm_win;
    uint16_t* deq_rows = reinterpret_cast<uint16_t*>(deq);
    if (pl.tc_deq == 1) {
        DeqGatherArgs d;
        d.cache = reinterpret_cast<const uint8_t*>(cache);
        d.window = reinterpret_cast<const uint8_t*>(window);
        d.rb = rb;
        d.n_cap = n_cap;
        d.n_win = n_win;
        d.q_pos = q_pos;
        d.win_pos0 = win_pos0;
        d.topk_idx = sparse ? topk_idx : nullptr;
        d.k = g.k;
        d.W = g.W;
        d.m = g.m;
        d.qps = Q / B;
        d.T_sel = pl.tc_T_sel;
        d.T = pl.tc_T;
        d.rows = (int64_t)Q * pl.tc_T * kRows;
        d.out = deq_rows;
        const int64_t blocks = (d.rows + kDeqThreads / 32 - 1) / (kDeqThreads / 32);
        dequant_gather_kernel<<<(unsigned)blocks, kDeqThreads, 0, st>>>(d);
        note_launch();
        const uint64_t dm[3] = {(uint64_t)kD, (uint64_t)pl.tc_T * kRows, (uint64_t)Q};
        const uint64_t sd[2] = {(uint64_t)kD * 2, (uint64_t)pl.tc_T * kRows * kD * 2};
        const uint32_t box[3] = {64, (uint32_t)kRows, 1};
        if (!make_tmap_bf16(&tm_sel, deq_rows, 3, dm, sd, box)) return cudaErrorInvalidValue;
        tm_win = tm_sel;  // never read
    } else {
        if (pl.tc_deq == 2) {  // every stored row, then the bf16 copies stand in for the rows
            const int64_t n_rows[2] = {(int64_t)B * n_cap, g.W > 0 ? (int64_t)B * n_win : 0};
            const void* src[2] = {cache, window};
            uint16_t* dst[2] = {deq_rows, deq_rows + n_rows[0] * kD};
            for (int j = 0; j < 2; j++) {
                if (n_rows[j] == 0) continue;
                const int64_t blocks = (n_rows[j] + kDeqThreads / 32 - 1) / (kDeqThreads / 32);
                dequant_rows_kernel<<<(unsigned)blocks, kDeqThreads, 0, st>>>(
                    reinterpret_cast<const uint8_t*>(src[j]), rb, n_rows[j], dst[j]);
                note_launch();
            }
            cache = dst[0];
            window = dst[1];
        }
        if (sparse) {
            const uint64_t d[2] = {(uint64_t)kD, (uint64_t)B * (uint64_t)n_cap};
            const uint64_t s[1] = {(uint64_t)kD * 2};
            const uint32_t box[2] = {64, 1};
            if (!make_tmap_bf16(&tm_sel, cache, 2, d, s, box)) return cudaErrorInvalidValue;
        } else {
            const uint64_t d[3] = {(uint64_t)kD, (uint64_t)n_cap, (uint64_t)B};
            const uint64_t s[2] = {(uint64_t)kD * 2, (uint64_t)n_cap * kD * 2};
            const uint32_t box[3] = {64, (uint32_t)kRows, 1};
            if (!make_tmap_bf16(&tm_sel, cache, 3, d, s, box)) return cudaErrorInvalidValue;
        }
        if (g.W > 0) {
            const uint64_t d[3] = {(uint64_t)kD, (uint64_t)n_win, (uint64_t)B};
            const uint64_t s[2] = {(uint64_t)kD * 2, (uint64_t)n_win * kD * 2};
            const uint32_t box[3] = {64, (uint32_t)kRows, 1};
            if (!make_tmap_bf16(&tm_win, window, 3, d, s, box)) return cudaErrorInvalidValue;
        } else {
            tm_win = tm_sel;  // never read
        }
    }
    AttTcArgs a;
    a.q = reinterpret_cast<const uint16_t*>(q);
    a.q_pos = q_pos;
    a.topk_idx = sparse ? topk_idx : nullptr;
    a.k = g.k;
    a.pre = pl.tc_deq == 1 ? 1 : 0;
    a.cache = reinterpret_cast<const uint8_t*>(cache);
    a.n_cap = n_cap;
    a.n_win = n_win;
    a.win_pos0 = win_pos0;
    a.W = g.W;
    a.m = g.m;
    a.qps = Q / B;
    a.eps = g.eps;
    a.scale_log2 = g.scale * kLog2e;
    a.T_sel = pl.tc_T_sel;
    a.T = pl.tc_T;
    a.total = pl.tc_total;
    a.grid = pl.tc_grid;
    a.qcta = pl.tc_qcta;
    a.qrem = pl.tc_qrem;
    a.qc = pl.tc_qc;
    a.seg = pl.tc_seg;
    a.nseg = pl.tc_nseg;
    a.S = pl.splits;
    a.part_o = part_o;
    a.part_ml = part_ml;
    a.nslots = nslots;
    a.sink = sink;
    a.out = reinterpret_cast<uint16_t*>(out);
    a.lse = lse;
    a.derotate = g.derotate;
    a.status = status;
    a.theta = rope_theta(g);
    {
        cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(attend_tc_kernel<true, true>), kSmem);
        if (e == cudaSuccess) e = set_smem_attr(reinterpret_cast<const void*>(attend_tc_kernel<true, false>), kSmem);
        if (e == cudaSuccess) e = set_smem_attr(reinterpret_cast<const void*>(attend_tc_kernel<false, true>), kSmem);
        if (e == cudaSuccess) e = set_smem_attr(reinterpret_cast<const void*>(attend_tc_kernel<false, false>), kSmem);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tm_q;
    {
        const uint64_t d[3] = {(uint64_t)kD, (uint64_t)kH, (uint64_t)Q};
        const uint64_t sd[2] = {(uint64_t)kD * 2, (uint64_t)kH * kD * 2};
        const uint32_t box[3] = {64, (uint32_t)kH, 1};
        if (!make_tmap_bf16(&tm_q, q, 3, d, sd, box)) return cudaErrorInvalidValue;
    }
    // the split issue layout where no tile is gathered; the lean build
    // where there are no fixed splits, no pre-gathered rows and the window
    // (if any) is a ring
    const bool split = a.pre || a.topk_idx == nullptr;
    const bool lean = a.seg == 0 && !a.pre && a.win_pos0 == nullptr;
    const dim3 grid(pl.tc_grid);
    cudaError_t e;
    if (split)
        e = lean ? launch_dependent(attend_tc_kernel<true, true>, grid, dim3(Roles<true>::kThreads), kSmem, st,
                                    tm_sel, tm_win, tm_q, a)
                 : launch_dependent(attend_tc_kernel<true, false>, grid, dim3(Roles<true>::kThreads), kSmem, st,
                                    tm_sel, tm_win, tm_q, a);
    else
        e = lean ? launch_dependent(attend_tc_kernel<false, true>, grid, dim3(Roles<false>::kThreads), kSmem, st,
                                    tm_sel, tm_win, tm_q, a)
                 : launch_dependent(attend_tc_kernel<false, false>, grid, dim3(Roles<false>::kThreads), kSmem, st,
                                    tm_sel, tm_win, tm_q, a);
    note_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csa
