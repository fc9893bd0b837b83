// k_attend_tc.cu -- CSA / HCA core attention on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), bf16 rows of 512 dims, 64 query heads.
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2: CSA Step 3 (multi-query attention
// over the top-k compressed blocks), HCA (dense attention over every block),
// and 四项关键 Trick: RMSNorm and partial RoPE on q, a sliding window of the
// last W raw tokens, a learnable sink in the softmax denominator.
//
// One query's row list is cut into tiles of 128 rows: ceil(k/128) tiles of
// selected blocks (CSA, gathered row by row with TMA gather4) or
// ceil(n_cap/128) tiles of consecutive blocks (HCA, TMA tiles), then
// ceil(W/128) window tiles.  The (query, tile) pairs are dealt out in
// contiguous, balanced ranges to one persistent CTA per SM; the run of one
// query's tiles inside a CTA is a segment, reduced to an unnormalised partial
// (m, l, o) that attend_combine_kernel merges with the sink.
//
// Per tile (one shared KV head, so key = value = row e_j):
//   S^T[128 rows, 64 heads] = E[128, 512] . Q'^T          (swap-AB: rows are M)
//   P = 2^(S^T * scale * log2 e - m)  (bf16, per head running reference m)
//   O^T[512, 64] += E^T[512, 128] . P^T                    (4 MMAs of M = 128)
// The tile stays in shared memory (4 slices of 128 rows x 128 dims, 128-byte
// swizzle) between the two products: E is the K-major A operand of the first
// and, read along its rows, the MN-major A operand of the second.  A slice is
// refilled with the next tile as soon as its PV product is done.  The running
// reference m is raised only when a tile's maximum exceeds it by more than
// 2^8; O^T (in TMEM) and the partial sums are then rescaled in place.
//
// Warp roles: warp 0 loads (TMA), warp 1 issues MMAs, warps 2..5 normalise
// and rotate q, run the softmax and write the partials.  Every wait is
// bounded; on a timeout the kernel sets CSA_DEV_TIMEOUT, every role leaves its
// loop, outstanding copies and MMAs are waited for and TMEM is freed.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa {

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

namespace {

constexpr int kD = 512;
constexpr int kH = 64;
constexpr int kRows = 128;
constexpr int kSlices = 4;                          // 128-dim slices of a tile
constexpr uint32_t kBoxBytes = kRows * 128;         // 128 rows x 64 dims (bf16)
constexpr uint32_t kSliceBytes = 2 * kBoxBytes;     // 128 rows x 128 dims
constexpr uint32_t kQBoxBytes = kH * 128;           // 64 heads x 64 dims
constexpr uint32_t kQBytes = 8 * kQBoxBytes;        // 64 heads x 512 dims
constexpr uint32_t kPBytes = kRows * kH * 2;        // 128 rows x 64 heads
constexpr size_t kSmem = 1024 + kSlices * kSliceBytes + kQBytes + kPBytes;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S^T: 64 columns
constexpr uint32_t kColO = 256;  // O^T: 4 x 64 columns
constexpr float kRescaleLog2 = 8.f;
constexpr int kBarSoftmax = 1;   // named barrier of the 4 softmax warps

struct AttTcArgs {
    const uint16_t* q;        // [Q, 64, 512] bf16
    const int64_t* q_pos;     // [Q]
    const int32_t* topk_idx;  // [Q, k]; nullptr: dense (HCA)
    int k;
    int64_t n_cap, n_win;
    const int64_t* win_pos0;  // [B]
    int W, m, qps;
    double base;
    float eps, scale_log2;
    int T_sel, T;             // tiles per query: selected / cache part, all
    int64_t total;            // Q * T
    int grid;
    int S;                    // partial slots per query
    float* part_o;            // [Q, S, 64, 512]
    float* part_ml;           // [Q, S, 64, 2]
    uint32_t* status;
};

// CTA that owns global tile g (CTA c owns [c*total/grid, (c+1)*total/grid)).
__device__ __forceinline__ int64_t cta_of(const AttTcArgs& a, int64_t g) {
    return ((g + 1) * a.grid - 1) / a.total;
}

struct QueryInfo {
    int64_t i, n_av;
    int seq;
};

__device__ __forceinline__ QueryInfo query_info(const AttTcArgs& a, int64_t qi) {
    QueryInfo r;
    r.i = a.q_pos[qi];
    r.seq = (int)(qi / a.qps);
    int64_t n = (r.i + 1) / a.m;
    if (n < 0) n = 0;
    r.n_av = n < a.n_cap ? n : a.n_cap;  // an overflow is flagged by the softmax warps
    return r;
}

// Whether tile lt of a query has any row that can be valid.  Every role
// evaluates the same predicate, so skipped tiles cost nothing anywhere.
__device__ __forceinline__ bool tile_live(const AttTcArgs& a, const QueryInfo& qi, int lt) {
    if (lt < a.T_sel) {
        if (a.topk_idx) return qi.n_av > 0;
        return (int64_t)lt * kRows < qi.n_av;
    }
    const int r0 = (lt - a.T_sel) * kRows;
    if (r0 >= a.W) return false;
    const int rlast = min(a.W, r0 + kRows) - 1;
    return qi.i - a.W + 1 + rlast >= 0;
}

// Last live tile of the segment [lt0, lt1) of a query, or -1.
__device__ __forceinline__ int last_live(const AttTcArgs& a, const QueryInfo& qi, int lt0, int lt1) {
    for (int lt = lt1 - 1; lt >= lt0; --lt)
        if (tile_live(a, qi, lt)) return lt;
    return -1;
}

// -------------------------------------------------------------- softmax helpers
// Reduce-scatter 64 per-lane values over the warp: afterwards lane l holds the
// reduction of entries 2l and 2l+1 over all 32 lanes.
template <bool kMax>
__device__ __forceinline__ float2 warp_reduce_scatter64(const float (&v)[64], int lane) {
    auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
    float a[32], b[16], c[8], d[4], e[2];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int j = 0; j < 32; j++) {
            float keep = up ? v[j + 32] : v[j], send = up ? v[j] : v[j + 32];
            a[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
        }
    }
    {
        const bool up = lane & 8;
#pragma unroll
        for (int j = 0; j < 16; j++) {
            float keep = up ? a[j + 16] : a[j], send = up ? a[j] : a[j + 16];
            b[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
        }
    }
    {
        const bool up = lane & 4;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float keep = up ? b[j + 8] : b[j], send = up ? b[j] : b[j + 8];
            c[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
        }
    }
    {
        const bool up = lane & 2;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float keep = up ? c[j + 4] : c[j], send = up ? c[j] : c[j + 4];
            d[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
        }
    }
    {
        const bool up = lane & 1;
#pragma unroll
        for (int j = 0; j < 2; j++) {
            float keep = up ? d[j + 2] : d[j], send = up ? d[j] : d[j + 2];
            e[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 1));
        }
    }
    return make_float2(e[0], e[1]);
}

__device__ __forceinline__ bool softmax_barrier_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(kBarSoftmax)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void softmax_barrier() { tc::named_barrier(kBarSoftmax, 128); }

// Wait by lane 0, verdict shared with the warp (tcgen05.ld is warp-wide).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status, int lane) {
    int ok = 1;
    if (lane == 0) ok = tc::mbar_wait(bar, parity, abort_flag, status) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)f32_to_bf16_rn(lo) | ((uint32_t)f32_to_bf16_rn(hi) << 16);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tm_sel,
                     const __grid_constant__ CUtensorMap tm_win, AttTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sE = sm;                              // kSlices x kSliceBytes
    uint8_t* sQ = sE + kSlices * kSliceBytes;      // 8 boxes of 64 heads x 64 dims
    uint8_t* sP = sQ + kQBytes;                    // 128 rows x 64 heads

    __shared__ __align__(8) uint64_t full[kSlices], empty[kSlices];
    __shared__ __align__(8) uint64_t s_full, p_full, o_full, q_full, mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_sh;
    __shared__ float red[4][kH];
    __shared__ float mref[kH], alph[kH];
    __shared__ float rope_cs[64];
    volatile int* abort_flag = &abort_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlices; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(&s_full, 1);
        tc::mbar_init(&p_full, 4);
        tc::mbar_init(&o_full, 1);
        tc::mbar_init(&q_full, 1);
        tc::mbar_init(&mma_done, 1);
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

    const int64_t g_begin = (int64_t)blockIdx.x * a.total / a.grid;
    const int64_t g_end = (int64_t)(blockIdx.x + 1) * a.total / a.grid;

    if (warp == 0) {
        // ------------------------------------------------------------ loads
        if (lane == 0) {
            tc::tma_prefetch_map(&tm_sel);
            if (a.W > 0) tc::tma_prefetch_map(&tm_win);
        }
        uint32_t tcount = 0;
        uint32_t fills[kSlices] = {0, 0, 0, 0};  // loads issued into each slot
        for (int64_t g = g_begin; g < g_end && !*abort_flag;) {
            const int64_t qi = g / a.T;
            const int64_t seg_end = min(g_end, (qi + 1) * a.T);
            const QueryInfo inf = query_info(a, qi);
            bool stop = false;
            for (int lt = (int)(g - qi * a.T); lt < (int)(seg_end - qi * a.T); ++lt) {
                if (!tile_live(a, inf, lt)) continue;
                // gathered rows of this lane (CSA selected tiles): rows 4*lane .. 4*lane+3
                int rows[4] = {0, 0, 0, 0};
                const bool gather = lt < a.T_sel && a.topk_idx != nullptr;
                if (gather) {
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const int p = lt * kRows + 4 * lane + j;
                        int64_t e = p < a.k ? (int64_t)a.topk_idx[qi * a.k + p] : -1;
                        if (e < 0 || e >= inf.n_av) e = 0;  // masked by the softmax warps
                        rows[j] = (int)((int64_t)inf.seq * a.n_cap + e);
                    }
                }
                for (int c = 0; c < kSlices; c++) {
                    if (!warp_wait(&empty[c], (tcount & 1u) ^ 1u, abort_flag, a.status, lane)) {
                        stop = true;
                        break;
                    }
                    uint8_t* dst = sE + c * kSliceBytes;
                    if (lane == 0) tc::mbar_arrive_expect_tx(&full[c], kSliceBytes);
                    __syncwarp();
                    if (gather) {
#pragma unroll
                        for (int b = 0; b < 2; b++)
                            tc::tma_gather4(dst + b * kBoxBytes + lane * 512, &tm_sel, &full[c],
                                            c * 128 + b * 64, rows[0], rows[1], rows[2], rows[3]);
                    } else if (lane == 0) {
                        int row0;
                        const CUtensorMap* map;
                        if (lt < a.T_sel) {
                            map = &tm_sel;
                            row0 = lt * kRows;
                        } else {
                            map = &tm_win;
                            row0 = (int)(inf.i - a.W + 1 + (int64_t)(lt - a.T_sel) * kRows -
                                         a.win_pos0[inf.seq]);
                        }
#pragma unroll
                        for (int b = 0; b < 2; b++)
                            tc::tma_load_3d(dst + b * kBoxBytes, map, &full[c], c * 128 + b * 64, row0,
                                            inf.seq);
                    }
                    ++fills[c];
                }
                if (stop) break;
                ++tcount;
            }
            if (stop) break;
            g = seg_end;
        }
        // Leave no copy in flight: the newest load of every slot must have
        // landed (at most one phase of a slot is ever outstanding).
        if (lane == 0) {
            for (int c = 0; c < kSlices; c++) {
                if (fills[c] == 0) continue;
                if (!tc::mbar_drain(&full[c], (fills[c] - 1u) & 1u)) atomicOr(a.status, CSA_DEV_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, kH, 0, 0);
            constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, kH, 1, 1);
            const uint32_t sE0 = tc::smem_u32(sE), sQ0 = tc::smem_u32(sQ), sP0 = tc::smem_u32(sP);
            uint32_t tcount = 0, nq = 0;
            bool stop = false;
            for (int64_t g = g_begin; g < g_end && !stop;) {
                const int64_t qi = g / a.T;
                const int64_t seg_end = min(g_end, (qi + 1) * a.T);
                const QueryInfo inf = query_info(a, qi);
                bool first = true;
                for (int lt = (int)(g - qi * a.T); lt < (int)(seg_end - qi * a.T); ++lt) {
                    if (!tile_live(a, inf, lt)) continue;
                    if (first) {
                        if (!tc::mbar_wait(&q_full, nq & 1u, abort_flag, a.status)) { stop = true; break; }
                        ++nq;
                    }
                    // S^T = E . Q'^T over the 512 dims
                    for (int c = 0; c < kSlices && !stop; c++) {
                        if (!tc::mbar_wait(&full[c], tcount & 1u, abort_flag, a.status)) { stop = true; break; }
                        tc::fence_after_sync();
                        const uint32_t slice = sE0 + c * kSliceBytes;
#pragma unroll
                        for (int j = 0; j < 8; j++) {
                            const int kg = 8 * c + j;
                            const uint64_t ad = tc::sdesc_sw128(slice + (j >> 2) * kBoxBytes + (j & 3) * 32, 16, 1024);
                            const uint64_t bd = tc::sdesc_sw128(sQ0 + (kg >> 2) * kQBoxBytes + (kg & 3) * 32, 16, 1024);
                            tc::mma_bf16_ss(tmem + kColS, ad, bd, idesc_qk, (c | j) != 0 ? 1u : 0u);
                        }
                    }
                    if (stop) break;
                    tc::mma_commit(&s_full);
                    if (!tc::mbar_wait(&p_full, tcount & 1u, abort_flag, a.status)) { stop = true; break; }
                    tc::fence_after_sync();
                    // O^T += E^T . P^T, one 128-dim slice at a time
                    for (int c = 0; c < kSlices; c++) {
                        const uint32_t slice = sE0 + c * kSliceBytes;
#pragma unroll
                        for (int kk = 0; kk < 8; kk++) {
                            const uint64_t ad = tc::sdesc_sw128(slice + kk * 2048, kBoxBytes, 1024);
                            const uint64_t bd = tc::sdesc_sw128(sP0 + kk * 2048, kBoxBytes, 1024);
                            tc::mma_bf16_ss(tmem + kColO + 64 * c, ad, bd, idesc_pv,
                                            (first && kk == 0) ? 0u : 1u);
                        }
                        tc::mma_commit(&empty[c]);
                    }
                    tc::mma_commit(&o_full);
                    first = false;
                    ++tcount;
                }
                g = seg_end;
            }
            // every MMA issued so far must be complete before TMEM is freed
            tc::mma_commit(&mma_done);
            if (!tc::mbar_drain(&mma_done, 0)) atomicOr(a.status, CSA_DEV_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int sw = warp - 2;                 // 0..3
        const int tid = threadIdx.x - 64;        // 0..127
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;     // row of the tile / dim of an O^T slice
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float kLn2 = 0.6931471805599453f;

        // q' = RoPE(RMSNorm(q), i) of query qi into sQ (bf16, 128-byte swizzle)
        auto prep_q = [&](int64_t qi) {
            const int64_t i = a.q_pos[qi];
            if (tid < 32) {
                float c, s;
                rope_cos_sin((double)i, tid, kRopeDims, a.base, &c, &s);
                rope_cs[2 * tid] = c;
                rope_cs[2 * tid + 1] = s;
            }
            softmax_barrier();
            for (int hh = 0; hh < 16; hh++) {
                const int h = sw * 16 + hh;
                const uint4* src = reinterpret_cast<const uint4*>(a.q + (qi * kH + h) * kD) + lane * 2;
                const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
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
                        const float c = rope_cs[2 * j], s = rope_cs[2 * j + 1];
                        const float x0 = x[2 * e], x1 = x[2 * e + 1];
                        x[2 * e] = x0 * c - x1 * s;
                        x[2 * e + 1] = x0 * s + x1 * c;
                    }
                }
                uint4 o0, o1;
                o0.x = pack_bf16x2(x[0], x[1]);
                o0.y = pack_bf16x2(x[2], x[3]);
                o0.z = pack_bf16x2(x[4], x[5]);
                o0.w = pack_bf16x2(x[6], x[7]);
                o1.x = pack_bf16x2(x[8], x[9]);
                o1.y = pack_bf16x2(x[10], x[11]);
                o1.z = pack_bf16x2(x[12], x[13]);
                o1.w = pack_bf16x2(x[14], x[15]);
                uint8_t* base = sQ + (lane >> 2) * kQBoxBytes + h * 128;
                const int ch = (lane & 3) * 2;
                *reinterpret_cast<uint4*>(base + (((ch) ^ (h & 7)) << 4)) = o0;
                *reinterpret_cast<uint4*>(base + (((ch + 1) ^ (h & 7)) << 4)) = o1;
            }
            tc::fence_proxy_async_smem();
            softmax_barrier();
            if (tid == 0) tc::mbar_arrive(&q_full);
        };

        // the next segment (from global tile g) with a live tile, or -1
        auto next_live_query = [&](int64_t g) -> int64_t {
            while (g < g_end) {
                const int64_t qi = g / a.T;
                const int64_t seg_end = min(g_end, (qi + 1) * a.T);
                const QueryInfo inf = query_info(a, qi);
                if (last_live(a, inf, (int)(g - qi * a.T), (int)(seg_end - qi * a.T)) >= 0) return qi;
                g = seg_end;
            }
            return -1;
        };

        {
            const int64_t q0 = next_live_query(g_begin);
            if (q0 >= 0) prep_q(q0);
        }
        uint32_t tcount = 0;
        bool stop = false;
        float l_part[kH];
        for (int64_t g = g_begin; g < g_end && !stop;) {
            const int64_t qi = g / a.T;
            const int64_t seg_end = min(g_end, (qi + 1) * a.T);
            const QueryInfo inf = query_info(a, qi);
            const int lt0 = (int)(g - qi * a.T), lt1 = (int)(seg_end - qi * a.T);
            const int lt_last = last_live(a, inf, lt0, lt1);
            if (tid == 0 && (inf.i + 1) / a.m > a.n_cap) atomicOr(a.status, CSA_DEV_BAD_POSITION);
            if (tid < kH) mref[tid] = -INFINITY;
#pragma unroll
            for (int h = 0; h < kH; h++) l_part[h] = 0.f;
            int seg_tiles = 0;
            for (int lt = lt0; lt <= lt_last; ++lt) {
                if (!tile_live(a, inf, lt)) continue;
                // row validity (and the device-side checks of the row list)
                bool valid;
                if (lt < a.T_sel) {
                    const int p = lt * kRows + row;
                    if (a.topk_idx) {
                        valid = false;
                        if (p < a.k) {
                            const int64_t e = a.topk_idx[qi * a.k + p];
                            if (e >= 0) {
                                if (e < inf.n_av) valid = true;
                                else atomicOr(a.status, CSA_DEV_BAD_TOPK_INDEX);
                            }
                        }
                    } else {
                        valid = p < inf.n_av;
                    }
                } else {
                    const int r = (lt - a.T_sel) * kRows + row;
                    const int64_t wpos = inf.i - a.W + 1 + r;
                    valid = false;
                    if (r < a.W && wpos >= 0) {
                        const int64_t wr = wpos - a.win_pos0[inf.seq];
                        if (wr >= 0 && wr < a.n_win) valid = true;
                        else atomicOr(a.status, CSA_DEV_BAD_WINDOW);
                    }
                }
                // all four warps leave together, or none does (named barriers follow)
                if (softmax_barrier_or(!warp_wait(&s_full, tcount & 1u, abort_flag, a.status, lane))) {
                    stop = true;
                    break;
                }
                tc::fence_after_sync();
                float x[kH];
                {
                    uint32_t r[64];
                    tc::tmem_ld64(tmem + lane_off + kColS, r);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < kH; h++) x[h] = valid ? __uint_as_float(r[h]) * a.scale_log2 : -INFINITY;
                }
                // per-head maximum of the tile, then the running reference
                const float2 mx = warp_reduce_scatter64<true>(x, lane);
                red[sw][2 * lane] = mx.x;
                red[sw][2 * lane + 1] = mx.y;
                softmax_barrier();
                bool mine = false;
                if (tid < kH) {
                    const float tm = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
                    const float mo = mref[tid];
                    float al = 1.f;
                    if (tm > mo + kRescaleLog2) {
                        al = (mo == -INFINITY) ? 0.f : exp2f(mo - tm);
                        mine = mo != -INFINITY;
                        mref[tid] = tm;
                    }
                    alph[tid] = al;
                }
                const bool resc = softmax_barrier_or(mine);
                if (resc) {
#pragma unroll
                    for (int h = 0; h < kH; h++) l_part[h] *= alph[h];
                    if (seg_tiles > 0) {  // O^T holds this segment's earlier tiles
                        for (int c = 0; c < kSlices; c++) {
                            uint32_t r[64];
                            tc::tmem_ld64(tmem + lane_off + kColO + 64 * c, r);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int h = 0; h < kH; h++) r[h] = __float_as_uint(__uint_as_float(r[h]) * alph[h]);
                            tc::tmem_st64(tmem + lane_off + kColO + 64 * c, r);
                        }
                        tc::tmem_st_wait();
                    }
                }
                // P row (bf16) into the MN-major B operand, 128-byte swizzle
                uint8_t* prow = sP + row * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ch++) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int h = ch * 8 + 2 * e;
                        const float m0 = mref[h], m1 = mref[h + 1];
                        const float p0 = (m0 == -INFINITY) ? 0.f : exp2f(x[h] - m0);
                        const float p1 = (m1 == -INFINITY) ? 0.f : exp2f(x[h + 1] - m1);
                        w[e] = pack_bf16x2(p0, p1);
                        l_part[h] += __uint_as_float(w[e] << 16);
                        l_part[h + 1] += __uint_as_float(w[e] & 0xffff0000u);
                    }
                    *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&p_full);
                ++seg_tiles;
                ++tcount;
                if (lt == lt_last) {
                    // every QK product of this segment is done: q' of the next one may go in
                    const int64_t qn = next_live_query(seg_end);
                    if (qn >= 0) prep_q(qn);
                }
            }
            if (stop) break;
            // ---------------------------------------------------- segment epilogue
            const int64_t slot = (int64_t)blockIdx.x - cta_of(a, qi * a.T);
            const float2 ls = warp_reduce_scatter64<false>(l_part, lane);
            red[sw][2 * lane] = ls.x;
            red[sw][2 * lane + 1] = ls.y;
            softmax_barrier();
            const int64_t pbase = (qi * a.S + slot) * kH;
            if (tid < kH) {
                const float l = (red[0][tid] + red[1][tid]) + (red[2][tid] + red[3][tid]);
                const float mr = mref[tid];
                a.part_ml[(pbase + tid) * 2] = (mr == -INFINITY) ? -INFINITY : mr * kLn2;
                a.part_ml[(pbase + tid) * 2 + 1] = l;
            }
            if (seg_tiles > 0) {
                if (softmax_barrier_or(!warp_wait(&o_full, (tcount - 1u) & 1u, abort_flag, a.status, lane))) {
                    stop = true;
                    break;
                }
                tc::fence_after_sync();
                for (int c = 0; c < kSlices; c++) {
                    uint32_t r[64];
                    tc::tmem_ld64(tmem + lane_off + kColO + 64 * c, r);
                    tc::tmem_ld_wait();
                    float* dst = a.part_o + pbase * kD + c * 128 + row;
#pragma unroll
                    for (int h = 0; h < kH; h++) dst[(int64_t)h * kD] = __uint_as_float(r[h]);
                }
                tc::fence_before_sync();
            } else {
                for (int c = 0; c < kSlices; c++) {
                    float* dst = a.part_o + pbase * kD + c * 128 + row;
#pragma unroll 8
                    for (int h = 0; h < kH; h++) dst[(int64_t)h * kD] = 0.f;
                }
            }
            softmax_barrier();  // red[] and mref[] are free again
            g = seg_end;
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
    if (g.act != CSA_BF16 || g.kv != CSA_BF16 || g.D != kD || g.R != 64 || H != kH) return false;
    if (!sparse && n_cap < kRows) return false;     // tile boxes of 128 rows
    if (sparse && (n_cap < 1 || g.k < 1)) return false;
    if (g.W > 0 && n_win < kRows) return false;
    return true;
}

void plan_attend_tc(const Geometry& g, bool sparse, int Q, int64_t n_cap, AttendPlan* pl) {
    pl->tc_T_sel = sparse ? (g.k + kRows - 1) / kRows : (int)((n_cap + kRows - 1) / kRows);
    pl->tc_T = pl->tc_T_sel + (g.W + kRows - 1) / kRows;
    pl->tc_total = (int64_t)Q * pl->tc_T;
    const int64_t sms = num_sms();
    pl->tc_grid = (int)(pl->tc_total < sms ? pl->tc_total : sms);
    int smax = 1;
    if (pl->tc_total > 0) {
        auto cta = [&](int64_t t) { return ((t + 1) * pl->tc_grid - 1) / pl->tc_total; };
        for (int64_t q = 0; q < Q; q++) {
            int n = (int)(cta((q + 1) * pl->tc_T - 1) - cta(q * pl->tc_T) + 1);
            if (n > smax) smax = n;
        }
    }
    pl->splits = smax;
}

cudaError_t launch_attend_tc(const Geometry& g, const AttendPlan& pl, bool sparse, const void* q,
                             int H, int B, int Q, const int64_t* q_pos, const void* cache,
                             int64_t n_cap, const int32_t* topk_idx, const void* window,
                             int64_t n_win, const int64_t* win_pos0, float* part_o,
                             float* part_ml, uint32_t* status, cudaStream_t st) {
    (void)H;
    if (pl.tc_total == 0) return cudaSuccess;
    CUtensorMap tm_sel, tm_win;
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
    AttTcArgs a;
    a.q = reinterpret_cast<const uint16_t*>(q);
    a.q_pos = q_pos;
    a.topk_idx = sparse ? topk_idx : nullptr;
    a.k = g.k;
    a.n_cap = n_cap;
    a.n_win = n_win;
    a.win_pos0 = win_pos0;
    a.W = g.W;
    a.m = g.m;
    a.qps = Q / B;
    a.base = (double)g.base;
    a.eps = g.eps;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.T_sel = pl.tc_T_sel;
    a.T = pl.tc_T;
    a.total = pl.tc_total;
    a.grid = pl.tc_grid;
    a.S = pl.splits;
    a.part_o = part_o;
    a.part_ml = part_ml;
    a.status = status;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    attend_tc_kernel<<<pl.tc_grid, kThreads, kSmem, st>>>(tm_sel, tm_win, a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa
