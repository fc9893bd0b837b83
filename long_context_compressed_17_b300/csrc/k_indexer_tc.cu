// k_indexer_tc.cu -- lightning-indexer scoring on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), for keys of 128 dims and 64 heads, in bf16
// or in E4M3 with one float32 scale per key (kind::f8f6f4 MMAs).
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 2: Lightning Indexer
// Top-K 选择": score_b = sum_h w_h * relu(q_h . k_b) over causally complete
// blocks.  The q.K products are a dense contraction, so they run as
//   D[128 keys, N] = K_tile[128 keys, 128 dims] x Q[N, 128 dims]^T
// with the keys as the M = 128 side (swap-AB: a decode query has only 64
// heads) and N = 64 * NQ columns for NQ queries of one sequence; the relu and
// the head-weighted sum run in the epilogue straight out of TMEM, one key per
// thread.  Decode (NQ = 1) is an HBM stream of the keys; prefill (NQ = 4)
// reuses every key tile for four queries per MMA.
//
// Persistent CTAs walk a contiguous range of (query group, key tile) units.
// Warp 0 issues TMA loads; the MMAs are issued by warp 1, or for NQ = 1 by
// warps 1 and 2 on alternate tiles; the other warps are the epilogue: for
// NQ = 1 two groups of four (one per TMEM lane quarter) on alternate
// accumulators, for NQ = 4 sixteen, where four warps share a quarter and take
// one of the four queries each (the epilogue, 256 values per key, would
// otherwise hold the tensor pipe back).  Every wait is bounded: on a timeout
// the kernel flags CSA_DEV_TIMEOUT, all roles leave their loops and TMEM is
// freed.
#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa {

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);
bool make_tmap_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box);

namespace {

constexpr int kHI = 64;            // indexer heads (per query)
constexpr int kDI = 128;           // indexer dim
constexpr int kTileKeys = 128;     // MMA M

// F8: keys and queries in E4M3 (kind::f8f6f4 MMAs, K = 32 per MMA), one
// float32 scale per key row and per query head (folded into the head
// weights); otherwise bf16 (kind::f16, K = 16).
template <int NQ, bool F8>
struct Cfg {
    static constexpr int kEB = F8 ? 1 : 2;              // bytes per element
    static constexpr uint32_t kStageBytes = kTileKeys * kDI * kEB;  // 32 KiB bf16 (two boxes), 16 KiB E4M3 (one)
    static constexpr int kKSteps = kDI * kEB / 32;      // MMAs per key tile: 32 bytes of K each
    static constexpr int N = NQ * kHI;                  // MMA N
    // key tiles and TMEM accumulators in flight: E4M3 tiles are half the bytes,
    // so twice as many are in flight for the same shared memory
    static constexpr int kStages = F8 ? 8 : 4;
    static constexpr int kAcc = NQ == 1 ? (F8 ? 8 : 4) : 2;
    static constexpr int kQBufs = NQ == 1 ? 2 : 1;
    // Epilogue warps: for NQ = 4, sixteen (four per TMEM lane quarter, one
    // query each); for NQ = 1, two groups of four that take alternate
    // accumulators (a tile's epilogue is latency-bound: two in flight).
    static constexpr int kEpiWarps = NQ == 1 ? 8 : 16;
    static constexpr int kEpiGroups = NQ == 1 ? 2 : 1;
    static constexpr int kQPerWarp = NQ * 4 * kEpiGroups / kEpiWarps;  // queries of a key per epilogue warp
    // MMA-issuing warps: a thread issuing tcgen05.mma back to back waits on
    // each instruction longer than an N = 64 product takes to run, so decode
    // has two issuers on alternate key tiles (even stage and accumulator
    // counts: each barrier still hears from one issuer only)
    static constexpr int kIssuers = NQ == 1 ? 2 : 1;
    static_assert(kStages % kIssuers == 0 && kAcc % kIssuers == 0, "issuers own whole stages");
    static constexpr int kEpi0 = 1 + kIssuers;          // first epilogue warp
    static constexpr int kThreads = 32 * kEpi0 + 32 * kEpiWarps;
    static constexpr uint32_t kQBytes = (uint32_t)N * kDI * kEB;
    static constexpr uint32_t kTmemCols = kAcc * N;     // 256 or 512
    static constexpr size_t kBarBytes = 512;
    static_assert((2 * kStages + 2 * kQBufs + 2 * kAcc) * 8 + 8 <= kBarBytes, "barrier area too small");
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kQBufs * kQBytes + kBarBytes;
    static constexpr uint32_t idesc = F8 ? tc::idesc_e4m3_f32(kTileKeys, N) : tc::idesc_bf16_f32(kTileKeys, N);
};

struct IdxArgs {
    const float* w_idx;    // [Q, 64] (F8: the head weights times the query head scales)
    const float* key_scales;  // F8: [B, n_cap] per key row; else nullptr
    const int64_t* q_pos;  // [Q]
    float* scores;         // [Q, ld]
    int64_t ld;
    int64_t n_cap;
    int qps;               // queries per sequence
    int m;
    int n_tiles;           // key tiles per query group
    int64_t total_units;   // groups * n_tiles
    uint32_t* status;
};

// Blocks a query group sees: the largest floor((i+1)/m) of its queries, capped.
template <int NQ>
__device__ __forceinline__ int64_t group_avail(const IdxArgs& a, int64_t g) {
    int64_t nav = 0;
#pragma unroll
    for (int qq = 0; qq < NQ; qq++) {
        int64_t n = (a.q_pos[g * NQ + qq] + 1) / a.m;
        nav = max(nav, min(n, a.n_cap));
    }
    return nav;
}

}  // namespace

template <int NQ, bool F8>
__global__ void __launch_bounds__(Cfg<NQ, F8>::kThreads, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_keys,
                      const __grid_constant__ CUtensorMap tm_q, IdxArgs a) {
    using C = Cfg<NQ, F8>;
    constexpr uint32_t kStageBytes = C::kStageBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = sm;
    uint8_t* sB = sA + C::kStages * kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::kQBufs * C::kQBytes);
    uint64_t* empty = full + C::kStages;
    uint64_t* qfull = empty + C::kStages;
    uint64_t* qempty = qfull + C::kQBufs;
    uint64_t* tfull = qempty + C::kQBufs;
    uint64_t* tempty = tfull + C::kAcc;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + C::kAcc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < C::kQBufs; b++) {
            tc::mbar_init(&qfull[b], 1);
            tc::mbar_init(&qempty[b], C::kIssuers);  // every issuer releases the queries
        }
        for (int c = 0; c < C::kAcc; c++) {
            tc::mbar_init(&tfull[c], 1);
            tc::mbar_init(&tempty[c], C::kEpiWarps / C::kEpiGroups);  // one arrival per warp of its group
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::fence_proxy_async_smem();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int64_t per = (a.total_units + gridDim.x - 1) / gridDim.x;
    const int64_t u0 = (int64_t)blockIdx.x * per;
    const int64_t u1 = min(a.total_units, u0 + per);
    // (query group, key tile) of unit u0; every role steps it along without dividing
    const int64_t g0 = u0 / a.n_tiles;
    const int64_t t0 = u0 - g0 * a.n_tiles;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        tc::tma_prefetch_map(&tm_keys);
        tc::tma_prefetch_map(&tm_q);
        int stage = 0;
        uint32_t phase = 0;
        int64_t cur_g = -1, last_loaded = -1, gnav = 0;
        int qloads = 0, seq = 0;
        const float* ksrow = nullptr;  // F8: the sequence's key scales
        int64_t g = g0;
        for (int64_t u = u0, t = t0; u < u1; ++u, ++t) {
            if (t == a.n_tiles) {
                t = 0;
                ++g;
            }
            if (g != cur_g) {
                cur_g = g;
                gnav = group_avail<NQ>(a, g);
                seq = (int)((g * NQ) / a.qps);
                if (F8) ksrow = a.key_scales + (int64_t)seq * a.n_cap;
            }
            if ((int64_t)t * kTileKeys >= gnav) continue;  // no complete block in this tile
            if (g != last_loaded) {
                const int qb = qloads % C::kQBufs;
                const uint32_t par = ((uint32_t)(qloads / C::kQBufs) & 1u) ^ 1u;
                if (!tc::mbar_wait(&qempty[qb], par, abort_flag, a.status)) break;
                tc::mbar_arrive_expect_tx(&qfull[qb], C::kQBytes);
                uint8_t* dst = sB + qb * C::kQBytes;
                tc::tma_load_2d(dst, &tm_q, &qfull[qb], 0, (int)(g * C::N));
                if (!F8) tc::tma_load_2d(dst + C::kQBytes / 2, &tm_q, &qfull[qb], 64, (int)(g * C::N));
                last_loaded = g;
                qloads++;
            }
            if (!tc::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) break;
            tc::mbar_arrive_expect_tx(&full[stage], kStageBytes);
            uint8_t* dst = sA + stage * kStageBytes;
            tc::tma_load_3d(dst, &tm_keys, &full[stage], 0, (int)(t * kTileKeys), seq);
            if (!F8) tc::tma_load_3d(dst + kStageBytes / 2, &tm_keys, &full[stage], 64, (int)(t * kTileKeys), seq);
            if (F8) {  // the tile's key scales head for L2 now: the epilogue reads them thousands of cycles later
                const int64_t k0 = t * kTileKeys, kn = min((int64_t)kTileKeys, a.n_cap - k0);
                for (int64_t o = 0; o < kn; o += 32) tc::prefetch_l2_line(ksrow + k0 + o);
                tc::prefetch_l2_line(ksrow + k0 + kn - 1);
            }
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    } else if (warp >= 1 && warp < C::kEpi0 && lane == 0) {
        // ------------------------------------------------ MMA issuers
        // Issuer `me` takes the live units j with j % kIssuers == me; every
        // issuer follows the query buffers through all of them.
        constexpr uint32_t idesc = C::idesc;
        const uint32_t me = (uint32_t)(warp - 1);
        uint32_t j = 0;  // live units so far
        int quses = 0, qb = 0;
        int64_t cur_g = -1, last_used = -1, gnav = 0;
        int64_t g = g0;
        for (int64_t u = u0, t = t0; u < u1; ++u, ++t) {
            if (t == a.n_tiles) {
                t = 0;
                ++g;
            }
            if (g != cur_g) {
                cur_g = g;
                gnav = group_avail<NQ>(a, g);
            }
            if ((int64_t)t * kTileKeys >= gnav) continue;
            if (g != last_used) {
                if (quses > 0) tc::mma_commit(&qempty[qb]);  // the old queries are free once read
                qb = quses % C::kQBufs;
                const uint32_t par = (uint32_t)(quses / C::kQBufs) & 1u;
                if (!tc::mbar_wait(&qfull[qb], par, abort_flag, a.status)) break;
                last_used = g;
                quses++;
            }
            const uint32_t jj = j++;
            if (jj % C::kIssuers != me) continue;
            const int stage = (int)(jj % C::kStages), acc = (int)(jj % C::kAcc);
            const uint32_t phase = (jj / C::kStages) & 1u, aphase = (jj / C::kAcc) & 1u;
            if (!tc::mbar_wait(&tempty[acc], aphase ^ 1u, abort_flag, a.status)) break;
            if (!tc::mbar_wait(&full[stage], phase, abort_flag, a.status)) break;
            tc::fence_after_sync();
            const uint32_t a_base = tc::smem_u32(sA + stage * kStageBytes);
            const uint32_t b_base = tc::smem_u32(sB + qb * C::kQBytes);
            const uint32_t d = tmem + (uint32_t)(acc * C::N);
#pragma unroll
            for (int kk = 0; kk < C::kKSteps; kk++) {
                if (F8) {  // one 128-byte row per key / head: 32 bytes of K per MMA
                    tc::mma_f8_ss(d, tc::sdesc_kmajor_sw128(a_base + (uint32_t)kk * 32u),
                                  tc::sdesc_kmajor_sw128(b_base + (uint32_t)kk * 32u), idesc, kk > 0 ? 1u : 0u);
                } else {   // two 64-dim boxes of 128-byte rows
                    const uint32_t ka = (uint32_t)(kk >> 2) * (kStageBytes / 2) + (uint32_t)(kk & 3) * 32u;
                    const uint32_t kb = (uint32_t)(kk >> 2) * (C::kQBytes / 2) + (uint32_t)(kk & 3) * 32u;
                    tc::mma_bf16_ss(d, tc::sdesc_kmajor_sw128(a_base + ka),
                                    tc::sdesc_kmajor_sw128(b_base + kb), idesc, kk > 0 ? 1u : 0u);
                }
            }
            tc::mma_commit(&empty[stage]);  // key tile free when these MMAs finish
            tc::mma_commit(&tfull[acc]);    // accumulator ready for the epilogue
        }
    } else if (warp >= C::kEpi0) {
        // ------------------------------------------------ epilogue: one key per thread
        const int quarter = warp & 3;          // TMEM lanes this warp may read
        const int row = quarter * 32 + lane;   // key within the tile
        static_assert(C::kQPerWarp == 1, "one query per epilogue warp");
        const int wq = (warp - C::kEpi0) >> 2;
        const int grp = C::kEpiGroups > 1 ? wq : 0;  // this warp takes the accumulators acc % groups == grp
        const int q0 = C::kEpiGroups > 1 ? 0 : wq;   // this warp's query within the query group
        int acc = 0;
        uint32_t aphase = 0;
        int64_t cur_g = -1, gnav = 0;
        int64_t nav[NQ];
        float* srow = a.scores;            // this warp's query's score row
        const float* krow = a.key_scales;  // F8: the sequence's key scales
        // the query's head weights: in registers for decode (loaded once per query
        // group), read through L1 per tile in prefill (the registers go to the
        // sixteen epilogue warps there)
        constexpr bool kWRegs = NQ == 1;
        float wr[kWRegs ? kHI : 1];
        int64_t g = g0;
        for (int64_t u = u0, t = t0; u < u1; ++u, ++t) {
            if (t == a.n_tiles) {
                t = 0;
                ++g;
            }
            if (g != cur_g) {
                cur_g = g;
                gnav = 0;
#pragma unroll
                for (int qq = 0; qq < NQ; qq++) {
                    nav[qq] = min((a.q_pos[g * NQ + qq] + 1) / a.m, a.n_cap);
                    gnav = max(gnav, nav[qq]);
                }
                if (NQ == 1) srow = a.scores + (g * NQ + q0) * a.ld;
                if (F8 && NQ == 1) krow = a.key_scales + (g * NQ / a.qps) * a.n_cap;
                if constexpr (kWRegs) {
                    const float4* w4 = reinterpret_cast<const float4*>(a.w_idx + (g * NQ + q0) * kHI);
#pragma unroll
                    for (int j4 = 0; j4 < kHI / 4; j4++) {
                        const float4 w = __ldg(w4 + j4);
                        wr[4 * j4] = w.x;
                        wr[4 * j4 + 1] = w.y;
                        wr[4 * j4 + 2] = w.z;
                        wr[4 * j4 + 3] = w.w;
                    }
                }
            }
            const int64_t key = (int64_t)t * kTileKeys + row;
            if (NQ != 1) srow = a.scores + (g * NQ + q0) * a.ld;
            if ((int64_t)t * kTileKeys >= gnav) {  // nothing complete in this tile
                if (key < a.n_cap && grp == 0) srow[key] = -INFINITY;
                continue;
            }
            if ((acc % C::kEpiGroups) != grp) {  // the other group's accumulator
                if (++acc == C::kAcc) {
                    acc = 0;
                    aphase ^= 1u;
                }
                continue;
            }
            // E4M3 keys: this key's scale is on its way while the accumulator is awaited
            // (prefill keeps no row pointer: its sixteen warps are short of registers)
            const float ksc = (F8 && key < a.n_cap)
                                  ? __ldg((NQ == 1 ? krow : a.key_scales + (g * NQ / a.qps) * a.n_cap) + key)
                                  : 1.f;
            // one lane waits, the whole warp follows its verdict (tcgen05.ld is warp-wide)
            int ok = 1;
            if (lane == 0) ok = tc::mbar_wait(&tfull[acc], aphase, abort_flag, a.status) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc::fence_after_sync();
            const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::N);
            {
                float acc4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
#pragma unroll
                for (int half = 0; half < 2; half++) {
                    float v[32];
                    tc::tmem_ld32(tbase + (uint32_t)(q0 * kHI + half * 32), v);
                    tc::tmem_ld_wait();
                    if constexpr (kWRegs) {
#pragma unroll
                        for (int j = 0; j < 32; j++) acc4[j & 3] = fmaf(wr[half * 32 + j], fmaxf(v[j], 0.f), acc4[j & 3]);
                    } else {
                        const float4* w4 = reinterpret_cast<const float4*>(a.w_idx + (g * NQ + q0) * kHI) + half * 8;
#pragma unroll
                        for (int j4 = 0; j4 < 8; j4++) {
                            const float4 w = __ldg(w4 + j4);
                            acc4[0] = fmaf(w.x, fmaxf(v[4 * j4 + 0], 0.f), acc4[0]);
                            acc4[1] = fmaf(w.y, fmaxf(v[4 * j4 + 1], 0.f), acc4[1]);
                            acc4[2] = fmaf(w.z, fmaxf(v[4 * j4 + 2], 0.f), acc4[2]);
                            acc4[3] = fmaf(w.w, fmaxf(v[4 * j4 + 3], 0.f), acc4[3]);
                        }
                    }
                }
                float s = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
                if (F8) s *= ksc;
                if (key < a.n_cap) srow[key] = key < nav[q0] ? s : -INFINITY;
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&tempty[acc]);
            if (++acc == C::kAcc) {
                acc = 0;
                aphase ^= 1u;
            }
        }
    }
    // ---------------------------------------------------- teardown
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int NQ, bool F8>
static cudaError_t run_indexer(const CUtensorMap& tm_keys, const CUtensorMap& tm_q, const IdxArgs& a, int grid,
                               cudaStream_t st) {
    using C = Cfg<NQ, F8>;
    {
        cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(indexer_tc_kernel<NQ, F8>), C::kSmem);
        if (e != cudaSuccess) return e;
    }
    indexer_tc_kernel<NQ, F8><<<grid, C::kThreads, C::kSmem, st>>>(tm_keys, tm_q, a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_indexer_tc(const Geometry& g, const void* q_idx, const float* w_idx, int HI,
                              int dI, const void* keys, const float* key_scales, int64_t n_cap, int B,
                              int Q, const int64_t* q_pos, uint32_t* status, float* scores, int64_t ld,
                              cudaStream_t st, bool* launched) {
    *launched = false;
    const bool f8 = key_scales != nullptr;  // q_idx: E4M3 codes, w_idx: weights x head scales
    if ((!f8 && g.act != CSA_BF16) || HI != kHI || dI != kDI || n_cap < kTileKeys || Q < 1) return cudaSuccess;
    if (((uintptr_t)w_idx & 15u) || (ld % 4) != 0) return cudaSuccess;
    const int qps = Q / B;
    const int NQ = (qps % 4 == 0) ? 4 : 1;
    const uint64_t eb = f8 ? 1 : 2;
    CUtensorMap tm_keys, tm_q;
    const uint64_t kd[3] = {(uint64_t)kDI, (uint64_t)n_cap, (uint64_t)B};
    const uint64_t ks[2] = {(uint64_t)kDI * eb, (uint64_t)n_cap * kDI * eb};
    const uint32_t kb[3] = {(uint32_t)(128 / eb), (uint32_t)kTileKeys, 1};  // 128-byte rows
    const uint64_t qd[2] = {(uint64_t)kDI, (uint64_t)Q * kHI};
    const uint64_t qs[1] = {(uint64_t)kDI * eb};
    const uint32_t qbox[2] = {(uint32_t)(128 / eb), (uint32_t)(NQ * kHI)};
    const bool maps = f8 ? (make_tmap_u8(&tm_keys, keys, 3, kd, ks, kb) && make_tmap_u8(&tm_q, q_idx, 2, qd, qs, qbox))
                         : (make_tmap_bf16(&tm_keys, keys, 3, kd, ks, kb) &&
                            make_tmap_bf16(&tm_q, q_idx, 2, qd, qs, qbox));
    if (!maps) return f8 ? cudaErrorInvalidValue : cudaSuccess;  // bf16: the CUDA-core path runs instead
    IdxArgs a;
    a.w_idx = w_idx;
    a.key_scales = key_scales;
    a.q_pos = q_pos;
    a.scores = scores;
    a.ld = ld;
    a.n_cap = n_cap;
    a.qps = qps;
    a.m = g.m;
    a.n_tiles = (int)((n_cap + kTileKeys - 1) / kTileKeys);
    a.total_units = (int64_t)(Q / NQ) * a.n_tiles;
    a.status = status;
    const int64_t sms = num_sms();
    const int grid = (int)(a.total_units < sms ? a.total_units : sms);
    cudaError_t e;
    if (NQ == 1)
        e = f8 ? run_indexer<1, true>(tm_keys, tm_q, a, grid, st) : run_indexer<1, false>(tm_keys, tm_q, a, grid, st);
    else
        e = f8 ? run_indexer<4, true>(tm_keys, tm_q, a, grid, st) : run_indexer<4, false>(tm_keys, tm_q, a, grid, st);
    if (e == cudaSuccess) *launched = true;
    return e;
}

}  // namespace csa
