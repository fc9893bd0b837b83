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
// the kernel flags CSA_DEV_TIMEOUT, all roles leave their loops, the copies
// and MMAs in flight are waited for (bounded too) and TMEM is freed.
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa {

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);
bool make_tmap_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box);
bool make_tmap_u8_linear(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides_bytes, const uint32_t* box);

namespace {

constexpr int kHI = 64;            // indexer heads (per query)
constexpr int kDI = 128;           // indexer dim
constexpr int kTileKeys = 128;     // MMA M

// Key formats: bf16 (kind::f16 MMAs, K = 16), E4M3 with one float32 scale
// per key (kind::f8f6f4 MMAs, K = 32; query heads in E4M3 with their scales
// folded into the head weights), or FP4: E2M1 codes with one power-of-two
// scale per 32 dims, expanded in shared memory to E4M3 codes with one
// power-of-two scale per key (exact: the packer keeps a key's block scales
// within 14 binades of its largest), then scored as E4M3 keys.
enum { kKeyBf16 = 0, kKeyE4m3 = 1, kKeyFp4 = 2 };
// A packed FP4 key tile: 128 keys x 64 code bytes, then 128 x 4 exponent bytes.
constexpr uint32_t kFp4TileBytes = kTileKeys * (kDI / 2) + kTileKeys * (kDI / 32);
static_assert(kFp4TileBytes == 8704 && kFp4TileBytes % 128 == 0, "FP4 tile layout");
constexpr int kFp4Rows = kFp4TileBytes / 128;  // 68 rows of 128 bytes

template <int NQ, int KF>
struct Cfg {
    static constexpr bool F8 = KF != kKeyBf16;          // E4M3 MMAs
    static constexpr bool F4 = KF == kKeyFp4;
    static constexpr int kEB = F8 ? 1 : 2;              // bytes per element
    static constexpr uint32_t kStageBytes = kTileKeys * kDI * kEB;  // 32 KiB bf16 (two boxes), 16 KiB E4M3 (one)
    static constexpr int kKSteps = kDI * kEB / 32;      // MMAs per key tile: 32 bytes of K each
    static constexpr int N = NQ * kHI;                  // MMA N
    // key tiles and TMEM accumulators in flight: E4M3 tiles are half the bytes,
    // so twice as many are in flight for the same shared memory; FP4 tiles
    // land in the raw ring (the HBM stream's depth) and spend only the
    // conversion-to-MMA span in a stage
    static constexpr int kStages = F4 ? 4 : (F8 ? 8 : 4);
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
    // FP4 -> E4M3 converters, one key a thread: groups of four warps on
    // alternate tiles (decode: two groups, or the conversion would fall
    // behind the HBM stream)
    static constexpr int kConvWarps = F4 ? (NQ == 1 ? 8 : 4) : 0;
    static constexpr int kConvGroups = kConvWarps / 4;
    static_assert(kConvGroups * 4 == kConvWarps, "whole converter groups");
    static constexpr int kConv0 = kEpi0 + kEpiWarps;
    static constexpr int kThreads = 32 * (kConv0 + kConvWarps);
    static constexpr uint32_t kQBytes = (uint32_t)N * kDI * kEB;
    static constexpr uint32_t kTmemCols = kAcc * N;     // 256 or 512
    static constexpr int kRawStages = F4 ? 12 : 0;      // packed FP4 tiles in flight (~104 KiB)
    static constexpr int kRawSlots = kRawStages / 2;    // ... loaded two consecutive live tiles a slot
    static constexpr int kScaleSlots = F4 ? kStages + kAcc : 0;  // per-key scales of the tiles in flight
    static constexpr size_t kBarBytes = 1024;
    static_assert((2 * kStages + 2 * kQBufs + 2 * kAcc + 2 * kRawSlots + kScaleSlots + kIssuers) * 8 + 8 <= kBarBytes,
                  "barrier area too small");
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kQBufs * kQBytes +
                                    (size_t)kRawStages * kFp4TileBytes + (size_t)kScaleSlots * kTileKeys * 4 +
                                    kBarBytes;
    static constexpr uint32_t idesc = F8 ? tc::idesc_e4m3_f32(kTileKeys, N) : tc::idesc_bf16_f32(kTileKeys, N);
};

struct IdxArgs {
    const float* w_idx;    // [Q, 64] (F8: the head weights times the query head scales)
    const float* key_scales;  // E4M3 keys: [B, n_cap] per key row; else nullptr
    const uint8_t* key_pack;  // FP4 keys: [B, n_tiles] packed tiles of kFp4TileBytes; else nullptr
    const int64_t* q_pos;  // [Q]
    float* scores;         // [Q, ld]
    int64_t ld;
    int64_t n_cap;
    int qps;               // queries per sequence
    int m;
    int n_tiles;           // key tiles per query group
    int64_t total_units;   // groups * n_tiles
    uint32_t* status;
    int withhold;          // test hook: the producer issues nothing (see csa_test_withhold_indexer_loads)
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

template <int NQ, int KF>
__global__ void __launch_bounds__(Cfg<NQ, KF>::kThreads, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_keys,
                      const __grid_constant__ CUtensorMap tm_q, IdxArgs a) {
    using C = Cfg<NQ, KF>;
    tc::grid_dep_launch();  // the selection after this kernel may be scheduled now
    constexpr bool F8 = C::F8;
    constexpr bool F4 = C::F4;
    constexpr uint32_t kStageBytes = C::kStageBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = sm;
    uint8_t* sB = sA + C::kStages * kStageBytes;
    uint8_t* sRaw = sB + C::kQBufs * C::kQBytes;                                   // FP4 packed tiles
    float* sKs = reinterpret_cast<float*>(sRaw + (size_t)C::kRawStages * kFp4TileBytes);  // FP4 key scales
    uint64_t* full = reinterpret_cast<uint64_t*>(sKs + C::kScaleSlots * kTileKeys);
    uint64_t* empty = full + C::kStages;
    uint64_t* qfull = empty + C::kStages;
    uint64_t* qempty = qfull + C::kQBufs;
    uint64_t* tfull = qempty + C::kQBufs;
    uint64_t* tempty = tfull + C::kAcc;
    uint64_t* rfull = tempty + C::kAcc;       // FP4: the packed tiles of a raw slot landed
    uint64_t* rempty = rfull + C::kRawSlots;  // FP4: both tiles of a raw slot read by the converters
    uint64_t* sfull = rempty + C::kRawSlots;  // FP4: key scales of a tile written
    uint64_t* idone = sfull + C::kScaleSlots;  // every MMA of an issuer done (before TMEM is freed)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(idone + C::kIssuers);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // FP4: E4M3 codes of the E2M1 magnitudes 0..7 times 2^sh for every shift
    // sh = -8 .. 6 a nonzero block can have (eight bytes per shift)
    __shared__ uint2 fp4_lut[15];
    if constexpr (F4) {
        if (threadIdx.x < 15) {
            const float kMag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
            uint32_t w[2] = {0u, 0u};
            for (int m = 1; m < 8; m++)
                w[m >> 2] |= (uint32_t)f32_to_e4m3_sat(ldexpf(kMag[m], (int)threadIdx.x - 8)) << (8 * (m & 3));
            fp4_lut[threadIdx.x] = make_uint2(w[0], w[1]);
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; s++) {
            tc::mbar_init(&full[s], F4 ? 4 : 1);  // FP4: every warp of a converter group
            tc::mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < C::kRawSlots; s++) {
            tc::mbar_init(&rfull[s], 1);
            tc::mbar_init(&rempty[s], 8);  // the four warps of each converter group
        }
        for (int s = 0; s < C::kScaleSlots; s++) tc::mbar_init(&sfull[s], 4);
        for (int i = 0; i < C::kIssuers; i++) tc::mbar_init(&idone[i], 1);
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

    if (warp == 0 && lane == 0 && !a.withhold) {
        // ------------------------------------------------ TMA producer
        // (under the test hook it issues nothing: no copy is ever in flight, the
        // issuers' bounded waits on the query and key tiles expire)
        tc::tma_prefetch_map(&tm_keys);
        tc::tma_prefetch_map(&tm_q);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t nraw = 0;  // FP4: packed tiles loaded
        uint32_t nkey = 0;  // key tiles loaded into the stages
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
                if (KF == kKeyE4m3) ksrow = a.key_scales + (int64_t)seq * a.n_cap;
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
            if constexpr (F4) {
                // Packed tiles, one TMA box of 68 rows of 128 bytes each, into
                // the raw ring two live tiles a slot (the second found ahead:
                // each producer pass costs far more than its copies), where the
                // converter warps expand them into stages.
                if ((nraw & 1u) == 0) {
                    const uint32_t pr = nraw >> 1;
                    const int rs = (int)(pr % C::kRawSlots);
                    if (!tc::mbar_wait(&rempty[rs], ((pr / C::kRawSlots) & 1u) ^ 1u, abort_flag, a.status)) break;
                    // the next live tile in this CTA's range, if any
                    int seq_n = seq;
                    int64_t t_n = t, g_n = g, nav_n = gnav;
                    bool has_next = false;
                    for (int64_t un = u + 1; un < u1; ++un) {
                        if (++t_n == a.n_tiles) {
                            t_n = 0;
                            ++g_n;
                            nav_n = group_avail<NQ>(a, g_n);
                            seq_n = (int)((g_n * NQ) / a.qps);
                        }
                        if (t_n * kTileKeys < nav_n) {
                            has_next = true;
                            break;
                        }
                    }
                    tc::mbar_arrive_expect_tx(&rfull[rs], kFp4TileBytes * (has_next ? 2u : 1u));
                    uint8_t* dst = sRaw + (size_t)rs * 2 * kFp4TileBytes;
                    tc::tma_load_2d(dst, &tm_keys, &rfull[rs], 0, (int)(((int64_t)seq * a.n_tiles + t) * kFp4Rows));
                    if (has_next)
                        tc::tma_load_2d(dst + kFp4TileBytes, &tm_keys, &rfull[rs], 0,
                                        (int)(((int64_t)seq_n * a.n_tiles + t_n) * kFp4Rows));
                }
                ++nraw;
                continue;
            }
            if (!tc::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) break;
            tc::mbar_arrive_expect_tx(&full[stage], kStageBytes);
            ++nkey;
            uint8_t* dst = sA + stage * kStageBytes;
            tc::tma_load_3d(dst, &tm_keys, &full[stage], 0, (int)(t * kTileKeys), seq);
            if (!F8) tc::tma_load_3d(dst + kStageBytes / 2, &tm_keys, &full[stage], 64, (int)(t * kTileKeys), seq);
            if (KF == kKeyE4m3) {  // the tile's key scales head for L2 now: the epilogue reads them thousands of cycles later
                const int64_t k0 = t * kTileKeys, kn = min((int64_t)kTileKeys, a.n_cap - k0);
                for (int64_t o = 0; o < kn; o += 32) tc::prefetch_l2_line(ksrow + k0 + o);
                tc::prefetch_l2_line(ksrow + k0 + kn - 1);
            }
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // Leave no copy in flight (a role that gave up may not have consumed
        // them): the newest load of every buffer must have landed.
        auto drain_newest = [&](uint64_t* bars, uint32_t loads, uint32_t n) {
            for (uint32_t s2 = 0; s2 < n && s2 < loads; s2++) {
                const uint32_t i = s2 + (loads - 1u - s2) / n * n;  // newest load into buffer s2
                if (!tc::mbar_drain(&bars[s2], (i / n) & 1u)) atomicOr(a.status, CSA_DEV_TIMEOUT);
            }
        };
        drain_newest(full, nkey, (uint32_t)C::kStages);
        drain_newest(qfull, (uint32_t)qloads, (uint32_t)C::kQBufs);
        if constexpr (F4) drain_newest(rfull, (nraw + 1u) >> 1, (uint32_t)C::kRawSlots);
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
        // every MMA this thread issued must be complete before TMEM is freed
        tc::mma_commit(&idone[me]);
        if (!tc::mbar_drain(&idone[me], 0)) atomicOr(a.status, CSA_DEV_TIMEOUT);
    } else if (warp >= C::kEpi0 && warp < C::kConv0) {
        // ------------------------------------------------ epilogue: one key per thread
        const int quarter = warp & 3;          // TMEM lanes this warp may read
        const int row = quarter * 32 + lane;   // key within the tile
        static_assert(C::kQPerWarp == 1, "one query per epilogue warp");
        const int wq = (warp - C::kEpi0) >> 2;
        const int grp = C::kEpiGroups > 1 ? wq : 0;  // this warp takes the accumulators acc % groups == grp
        const int q0 = C::kEpiGroups > 1 ? 0 : wq;   // this warp's query within the query group
        int acc = 0;
        uint32_t aphase = 0;
        uint32_t jl = 0;  // live units so far (FP4: the key-scale slot is jl % kScaleSlots)
        int64_t cur_g = -1, gnav = 0;
        int64_t nav[NQ];
        float* srow = a.scores;            // this warp's query's score row
        const float* krow = a.key_scales;  // F8: the sequence's key scales
        // the query's head weights: in registers for decode (loaded once per query
        // group), read through L1 per tile in prefill (the registers go to the
        // sixteen epilogue warps there)
        constexpr bool kWRegs = NQ == 1 && !F4;  // FP4: the converter warps leave 96 registers
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
            const uint32_t jj = jl++;
            if ((acc % C::kEpiGroups) != grp) {  // the other group's accumulator
                if (++acc == C::kAcc) {
                    acc = 0;
                    aphase ^= 1u;
                }
                continue;
            }
            // E4M3 keys: this key's scale is on its way while the accumulator is awaited
            // (prefill keeps no row pointer: its sixteen warps are short of registers)
            float ksc = (KF == kKeyE4m3 && key < a.n_cap)
                            ? __ldg((NQ == 1 ? krow : a.key_scales + (g * NQ / a.qps) * a.n_cap) + key)
                            : 1.f;
            if constexpr (F4) {  // the power-of-two scale the converters chose for this key
                // every lane waits (each acquires the converters' writes it reads)
                const int slot = (int)(jj % C::kScaleSlots);
                const int oks = tc::mbar_wait(&sfull[slot], (jj / C::kScaleSlots) & 1u, abort_flag, a.status) ? 1 : 0;
                if (!__all_sync(0xffffffffu, oks)) break;
                ksc = sKs[slot * kTileKeys + row];
            }
            // one lane waits, the whole warp follows its verdict (tcgen05.ld is warp-wide)
            int ok = 1;
            if (lane == 0) ok = tc::mbar_wait(&tfull[acc], aphase, abort_flag, a.status) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc::fence_after_sync();
            const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::N);
            {
                float acc4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
                if constexpr (F4) {
                    // sixteen heads a load, their weights through L1 (the
                    // converter warps leave the epilogue 96 registers a thread)
                    const float4* w4 = reinterpret_cast<const float4*>(a.w_idx + (g * NQ + q0) * kHI);
#pragma unroll
                    for (int qt = 0; qt < 4; qt++) {
                        float v[16];
                        tc::tmem_ld16(tbase + (uint32_t)(q0 * kHI + qt * 16), v);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int j4 = 0; j4 < 4; j4++) {
                            const float4 w = __ldg(w4 + qt * 4 + j4);
                            acc4[0] = fmaf(w.x, fmaxf(v[4 * j4 + 0], 0.f), acc4[0]);
                            acc4[1] = fmaf(w.y, fmaxf(v[4 * j4 + 1], 0.f), acc4[1]);
                            acc4[2] = fmaf(w.z, fmaxf(v[4 * j4 + 2], 0.f), acc4[2]);
                            acc4[3] = fmaf(w.w, fmaxf(v[4 * j4 + 3], 0.f), acc4[3]);
                        }
                    }
                } else
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
                if (F8) s *= ksc;  // E4M3: the stored per-key scale; FP4: the converted key's 2^E
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
    if constexpr (F4) {
        if (warp >= C::kConv0) {
            // ------------------------------------------------ FP4 -> E4M3 converters
            // Thread k of the four converter warps expands key k of every tile:
            // E = the largest exponent of its blocks with a nonzero code, the
            // key's scale 2^(E - 6) (its largest value 6 * 2^E lands on
            // 384 <= 448), and block j's codes become the E4M3 codes of
            // e2m1 * 2^(e_j - E + 6): an 8-entry magnitude table per block
            // (exact conversions), looked up four codes at a time with byte
            // permutes, the signs moved from bit 3 of each nibble to bit 7 of
            // each byte with the permute's sign-replicate selectors.  The row
            // is written with the 128-byte swizzle of a TMA tile load.  A block
            // whose codes are all zero may have any shift: its table is never
            // read beyond entry 0, so the shift is clamped into the table.
            const int k = ((warp - C::kConv0) & 3) * 32 + lane;
            const uint32_t grp = (uint32_t)((warp - C::kConv0) >> 2);  // takes tiles jj = grp mod kConvGroups
            uint32_t j = 0;
            int64_t cur_g = -1, gnav = 0;
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
                const uint32_t jj = j++;
                if (jj % C::kConvGroups != grp) continue;
                const int stage = (int)(jj % C::kStages), rs = (int)((jj >> 1) % C::kRawSlots);
                const int slot = (int)(jj % C::kScaleSlots);
                if (!tc::mbar_wait(&rfull[rs], ((jj >> 1) / C::kRawSlots) & 1u, abort_flag, a.status)) break;
                if (!tc::mbar_wait(&empty[stage], ((jj / C::kStages) & 1u) ^ 1u, abort_flag, a.status)) break;
                const uint8_t* raw = sRaw + ((size_t)rs * 2 + (jj & 1u)) * kFp4TileBytes;
                // chunk c = block c (32 codes); static indices keep cw in
                // registers (a lane-dependent index would put it in local memory)
                uint4 cw[4];
#pragma unroll
                for (int c = 0; c < 4; c++) cw[c] = *reinterpret_cast<const uint4*>(raw + k * 64 + c * 16);
                const uint32_t ex = *reinterpret_cast<const uint32_t*>(raw + kTileKeys * 64 + k * 4);
                int E = -1000;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const uint32_t nzm = (cw[c].x | cw[c].y | cw[c].z | cw[c].w) & 0x77777777u;
                    const int ej = (int)((ex >> (8 * c)) & 0xFFu) - 127;
                    if (nzm != 0u && ej > E) E = ej;
                }
                if (E == -1000) E = 0;  // no nonzero code: any scale
                const int Ek = E - 6;
                uint8_t* row = sA + stage * kStageBytes + k * 128;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int sh = min(6, max(-8, (int)((ex >> (8 * c)) & 0xFFu) - 127 - Ek));
                    const uint2 lt = fp4_lut[sh + 8];
                    const uint32_t lut[2] = {lt.x, lt.y};
                    const uint32_t w[4] = {cw[c].x, cw[c].y, cw[c].z, cw[c].w};
                    uint32_t o[8];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const uint32_t wl = w[i] << 4;
                        uint32_t sg0, sg1;
                        asm("prmt.b32 %0, %1, %2, 0xD9C8;" : "=r"(sg0) : "r"(wl), "r"(w[i]));
                        asm("prmt.b32 %0, %1, %2, 0xFBEA;" : "=r"(sg1) : "r"(wl), "r"(w[i]));
                        o[2 * i] = __byte_perm(lut[0], lut[1], w[i] & 0x7777u) | (sg0 & 0x80808080u);
                        o[2 * i + 1] = __byte_perm(lut[0], lut[1], (w[i] >> 16) & 0x7777u) | (sg1 & 0x80808080u);
                    }
                    // dims 32c .. 32c+15 are chunk 2c of the row, 32c+16 .. chunk 2c+1
                    *reinterpret_cast<uint4*>(row + (((2 * c) ^ (k & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4*>(row + (((2 * c + 1) ^ (k & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
                sKs[slot * kTileKeys + k] = ldexpf(1.f, Ek);
                tc::fence_proxy_async_smem();  // the rows are read by the MMAs (async proxy)
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&full[stage]);
                    tc::mbar_arrive(&sfull[slot]);
                    tc::mbar_arrive(&rempty[rs]);
                }
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

template <int NQ, int KF>
static cudaError_t run_indexer(const CUtensorMap& tm_keys, const CUtensorMap& tm_q, const IdxArgs& a, int grid,
                               cudaStream_t st) {
    using C = Cfg<NQ, KF>;
    {
        cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(indexer_tc_kernel<NQ, KF>), C::kSmem);
        if (e != cudaSuccess) return e;
    }
    indexer_tc_kernel<NQ, KF><<<grid, C::kThreads, C::kSmem, st>>>(tm_keys, tm_q, a);
    note_launch();
    return cudaGetLastError();
}

static std::atomic<int> g_withhold{0};

void set_indexer_withhold(int on) { g_withhold.store(on ? 1 : 0, std::memory_order_relaxed); }

// kf: kKeyBf16 (keys bf16 [B, n_cap, 128]), kKeyE4m3 (key codes [B, n_cap, 128]
// + key_scales), kKeyFp4 (keys: packed tiles [B, ceil(n_cap/128)]).  For the
// 8-bit formats q_idx holds the query codes and w_idx the head weights times
// the query head scales.
static cudaError_t launch_indexer_tc_kf(const Geometry& g, int kf, const void* q_idx, const float* w_idx, int HI,
                                        int dI, const void* keys, const float* key_scales, int64_t n_cap, int B,
                                        int Q, const int64_t* q_pos, uint32_t* status, float* scores, int64_t ld,
                                        cudaStream_t st, bool* launched) {
    *launched = false;
    const bool f8 = kf != kKeyBf16;
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
    bool maps;
    if (kf == kKeyFp4) {
        // packed tiles as rows of 128 bytes, one box of kFp4Rows rows a tile,
        // copied linearly (tiled TMA moves them several times faster than
        // one bulk copy a tile)
        const uint64_t pd[2] = {128, (uint64_t)B * (uint64_t)((n_cap + kTileKeys - 1) / kTileKeys) * kFp4Rows};
        const uint64_t ps[1] = {128};
        const uint32_t pbox[2] = {128, (uint32_t)kFp4Rows};
        maps = make_tmap_u8_linear(&tm_keys, keys, 2, pd, ps, pbox) && make_tmap_u8(&tm_q, q_idx, 2, qd, qs, qbox);
    } else if (f8) {
        maps = make_tmap_u8(&tm_keys, keys, 3, kd, ks, kb) && make_tmap_u8(&tm_q, q_idx, 2, qd, qs, qbox);
    } else {
        maps = make_tmap_bf16(&tm_keys, keys, 3, kd, ks, kb) && make_tmap_bf16(&tm_q, q_idx, 2, qd, qs, qbox);
    }
    if (!maps) return f8 ? cudaErrorInvalidValue : cudaSuccess;  // bf16: the CUDA-core path runs instead
    IdxArgs a;
    a.w_idx = w_idx;
    a.key_scales = kf == kKeyE4m3 ? key_scales : nullptr;
    a.key_pack = kf == kKeyFp4 ? reinterpret_cast<const uint8_t*>(keys) : nullptr;
    a.q_pos = q_pos;
    a.scores = scores;
    a.ld = ld;
    a.n_cap = n_cap;
    a.qps = qps;
    a.m = g.m;
    a.n_tiles = (int)((n_cap + kTileKeys - 1) / kTileKeys);
    a.total_units = (int64_t)(Q / NQ) * a.n_tiles;
    a.status = status;
    a.withhold = g_withhold.load(std::memory_order_relaxed);
    const int64_t sms = num_sms();
    const int grid = (int)(a.total_units < sms ? a.total_units : sms);
    cudaError_t e;
    if (kf == kKeyFp4)
        e = NQ == 1 ? run_indexer<1, kKeyFp4>(tm_keys, tm_q, a, grid, st) : run_indexer<4, kKeyFp4>(tm_keys, tm_q, a, grid, st);
    else if (kf == kKeyE4m3)
        e = NQ == 1 ? run_indexer<1, kKeyE4m3>(tm_keys, tm_q, a, grid, st) : run_indexer<4, kKeyE4m3>(tm_keys, tm_q, a, grid, st);
    else
        e = NQ == 1 ? run_indexer<1, kKeyBf16>(tm_keys, tm_q, a, grid, st) : run_indexer<4, kKeyBf16>(tm_keys, tm_q, a, grid, st);
    if (e == cudaSuccess) *launched = true;
    return e;
}

cudaError_t launch_indexer_tc(const Geometry& g, const void* q_idx, const float* w_idx, int HI,
                              int dI, const void* keys, const float* key_scales, int64_t n_cap, int B,
                              int Q, const int64_t* q_pos, uint32_t* status, float* scores, int64_t ld,
                              cudaStream_t st, bool* launched) {
    return launch_indexer_tc_kf(g, key_scales != nullptr ? kKeyE4m3 : kKeyBf16, q_idx, w_idx, HI, dI, keys,
                                key_scales, n_cap, B, Q, q_pos, status, scores, ld, st, launched);
}

cudaError_t launch_indexer_tc_fp4(const Geometry& g, const uint8_t* q8, const float* w_eff, const uint8_t* key_pack,
                                  int64_t n_cap, int B, int Q, const int64_t* q_pos, uint32_t* status,
                                  float* scores, int64_t ld, cudaStream_t st, bool* launched) {
    return launch_indexer_tc_kf(g, kKeyFp4, q8, w_eff, kHI, kDI, key_pack, nullptr, n_cap, B, Q, q_pos, status,
                                scores, ld, st, launched);
}

}  // namespace csa
