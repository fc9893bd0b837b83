// k_out_proj.cu -- grouped output projection on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA).
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 4: Grouped Output
// Projection": the 512-dim heads are projected in groups to cut the cost.  The
// H heads form G consecutive groups; group g's concatenated head outputs x_g
// (K = H/G * D values a query) are projected by its own matrix W_g [d_g, K]:
//   out[q, g*d_g + n] = sum_k x_g[q, k] * W_g[n, k]
// a block-diagonal projection, G times cheaper than a dense one of the same
// output width.  Each group is a dense bf16 GEMM with fp32 accumulation:
// tiles of 128 queries x BN outputs, K in stages of 64 (128-byte rows, the
// 128-byte swizzle) loaded by TMA into a four-stage ring, M = 128 x N = BN
// MMAs issued by one thread into a TMEM accumulator, and four epilogue warps
// (one per TMEM lane quarter) converting a row's outputs to bf16.  Decode
// (a few dozen queries) streams the weights with narrow tiles (BN = 64) and,
// given a float32 scratch, splits each group's K over four CTAs whose
// products are added there atomically and rounded to bf16 by a second pass,
// so that 256 CTAs share the stream; prefill uses BN = 256.  Query rows past
// Q read as zeros (TMA fill) and are not stored.  Every wait is bounded: on a
// timeout the kernel flags CSA_DEV_TIMEOUT, every role leaves, outstanding
// MMAs are waited for and TMEM is freed.
#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa {

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

namespace {

constexpr int kBM = 128;  // queries per tile (MMA M)
constexpr int kBK = 64;   // K per stage: one 128-byte row of bf16
constexpr int kOpStages = 4;
constexpr int kOpThreads = 64 + 128;

template <int BN>
struct OpCfg {
    static constexpr uint32_t kABytes = kBM * kBK * 2;
    static constexpr uint32_t kBBytes = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr size_t kSmem = 1024 + (size_t)kOpStages * kStageBytes;
    static constexpr uint32_t kTmemCols = BN;  // a power of two >= 32
    static constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, BN);
};

struct OpArgs {
    uint16_t* out;  // [Q, G * d_g] bf16
    float* acc;     // split K: [Q, G * d_g] float32 sums (zeroed first); else nullptr
    int Q, d_g, K;  // K = H/G * D
    int splits;     // CTAs a group's K is split over (grid z = G * splits)
    int64_t ldo;    // G * d_g
    uint32_t* status;
};

}  // namespace

template <int BN>
__global__ void __launch_bounds__(kOpThreads, 1)
    out_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ OpArgs a) {
    using C = OpCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[kOpStages], empty[kOpStages], acc_full, mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_sh;
    volatile int* abort_flag = &abort_sh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * BN, g = blockIdx.z / a.splits;
    const int split = blockIdx.z % a.splits;
    const int nk = a.K / kBK / a.splits;  // K steps of this CTA, from kt0
    const int kt0 = split * nk;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kOpStages; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(&acc_full, 1);
        tc::mbar_init(&mma_done, 1);
        abort_sh = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_slot, C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        tc::tma_prefetch_map(&tm_x);
        tc::tma_prefetch_map(&tm_w);
        uint32_t issued = 0;
        for (int kt = 0; kt < nk; kt++) {
            const int s = kt % kOpStages;
            if (!tc::mbar_wait(&empty[s], ((kt / kOpStages) & 1u) ^ 1u, abort_flag, a.status)) break;
            tc::mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            uint8_t* st = sm + s * C::kStageBytes;
            tc::tma_load_2d(st, &tm_x, &full[s], g * a.K + (kt0 + kt) * kBK, m0);
            tc::tma_load_3d(st + C::kABytes, &tm_w, &full[s], (kt0 + kt) * kBK, n0, g);
            ++issued;
        }
        // leave no copy in flight: every stage's newest fill has landed
        for (uint32_t kt = issued > kOpStages ? issued - kOpStages : 0; kt < issued; kt++)
            if (!tc::mbar_drain(&full[kt % kOpStages], (kt / kOpStages) & 1u)) atomicOr(a.status, CSA_DEV_TIMEOUT);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issue
        for (int kt = 0; kt < nk; kt++) {
            const int s = kt % kOpStages;
            if (!tc::mbar_wait(&full[s], (kt / kOpStages) & 1u, abort_flag, a.status)) break;
            tc::fence_after_sync();
            const uint32_t sa = tc::smem_u32(sm + s * C::kStageBytes);
            const uint32_t sb = sa + C::kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; kk++)
                tc::mma_bf16_ss(tmem, tc::sdesc_kmajor_sw128(sa + kk * 32), tc::sdesc_kmajor_sw128(sb + kk * 32),
                                C::idesc, (kt | kk) != 0 ? 1u : 0u);
            tc::mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        tc::mma_commit(&acc_full);
        // every MMA issued must be complete before TMEM is freed
        tc::mma_commit(&mma_done);
        if (!tc::mbar_drain(&mma_done, 0)) atomicOr(a.status, CSA_DEV_TIMEOUT);
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue: one query row per thread
        const int quarter = warp & 3;
        const int row = m0 + quarter * 32 + lane;
        int ok = 1;
        if (lane == 0) ok = tc::mbar_wait(&acc_full, 0, abort_flag, a.status) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && !*abort_flag) {
            tc::fence_after_sync();
            uint16_t* dst = a.out + (int64_t)row * a.ldo + (int64_t)g * a.d_g + n0;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                tc::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
                tc::tmem_ld_wait();
                if (a.acc != nullptr) {
                    if (row < a.Q && n0 + c0 < a.d_g) {  // this split's share of the sum
                        float* dacc = a.acc + (int64_t)row * a.ldo + (int64_t)g * a.d_g + n0 + c0;
#pragma unroll
                        for (int j = 0; j < 32; j++) atomicAdd(dacc + j, v[j]);
                    }
                } else if (row < a.Q && n0 + c0 < a.d_g) {
                    uint32_t p[16];
#pragma unroll
                    for (int j = 0; j < 16; j++)
                        p[j] = (uint32_t)f32_to_bf16_rn(v[2 * j]) | ((uint32_t)f32_to_bf16_rn(v[2 * j + 1]) << 16);
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                    for (int j = 0; j < 4; j++) d4[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
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

// Decode-sized calls with a float32 scratch: the weights are the M = 128 side
// (swap-AB: D^T[128 outputs, NQ queries] = W_g tile x X_g^T), so every byte a
// stage holds is used (the query side is NQ rows, not a 128-row tile of
// which most rows are past Q), and each group's K is split over `splits`
// CTAs whose products are added atomically in the scratch.  Same roles as
// above; the epilogue thread of TMEM lane r owns output r of the tile and
// adds its NQ query values (lanes hold consecutive outputs: coalesced).
constexpr int kSwStages = 5;

template <int NQ>
struct SwCfg {
    static constexpr uint32_t kWBytes = kBM * kBK * 2;  // 128 outputs x 64 K
    static constexpr uint32_t kXBytes = NQ * kBK * 2;   // NQ queries x 64 K
    static constexpr uint32_t kStageBytes = kWBytes + kXBytes;
    static constexpr size_t kSmem = 1024 + (size_t)kSwStages * kStageBytes;
    static constexpr uint32_t kTmemCols = NQ;  // a power of two >= 32
    static constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, NQ);
};

template <int NQ>
__global__ void __launch_bounds__(kOpThreads, 1)
    out_proj_swap_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                         const __grid_constant__ OpArgs a) {
    using C = SwCfg<NQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[kSwStages], empty[kSwStages], acc_full, mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_sh;
    volatile int* abort_flag = &abort_sh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = blockIdx.x * kBM, g = blockIdx.y, split = blockIdx.z;
    const int nk = a.K / kBK / a.splits;  // K steps of this CTA, from kt0
    const int kt0 = split * nk;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSwStages; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(&acc_full, 1);
        tc::mbar_init(&mma_done, 1);
        abort_sh = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_slot, C::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        tc::tma_prefetch_map(&tm_x);
        tc::tma_prefetch_map(&tm_w);
        uint32_t issued = 0;
        for (int kt = 0; kt < nk; kt++) {
            const int s = kt % kSwStages;
            if (!tc::mbar_wait(&empty[s], ((kt / kSwStages) & 1u) ^ 1u, abort_flag, a.status)) break;
            tc::mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            uint8_t* st = sm + s * C::kStageBytes;
            tc::tma_load_3d(st, &tm_w, &full[s], (kt0 + kt) * kBK, o0, g);
            tc::tma_load_2d(st + C::kWBytes, &tm_x, &full[s], g * a.K + (kt0 + kt) * kBK, 0);
            ++issued;
        }
        for (uint32_t kt = issued > kSwStages ? issued - kSwStages : 0; kt < issued; kt++)
            if (!tc::mbar_drain(&full[kt % kSwStages], (kt / kSwStages) & 1u)) atomicOr(a.status, CSA_DEV_TIMEOUT);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issue
        for (int kt = 0; kt < nk; kt++) {
            const int s = kt % kSwStages;
            if (!tc::mbar_wait(&full[s], (kt / kSwStages) & 1u, abort_flag, a.status)) break;
            tc::fence_after_sync();
            const uint32_t sw = tc::smem_u32(sm + s * C::kStageBytes);
            const uint32_t sx = sw + C::kWBytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; kk++)
                tc::mma_bf16_ss(tmem, tc::sdesc_kmajor_sw128(sw + kk * 32), tc::sdesc_kmajor_sw128(sx + kk * 32),
                                C::idesc, (kt | kk) != 0 ? 1u : 0u);
            tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(&acc_full);
        tc::mma_commit(&mma_done);
        if (!tc::mbar_drain(&mma_done, 0)) atomicOr(a.status, CSA_DEV_TIMEOUT);
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue: output o0 + r, r = this thread's TMEM lane
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        int ok = 1;
        if (lane == 0) ok = tc::mbar_wait(&acc_full, 0, abort_flag, a.status) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && !*abort_flag) {
            tc::fence_after_sync();
            float* dacc = a.acc + (int64_t)g * a.d_g + o0 + r;
#pragma unroll 1
            for (int q0 = 0; q0 < NQ; q0 += 32) {
                float v[32];
                tc::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)q0, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; j++)
                    if (q0 + j < a.Q) atomicAdd(dacc + (int64_t)(q0 + j) * a.ldo, v[j]);
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

// The split products' float32 sums rounded to bf16 (n values).
__global__ void __launch_bounds__(256) out_proj_round_kernel(const float* __restrict__ acc,
                                                             uint16_t* __restrict__ out, int64_t n) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i + 3 < n) {
        const float4 v = *reinterpret_cast<const float4*>(acc + i);
        *reinterpret_cast<uint2*>(out + i) =
            make_uint2((uint32_t)f32_to_bf16_rn(v.x) | ((uint32_t)f32_to_bf16_rn(v.y) << 16),
                       (uint32_t)f32_to_bf16_rn(v.z) | ((uint32_t)f32_to_bf16_rn(v.w) << 16));
    } else {
        for (int64_t j = i; j < n; j++) out[j] = f32_to_bf16_rn(acc[j]);
    }
}

bool out_proj_supported(int H, int D, int G, int d_g) {
    if (G < 1 || H % G != 0) return false;
    const int K = H / G * D;
    return K % kBK == 0 && d_g >= 64 && d_g % 64 == 0;
}

cudaError_t launch_out_proj(const void* o, int Q, int H, int D, int G, const void* w, int d_g, void* out,
                            float* acc, uint32_t* status, cudaStream_t st) {
    if (Q == 0) return cudaSuccess;
    const int K = H / G * D;
    const int64_t n_out = (int64_t)Q * G * d_g;
    if (acc != nullptr && Q <= kBM && d_g % kBM == 0) {
        // swap-AB, K split so that the grid covers the SMs about twice
        int splits = 1;
        const int64_t tiles = (int64_t)(d_g / kBM) * G, want = 2LL * num_sms();
        while (splits < 16 && tiles * splits * 2 <= want && (K / kBK) % (splits * 2) == 0) splits *= 2;
        const int nq = Q <= 32 ? 32 : (Q <= 64 ? 64 : 128);
        CUtensorMap tm_x, tm_w;
        {
            const uint64_t d[2] = {(uint64_t)H * D, (uint64_t)Q};
            const uint64_t sd[1] = {(uint64_t)H * D * 2};
            const uint32_t box[2] = {(uint32_t)kBK, (uint32_t)nq};
            if (!make_tmap_bf16(&tm_x, o, 2, d, sd, box)) return cudaErrorInvalidValue;
        }
        {
            const uint64_t d[3] = {(uint64_t)K, (uint64_t)d_g, (uint64_t)G};
            const uint64_t sd[2] = {(uint64_t)K * 2, (uint64_t)d_g * K * 2};
            const uint32_t box[3] = {(uint32_t)kBK, (uint32_t)kBM, 1};
            if (!make_tmap_bf16(&tm_w, w, 3, d, sd, box)) return cudaErrorInvalidValue;
        }
        OpArgs a;
        a.out = reinterpret_cast<uint16_t*>(out);
        a.acc = acc;
        a.Q = Q;
        a.d_g = d_g;
        a.K = K;
        a.splits = splits;
        a.ldo = (int64_t)G * d_g;
        a.status = status;
        cudaError_t e = cudaMemsetAsync(acc, 0, (size_t)n_out * sizeof(float), st);
        if (e != cudaSuccess) return e;
        const dim3 grid((unsigned)(d_g / kBM), (unsigned)G, (unsigned)splits);
        if (nq == 32) {
            e = set_smem_attr(reinterpret_cast<const void*>(out_proj_swap_kernel<32>), SwCfg<32>::kSmem);
            if (e == cudaSuccess)
                out_proj_swap_kernel<32><<<grid, kOpThreads, SwCfg<32>::kSmem, st>>>(tm_x, tm_w, a);
        } else if (nq == 64) {
            e = set_smem_attr(reinterpret_cast<const void*>(out_proj_swap_kernel<64>), SwCfg<64>::kSmem);
            if (e == cudaSuccess)
                out_proj_swap_kernel<64><<<grid, kOpThreads, SwCfg<64>::kSmem, st>>>(tm_x, tm_w, a);
        } else {
            e = set_smem_attr(reinterpret_cast<const void*>(out_proj_swap_kernel<128>), SwCfg<128>::kSmem);
            if (e == cudaSuccess)
                out_proj_swap_kernel<128><<<grid, kOpThreads, SwCfg<128>::kSmem, st>>>(tm_x, tm_w, a);
        }
        if (e != cudaSuccess) return e;
        note_launch();
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const int64_t blocks = (n_out + 4 * 256 - 1) / (4 * 256);
        out_proj_round_kernel<<<(unsigned)blocks, 256, 0, st>>>(acc, reinterpret_cast<uint16_t*>(out), n_out);
        note_launch();
        return cudaGetLastError();
    }
    const int splits = 1;
    acc = nullptr;
    // narrow tiles for a few queries (more CTAs stream the weights), wide ones otherwise
    const bool narrow = Q <= kBM || d_g % 256 != 0;
    CUtensorMap tm_x, tm_w;
    {
        const uint64_t d[2] = {(uint64_t)H * D, (uint64_t)Q};
        const uint64_t s[1] = {(uint64_t)H * D * 2};
        const uint32_t box[2] = {(uint32_t)kBK, (uint32_t)kBM};
        if (!make_tmap_bf16(&tm_x, o, 2, d, s, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t d[3] = {(uint64_t)K, (uint64_t)d_g, (uint64_t)G};
        const uint64_t s[2] = {(uint64_t)K * 2, (uint64_t)d_g * K * 2};
        const uint32_t box[3] = {(uint32_t)kBK, narrow ? 64u : 256u, 1};
        if (!make_tmap_bf16(&tm_w, w, 3, d, s, box)) return cudaErrorInvalidValue;
    }
    OpArgs a;
    a.out = reinterpret_cast<uint16_t*>(out);
    a.acc = acc;
    a.Q = Q;
    a.d_g = d_g;
    a.K = K;
    a.splits = splits;
    a.ldo = (int64_t)G * d_g;
    a.status = status;
    const dim3 grid((unsigned)((Q + kBM - 1) / kBM), (unsigned)(d_g / (narrow ? 64 : 256)), (unsigned)(G * splits));
    cudaError_t e;
    if (narrow) {
        e = set_smem_attr(reinterpret_cast<const void*>(out_proj_kernel<64>), OpCfg<64>::kSmem);
        if (e != cudaSuccess) return e;
        out_proj_kernel<64><<<grid, kOpThreads, OpCfg<64>::kSmem, st>>>(tm_x, tm_w, a);
    } else {
        e = set_smem_attr(reinterpret_cast<const void*>(out_proj_kernel<256>), OpCfg<256>::kSmem);
        if (e != cudaSuccess) return e;
        out_proj_kernel<256><<<grid, kOpThreads, OpCfg<256>::kSmem, st>>>(tm_x, tm_w, a);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa
