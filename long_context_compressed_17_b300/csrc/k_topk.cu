// k_topk.cu -- exact top-k selection over indexer scores.
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 2": keep the top-K
// compressed blocks per query; ties go to the lower block index.  The scores
// are mapped to order-preserving 32-bit keys and a radix select (four 8-bit
// digits, most significant first) finds the k-th largest key T.  Every block
// with key > T is kept, and of the blocks with key == T the lowest indices
// fill the remaining slots.  The output lists the kept blocks in ascending
// index order.
//
// One CTA of 1024 threads per query row; each thread owns a contiguous index
// range so that the final compaction preserves index order with one block scan.
#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int kTopkThreads = 1024;

// Order-preserving key of a float score (both zeros share one key).
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f == 0.f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan over the CTA (kTopkThreads threads); returns the prefix and
// writes the total to *total.  `sw` holds 32 ints of shared scratch.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sw, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) sw[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = sw[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sw[lane] = w;  // inclusive per-warp totals
    }
    __syncthreads();
    int before = (warp > 0 ? sw[warp - 1] : 0) + x - v;
    *total = sw[31];
    return before;
}

__global__ void __launch_bounds__(kTopkThreads)
    topk_radix_kernel(const float* __restrict__ scores, int64_t n_cap_pad, int64_t n_cap,
                      const int64_t* __restrict__ q_pos, int m, int k, int32_t* __restrict__ idx,
                      float* __restrict__ sel) {
    __shared__ int hist[256];
    __shared__ int sw[32];
    __shared__ uint32_t s_digit;
    __shared__ int s_above;
    const int tid = threadIdx.x;
    const int64_t q = blockIdx.x;
    const float* s = scores + q * n_cap_pad;
    int32_t* oi = idx + q * k;
    float* os = sel ? sel + q * k : nullptr;
    int64_t n = (q_pos[q] + 1) / m;
    if (n > n_cap) n = n_cap;  // flagged by the indexer
    if (n < 0) n = 0;

    if (n <= k) {  // every complete block is kept
        for (int64_t j = tid; j < k; j += kTopkThreads) {
            oi[j] = j < n ? (int32_t)j : -1;
            if (os) os[j] = j < n ? s[j] : -INFINITY;
        }
        return;
    }

    const int64_t per = (n + kTopkThreads - 1) / kTopkThreads;
    const int64_t lo = tid * per;
    const int64_t hi = min(n, lo + per);
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        for (int64_t j = lo; j < hi; j++) {
            uint32_t u = score_key(s[j]);
            if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns digits 8l .. 8l+7; suffix sums from the top digit down
            int c[8], loc = 0;
#pragma unroll
            for (int e = 0; e < 8; e++) {
                c[e] = hist[8 * tid + e];
                loc += c[e];
            }
            int suf = loc;  // inclusive suffix over lanes >= tid
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_down_sync(0xffffffffu, suf, o);
                if (tid + o < 32) suf += y;
            }
            int above = suf - loc;  // keys with a digit in higher lanes
#pragma unroll
            for (int e = 7; e >= 0; e--) {
                if (above < remaining && above + c[e] >= remaining) {
                    s_digit = (uint32_t)(8 * tid + e);
                    s_above = above;
                }
                above += c[e];
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 255u << shift;
        remaining -= s_above;
        __syncthreads();
    }
    const uint32_t T = prefix;  // key of the k-th largest score
    // remaining = number of blocks with key == T that are kept (lowest indices)
    int gt = 0, eq = 0;
    for (int64_t j = lo; j < hi; j++) {
        uint32_t u = score_key(s[j]);
        gt += (u > T);
        eq += (u == T);
    }
    int tot;
    int eq_before = block_exclusive_scan(eq, sw, &tot);
    int take = min(max(remaining - eq_before, 0), eq);
    int out_pos = block_exclusive_scan(gt + take, sw, &tot);
    for (int64_t j = lo; j < hi; j++) {
        float f = s[j];
        uint32_t u = score_key(f);
        bool keep = u > T;
        if (u == T && take > 0) {
            keep = true;
            take--;
        }
        if (keep) {
            oi[out_pos] = (int32_t)j;
            if (os) os[out_pos] = f;
            out_pos++;
        }
    }
}

cudaError_t launch_topk(const Geometry& g, const float* scores, int64_t ld, int64_t n_cap, int Q,
                        const int64_t* q_pos, int32_t* idx, float* sel, cudaStream_t st) {
    if (Q == 0) return cudaSuccess;
    topk_radix_kernel<<<Q, kTopkThreads, 0, st>>>(scores, ld, n_cap, q_pos, g.m, g.k, idx, sel);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa
