// k_compress.cu -- block compressor (softmax pooling + RMSNorm + partial RoPE)
// and the cache-row writer.
//
// Block compression follows "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA
// "Step 1: KV 压缩" (every m tokens pooled into one entry by an attention-like
// mechanism with learnable weights) and HCA (m' = 128); the entry is
// RMSNorm-ed and rotated on its last 64 dims at the block's last position
// (四项关键 Trick).  The mixed FP8/BF16 row format follows
// "DeepSeek-V4 技术报告深度解析" §2.1.4 "KV 缓存精度".
//
// Both kernels are HBM streams with a few FLOPs per byte: plain CUDA-core code,
// coalesced row reads, one CTA per output entry; the compressor stages its
// block of raw rows in shared memory so HBM is read once.
#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa {

constexpr int kCompressThreads = 256;

// This thread's RoPE frequency when it is one of the 32 that rotate a pair.
__device__ __forceinline__ double rope_theta_of(const RopeTheta& theta) {
    return threadIdx.x < kRopeDims / 2 ? theta.t[threadIdx.x] : 0.0;
}
constexpr size_t kCompressStageMax = 160 * 1024;  // raw block staged in smem up to this size

// row[0, D) holds a pooled vector (shared memory) and ss each thread's partial
// sum of its squares: RMSNorm it, rotate its last 64 dims at position pos and
// store it into a cache row at dst (whole CTA; red: 32 floats of scratch;
// theta_j: thread j < 32's RoPE frequency).  Out of line: the kernels call it
// from up to four places, and the inlined copies (with the sine, cosine and
// FP8 packing code) made them 77-111 KB of code that each CTA runs once.
template <int NT>
__device__ __noinline__ void norm_rope_store(float* row, float ss, float* red, int D, float eps, double pos,
                                             double theta_j, int kvfmt, uint8_t* dst) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nwarps = NT / 32;
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float tot = 0.f;
        for (int w = 0; w < nwarps; w++) tot += red[w];
        red[31] = 1.f / sqrtf(tot / (float)D + eps);
    }
    __syncthreads();
    const float rn = red[31];
    for (int d = tid; d < D; d += NT) row[d] *= rn;
    __syncthreads();
    if (tid < kRopeDims / 2) {
        const int j = tid;
        float c, s;
        rope_cs(pos, theta_j, &c, &s);
        const int d0 = D - kRopeDims + 2 * j;
        const float x0 = row[d0], x1 = row[d0 + 1];
        row[d0] = x0 * c - x1 * s;
        row[d0 + 1] = x0 * s + x1 * c;
    }
    __syncthreads();
    if (warp == 0) warp_pack_row(row, D, kvfmt, dst);
}

// The window row of raw token `tok` (RMSNorm, RoPE at pos; what the
// compressor with m = 1 writes), through row[0, D).
template <int NT>
__device__ void window_row(const uint8_t* tok, int act, float* row, float* red, int D, float eps, double pos,
                           const RopeTheta& theta, int kvfmt, uint8_t* dst) {
    float ss = 0.f;
    for (int d = threadIdx.x; d < D; d += NT) {
        const float c = load_act(tok, act, d);
        row[d] = c;
        ss = fmaf(c, c, ss);
    }
    norm_rope_store<NT>(row, ss, red, D, eps, pos, rope_theta_of(theta), kvfmt, dst);
}

// The block of m raw rows at src (shared memory or global) pooled into one
// entry and stored at dst: pooling scores z_t = kv_t . w_z + bias[t], softmax
// over the block, the weighted sum, RMSNorm and RoPE at `pos` (whole CTA; z:
// m floats, row: D floats, red: 32 floats of shared scratch).  m = 1 is a
// window row: its single weight is exactly 1.
template <int NT>
__device__ __forceinline__ void pool_block_store(const uint8_t* src, int act, int64_t act_row_bytes, int D, int m,
                                                 const float* __restrict__ w_z, const float* __restrict__ bias,
                                                 float* z, float* row, float* red, float eps, double pos,
                                                 const RopeTheta& theta, int kvfmt, uint8_t* dst) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nwarps = NT / 32;
    if (m == 1) {
        // a single token: its pooling weight is exactly 1 (window rows)
        if (tid == 0) z[0] = 1.f;
        __syncthreads();
    } else {
        // pooling scores z_t = kv_t . w_z + bias[t mod m]   (blocks start at multiples of m)
        for (int t = warp; t < m; t += nwarps) {
            const uint8_t* r = src + t * act_row_bytes;
            float acc = 0.f;
            for (int d = lane; d < D; d += 32) acc = fmaf(load_act(r, act, d), __ldg(w_z + d), acc);
            acc = warp_sum(acc);
            if (lane == 0) z[t] = acc + bias[t];
        }
        __syncthreads();
        // softmax over the block's tokens: z <- alpha
        if (warp == 0) {
            float zmax = -INFINITY;
            for (int t = lane; t < m; t += 32) zmax = fmaxf(zmax, z[t]);
            zmax = warp_max(zmax);
            float den = 0.f;
            for (int t = lane; t < m; t += 32) den += expf(z[t] - zmax);
            den = warp_sum(den);
            const float inv = 1.f / den;
            for (int t = lane; t < m; t += 32) z[t] = expf(z[t] - zmax) * inv;
        }
        __syncthreads();
    }
    // pooled vector and its sum of squares
    float ss = 0.f;
    for (int d = tid; d < D; d += NT) {
        float c = 0.f;
        for (int t = 0; t < m; t++) c = fmaf(z[t], load_act(src + t * act_row_bytes, act, d), c);
        row[d] = c;
        ss = fmaf(c, c, ss);
    }
    // RMSNorm, partial RoPE at the block's last position, store
    norm_rope_store<NT>(row, ss, red, D, eps, pos, rope_theta_of(theta), kvfmt, dst);
}

// grid (n_blocks_out, B).  Dynamic smem: (m + D + 32) floats, rounded up to
// 16 bytes, then (when `staged`) the block's m raw rows.
__global__ void __launch_bounds__(kCompressThreads)
    compress_kernel(const uint8_t* __restrict__ kv, int act, int64_t act_row_bytes,
                    int64_t kv_seq_bytes, int D, int m, int64_t pos0,
                    const float* __restrict__ w_z, const float* __restrict__ bias,
                    uint8_t* __restrict__ out, int kvfmt, int64_t kv_row_bytes,
                    int64_t out_seq_bytes, float eps, RopeTheta theta, int staged,
                    uint8_t* __restrict__ win_out, int64_t win_seq_bytes) {
    extern __shared__ __align__(16) float sm[];
    float* z = sm;            // [m] scores, then pooling weights
    float* row = sm + m;      // [D]
    float* red = row + D;     // [32]
    uint8_t* stage = reinterpret_cast<uint8_t*>(sm + ((m + D + 32 + 3) & ~3));
    const int tid = threadIdx.x;
    const int64_t b = blockIdx.x;
    const uint8_t* blk = kv + blockIdx.y * kv_seq_bytes + b * m * act_row_bytes;
    const uint8_t* src = blk;
    if (staged) {  // one coalesced pass over HBM; both sweeps below read smem
        const int64_t n16 = (int64_t)m * act_row_bytes / 16;
        const uint4* g = reinterpret_cast<const uint4*>(blk);
        uint4* s = reinterpret_cast<uint4*>(stage);
        for (int64_t i = tid; i < n16; i += kCompressThreads) s[i] = __ldg(g + i);
        __syncthreads();
        src = stage;
    }
    const double pos = (double)(pos0 + b * m + m - 1);
    pool_block_store<kCompressThreads>(src, act, act_row_bytes, D, m, w_z, bias, z, row, red, eps, pos, theta, kvfmt,
                     out + blockIdx.y * out_seq_bytes + b * kv_row_bytes);
    if (win_out != nullptr) {  // the window row of the block's last token
        __syncthreads();       // `row` is free again
        window_row<kCompressThreads>(src + (m - 1) * act_row_bytes, act, row, red, D, eps, pos, theta, kvfmt,
                   win_out + blockIdx.y * win_seq_bytes + b * kv_row_bytes);
    }
}

// Large blocks (HCA's m = 128) are split over a cluster of kSplit CTAs, each
// pooling m / kSplit tokens with its own softmax reference:
//   M_r = max z_t, S_r = sum e^(z_t - M_r), P_r = sum e^(z_t - M_r) kv_t
// (t in slice r).  Every CTA stores (M_r, S_r, P_r) into slot r of CTA 0's
// shared memory; after the cluster barrier CTA 0 merges them,
//   pooled = sum_r e^(M_r - M) P_r / sum_r e^(M_r - M) S_r,  M = max_r M_r,
// and finishes the entry as compress_kernel does (its pooled row goes where
// its raw slice was).  grid (n_blocks_out * kSplit, B), clusters of (kSplit,
// 1, 1).  Dynamic smem: the slice's raw rows (at least D floats), then
// m / kSplit scores, then kSplit slots of (4 + D) floats, then 32 floats.
constexpr int kSplit = 8;

// Shared memory of a cluster CTA: the slice's raw rows (at least D floats),
// then m / kSplit scores, then kSplit slots of (4 + D) floats, then 32 floats.
struct ClusterSmem {
    uint8_t* stage;
    float *z, *slots, *red;
    __device__ ClusterSmem(float* sm, int mt, int64_t act_row_bytes, int D) {
        const size_t slice_bytes = (size_t)mt * act_row_bytes;
        stage = reinterpret_cast<uint8_t*>(sm);
        z = reinterpret_cast<float*>(stage + ((slice_bytes + 15) & ~(size_t)15));
        slots = z + ((mt + 3) & ~3);  // [kSplit][4 + D]
        red = slots + kSplit * (4 + D);
    }
};

// The pooling of one block by a cluster of kSplit CTAs, CTA `rank` holding
// raw tokens rank*mt .. rank*mt+mt-1 of the block in c.stage (visible to the
// CTA).  CTA 0 stores the entry at entry_dst; CTA kSplit-1 stores the window
// row of the block's last token at win_dst (when not null).  Every CTA of the
// cluster must call this (one cluster barrier).
__device__ __forceinline__ void cluster_pool_store(const ClusterSmem& c, int rank, int act, int64_t act_row_bytes,
                                                   int D, int m, const float* __restrict__ w_z,
                                                   const float* __restrict__ bias, float eps, double pos,
                                                   const RopeTheta& theta, int kvfmt, uint8_t* entry_dst,
                                                   uint8_t* win_dst) {
    const int mt = m / kSplit;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nwarps = kCompressThreads / 32;
    const int t0 = rank * mt;  // first token of the slice within the block
    uint8_t* stage = c.stage;
    float* z = c.z;
    float* slots = c.slots;
    float* red = c.red;
    for (int t = warp; t < mt; t += nwarps) {
        const uint8_t* r = stage + t * act_row_bytes;
        float acc = 0.f;
        for (int d = lane; d < D; d += 32) acc = fmaf(load_act(r, act, d), __ldg(w_z + d), acc);
        acc = warp_sum(acc);
        if (lane == 0) z[t] = acc + bias[t0 + t];
    }
    __syncthreads();
    float zmax = -INFINITY;
    for (int t = 0; t < mt; t++) zmax = fmaxf(zmax, z[t]);  // every thread: mt is small
    __syncthreads();
    if (tid < mt) z[tid] = expf(z[tid] - zmax);
    __syncthreads();
    float zsum = 0.f;
    for (int t = 0; t < mt; t++) zsum += z[t];
    // this slice's (M_r, S_r, P_r) into slot `rank` of CTA 0
    const uint32_t slot0 = tc::mapa_shared(tc::smem_u32(slots + rank * (4 + D)), 0);
    for (int d4 = tid; d4 < D / 4; d4 += kCompressThreads) {
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            float cc = 0.f;
            for (int t = 0; t < mt; t++) cc = fmaf(z[t], load_act(stage + t * act_row_bytes, act, 4 * d4 + e), cc);
            p[e] = cc;
        }
        tc::st_cluster_v4(slot0 + 16u * (1 + d4), make_uint4(__float_as_uint(p[0]), __float_as_uint(p[1]),
                                                               __float_as_uint(p[2]), __float_as_uint(p[3])));
    }
    if (tid == 0)
        tc::st_cluster_v4(slot0, make_uint4(__float_as_uint(zmax), __float_as_uint(zsum), 0u, 0u));
    tc::cluster_sync();  // every slot of CTA 0 is written and visible
    if (rank == kSplit - 1 && win_dst != nullptr) {
        // the window row of the block's last token, the last row of this slice;
        // this CTA's own slots are unused and hold the row
        window_row<kCompressThreads>(stage + (mt - 1) * act_row_bytes, act, slots, red, D, eps, pos, theta, kvfmt,
                                     win_dst);
        return;
    }
    if (rank != 0) return;
    float* row = reinterpret_cast<float*>(stage);  // the raw slice is no longer needed
    float M = -INFINITY;
    for (int r = 0; r < kSplit; r++) M = fmaxf(M, slots[r * (4 + D)]);
    float S = 0.f;
    for (int r = 0; r < kSplit; r++) S += slots[r * (4 + D) + 1] * expf(slots[r * (4 + D)] - M);
    const float invS = 1.f / S;
    // merged pooled vector and its sum of squares
    float ss = 0.f;
    for (int d = tid; d < D; d += kCompressThreads) {
        float cc = 0.f;
        for (int r = 0; r < kSplit; r++) cc = fmaf(slots[r * (4 + D) + 4 + d], expf(slots[r * (4 + D)] - M), cc);
        cc *= invS;
        row[d] = cc;
        ss = fmaf(cc, cc, ss);
    }
    norm_rope_store<kCompressThreads>(row, ss, red, D, eps, pos, rope_theta_of(theta), kvfmt, entry_dst);
}

__global__ void __launch_bounds__(kCompressThreads)
    compress_cluster_kernel(const uint8_t* __restrict__ kv, int act, int64_t act_row_bytes,
                            int64_t kv_seq_bytes, int D, int m, int64_t pos0,
                            const float* __restrict__ w_z, const float* __restrict__ bias,
                            uint8_t* __restrict__ out, int kvfmt, int64_t kv_row_bytes,
                            int64_t out_seq_bytes, float eps, RopeTheta theta,
                            uint8_t* __restrict__ win_out, int64_t win_seq_bytes) {
    extern __shared__ __align__(16) float sm[];
    const int mt = m / kSplit;                          // tokens of this CTA
    const int rank = (int)tc::cluster_ctarank();        // == blockIdx.x % kSplit
    const int64_t b = blockIdx.x / kSplit;              // output entry
    const ClusterSmem c(sm, mt, act_row_bytes, D);
    {
        const uint4* g = reinterpret_cast<const uint4*>(kv + blockIdx.y * kv_seq_bytes +
                                                        (b * m + rank * mt) * act_row_bytes);
        uint4* st = reinterpret_cast<uint4*>(c.stage);
        const int64_t n16 = (int64_t)mt * act_row_bytes / 16;
        for (int64_t i = threadIdx.x; i < n16; i += kCompressThreads) st[i] = __ldg(g + i);
    }
    __syncthreads();
    cluster_pool_store(c, rank, act, act_row_bytes, D, m, w_z, bias, eps, (double)(pos0 + b * m + m - 1), theta,
                       kvfmt, out + blockIdx.y * out_seq_bytes + b * kv_row_bytes,
                       win_out != nullptr ? win_out + blockIdx.y * win_seq_bytes + b * kv_row_bytes : nullptr);
}

// ---------------------------------------------------------------- decode append
// One decode step's cache maintenance for a ragged batch: sequence s's newest
// token sits at position t = pos[s].  Its raw row goes to slot t mod m of the
// sequence's raw ring (the tokens of its current block, position p at slot
// p mod m), its window row RoPE(RMSNorm(kv_t), t) to row t mod n_win of the
// window ring, and when it completes a block (t + 1 a multiple of m) the
// block -- ring slots 0 .. m-2 and the new token -- is pooled into cache
// entry (t + 1)/m - 1.  The pooling and the window row are the compressor's
// own code (pool_block_store / cluster_pool_store, window_row).
struct DecodeAppend {
    const int64_t* pos;     // [B]
    const uint8_t* tok;     // [B] raw rows of the newest tokens (act format)
    uint8_t* ring;          // [B, m] raw rows (act format); nullptr when m == 1
    uint8_t* cache;         // [B, n_cap] stored rows
    int64_t n_cap;
    uint8_t* window;        // [B, n_win] stored rows; nullptr: no window
    int64_t n_win;
    uint32_t* status;
};

// Position checks of the step: the token's slot in its block and whether it
// completes a block whose entry fits in the cache (flagged otherwise).
__device__ __forceinline__ bool append_completes(const DecodeAppend& d, int64_t t, int m, bool report) {
    if ((t + 1) % m != 0) return false;
    if ((t + 1) / m > d.n_cap) {
        if (report) atomicOr(d.status, CSA_DEV_BAD_POSITION);
        return false;
    }
    return true;
}

// grid (B); dynamic smem: (m + D + 32) floats rounded up to 16 bytes, then m raw rows.
// kAppendThreads threads and at most 48 registers each: a CTA fits on an SM
// beside one of the indexer or the top-k, which the append runs beside.
constexpr int kAppendThreads = 128;
__global__ void __launch_bounds__(kAppendThreads, 10)
    append_step_kernel(const DecodeAppend d, int act, int64_t act_row_bytes, int D, int m,
                       const float* __restrict__ w_z, const float* __restrict__ bias, int kvfmt,
                       int64_t kv_row_bytes, float eps, RopeTheta theta) {
    extern __shared__ __align__(16) float sm[];
    float* z = sm;
    float* row = sm + m;
    float* red = row + D;
    uint8_t* stage = reinterpret_cast<uint8_t*>(sm + ((m + D + 32 + 3) & ~3));
    const int tid = threadIdx.x;
    const int64_t s = blockIdx.x;
    const int64_t t = d.pos[s];
    if (t < 0) {
        if (tid == 0) atomicOr(d.status, CSA_DEV_BAD_POSITION);
        return;
    }
    const bool complete = append_completes(d, t, m, tid == 0);
    const int64_t n16 = act_row_bytes / 16;
    uint4* last = reinterpret_cast<uint4*>(stage + (m - 1) * act_row_bytes);
    {
        const uint4* g = reinterpret_cast<const uint4*>(d.tok + s * act_row_bytes);
        for (int64_t i = tid; i < n16; i += kAppendThreads) last[i] = __ldg(g + i);
    }
    if (complete && m > 1) {  // the block's earlier tokens, written by earlier steps
        const uint4* g = reinterpret_cast<const uint4*>(d.ring + s * m * act_row_bytes);
        uint4* st = reinterpret_cast<uint4*>(stage);
        for (int64_t i = tid; i < (int64_t)(m - 1) * n16; i += kAppendThreads) st[i] = __ldg(g + i);
    }
    __syncthreads();
    if (m > 1) {  // the new token into its slot of the raw ring
        uint4* g = reinterpret_cast<uint4*>(d.ring + (s * m + t % m) * act_row_bytes);
        for (int64_t i = tid; i < n16; i += kAppendThreads) g[i] = last[i];
    }
    if (complete) {
        pool_block_store<kAppendThreads>(stage, act, act_row_bytes, D, m, w_z, bias, z, row, red, eps, (double)t, theta, kvfmt,
                         d.cache + (s * d.n_cap + (t + 1) / m - 1) * kv_row_bytes);
        __syncthreads();  // `row` is free again
    }
    if (d.window != nullptr)
        window_row<kAppendThreads>(stage + (m - 1) * act_row_bytes, act, row, red, D, eps, (double)t, theta, kvfmt,
                   d.window + (s * d.n_win + t % d.n_win) * kv_row_bytes);
}

// The same for blocks split over a cluster of kSplit CTAs: grid (kSplit, B),
// clusters of (kSplit, 1, 1).  A step that completes no block is done by the
// last CTA alone (ring slot and window row); the others leave at once.  Every
// branch before the cluster barrier depends on the sequence only, so all CTAs
// of a cluster take it together.
__global__ void __launch_bounds__(kCompressThreads)
    append_cluster_kernel(const DecodeAppend d, int act, int64_t act_row_bytes, int D, int m,
                          const float* __restrict__ w_z, const float* __restrict__ bias, int kvfmt,
                          int64_t kv_row_bytes, float eps, RopeTheta theta) {
    extern __shared__ __align__(16) float sm[];
    const int mt = m / kSplit;
    const int rank = (int)tc::cluster_ctarank();
    const int64_t s = blockIdx.y;
    const int64_t t = d.pos[s];
    const int tid = threadIdx.x;
    if (t < 0) {
        if (rank == 0 && tid == 0) atomicOr(d.status, CSA_DEV_BAD_POSITION);
        return;
    }
    const bool complete = append_completes(d, t, m, rank == 0 && tid == 0);
    const ClusterSmem c(sm, mt, act_row_bytes, D);
    const int64_t n16 = act_row_bytes / 16;
    const uint4* tok = reinterpret_cast<const uint4*>(d.tok + s * act_row_bytes);
    uint4* slot = reinterpret_cast<uint4*>(d.ring + (s * m + t % m) * act_row_bytes);
    uint8_t* win_dst = d.window != nullptr ? d.window + (s * d.n_win + t % d.n_win) * kv_row_bytes : nullptr;
    if (!complete) {
        if (rank != kSplit - 1) return;
        uint4* st = reinterpret_cast<uint4*>(c.stage);
        for (int64_t i = tid; i < n16; i += kCompressThreads) st[i] = __ldg(tok + i);
        __syncthreads();
        for (int64_t i = tid; i < n16; i += kCompressThreads) slot[i] = st[i];
        if (win_dst != nullptr)
            window_row<kCompressThreads>(c.stage, act, c.slots, c.red, D, eps, (double)t, theta, kvfmt, win_dst);
        return;
    }
    {  // slice rank of the block: ring slots rank*mt .. ; the last is the new token
        const uint4* g = reinterpret_cast<const uint4*>(d.ring + (s * m + rank * mt) * act_row_bytes);
        uint4* st = reinterpret_cast<uint4*>(c.stage);
        const int64_t n_ring = (int64_t)(rank == kSplit - 1 ? mt - 1 : mt) * n16;
        for (int64_t i = tid; i < n_ring; i += kCompressThreads) st[i] = __ldg(g + i);
        if (rank == kSplit - 1)
            for (int64_t i = tid; i < n16; i += kCompressThreads) st[n_ring + i] = __ldg(tok + i);
    }
    __syncthreads();
    if (rank == kSplit - 1) {
        const uint4* st = reinterpret_cast<const uint4*>(c.stage + (mt - 1) * act_row_bytes);
        for (int64_t i = tid; i < n16; i += kCompressThreads) slot[i] = st[i];
    }
    cluster_pool_store(c, rank, act, act_row_bytes, D, m, w_z, bias, eps, (double)t, theta, kvfmt,
                       d.cache + (s * d.n_cap + (t + 1) / m - 1) * kv_row_bytes, win_dst);
}

// one warp per row; dynamic smem: 4 warps x D floats
__global__ void __launch_bounds__(128)
    pack_kernel(const float* __restrict__ src, int64_t n, int D, int kvfmt, int64_t rb,
                uint8_t* __restrict__ dst) {
    extern __shared__ float sm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* row = sm + warp * D;
    int64_t r = (int64_t)blockIdx.x * 4 + warp;
    if (r >= n) return;
    for (int d = lane; d < D; d += 32) row[d] = src[r * D + d];
    __syncwarp();
    warp_pack_row(row, D, kvfmt, dst + r * rb);
}

cudaError_t launch_cache_pack(const Geometry& g, const float* src, int64_t n, void* dst,
                              cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 3) / 4;
    pack_kernel<<<(unsigned)blocks, 128, 4 * g.D * sizeof(float), st>>>(
        src, n, g.D, g.kv, g.kv_row_bytes, reinterpret_cast<uint8_t*>(dst));
    note_launch();
    return cudaGetLastError();
}

// Shared memory of the decode append: the cluster form for blocks of 64+
// tokens that split into kSplit slices of at least D floats, else one CTA per
// sequence staging the whole block (0: the block does not fit).
static size_t append_cluster_smem(const Geometry& g) {
    const int64_t act_rb = row_bytes(g.act, g.D);
    if (g.m < 64 || g.m % kSplit != 0) return 0;
    const int mt = g.m / kSplit;
    const size_t slice = ((size_t)mt * act_rb + 15) & ~(size_t)15;
    const size_t smem = slice + (size_t)(((mt + 3) & ~3) + kSplit * (4 + g.D) + 32) * sizeof(float);
    return (slice >= (size_t)g.D * sizeof(float) && smem <= 200 * 1024) ? smem : 0;
}

static size_t append_single_smem(const Geometry& g) {
    const size_t smem = (size_t)((g.m + g.D + 32 + 3) & ~3) * sizeof(float) + (size_t)g.m * row_bytes(g.act, g.D);
    return smem <= 200 * 1024 ? smem : 0;
}

bool decode_append_supported(const Geometry& g) { return append_cluster_smem(g) > 0 || append_single_smem(g) > 0; }

cudaError_t launch_decode_append(const Geometry& g, const void* tok, int B, const int64_t* pos, void* ring,
                                 const float* w_z, const float* bias, void* cache, int64_t n_cap, void* window,
                                 int64_t n_win, uint32_t* status, cudaStream_t st) {
    if (B == 0) return cudaSuccess;
    DecodeAppend d;
    d.pos = pos;
    d.tok = reinterpret_cast<const uint8_t*>(tok);
    d.ring = reinterpret_cast<uint8_t*>(ring);
    d.cache = reinterpret_cast<uint8_t*>(cache);
    d.n_cap = n_cap;
    d.window = (g.W > 0 && n_win > 0) ? reinterpret_cast<uint8_t*>(window) : nullptr;
    d.n_win = n_win;
    d.status = status;
    const int64_t act_rb = row_bytes(g.act, g.D);
    const size_t csm = append_cluster_smem(g);
    if (csm > 0) {
        cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(append_cluster_kernel), csm);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)kSplit, (unsigned)B, 1);
        cfg.blockDim = dim3(kCompressThreads, 1, 1);
        cfg.dynamicSmemBytes = csm;
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = kSplit;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, append_cluster_kernel, d, (int)g.act, act_rb, g.D, g.m, w_z, bias,
                               (int)g.kv, g.kv_row_bytes, g.eps, rope_theta(g));
        note_launch();
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const size_t smem = append_single_smem(g);
    if (smem == 0) return cudaErrorInvalidValue;  // refused earlier by the C ABI
    if (smem > 48 * 1024) {
        cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(append_step_kernel), smem);
        if (e != cudaSuccess) return e;
    }
    append_step_kernel<<<(unsigned)B, kAppendThreads, smem, st>>>(d, g.act, act_rb, g.D, g.m, w_z, bias, g.kv,
                                                                    g.kv_row_bytes, g.eps, rope_theta(g));
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_compress(const Geometry& g, const void* kv, int B, int64_t T,
                            int64_t kv_stride, int64_t pos0, const float* w_z, const float* bias,
                            void* out, int64_t out_stride, void* win_out, int64_t win_stride,
                            cudaStream_t st) {
    int64_t nb = T / g.m;
    if (nb == 0 || B == 0) return cudaSuccess;
    int64_t act_rb = row_bytes(g.act, g.D);
    if (g.m >= 64 && g.m % kSplit == 0 && nb * kSplit <= 0x7fffffff) {
        const int mt = g.m / kSplit;
        const size_t slice = ((size_t)mt * act_rb + 15) & ~(size_t)15;
        const size_t smem = slice + (size_t)(((mt + 3) & ~3) + kSplit * (4 + g.D) + 32) * sizeof(float);
        if (slice >= (size_t)g.D * sizeof(float) && smem <= 200 * 1024) {
            {
                cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(compress_cluster_kernel), smem);
                if (e != cudaSuccess) return e;
            }
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(nb * kSplit), (unsigned)B, 1);
            cfg.blockDim = dim3(kCompressThreads, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = st;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = kSplit;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            cudaError_t e = cudaLaunchKernelEx(
                &cfg, compress_cluster_kernel, reinterpret_cast<const uint8_t*>(kv), (int)g.act, act_rb,
                kv_stride * act_rb, g.D, g.m, pos0, w_z, bias, reinterpret_cast<uint8_t*>(out), (int)g.kv,
                g.kv_row_bytes, out_stride * g.kv_row_bytes, g.eps, rope_theta(g),
                reinterpret_cast<uint8_t*>(win_out), win_stride * g.kv_row_bytes);
            note_launch();
            if (e != cudaSuccess) return e;
            return cudaGetLastError();
        }
    }
    size_t smem = (size_t)((g.m + g.D + 32 + 3) & ~3) * sizeof(float);
    const size_t blk_bytes = (size_t)g.m * (size_t)act_rb;
    const int staged = blk_bytes <= kCompressStageMax ? 1 : 0;
    if (staged) smem += blk_bytes;
    if (smem > 48 * 1024) {
        cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(compress_kernel), smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)nb, (unsigned)B);
    compress_kernel<<<grid, kCompressThreads, smem, st>>>(
        reinterpret_cast<const uint8_t*>(kv), g.act, act_rb, kv_stride * act_rb, g.D, g.m, pos0,
        w_z, bias, reinterpret_cast<uint8_t*>(out), g.kv, g.kv_row_bytes,
        out_stride * g.kv_row_bytes, g.eps, rope_theta(g), staged, reinterpret_cast<uint8_t*>(win_out),
        win_stride * g.kv_row_bytes);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa
