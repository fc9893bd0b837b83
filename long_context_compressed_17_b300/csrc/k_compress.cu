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
constexpr size_t kCompressStageMax = 160 * 1024;  // raw block staged in smem up to this size

// row[0, D) holds a pooled vector (shared memory) and ss each thread's partial
// sum of its squares: RMSNorm it, rotate its last 64 dims at position pos and
// store it into a cache row at dst (whole CTA; red: 32 floats of scratch).
__device__ void norm_rope_store(float* row, float ss, float* red, int D, float eps, double pos,
                                const RopeTheta& theta, int kvfmt, uint8_t* dst) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nwarps = kCompressThreads / 32;
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
    for (int d = tid; d < D; d += kCompressThreads) row[d] *= rn;
    __syncthreads();
    if (tid < kRopeDims / 2) {
        const int j = tid;
        float c, s;
        rope_cs(pos, theta.t[j], &c, &s);
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
__device__ void window_row(const uint8_t* tok, int act, float* row, float* red, int D, float eps, double pos,
                           const RopeTheta& theta, int kvfmt, uint8_t* dst) {
    float ss = 0.f;
    for (int d = threadIdx.x; d < D; d += kCompressThreads) {
        const float c = load_act(tok, act, d);
        row[d] = c;
        ss = fmaf(c, c, ss);
    }
    norm_rope_store(row, ss, red, D, eps, pos, theta, kvfmt, dst);
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
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nwarps = kCompressThreads / 32;
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

    if (m == 1) {
        // a single token: its pooling weight is exactly 1 (window rows)
        if (tid == 0) z[0] = 1.f;
        __syncthreads();
    } else {
        // pooling scores z_t = kv_t . w_z + bias[t mod m]   (pos0 is a multiple of m)
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
    for (int d = tid; d < D; d += kCompressThreads) {
        float c = 0.f;
        for (int t = 0; t < m; t++) c = fmaf(z[t], load_act(src + t * act_row_bytes, act, d), c);
        row[d] = c;
        ss = fmaf(c, c, ss);
    }
    // RMSNorm, partial RoPE at the block's last position, store
    const double pos = (double)(pos0 + b * m + m - 1);
    norm_rope_store(row, ss, red, D, eps, pos, theta, kvfmt, out + blockIdx.y * out_seq_bytes + b * kv_row_bytes);
    if (win_out != nullptr) {  // the window row of the block's last token
        __syncthreads();       // `row` is free again
        window_row(src + (m - 1) * act_row_bytes, act, row, red, D, eps, pos, theta, kvfmt,
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
    const size_t slice_bytes = (size_t)mt * act_row_bytes;
    uint8_t* stage = reinterpret_cast<uint8_t*>(sm);
    float* z = reinterpret_cast<float*>(stage + ((slice_bytes + 15) & ~(size_t)15));
    float* slots = z + ((mt + 3) & ~3);                 // [kSplit][4 + D]
    float* red = slots + kSplit * (4 + D);              // [32]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nwarps = kCompressThreads / 32;
    const int t0 = rank * mt;                           // first token of the slice within the block
    {
        const uint4* g = reinterpret_cast<const uint4*>(kv + blockIdx.y * kv_seq_bytes +
                                                        (b * m + t0) * act_row_bytes);
        uint4* s = reinterpret_cast<uint4*>(stage);
        const int64_t n16 = (int64_t)slice_bytes / 16;
        for (int64_t i = tid; i < n16; i += kCompressThreads) s[i] = __ldg(g + i);
    }
    __syncthreads();
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
            float c = 0.f;
            for (int t = 0; t < mt; t++) c = fmaf(z[t], load_act(stage + t * act_row_bytes, act, 4 * d4 + e), c);
            p[e] = c;
        }
        tc::st_cluster_v4(slot0 + 16u * (1 + d4), make_uint4(__float_as_uint(p[0]), __float_as_uint(p[1]),
                                                               __float_as_uint(p[2]), __float_as_uint(p[3])));
    }
    if (tid == 0)
        tc::st_cluster_v4(slot0, make_uint4(__float_as_uint(zmax), __float_as_uint(zsum), 0u, 0u));
    tc::cluster_sync();  // every slot of CTA 0 is written and visible
    const double pos = (double)(pos0 + b * m + m - 1);
    if (rank == kSplit - 1 && win_out != nullptr) {
        // the window row of the block's last token, the last row of this slice;
        // this CTA's own slots are unused and hold the row
        window_row(stage + (mt - 1) * act_row_bytes, act, slots, red, D, eps, pos, theta, kvfmt,
                   win_out + blockIdx.y * win_seq_bytes + b * kv_row_bytes);
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
        float c = 0.f;
        for (int r = 0; r < kSplit; r++) c = fmaf(slots[r * (4 + D) + 4 + d], expf(slots[r * (4 + D)] - M), c);
        c *= invS;
        row[d] = c;
        ss = fmaf(c, c, ss);
    }
    norm_rope_store(row, ss, red, D, eps, pos, theta, kvfmt, out + blockIdx.y * out_seq_bytes + b * kv_row_bytes);
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
