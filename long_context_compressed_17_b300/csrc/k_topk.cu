// k_topk.cu -- exact top-k selection over indexer scores.
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 2": keep the top-K
// compressed blocks per query; ties go to the lower block index, so the
// order is the total order (score descending, index ascending).  Scores are
// mapped to order-preserving 32-bit keys; a radix select (four 8-bit digits,
// most significant first) over keys held in shared memory finds the k-th
// largest key T; every block with key > T is kept, and of the blocks with
// key == T the lowest indices fill the remaining slots.  The output lists the
// kept blocks in ascending index order.
//
// Two stages.  A query's n complete blocks are cut into max(1, n / C) chunks
// of C scores, the last one taking the remainder (C <= size < 2C); one CTA
// per (chunk, query) selects the chunk's own top k.  Because the order is
// total, the query's top k is a subset of the union of the chunks' top k.
// With a single chunk that selection is already the answer; otherwise each
// chunk CTA writes its k candidates (keys, then indices, in index order) over
// the start of its own chunk of the score row (C >= 2k, so they fit) -- the
// scores are consumed -- and one CTA per query selects the final k.
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kChunkThreads = 512;
constexpr int kMergeThreads = 1024;
constexpr int kMaxSingle = 32768;       // one chunk per query up to this many blocks (128 KiB of keys)
constexpr int kMinChunk = 8192;         // C when queries are split
constexpr int kMaxChunk = 16384;        // largest C (a chunk holds < 2C keys)

// Order-preserving key of a float score (both zeros share one key).
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f == 0.f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Exclusive scan over the CTA; returns the prefix, writes the total.
// `sw` holds 32 ints of shared scratch.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sw, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
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
        int w = lane < nw ? sw[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sw[lane] = w;  // inclusive per-warp totals
    }
    __syncthreads();
    const int before = (warp > 0 ? sw[warp - 1] : 0) + x - v;
    *total = sw[nw - 1];
    return before;
}

struct Select {
    uint32_t T;   // key of the k-th largest
    int take_eq;  // how many keys equal to T are kept (the lowest indices)
};

// Radix select of the k-th largest of keys[0, n) (shared memory), 0 < k < n.
__device__ Select block_radix_select(const uint32_t* keys, int n, int k, int* hist, uint32_t* s_digit,
                                     int* s_above) {
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint32_t u = keys[i];
            if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l owns digits 8l .. 8l+7; suffix sums from the top digit down
            const int l = threadIdx.x;
            int c[8], loc = 0;
#pragma unroll
            for (int e = 0; e < 8; e++) {
                c[e] = hist[8 * l + e];
                loc += c[e];
            }
            int suf = loc;  // inclusive suffix over lanes >= l
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_down_sync(0xffffffffu, suf, o);
                if (l + o < 32) suf += y;
            }
            int above = suf - loc;  // keys with a digit in higher lanes
#pragma unroll
            for (int e = 7; e >= 0; e--) {
                if (above < remaining && above + c[e] >= remaining) {
                    *s_digit = (uint32_t)(8 * l + e);
                    *s_above = above;
                }
                above += c[e];
            }
        }
        __syncthreads();
        prefix |= *s_digit << shift;
        mask |= 255u << shift;
        remaining -= *s_above;
        __syncthreads();
    }
    return Select{prefix, remaining};
}

// Keep the top `k` of keys[0, n) in index order: calls emit(pos, i) for the
// kept entries with pos = 0 .. k-1 ascending in i.  The keys are swept in
// block-wide rounds (thread t reads entry r + t: no bank conflicts); one scan
// of the packed (greater, equal) counts per round places every kept entry.
template <class Emit>
__device__ void block_compact(const uint32_t* keys, int n, Select sel, int* sw, Emit emit) {
    int base = 0, eq_left = sel.take_eq;
    for (int r0 = 0; r0 < n; r0 += blockDim.x) {
        const int i = r0 + threadIdx.x;
        const uint32_t u = i < n ? keys[i] : 0u;
        const int gt = (i < n && u > sel.T) ? 1 : 0;
        const int eq = (i < n && u == sel.T) ? 1 : 0;
        int tot;
        const int before = block_exclusive_scan(gt | (eq << 16), sw, &tot);
        const int gt_before = before & 0xffff, eq_before = before >> 16;
        if (gt || (eq && eq_before < eq_left)) emit(base + gt_before + min(eq_before, eq_left), i);
        const int eq_tot = tot >> 16;
        base += (tot & 0xffff) + min(eq_tot, eq_left);
        eq_left -= min(eq_tot, eq_left);
    }
}

__device__ __forceinline__ int64_t n_complete(const int64_t* q_pos, int64_t q, int m, int64_t n_cap) {
    int64_t n = (q_pos[q] + 1) / m;
    if (n > n_cap) n = n_cap;  // flagged by the indexer
    return n < 0 ? 0 : n;
}

__device__ __forceinline__ int64_t n_chunks(int64_t n, int chunk) {
    const int64_t c = n / chunk;
    return c > 1 ? c : 1;
}

// Stage 1: grid (max chunks, Q).  Writes the final selection when the query
// has one chunk, its candidates otherwise.
__global__ void __launch_bounds__(kChunkThreads)
    topk_chunk_kernel(float* __restrict__ scores, int64_t ld, int64_t n_cap,
                      const int64_t* __restrict__ q_pos, int m, int k, int chunk,
                      int32_t* __restrict__ idx, float* __restrict__ sel) {
    extern __shared__ uint32_t keys[];  // [< 2 * chunk] (or the whole row)
    __shared__ int hist[256];
    __shared__ int sw[32];
    __shared__ uint32_t s_digit;
    __shared__ int s_above;
    const int64_t q = blockIdx.y;
    const int64_t n = n_complete(q_pos, q, m, n_cap);
    const int64_t nch = n_chunks(n, chunk);
    if ((int64_t)blockIdx.x >= nch) return;
    float* row = scores + q * ld;
    if (nch == 1) {
        // a single chunk: this CTA writes the answer
        int32_t* oi = idx + q * k;
        float* os = sel ? sel + q * k : nullptr;
        const int nc = (int)n;
        if (nc <= k) {
            for (int j = threadIdx.x; j < k; j += blockDim.x) {
                oi[j] = j < nc ? j : -1;
                if (os) os[j] = j < nc ? row[j] : -INFINITY;
            }
            return;
        }
        for (int i = threadIdx.x; i < nc; i += blockDim.x) keys[i] = score_key(row[i]);
        __syncthreads();
        const Select s = block_radix_select(keys, nc, k, hist, &s_digit, &s_above);
        block_compact(keys, nc, s, sw, [&](int pos, int i) {
            oi[pos] = i;
            if (os) os[pos] = key_score(keys[i]);
        });
        return;
    }
    const int64_t lo = (int64_t)blockIdx.x * chunk;
    const int nc = (int)((int64_t)blockIdx.x == nch - 1 ? n - lo : chunk);  // chunk <= nc < 2 chunk
    for (int i = threadIdx.x; i < nc; i += blockDim.x) keys[i] = score_key(row[lo + i]);
    __syncthreads();  // the chunk is in smem: its region of the row may be overwritten
    uint32_t* ck = reinterpret_cast<uint32_t*>(row + lo);      // [k] candidate keys
    int32_t* cidx = reinterpret_cast<int32_t*>(row + lo + k);  // [k] candidate indices
    const Select s = block_radix_select(keys, nc, k, hist, &s_digit, &s_above);
    block_compact(keys, nc, s, sw, [&](int pos, int i) {
        ck[pos] = keys[i];
        cidx[pos] = (int32_t)(lo + i);
    });
}

// Stage 2: one CTA per query with more than one chunk; chunk c's k
// candidates sit at row[c*chunk ..]: k keys, then k indices.
__global__ void __launch_bounds__(kMergeThreads)
    topk_merge_kernel(const float* __restrict__ scores, int64_t ld, int64_t n_cap,
                      const int64_t* __restrict__ q_pos, int m, int k, int chunk,
                      int32_t* __restrict__ idx, float* __restrict__ sel) {
    extern __shared__ uint32_t keys[];  // [nchunks * k]
    __shared__ int hist[256];
    __shared__ int sw[32];
    __shared__ uint32_t s_digit;
    __shared__ int s_above;
    const int64_t q = blockIdx.x;
    const int64_t n = n_complete(q_pos, q, m, n_cap);
    const int64_t nch = n_chunks(n, chunk);
    if (nch <= 1) return;
    const float* row = scores + q * ld;
    const int C = (int)(nch * k);
    for (int i = threadIdx.x; i < C; i += blockDim.x)
        keys[i] = reinterpret_cast<const uint32_t*>(row + (int64_t)(i / k) * chunk)[i % k];
    __syncthreads();
    int32_t* oi = idx + q * k;
    float* os = sel ? sel + q * k : nullptr;
    const Select s = block_radix_select(keys, C, k, hist, &s_digit, &s_above);
    block_compact(keys, C, s, sw, [&](int pos, int i) {
        oi[pos] = reinterpret_cast<const int32_t*>(row + (int64_t)(i / k) * chunk + k)[i % k];
        if (os) os[pos] = key_score(keys[i]);
    });
}

}  // namespace

// Chunk size C for n_cap blocks and Q queries, or 0 when the selection does
// not fit in shared memory.
int64_t topk_chunk(int64_t n_cap, int Q, int k) {
    const int64_t sms = num_sms();
    if (n_cap <= kMaxSingle && ((int64_t)Q >= 2 * sms || n_cap < 2 * kMinChunk))
        return n_cap > 0 ? n_cap : 1;  // one chunk per query
    int64_t chunk = kMinChunk;
    while (chunk < kMaxChunk && (int64_t)Q * (n_cap / chunk) > 4 * sms) chunk *= 2;
    while (chunk < 2 * (int64_t)k) chunk *= 2;
    // the merge holds max(1, n_cap / C) * k keys in shared memory
    while ((n_cap / chunk) * (int64_t)k * 4 > 200 * 1024 && chunk <= kMaxChunk) chunk *= 2;
    if (chunk > kMaxChunk) return 0;
    return chunk;
}

size_t topk_chunk_smem(int64_t n_cap, int64_t chunk) {
    const int64_t keys = chunk >= n_cap ? n_cap : 2 * chunk - 1;
    return (size_t)(keys > 0 ? keys : 1) * sizeof(uint32_t);
}

cudaError_t launch_topk(const Geometry& g, float* scores, int64_t ld, int64_t n_cap, int Q,
                        const int64_t* q_pos, int32_t* idx, float* sel, cudaStream_t st) {
    if (Q == 0) return cudaSuccess;
    const int k = g.k;
    const int64_t chunk = topk_chunk(n_cap, Q, k);
    if (chunk == 0) return cudaErrorInvalidValue;  // rejected earlier by the C ABI
    const int64_t max_chunks = n_cap / chunk > 1 ? n_cap / chunk : 1;
    const size_t smem1 = topk_chunk_smem(n_cap, chunk);
    static int attr1 = 0;
    if ((int)smem1 > attr1) {
        cudaError_t e = cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem1);
        if (e != cudaSuccess) return e;
        attr1 = (int)smem1;
    }
    dim3 grid1((unsigned)max_chunks, (unsigned)Q);
    topk_chunk_kernel<<<grid1, kChunkThreads, smem1, st>>>(scores, ld, n_cap, q_pos, g.m, k, (int)chunk, idx, sel);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || max_chunks <= 1) return e;
    const size_t smem2 = (size_t)max_chunks * k * sizeof(uint32_t);
    static int attr2 = 0;
    if ((int)smem2 > attr2) {
        e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
        if (e != cudaSuccess) return e;
        attr2 = (int)smem2;
    }
    topk_merge_kernel<<<(unsigned)Q, kMergeThreads, smem2, st>>>(scores, ld, n_cap, q_pos, g.m, k, (int)chunk, idx, sel);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa
