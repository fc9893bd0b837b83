// k_topk.cu -- exact top-k selection over indexer scores.
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 2": keep the top-K
// compressed blocks per query; ties go to the lower block index, so the
// order is the total order (score descending, index ascending).  Scores are
// mapped to order-preserving 32-bit keys.  A radix select over keys held in
// shared memory finds the k-th largest key T: the keys' common leading bits
// are skipped (block min / max), then 11-bit digits are resolved from the
// first differing bit down, each pass over the keys that still match the
// resolved prefix (copied to a short candidate list once they fit).  Every
// block with key > T is kept, and of the blocks with key == T the lowest
// indices fill the remaining slots; the kept blocks are listed in ascending
// index order by a warp-segmented compaction (ballots within a warp, one
// exclusive scan over the warps).
//
// Two stages.  A query's n complete blocks are cut into ceil(n / C) chunks
// of equal size (up to one), each of at least C / 2 >= 2k scores; one CTA per
// (chunk, query) selects the chunk's own top k.  Because the order is total,
// the query's top k is a subset of the union of the chunks' top k.  With a
// single chunk that selection is already the answer; otherwise each chunk CTA
// writes its k candidates (keys, then indices, in index order) over the
// start of its own chunk of the score row -- the scores are consumed -- and
// one CTA per query selects the final k from the concatenated candidates
// (still in ascending index order).
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kDigitBits = 11;
constexpr int kBins = 1 << kDigitBits;  // two bins per thread in the digit search
constexpr int kChunk = 32768;           // C: most scores one CTA holds (128 KiB of keys)
constexpr int kCandCap = 4096;          // a digit's keys are copied out once this few
constexpr int kMergeKeys = 40960;       // most candidates one merge CTA holds (160 KiB)

// Order-preserving key of a float score (both zeros share one key).
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f == 0.f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Shared scratch of one selection (besides the keys).
struct Scratch {
    int hist[kBins];
    uint32_t cand[kCandCap];
    uint32_t red[2][kWarps];
    int wcnt[2][kWarps];
    int scan[kWarps];
    int n_cand;
    int digit, above;
};

// Exclusive scan of one int per thread over the CTA; returns the prefix.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sw) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sw[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = sw[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sw[lane] = w;  // inclusive per-warp totals
    }
    __syncthreads();
    const int before = (warp > 0 ? sw[warp - 1] : 0) + x - v;
    __syncthreads();  // sw is free for the next scan
    return before;
}

struct Select {
    uint32_t T;   // key of the k-th largest
    int take_eq;  // how many keys equal to T are kept (the lowest indices)
};

// Each thread's smallest / largest key -> the CTA's (every thread).
__device__ __forceinline__ void block_minmax(uint32_t& lo, uint32_t& hi, Scratch& s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
        s.red[0][warp] = lo;
        s.red[1][warp] = hi;
    }
    __syncthreads();
    lo = s.red[0][lane];
    hi = s.red[1][lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
}

// Radix select of the k-th largest of keys[0, n) (shared memory), 0 < k <= n,
// given the smallest and largest key (the bits all keys share are skipped).
__device__ Select radix_select(const uint32_t* keys, int n, int k, uint32_t lo, uint32_t hi, Scratch& s) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (lo == hi) return Select{hi, k};
    int top = 31 - __clz(lo ^ hi);  // highest bit in which keys differ
    uint32_t prefix = top == 31 ? 0u : (hi & ~((2u << top) - 1u));
    int remaining = k;
    const uint32_t* src = keys;  // the keys matching the prefix are among src[0, m)
    int m = n;
    for (;;) {
        const int shift = top >= kDigitBits - 1 ? top - (kDigitBits - 1) : 0;
        const uint32_t himask = top == 31 ? 0u : ~((2u << top) - 1u);
        for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0;
        __syncthreads();
#pragma unroll 4
        for (int i = tid; i < m; i += kThreads) {
            const uint32_t u = src[i];
            if ((u & himask) == prefix) atomicAdd(&s.hist[(u >> shift) & (kBins - 1)], 1);
        }
        __syncthreads();
        // the digit d with (keys above d) < remaining <= (keys at or above d):
        // thread t holds bins 2047-2t and 2046-2t, counted from the top bin
        const int b0 = kBins - 1 - 2 * tid, b1 = b0 - 1;
        const int c0 = s.hist[b0], c1 = s.hist[b1];
        const int before = block_exclusive_scan(c0 + c1, s.scan);
        if (before < remaining && before + c0 >= remaining) {
            s.digit = b0;
            s.above = before;
        } else if (before + c0 < remaining && before + c0 + c1 >= remaining) {
            s.digit = b1;
            s.above = before + c0;
        }
        __syncthreads();
        const int d = s.digit, cnt = s.hist[d];
        remaining -= s.above;
        prefix |= (uint32_t)d << shift;
        if (shift == 0) return Select{prefix, remaining};
        top = shift - 1;
        if (cnt <= kCandCap && src != s.cand) {
            // the keys of digit d go to the candidate list (their order is irrelevant)
            if (tid == 0) s.n_cand = 0;
            __syncthreads();
            const uint32_t newmask = ~((2u << top) - 1u);
#pragma unroll 4
            for (int i0 = 0; i0 < m; i0 += kThreads) {
                const int i = i0 + tid;
                const uint32_t u = i < m ? src[i] : 0u;
                const bool hit = i < m && (u & newmask) == prefix;
                const uint32_t bal = __ballot_sync(0xffffffffu, hit);
                int base = 0;
                if (lane == 0 && bal) base = atomicAdd(&s.n_cand, __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (hit) s.cand[base + __popc(bal & ((1u << lane) - 1u))] = u;
            }
            __syncthreads();
            src = s.cand;
            m = s.n_cand;
        }
        __syncthreads();  // digit, above and hist are rewritten by the next pass
    }
}

// Keep the top `k` of keys[0, n) in index order: calls emit(pos, i) for the
// kept entries with pos = 0 .. k-1 ascending in i.  Warp w sweeps the
// contiguous range [w*seg, (w+1)*seg) twice: once to count, once to place.
template <class Emit>
__device__ void block_compact(const uint32_t* keys, int n, Select sel, Scratch& s, Emit emit) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
    const int i0 = warp * seg, i1 = min(n, i0 + seg);
    int gt = 0, eq = 0;
#pragma unroll 4
    for (int r = i0; r < i1; r += 32) {
        const int i = r + lane;
        const uint32_t u = i < i1 ? keys[i] : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, i < i1 && u > sel.T));
        eq += __popc(__ballot_sync(0xffffffffu, i < i1 && u == sel.T));
    }
    if (lane == 0) {
        s.wcnt[0][warp] = gt;
        s.wcnt[1][warp] = eq;
    }
    __syncthreads();
    if (warp == 0) {
        const int g0 = s.wcnt[0][lane], e0 = s.wcnt[1][lane];
        int g = g0, e = e0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yg = __shfl_up_sync(0xffffffffu, g, o), ye = __shfl_up_sync(0xffffffffu, e, o);
            if (lane >= o) {
                g += yg;
                e += ye;
            }
        }
        s.wcnt[0][lane] = g - g0;  // exclusive
        s.wcnt[1][lane] = e - e0;
    }
    __syncthreads();
    int gt_base = s.wcnt[0][warp], eq_base = s.wcnt[1][warp];
    const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll 4
    for (int r = i0; r < i1; r += 32) {
        const int i = r + lane;
        const uint32_t u = i < i1 ? keys[i] : 0u;
        const bool is_gt = i < i1 && u > sel.T, is_eq = i < i1 && u == sel.T;
        const uint32_t bg = __ballot_sync(0xffffffffu, is_gt), be = __ballot_sync(0xffffffffu, is_eq);
        const int g_before = gt_base + __popc(bg & lt_mask), e_before = eq_base + __popc(be & lt_mask);
        if (is_gt || (is_eq && e_before < sel.take_eq)) emit(g_before + min(e_before, sel.take_eq), i);
        gt_base += __popc(bg);
        eq_base += __popc(be);
    }
}

// keys[i] = score_key(src[i]) for i < n: 16-byte loads (every one issued
// before any is used) when src is 16-byte aligned, else 4-byte loads.
template <int kBatch>
__device__ __forceinline__ void load_keys(const float* src, int n, uint32_t* keys, uint32_t& lo, uint32_t& hi) {
    lo = 0xffffffffu;
    hi = 0u;
    auto put = [&](int i, uint32_t q) {
        keys[i] = q;
        lo = min(lo, q);
        hi = max(hi, q);
    };
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        const float4* v = reinterpret_cast<const float4*>(src);
        uint4* kv = reinterpret_cast<uint4*>(keys);
        const int n4 = n / 4;
        for (int j0 = threadIdx.x; j0 < n4; j0 += kBatch * kThreads) {
            float4 f[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; u++)
                if (j0 + u * kThreads < n4) f[u] = __ldg(v + j0 + u * kThreads);
#pragma unroll
            for (int u = 0; u < kBatch; u++)
                if (j0 + u * kThreads < n4) {
                    const uint4 q = make_uint4(score_key(f[u].x), score_key(f[u].y), score_key(f[u].z),
                                               score_key(f[u].w));
                    kv[j0 + u * kThreads] = q;
                    lo = min(min(lo, min(q.x, q.y)), min(q.z, q.w));
                    hi = max(max(hi, max(q.x, q.y)), max(q.z, q.w));
                }
        }
        for (int i = 4 * n4 + threadIdx.x; i < n; i += kThreads) put(i, score_key(src[i]));
    } else {
#pragma unroll 8
        for (int i = threadIdx.x; i < n; i += kThreads) put(i, score_key(src[i]));
    }
}

__device__ __forceinline__ int64_t n_complete(const int64_t* q_pos, int64_t q, int m, int64_t n_cap) {
    int64_t n = (q_pos[q] + 1) / m;
    if (n > n_cap) n = n_cap;  // flagged by the indexer
    return n < 0 ? 0 : n;
}

__device__ __forceinline__ int64_t n_chunks(int64_t n) { return n > kChunk ? (n + kChunk - 1) / kChunk : 1; }

// Chunk c of nch over n blocks: [c*n/nch, (c+1)*n/nch).
__device__ __forceinline__ int64_t chunk_lo(int64_t c, int64_t n, int64_t nch) { return c * n / nch; }

// Stage 1: grid (max chunks, Q).  Writes the final selection when the query
// has one chunk, its candidates otherwise.  kMinBlocks = 2 when two CTAs fit
// an SM (chunks of at most ~21K scores: one CTA's selection passes overlap
// the other's loads), at the price of 32 registers a thread; else 1.
template <int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    topk_chunk_kernel(float* __restrict__ scores, int64_t ld, int64_t n_cap,
                      const int64_t* __restrict__ q_pos, int m, int k,
                      int32_t* __restrict__ idx, float* __restrict__ sel) {
    constexpr int kLoadBatch = kMinBlocks == 2 ? 2 : 8;  // 16-byte loads in flight per thread
    extern __shared__ uint32_t keys[];  // [<= kChunk]
    __shared__ Scratch s;
    const int64_t q = blockIdx.y;
    const int64_t n = n_complete(q_pos, q, m, n_cap);
    const int64_t nch = n_chunks(n);
    if ((int64_t)blockIdx.x >= nch) return;
    float* row = scores + q * ld;
    const int64_t lo = chunk_lo(blockIdx.x, n, nch);
    const int nc = (int)(chunk_lo(blockIdx.x + 1, n, nch) - lo);
    if (nch == 1) {
        // a single chunk: this CTA writes the answer
        int32_t* oi = idx + q * k;
        float* os = sel ? sel + q * k : nullptr;
        if (nc <= k) {
            for (int j = threadIdx.x; j < k; j += kThreads) {
                oi[j] = j < nc ? j : -1;
                if (os) os[j] = j < nc ? row[j] : -INFINITY;
            }
            return;
        }
        uint32_t lo_k, hi_k;
        load_keys<kLoadBatch>(row, nc, keys, lo_k, hi_k);
        block_minmax(lo_k, hi_k, s);  // also makes the keys visible to the CTA
        const Select t = radix_select(keys, nc, k, lo_k, hi_k, s);
        block_compact(keys, nc, t, s, [&](int pos, int i) {
            oi[pos] = i;
            if (os) os[pos] = key_score(keys[i]);
        });
        return;
    }
    uint32_t lo_k, hi_k;
    load_keys<kLoadBatch>(row + lo, nc, keys, lo_k, hi_k);
    block_minmax(lo_k, hi_k, s);  // the chunk is in smem: its region of the row may be overwritten
    uint32_t* ck = reinterpret_cast<uint32_t*>(row + lo);      // [k] candidate keys
    int32_t* cidx = reinterpret_cast<int32_t*>(row + lo + k);  // [k] candidate indices
    const Select t = radix_select(keys, nc, k, lo_k, hi_k, s);
    block_compact(keys, nc, t, s, [&](int pos, int i) {
        ck[pos] = keys[i];
        cidx[pos] = (int32_t)(lo + i);
    });
}

// Stage 2: one CTA per query with more than one chunk; chunk c's k
// candidates sit at the start of its range of the row: k keys, then k
// indices.
__global__ void __launch_bounds__(kThreads, 1)
    topk_merge_kernel(const float* __restrict__ scores, int64_t ld, int64_t n_cap,
                      const int64_t* __restrict__ q_pos, int m, int k,
                      int32_t* __restrict__ idx, float* __restrict__ sel) {
    extern __shared__ uint32_t keys[];  // [nchunks * k]
    __shared__ Scratch s;
    const int64_t q = blockIdx.x;
    const int64_t n = n_complete(q_pos, q, m, n_cap);
    const int64_t nch = n_chunks(n);
    if (nch <= 1) return;
    const float* row = scores + q * ld;
    const int C = (int)(nch * k);
    uint32_t lo_k = 0xffffffffu, hi_k = 0u;
    for (int64_t c = 0; c < nch; c++) {  // chunk c's k candidate keys
        const uint32_t* ck = reinterpret_cast<const uint32_t*>(row + chunk_lo(c, n, nch));
#pragma unroll 4
        for (int j = threadIdx.x; j < k; j += kThreads) {
            const uint32_t u = ck[j];
            keys[c * k + j] = u;
            lo_k = min(lo_k, u);
            hi_k = max(hi_k, u);
        }
    }
    block_minmax(lo_k, hi_k, s);  // also makes the keys visible to the CTA
    int32_t* oi = idx + q * k;
    float* os = sel ? sel + q * k : nullptr;
    const Select t = radix_select(keys, C, k, lo_k, hi_k, s);
    block_compact(keys, C, t, s, [&](int pos, int i) {
        oi[pos] = reinterpret_cast<const int32_t*>(row + chunk_lo(i / k, n, nch) + k)[i % k];
        if (os) os[pos] = key_score(keys[i]);
    });
}

}  // namespace

// Chunk size for n_cap blocks, or 0 when the selection does not fit in
// shared memory (the merge holds ceil(n_cap / C) * k keys) or a chunk could
// not hold its k candidates twice over.
int64_t topk_chunk(int64_t n_cap, int Q, int k) {
    (void)Q;
    if (n_cap <= kChunk) return n_cap > 0 ? n_cap : 1;  // one chunk per query
    const int64_t nch = (n_cap + kChunk - 1) / kChunk;
    if (nch * (int64_t)k > kMergeKeys || 2 * (int64_t)k > kChunk / 2) return 0;
    return kChunk;
}

cudaError_t launch_topk(const Geometry& g, float* scores, int64_t ld, int64_t n_cap, int Q,
                        const int64_t* q_pos, int32_t* idx, float* sel, cudaStream_t st) {
    if (Q == 0) return cudaSuccess;
    const int k = g.k;
    if (topk_chunk(n_cap, Q, k) == 0) return cudaErrorInvalidValue;  // rejected earlier by the C ABI
    const int64_t max_chunks = n_cap > kChunk ? (n_cap + kChunk - 1) / kChunk : 1;
    const size_t smem1 = (size_t)(n_cap < kChunk ? (n_cap > 0 ? n_cap : 1) : kChunk) * sizeof(uint32_t);
    // two CTAs an SM when both fit in its 228 KiB of shared memory
    const bool two = smem1 + sizeof(Scratch) + 1024 <= 114 * 1024;
    static int attr1[2] = {0, 0};
    if ((int)smem1 > attr1[two]) {
        cudaError_t e = two ? cudaFuncSetAttribute(topk_chunk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem1)
                            : cudaFuncSetAttribute(topk_chunk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem1);
        if (e != cudaSuccess) return e;
        attr1[two] = (int)smem1;
    }
    dim3 grid1((unsigned)max_chunks, (unsigned)Q);
    if (two)
        topk_chunk_kernel<2><<<grid1, kThreads, smem1, st>>>(scores, ld, n_cap, q_pos, g.m, k, idx, sel);
    else
        topk_chunk_kernel<1><<<grid1, kThreads, smem1, st>>>(scores, ld, n_cap, q_pos, g.m, k, idx, sel);
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
    topk_merge_kernel<<<(unsigned)Q, kThreads, smem2, st>>>(scores, ld, n_cap, q_pos, g.m, k, idx, sel);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa
