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
//
// When few queries each hold one chunk (decode), a cluster of four CTAs
// selects each query instead: every CTA holds a quarter of the row, the radix
// passes sum the four histograms over distributed shared memory (each CTA
// then takes the same decisions), and each CTA lists its kept blocks after
// those of the CTAs before it.
#include <cstddef>

#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kDigitBits = 11;
constexpr int kBins = 1 << kDigitBits;  // two bins per thread in the digit search
constexpr int kChunk = 32768;           // C: most scores one CTA holds (128 KiB of keys)
constexpr int kCandCap = 4096;          // a digit's keys are copied out once this few
constexpr int kMergeKeys = 40960;       // most candidates one merge CTA holds (160 KiB)
constexpr int kClusterCS = 4;           // CTAs selecting one query together when queries are few
constexpr int kClusterMinKeys = 4096;   // ... and its row holds at least this many scores

// Order-preserving key of a float score (both zeros share one key).
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f == 0.f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Shared scratch of one selection (besides the keys).  CS > 1: the CTA is
// one of a cluster of CS that select one query's top k together, each over
// a slice of its scores; the histograms alternate between two buffers so
// that one cluster barrier a pass suffices, and ctot is read by the other
// CTAs of the cluster.
template <int CS>
struct __align__(16) TopkScratch {
    int hist[CS > 1 ? 2 : 1][kBins];  // 16-byte aligned: bins 2i, 2i+1 load as one pair
    uint32_t cand[kCandCap];
    uint32_t red[2][kWarps];
    int wcnt[2][kWarps];
    int scan[kWarps];
    int n_cand;
    int digit, above, dcount;  // selected digit, keys above it, keys in it (whole cluster)
    int ctot[2];               // this CTA's kept keys above / equal to T
    uint32_t bcast[2];         // cluster-wide values read by warp 0, for the CTA
};
using Scratch = TopkScratch<1>;
// pairs read with one 8-byte load from another CTA of the cluster
static_assert(offsetof(TopkScratch<4>, ctot) % 8 == 0, "ctot must be 8-byte aligned");
static_assert(offsetof(TopkScratch<4>, hist) % 16 == 0 && (kBins * sizeof(int)) % 8 == 0,
              "histogram pairs must be 8-byte aligned");

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
    uint32_t T;   // the k-th largest key, or the least key of the last digit's bin when all of it is kept
    int take_eq;  // how many keys equal to T are kept (the lowest indices); every key above T is kept
};

// Warp sweeps over keys in shared memory: warp w owns the contiguous range
// [w*seg, (w+1)*seg) (seg a multiple of 128, so with a 16-byte aligned key
// array every group of four starts 16-byte aligned) and covers 128 keys per
// step, lane l keys 4l .. 4l+3 of the step.
__device__ __forceinline__ int sweep_seg(int n) { return ((n + kWarps - 1) / kWarps + 127) & ~127; }

// The four keys at i .. i+3 that lie below i1 (one 16-byte load when all do);
// valid bit e says whether key i+e exists.
__device__ __forceinline__ uint32_t load4(const uint32_t* keys, int i, int i1, uint32_t (&u)[4]) {
    if (i + 3 < i1) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
        u[0] = v.x;
        u[1] = v.y;
        u[2] = v.z;
        u[3] = v.w;
        return 0xfu;
    }
    uint32_t valid = 0;
#pragma unroll
    for (int e = 0; e < 4; e++) {
        u[e] = 0u;
        if (i + e < i1) {
            u[e] = keys[i + e];
            valid |= 1u << e;
        }
    }
    return valid;
}

// Inclusive sum over the lanes of a warp.
__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Each thread's smallest / largest key -> the CTA's (every thread).
template <class S>
__device__ __forceinline__ void block_minmax(uint32_t& lo, uint32_t& hi, S& s) {
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

// Radix select of the k-th largest of the keys, 0 < k <= their number,
// given the smallest and largest key (the bits all keys share are skipped).
// CS == 1: keys[0, n) in this CTA's shared memory.  CS > 1: every CTA of the
// cluster holds its slice in keys[0, n), lo / hi are the cluster's, and each
// pass sums the CTAs' histograms, so that every CTA takes the same
// decisions (and the same cluster barriers).
template <int CS, class S>
__device__ Select radix_select(const uint32_t* keys, int n, int k, uint32_t lo, uint32_t hi, S& s) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (lo == hi) return Select{hi, k};
    int top = 31 - __clz(lo ^ hi);  // highest bit in which keys differ
    uint32_t prefix = top == 31 ? 0u : (hi & ~((2u << top) - 1u));
    int remaining = k;
    const uint32_t* src = keys;  // the keys matching the prefix are among src[0, m)
    int m = n;
    for (int pass = 0;; ++pass) {
        int* hist = s.hist[CS > 1 ? (pass & 1) : 0];
        const int shift = top >= kDigitBits - 1 ? top - (kDigitBits - 1) : 0;
        const uint32_t himask = top == 31 ? 0u : ~((2u << top) - 1u);
        for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
        __syncthreads();
#pragma unroll 4
        for (int i = tid; i < m; i += kThreads) {
            const uint32_t u = src[i];
            if ((u & himask) == prefix) atomicAdd(&hist[(u >> shift) & (kBins - 1)], 1);
        }
        __syncthreads();
        // the digit d with (keys above d) < remaining <= (keys at or above d):
        // thread t holds bins 2047-2t and 2046-2t, counted from the top bin
        const int b0 = kBins - 1 - 2 * tid, b1 = b0 - 1;
        int c0, c1;
        if constexpr (CS == 1) {
            c0 = hist[b0];
            c1 = hist[b1];
        } else {
            tc::cluster_sync();  // every CTA's histogram of this pass is complete
            c0 = c1 = 0;
            const uint32_t a = tc::smem_u32(&hist[b1]);  // bins b1 (even), b0 = b1 + 1
#pragma unroll
            for (int r = 0; r < CS; r++) {
                const uint2 v = tc::ld_cluster_v2_u32(tc::mapa_shared(a, (uint32_t)r));
                c1 += (int)v.x;
                c0 += (int)v.y;
            }
        }
        const int before = block_exclusive_scan(c0 + c1, s.scan);
        if (before < remaining && before + c0 >= remaining) {
            s.digit = b0;
            s.above = before;
            s.dcount = c0;
        } else if (before + c0 < remaining && before + c0 + c1 >= remaining) {
            s.digit = b1;
            s.above = before + c0;
            s.dcount = c1;
        }
        __syncthreads();
        const int d = s.digit, cnt = s.dcount;
        remaining -= s.above;
        prefix |= (uint32_t)d << shift;
        // Done at the last digit, or when digit d holds exactly the keys still
        // needed: then the k-th largest key is the smallest of them, every key
        // at or above T = prefix (its lower bits zero) is kept, and there are
        // k of them, so the set is the exact one and has no tie to break.
        if (shift == 0 || cnt == remaining) return Select{prefix, remaining};
        top = shift - 1;
        // (a cluster's CTAs hold a quarter of the row each: their later
        // passes sweep their own keys again, cheaper than copying them out)
        if (CS == 1 && cnt <= kCandCap && src != s.cand) {
            // the keys of digit d go to the candidate list (their order is
            // irrelevant): each warp counts its range's hits, takes its place
            // in the list with one atomic, then writes them
            if (tid == 0) s.n_cand = 0;
            __syncthreads();
            const uint32_t newmask = ~((2u << top) - 1u);
            const int seg = sweep_seg(m), warp = tid >> 5;
            const int i0 = warp * seg, i1 = min(m, i0 + seg);
            int hits = 0;
            for (int r = i0; r < i1; r += 128) {
                uint32_t u[4];
                const uint32_t valid = load4(src, r + 4 * lane, i1, u);
#pragma unroll
                for (int e = 0; e < 4; e++) hits += ((valid >> e) & 1u) && (u[e] & newmask) == prefix;
            }
            hits = (int)__reduce_add_sync(0xffffffffu, (uint32_t)hits);
            int base = 0;
            if (lane == 0 && hits) base = atomicAdd(&s.n_cand, hits);
            base = __shfl_sync(0xffffffffu, base, 0);
            if (hits) {
                for (int r = i0; r < i1; r += 128) {
                    uint32_t u[4];
                    const uint32_t valid = load4(src, r + 4 * lane, i1, u);
                    uint32_t h = 0;
#pragma unroll
                    for (int e = 0; e < 4; e++) h += ((valid >> e) & 1u) && (u[e] & newmask) == prefix;
                    const uint32_t incl = warp_inclusive_sum(h);
                    int pos = base + (int)(incl - h);
#pragma unroll
                    for (int e = 0; e < 4; e++)
                        if (((valid >> e) & 1u) && (u[e] & newmask) == prefix) s.cand[pos++] = u[e];
                    base += (int)__shfl_sync(0xffffffffu, incl, 31);
                }
            }
            __syncthreads();
            src = s.cand;
            m = s.n_cand;
        }
        __syncthreads();  // digit, above and hist are rewritten by the next pass
    }
}

// Keep the top `k` of keys[0, n) in index order: calls emit(pos, i) for the
// kept entries with pos = 0 .. k-1 ascending in i.  Each warp sweeps its
// range twice (see sweep_seg): once to count the keys above T and equal to
// T, once to place them, with one packed (above << 16 | equal) scan over the
// lanes per 128 keys.  keys must be 16-byte aligned.
// CS > 1: the kept keys of the CTAs before this one in the cluster come first.
template <int CS, class S, class Emit>
__device__ void block_compact(const uint32_t* keys, int n, Select sel, S& s, Emit emit) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = sweep_seg(n);
    const int i0 = warp * seg, i1 = min(n, i0 + seg);
    // per lane and step: keys above T and equal to T, packed (each <= 4)
    auto counts = [&](const uint32_t (&u)[4], uint32_t valid) {
        uint32_t c = 0;
#pragma unroll
        for (int e = 0; e < 4; e++)
            if ((valid >> e) & 1u) c += u[e] > sel.T ? (1u << 16) : (u[e] == sel.T ? 1u : 0u);
        return c;
    };
    uint32_t tot = 0;
    for (int r = i0; r < i1; r += 128) {
        uint32_t u[4];
        const uint32_t valid = load4(keys, r + 4 * lane, i1, u);
        tot += counts(u, valid);
    }
    tot = __reduce_add_sync(0xffffffffu, tot);  // a warp's range holds < 65536 keys
    if (lane == 0) {
        s.wcnt[0][warp] = (int)(tot >> 16);
        s.wcnt[1][warp] = (int)(tot & 0xffffu);
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
        if (CS > 1 && lane == 31) {
            s.ctot[0] = g;
            s.ctot[1] = e;
        }
    }
    __syncthreads();
    int gt_base = s.wcnt[0][warp], eq_base = s.wcnt[1][warp];
    if constexpr (CS > 1) {
        tc::cluster_sync();  // every CTA's totals are visible
        if (warp == 0) {  // the kept keys of the CTAs before this one
            const uint32_t rank = tc::cluster_ctarank();
            uint32_t g = 0, e = 0;
            if ((uint32_t)lane < rank) {
                const uint2 v = tc::ld_cluster_v2_u32(tc::mapa_shared(tc::smem_u32(&s.ctot[0]), (uint32_t)lane));
                g = v.x;
                e = v.y;
            }
            g = __reduce_add_sync(0xffffffffu, g);
            e = __reduce_add_sync(0xffffffffu, e);
            if (lane == 0) {
                s.bcast[0] = g;
                s.bcast[1] = e;
            }
        }
        __syncthreads();
        gt_base += (int)s.bcast[0];
        eq_base += (int)s.bcast[1];
    }
    for (int r = i0; r < i1; r += 128) {
        uint32_t u[4];
        const int i = r + 4 * lane;
        const uint32_t valid = load4(keys, i, i1, u);
        const uint32_t c = counts(u, valid);
        const uint32_t incl = warp_inclusive_sum(c);
        const uint32_t excl = incl - c;
        int g = gt_base + (int)(excl >> 16), e = eq_base + (int)(excl & 0xffffu);
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (!((valid >> q) & 1u)) continue;
            if (u[q] > sel.T) {
                emit(g + min(e, sel.take_eq), i + q);
                ++g;
            } else if (u[q] == sel.T) {
                if (e < sel.take_eq) emit(g + e, i + q);
                ++e;
            }
        }
        const uint32_t step = __shfl_sync(0xffffffffu, incl, 31);
        gt_base += (int)(step >> 16);
        eq_base += (int)(step & 0xffffu);
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
    extern __shared__ __align__(16) uint32_t keys[];  // [<= kChunk], 16-byte aligned
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
        const Select t = radix_select<1>(keys, nc, k, lo_k, hi_k, s);
        block_compact<1>(keys, nc, t, s, [&](int pos, int i) {
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
    const Select t = radix_select<1>(keys, nc, k, lo_k, hi_k, s);
    block_compact<1>(keys, nc, t, s, [&](int pos, int i) {
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
    extern __shared__ __align__(16) uint32_t keys[];  // [nchunks * k], 16-byte aligned
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
    const Select t = radix_select<1>(keys, C, k, lo_k, hi_k, s);
    block_compact<1>(keys, C, t, s, [&](int pos, int i) {
        oi[pos] = reinterpret_cast<const int32_t*>(row + chunk_lo(i / k, n, nch) + k)[i % k];
        if (os) os[pos] = key_score(keys[i]);
    });
}

// One query's row of at most kChunk scores selected by a cluster of CS CTAs
// (grid (CS, Q), clusters of (CS, 1, 1)): CTA r holds the keys of
// [b(r), b(r+1)), b(r) = r*n/CS rounded down to a multiple of 4 (b(CS) = n),
// and writes the kept ones of its slice after those of the CTAs before it.
// Every branch between cluster barriers depends on n, k or cluster-wide
// counts only, so all CTAs of a cluster pass the same barriers.
template <int CS>
__global__ void __launch_bounds__(kThreads, 1)
    topk_cluster_kernel(const float* __restrict__ scores, int64_t ld, int64_t n_cap,
                        const int64_t* __restrict__ q_pos, int m, int k,
                        int32_t* __restrict__ idx, float* __restrict__ sel) {
    extern __shared__ __align__(16) uint32_t keys[];  // [<= kChunk / CS + 4], 16-byte aligned
    __shared__ TopkScratch<CS> s;
    tc::grid_dep_wait();    // the scores of the kernel before (a programmatic dependent launch)
    tc::grid_dep_launch();  // ... and the attention after may be scheduled now
    const int rank = (int)tc::cluster_ctarank();
    const int64_t q = blockIdx.y;
    const int n = (int)n_complete(q_pos, q, m, n_cap);
    const float* row = scores + q * ld;
    int32_t* oi = idx + q * k;
    float* os = sel ? sel + q * k : nullptr;
    if (n <= k) {  // every block is kept (the same decision in every CTA)
        if (rank == 0)
            for (int j = threadIdx.x; j < k; j += kThreads) {
                oi[j] = j < n ? j : -1;
                if (os) os[j] = j < n ? row[j] : -INFINITY;
            }
        return;
    }
    auto bnd = [&](int r) { return r == CS ? n : (int)(((int64_t)r * n / CS) & ~(int64_t)3); };
    const int lo = bnd(rank), nc = bnd(rank + 1) - lo;
    uint32_t lo_k, hi_k;
    load_keys<8>(row + lo, nc, keys, lo_k, hi_k);
    __syncthreads();  // the keys are visible to the CTA
    // No cluster-wide min / max: the radix starts at the top bit.  Agreeing on
    // a common prefix costs a cluster barrier, and indexer scores spread over
    // too many bits for a skipped prefix to save a pass.
    const Select t = radix_select<CS>(keys, nc, k, 0u, 0xffffffffu, s);
    block_compact<CS>(keys, nc, t, s, [&](int pos, int i) {
        oi[pos] = lo + i;
        if (os) os[pos] = key_score(keys[i]);
    });
    tc::cluster_sync();  // no CTA leaves while another may still read its shared memory
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
    if (n_cap <= kChunk && n_cap >= kClusterMinKeys && (int64_t)Q * kClusterCS <= 2LL * num_sms()) {
        // few queries of one chunk each (decode): kClusterCS CTAs a query
        const size_t smem = ((size_t)(n_cap / kClusterCS + 4) * sizeof(uint32_t) + 15) & ~(size_t)15;
        {
            cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(topk_cluster_kernel<kClusterCS>), smem);
            if (e != cudaSuccess) return e;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)kClusterCS, (unsigned)Q, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute at[2];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = kClusterCS;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dep_wait
        at[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 2;
        cudaError_t e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel<kClusterCS>, (const float*)scores, ld, n_cap,
                                           q_pos, g.m, k, idx, sel);
        note_launch();
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const int64_t max_chunks = n_cap > kChunk ? (n_cap + kChunk - 1) / kChunk : 1;
    const size_t smem1 = ((size_t)(n_cap < kChunk ? (n_cap > 0 ? n_cap : 1) : kChunk) * sizeof(uint32_t) + 15) & ~(size_t)15;
    // two CTAs an SM when both fit in its 228 KiB of shared memory
    const bool two = smem1 + sizeof(Scratch) + 1024 <= 114 * 1024;
    {
        cudaError_t e = two ? set_smem_attr(reinterpret_cast<const void*>(topk_chunk_kernel<2>), smem1)
                            : set_smem_attr(reinterpret_cast<const void*>(topk_chunk_kernel<1>), smem1);
        if (e != cudaSuccess) return e;
    }
    dim3 grid1((unsigned)max_chunks, (unsigned)Q);
    if (two)
        topk_chunk_kernel<2><<<grid1, kThreads, smem1, st>>>(scores, ld, n_cap, q_pos, g.m, k, idx, sel);
    else
        topk_chunk_kernel<1><<<grid1, kThreads, smem1, st>>>(scores, ld, n_cap, q_pos, g.m, k, idx, sel);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || max_chunks <= 1) return e;
    const size_t smem2 = ((size_t)max_chunks * k * sizeof(uint32_t) + 15) & ~(size_t)15;
    e = set_smem_attr(reinterpret_cast<const void*>(topk_merge_kernel), smem2);
    if (e != cudaSuccess) return e;
    topk_merge_kernel<<<(unsigned)Q, kThreads, smem2, st>>>(scores, ld, n_cap, q_pos, g.m, k, idx, sel);
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa
