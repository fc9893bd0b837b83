// k_attend.cu -- CSA / HCA core attention, CUDA-core path, and the split-K
// log-sum-exp combine shared by every attention path.
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2: CSA Step 3 (multi-query attention
// over the top-k blocks), HCA (dense attention over every compressed block),
// and 四项关键 Trick: RMSNorm on q and KV, partial RoPE on the last 64 dims and
// RoPE at -i on the output, a sliding window of the last 128 raw tokens, and a
// learnable sink logit in the softmax denominator.
//
// A query's rows form one list: [selected blocks (CSA) | every block (HCA)]
// followed by the W window positions i-W+1 .. i.  The list is cut into
// `splits` contiguous ranges; each CTA reduces one range for a group of heads
// into an unnormalised partial (m, l, o) and attend_combine_kernel merges the
// partials, adds the sink once and applies the output rotation.  The split
// count depends on the list length and the SM count only, never on the batch
// composition of a single query.
#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa {

constexpr int kAttThreads = 256;
constexpr int kAttRows = 32;

struct AttendArgs {
    const uint8_t* q;
    int act;
    int H, qps;
    const int64_t* q_pos;
    const uint8_t* cache;
    int64_t n_cap;
    int64_t rb;  // stored row bytes
    int kvfmt;
    const int32_t* topk_idx;  // nullptr: dense (HCA)
    int k;
    const uint8_t* window;
    int64_t n_win;
    const int64_t* win_pos0;  // nullptr: the window is a ring (position p at row p mod n_win)
    int W, m, R;
    RopeTheta theta;
    float eps, scale;
    float* part_o;   // [Q, S, H, D]
    float* part_ml;  // [Q, S, H, 2]
    int S;
    int64_t list_base;  // k (CSA) or n_cap (HCA): list position of the first window row
    int64_t rows_per_split;
    uint32_t* status;
};

// Resolve list position p of query (seq, i) to a stored row, or nullptr when
// the row is masked (padding, not yet complete, before position 0).
__device__ __forceinline__ const uint8_t* resolve_row(const AttendArgs& a, int64_t qi, int seq,
                                                      int64_t i, int64_t n_av, int64_t p) {
    if (p < a.list_base) {
        int64_t e;
        if (a.topk_idx) {
            e = a.topk_idx[qi * a.k + p];
            if (e < 0) return nullptr;
            if (e >= n_av) {
                atomicOr(a.status, CSA_DEV_BAD_TOPK_INDEX);
                return nullptr;
            }
        } else {
            e = p;
            if (e >= n_av) return nullptr;
        }
        return a.cache + ((int64_t)seq * a.n_cap + e) * a.rb;
    }
    int64_t wpos = i - a.W + 1 + (p - a.list_base);
    if (wpos < 0) return nullptr;
    if (a.win_pos0 == nullptr)  // ring window: position p at row p mod n_win (n_win >= W)
        return a.window + ((int64_t)seq * a.n_win + wpos % a.n_win) * a.rb;
    int64_t wr = wpos - a.win_pos0[seq];
    if (wr < 0 || wr >= a.n_win) {
        atomicOr(a.status, CSA_DEV_BAD_WINDOW);
        return nullptr;
    }
    return a.window + ((int64_t)seq * a.n_win + wr) * a.rb;
}

// Normalise and rotate the query heads [h0, h0+nh) into qs (float32).
__device__ inline void prepare_q(const AttendArgs& a, int64_t qi, int64_t i, int h0, int nh, int D,
                                 float* qs, float* cs) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int j = tid; j < a.R / 2; j += blockDim.x) rope_cs((double)i, a.theta.t[j], &cs[2 * j], &cs[2 * j + 1]);
    const int act_es = a.act == CSA_F32 ? 4 : 2;
    for (int h = warp; h < nh; h += blockDim.x / 32) {
        const uint8_t* qr = a.q + ((int64_t)qi * a.H + h0 + h) * D * act_es;
        float ss = 0.f;
        for (int d = lane; d < D; d += 32) {
            float x = load_act(qr, a.act, d);
            qs[h * D + d] = x;
            ss = fmaf(x, x, ss);
        }
        ss = warp_sum(ss);
        float r = 1.f / sqrtf(ss / (float)D + a.eps);
        for (int d = lane; d < D; d += 32) qs[h * D + d] *= r;
    }
    __syncthreads();
    for (int e = tid; e < nh * (a.R / 2); e += blockDim.x) {
        int h = e / (a.R / 2), j = e % (a.R / 2);
        float c = cs[2 * j], s = cs[2 * j + 1];
        float* x = qs + h * D + D - a.R + 2 * j;
        float x0 = x[0], x1 = x[1];
        x[0] = x0 * c - x1 * s;
        x[1] = x0 * s + x1 * c;
    }
    __syncthreads();
}

template <int D, int HG>
__global__ void __launch_bounds__(kAttThreads) attend_generic_kernel(AttendArgs a) {
    constexpr int TPH = kAttThreads / HG;   // threads per head in the PV update
    constexpr int OPT = D / TPH;            // output dims per thread
    constexpr int ES = D + 1;               // padded row stride (bank-conflict free)
    extern __shared__ float sm[];
    float* qs = sm;                          // [HG][D]
    float* es = qs + HG * D;                 // [kAttRows][ES]
    float* pr = es + kAttRows * ES;          // [HG][kAttRows]
    float* mh = pr + HG * kAttRows;          // [HG]
    float* lh = mh + HG;                     // [HG]
    float* al = lh + HG;                     // [HG]
    float* cs = al + HG;                     // [R]
    const uint8_t** rp = reinterpret_cast<const uint8_t**>(cs + 64);  // [kAttRows]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.z, h0 = blockIdx.y * HG;
    const int64_t qi = blockIdx.x;
    const int seq = (int)(qi / a.qps);
    const int64_t i = a.q_pos[qi];
    int64_t n_av = (i + 1) / a.m;
    if (n_av > a.n_cap) {
        if (tid == 0) atomicOr(a.status, CSA_DEV_BAD_POSITION);
        n_av = a.n_cap;
    }
    prepare_q(a, qi, i, h0, HG, D, qs, cs);
    if (tid < HG) {
        mh[tid] = -INFINITY;
        lh[tid] = 0.f;
    }
    float o[OPT];
#pragma unroll
    for (int u = 0; u < OPT; u++) o[u] = 0.f;
    const int hl = tid / TPH, dl = tid % TPH;

    const int64_t list_len = a.list_base + a.W;
    const int64_t r0 = (int64_t)split * a.rows_per_split;
    const int64_t r1 = min(list_len, r0 + a.rows_per_split);
    for (int64_t t0 = r0; t0 < r1; t0 += kAttRows) {
        if (tid < kAttRows) {
            int64_t p = t0 + tid;
            rp[tid] = (p < r1) ? resolve_row(a, qi, seq, i, n_av, p) : nullptr;
        }
        __syncthreads();
        for (int e = tid; e < kAttRows * D; e += kAttThreads) {
            int r = e / D, d = e % D;
            const uint8_t* row = rp[r];
            es[r * ES + d] = row ? load_kv(row, a.kvfmt, D, d) : 0.f;
        }
        __syncthreads();
        for (int h = warp; h < HG; h += kAttThreads / 32) {
            float s = 0.f;
            const float* qh = qs + h * D;
            const float* er = es + lane * ES;
#pragma unroll 8
            for (int d = 0; d < D; d++) s = fmaf(qh[d], er[d], s);
            s = rp[lane] ? s * a.scale : -INFINITY;
            float mt = warp_max(s);
            float m_old = mh[h];
            float m_new = fmaxf(m_old, mt);
            float p = (m_new == -INFINITY) ? 0.f : expf(s - m_new);
            float alpha = (m_new == -INFINITY) ? 1.f : expf(m_old - m_new);
            float ps = warp_sum(p);
            pr[h * kAttRows + lane] = p;
            if (lane == 0) {
                mh[h] = m_new;
                lh[h] = lh[h] * alpha + ps;
                al[h] = alpha;
            }
        }
        __syncthreads();
        const float alpha = al[hl];
#pragma unroll
        for (int u = 0; u < OPT; u++) o[u] *= alpha;
        for (int r = 0; r < kAttRows; r++) {
            float p = pr[hl * kAttRows + r];
            const float* er = es + r * ES + dl;
#pragma unroll
            for (int u = 0; u < OPT; u++) o[u] = fmaf(p, er[u * TPH], o[u]);
        }
        __syncthreads();
    }
    const int64_t pbase = ((qi * a.S + split) * a.H + h0 + hl);
#pragma unroll
    for (int u = 0; u < OPT; u++) a.part_o[pbase * D + dl + u * TPH] = o[u];
    if (tid < HG) {
        int64_t pb = ((qi * a.S + split) * a.H + h0 + tid) * 2;
        a.part_ml[pb] = mh[tid];
        a.part_ml[pb + 1] = lh[tid];
    }
}

// Merge split partials, add the sink, normalise, rotate by -i and store.
// One warp per (query, head) item, four warps a block; lane l owns the
// float4 chunks l, l+32, l+64, l+96 of the row (dims 4c .. 4c+3 of chunk c,
// D <= 512), so the item's scalar work (the slot weights, the denominator,
// the rotation) is done once for the whole row.  The rows of the first
// kRing slots are requested at once (before the count of slots is known
// where it is read from memory: slots below S_alloc are inside the
// allocation), and every later slot's row kRing slots ahead of its use.
//   CUDA-core kernel, or fixed splits (tiles == 0): Q*H items, query q has
//   S_alloc partials.
//   Tensor-core kernel (tiles > 0): the CTAs own contiguous ranges of all
//   queries' tile lists (tiles per query) as TileDeal{total, tiles, grid,
//   qcta, qrem, qc} deals them; only a query cut by a CTA boundary has
//   partials (one per CTA meeting it, nslots[q] of them, written by the CTA
//   holding its first tile), every other query was finished by its only CTA
//   (nslots[q] = 0).  With by_query item (q, h) takes query q if it was cut;
//   otherwise there are (grid-1)*H items and item (b-1, h) handles the query
//   cut by boundary b, if b is the first boundary inside it.
constexpr int kCombineWarps = 4;

// The query cut by CTA boundary b (first tile of CTA b inside it) whose
// first boundary it is, and its partial count, or qi = -1 (the boundary
// falls between queries, or the query was met at an earlier boundary).  Out
// of line: only prefill-sized batches take it, and inlined it was 40% of the
// combine's code.  Tile counts are below 2^31.
__device__ __noinline__ void boundary_query(int64_t b, int64_t tiles, int64_t total, int grid, int qcta, int qrem,
                                            int qc, int64_t* qi_out, int* sq_out) {
    const TileDeal deal{total, tiles, grid, qcta, qrem, qc};
    const int64_t g = deal.begin(b);  // first tile of CTA b
    const uint32_t qi = (uint32_t)g / (uint32_t)tiles;
    *qi_out = -1;
    if ((int64_t)qi * tiles == g) return;  // the boundary falls between queries
    const int64_t c0 = deal.cta_of((int64_t)qi * tiles);
    if (c0 + 1 != b) return;               // handled at the query's first boundary
    *qi_out = qi;
    *sq_out = (int)(deal.cta_of(((int64_t)qi + 1) * tiles - 1) - c0 + 1);
}

__global__ void __launch_bounds__(32 * kCombineWarps)
    attend_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                          const int32_t* __restrict__ nslots, int S_alloc, int H, int D,
                          const float* __restrict__ sink, const int64_t* __restrict__ q_pos, int derotate,
                          void* __restrict__ out, int act, float* __restrict__ lse, int64_t tiles, int64_t total,
                          int grid, int qcta, int qrem, int qc, int by_query, int64_t items, RopeTheta theta) {
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (item >= items) return;
    const int h = (int)((uint32_t)item % (uint32_t)H);  // items < 2^31
    const int64_t unit = (int64_t)((uint32_t)item / (uint32_t)H);
    int64_t qi = unit;
    int Sq = S_alloc;  // an upper bound until nslots is read
    if (tiles > 0 && !by_query) {
        boundary_query(unit + 1, tiles, total, grid, qcta, qrem, qc, &qi, &Sq);
        if (qi < 0) return;
    }
    const int S = S_alloc;
    const float* ml = part_ml + (qi * S * H + h) * 2;  // slot s: ml[s * 2H], ml[s * 2H + 1]
    const int64_t mstep = (int64_t)H * 2;
    const float4* po = reinterpret_cast<const float4*>(part_o + (qi * S * H + h) * D);  // slot s: po[s * H*D/4]
    const int64_t ostep = (int64_t)H * D / 4;
    constexpr int kC = 4;     // chunks a lane (D / 4 <= 128)
    constexpr int kRing = 4;  // slots whose rows are in flight
    const int nc = D / 4;
    float4 v[kRing][kC];
    auto request = [&](int s2, float4* r) {  // slot s2's row into ring entry r
#pragma unroll
        for (int k = 0; k < kC; k++)
            if (lane + 32 * k < nc) r[k] = __ldg(po + s2 * ostep + lane + 32 * k);
    };
#pragma unroll
    for (int j = 0; j < kRing; j++)
        if (j < Sq) request(j, v[j]);
    const int64_t i = q_pos[qi];
    const float sk = sink[h];
    if (tiles > 0 && by_query) {
        Sq = nslots[qi];
        if (Sq == 0) return;                     // finished by its only CTA
    }
    // RoPE at -i for pair `lane` of the rotated dims (the same for every head)
    float rc = 1.f, rs = 0.f;
    if (derotate) rope_cs(-(double)i, theta.t[lane], &rc, &rs);
    float mstar = sk;
    for (int s2 = lane; s2 < Sq; s2 += 32) mstar = fmaxf(mstar, __ldg(ml + s2 * mstep));
    mstar = warp_max(mstar);
    auto weight = [&](int s2) {
        const float m0 = __ldg(ml + s2 * mstep);
        return (mstar == -INFINITY || m0 == -INFINITY) ? 0.f : expf(m0 - mstar);
    };
    float l = 0.f;
    for (int s2 = lane; s2 < Sq; s2 += 32) l += weight(s2) * __ldg(ml + s2 * mstep + 1);
    l = warp_sum(l);
    if (mstar != -INFINITY && sk != -INFINITY) l += expf(sk - mstar);
    if (lane == 0 && lse) lse[qi * H + h] = l > 0.f ? mstar + logf(l) : -INFINITY;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    // slot weights in slot order; a slot of weight 0 is not added (its values
    // are never used, whatever they hold)
    float4 acc[kC];
#pragma unroll
    for (int k = 0; k < kC; k++) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < Sq; s0 += kRing) {
#pragma unroll
        for (int j = 0; j < kRing; j++) {
            const int s2 = s0 + j;
            if (s2 >= Sq) break;
            const float w = weight(s2);
            if (w != 0.f) {
#pragma unroll
                for (int k = 0; k < kC; k++) {
                    acc[k].x = fmaf(w, v[j][k].x, acc[k].x);
                    acc[k].y = fmaf(w, v[j][k].y, acc[k].y);
                    acc[k].z = fmaf(w, v[j][k].z, acc[k].z);
                    acc[k].w = fmaf(w, v[j][k].w, acc[k].w);
                }
            }
            if (s2 + kRing < Sq) request(s2 + kRing, v[j]);  // slot s2's entry is free again
        }
    }
    // the rotated dims D-64 .. D-1 are chunks (D-64)/4 .. D/4-1: lanes 16..31
    // of one k, whose pairs are 2(lane-16) and 2(lane-16)+1
    const int p0 = 2 * (lane & 15);
    const float c0 = __shfl_sync(0xffffffffu, rc, p0), s0 = __shfl_sync(0xffffffffu, rs, p0);
    const float c1 = __shfl_sync(0xffffffffu, rc, p0 + 1), s1 = __shfl_sync(0xffffffffu, rs, p0 + 1);
#pragma unroll
    for (int k = 0; k < kC; k++) {
        const int c = lane + 32 * k;
        if (c >= nc) break;
        float o[4] = {acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv};
        if (derotate && 4 * c >= D - kRopeDims) {
            const float x0 = o[0], x1 = o[1], x2 = o[2], x3 = o[3];
            o[0] = x0 * c0 - x1 * s0;
            o[1] = x0 * s0 + x1 * c0;
            o[2] = x2 * c1 - x3 * s1;
            o[3] = x2 * s1 + x3 * c1;
        }
        if (act == CSA_F32) {
            reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (qi * H + h) * D)[c] =
                make_float4(o[0], o[1], o[2], o[3]);
        } else {
            uint2 pk;
            pk.x = (uint32_t)f32_to_bf16_rn(o[0]) | ((uint32_t)f32_to_bf16_rn(o[1]) << 16);
            pk.y = (uint32_t)f32_to_bf16_rn(o[2]) | ((uint32_t)f32_to_bf16_rn(o[3]) << 16);
            reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(out) + (qi * H + h) * D)[c] = pk;
        }
    }
}

cudaError_t launch_attend_tc(const Geometry& g, const AttendPlan& pl, bool sparse, const void* q,
                             int H, int B, int Q, const int64_t* q_pos, const void* cache,
                             int64_t n_cap, const int32_t* topk_idx, const void* window,
                             int64_t n_win, const int64_t* win_pos0, const float* sink,
                             void* out, float* lse, float* part_o, float* part_ml, int32_t* nslots,
                             uint8_t* deq, uint32_t* status, cudaStream_t st);

template <int D, int HG>
static cudaError_t run_generic(const AttendArgs& a, int Q, int H, cudaStream_t st) {
    size_t smem = (size_t)(HG * D + kAttRows * (D + 1) + HG * kAttRows + 3 * HG + 64) * sizeof(float) +
                  kAttRows * sizeof(void*);
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(attend_generic_kernel<D, HG>), smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)Q, (unsigned)(H / HG), (unsigned)a.S);
    attend_generic_kernel<D, HG><<<grid, kAttThreads, smem, st>>>(a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_attend(const Geometry& g, const AttendPlan& pl, bool sparse, const void* q,
                          int H, int B, int Q, const int64_t* q_pos, const void* cache,
                          int64_t n_cap, const int32_t* topk_idx, const void* window,
                          int64_t n_win, const int64_t* win_pos0, const float* sink, void* out,
                          float* lse, uint8_t* ws, uint32_t* status, cudaStream_t st) {
    if (Q == 0) return cudaSuccess;
    float* part_o = reinterpret_cast<float*>(ws + pl.part_o_off);
    float* part_ml = reinterpret_cast<float*>(ws + pl.part_ml_off);
    int32_t* nslots = pl.nslots_off ? reinterpret_cast<int32_t*>(ws + pl.nslots_off) : nullptr;
    cudaError_t e;
    if (pl.use_tc) {
        e = launch_attend_tc(g, pl, sparse, q, H, B, Q, q_pos, cache, n_cap, topk_idx, window,
                             n_win, win_pos0, sink, out, lse, part_o, part_ml, nslots, ws + pl.deq_off, status, st);
    } else {
        AttendArgs a;
        a.q = reinterpret_cast<const uint8_t*>(q);
        a.act = g.act;
        a.H = H;
        a.qps = Q / B;
        a.q_pos = q_pos;
        a.cache = reinterpret_cast<const uint8_t*>(cache);
        a.n_cap = n_cap;
        a.rb = g.kv_row_bytes;
        a.kvfmt = g.kv;
        a.topk_idx = sparse ? topk_idx : nullptr;
        a.k = g.k;
        a.window = reinterpret_cast<const uint8_t*>(window);
        a.n_win = n_win;
        a.win_pos0 = win_pos0;
        a.W = g.W;
        a.m = g.m;
        a.R = g.R;
        a.theta = rope_theta(g);
        a.eps = g.eps;
        a.scale = g.scale;
        a.part_o = part_o;
        a.part_ml = part_ml;
        a.S = pl.splits;
        a.list_base = sparse ? g.k : n_cap;
        a.rows_per_split = pl.rows_per_split;
        a.status = status;
        const int HG = pl.head_group;
        if (g.D == 512 && HG == 16) e = run_generic<512, 16>(a, Q, H, st);
        else if (g.D == 512 && HG == 8) e = run_generic<512, 8>(a, Q, H, st);
        else if (g.D == 256 && HG == 16) e = run_generic<256, 16>(a, Q, H, st);
        else if (g.D == 256 && HG == 8) e = run_generic<256, 8>(a, Q, H, st);
        else if (g.D == 128 && HG == 16) e = run_generic<128, 16>(a, Q, H, st);
        else if (g.D == 128 && HG == 8) e = run_generic<128, 8>(a, Q, H, st);
        else return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    // tensor-core kernel with ranges: an item per (query, head) when there
    // are no more queries than CTA boundaries (or the ranges are
    // query-aligned), else per (boundary, head).  Fixed splits (and the
    // CUDA-core kernel): every query has pl.splits partials, merged in split
    // order by an item per (query, head).
    const bool ranges = pl.use_tc && pl.tc_seg == 0;
    const int by_query = ranges && (Q <= pl.tc_grid - 1 || pl.tc_qcta > 0);
    const int64_t items = (!ranges || by_query) ? (int64_t)Q * H : (int64_t)(pl.tc_grid - 1) * H;
    if (items == 0) return cudaSuccess;  // every query was finished by its only CTA
    if (g.D % 128 != 0 || g.D > 512) return cudaErrorInvalidValue;  // the combine's lane layout
    if (items >= (1LL << 31)) return cudaErrorInvalidValue;         // its item arithmetic is 32-bit
    const int64_t blocks = (items + kCombineWarps - 1) / kCombineWarps;
    // launched in stream order: as a programmatic dependent of the attention
    // kernel it took 2-4 us longer a step (CSA decode 128K, HCA decode 1M)
    attend_combine_kernel<<<dim3((unsigned)blocks), dim3(32 * kCombineWarps), 0, st>>>(part_o, part_ml,
        ranges && by_query ? nslots : nullptr, pl.splits, H, g.D, sink, q_pos, g.derotate, out, g.act, lse,
        ranges ? (int64_t)pl.tc_T : 0, pl.tc_total, pl.tc_grid,
        pl.tc_qcta, pl.tc_qrem, pl.tc_qc, by_query, items, rope_theta(g));
    note_launch();
    return cudaGetLastError();
}

}  // namespace csa
