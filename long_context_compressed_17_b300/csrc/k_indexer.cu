// k_indexer.cu -- lightning-indexer scoring, CUDA-core path.
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 2: Lightning Indexer
// Top-K 选择": a light indexer scores every compressed block per query.
// score_b = sum_h w_h * relu(q_h . k_b) over causally complete blocks
// (b*m + m - 1 <= i); other blocks get -inf so the selection skips them.
//
// This path serves every shape (fp32 and bf16, idx_dim 64 or 128).  The
// tensor-core path for bf16 / idx_dim 128 lives in k_indexer_tc.cu.
#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int kIdxTile = 128;  // keys per CTA, one per thread

template <int DI>
__global__ void __launch_bounds__(kIdxTile)
    indexer_generic_kernel(const uint8_t* __restrict__ q_idx, const float* __restrict__ w_idx,
                           int HI, const uint8_t* __restrict__ keys, int act, int64_t n_cap,
                           int qps, int q_per_cta, const int64_t* __restrict__ q_pos, int m,
                           float* __restrict__ scores, int64_t n_cap_pad,
                           uint32_t* __restrict__ status) {
    extern __shared__ float sm[];
    float* qs = sm;               // [HI][DI]
    float* ws = sm + HI * DI;     // [HI]
    const int tid = threadIdx.x;
    const int64_t j = (int64_t)blockIdx.x * kIdxTile + tid;
    const int q0 = blockIdx.y * q_per_cta;
    const int seq = q0 / qps;
    const int act_es = (act == CSA_F32) ? 4 : 2;

    float kreg[DI];
    if (j < n_cap) {
        const uint8_t* kr = keys + ((int64_t)seq * n_cap + j) * DI * act_es;
#pragma unroll
        for (int d = 0; d < DI; d++) kreg[d] = load_act(kr, act, d);
    }
    for (int qq = 0; qq < q_per_cta; qq++) {
        const int q = q0 + qq;
        __syncthreads();
        const uint8_t* qr = q_idx + (int64_t)q * HI * DI * act_es;
        for (int e = tid; e < HI * DI; e += kIdxTile) qs[e] = load_act(qr, act, e);
        for (int h = tid; h < HI; h += kIdxTile) ws[h] = w_idx[(int64_t)q * HI + h];
        __syncthreads();
        int64_t n_av = (q_pos[q] + 1) / m;
        if (n_av > n_cap) {
            if (tid == 0 && blockIdx.x == 0) atomicOr(status, CSA_DEV_BAD_POSITION);
            n_av = n_cap;
        }
        if (j >= n_cap) continue;
        float s = -INFINITY;
        if (j < n_av) {
            s = 0.f;
            for (int h = 0; h < HI; h++) {
                float dot = 0.f;
#pragma unroll
                for (int d = 0; d < DI; d++) dot = fmaf(qs[h * DI + d], kreg[d], dot);
                s = fmaf(ws[h], fmaxf(dot, 0.f), s);
            }
        }
        scores[(int64_t)q * n_cap_pad + j] = s;
    }
}

cudaError_t launch_indexer_tc(const Geometry& g, const void* q_idx, const float* w_idx, int HI,
                              int dI, const void* keys, int64_t n_cap, int B, int Q,
                              const int64_t* q_pos, uint32_t* status, float* scores, int64_t ld,
                              cudaStream_t st, bool* launched);

cudaError_t launch_indexer(const Geometry& g, const void* q_idx, const float* w_idx, int HI,
                           int dI, const void* keys, int64_t n_cap, int B, int Q,
                           const int64_t* q_pos, uint32_t* status, float* scores, int64_t ld,
                           cudaStream_t st) {
    if (Q == 0 || n_cap == 0) return cudaSuccess;
    bool launched = false;
    cudaError_t e = launch_indexer_tc(g, q_idx, w_idx, HI, dI, keys, n_cap, B, Q, q_pos, status,
                                      scores, ld, st, &launched);
    if (launched || e != cudaSuccess) return e;
    const int qps = Q / B;
    int qpc = 1;
    for (int c : {32, 16, 8, 4, 2})
        if (qps % c == 0) {
            qpc = c;
            break;
        }
    dim3 grid((unsigned)((n_cap + kIdxTile - 1) / kIdxTile), (unsigned)(Q / qpc));
    size_t smem = (size_t)(HI * dI + HI) * sizeof(float);
    auto run = [&](auto kern) -> cudaError_t {
        if (smem > 48 * 1024) {
            cudaError_t a = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (a != cudaSuccess) return a;
        }
        kern<<<grid, kIdxTile, smem, st>>>(reinterpret_cast<const uint8_t*>(q_idx), w_idx, HI,
                                           reinterpret_cast<const uint8_t*>(keys), g.act, n_cap,
                                           qps, qpc, q_pos, g.m, scores, ld, status);
        note_launch();
        return cudaGetLastError();
    };
    return dI == 64 ? run(indexer_generic_kernel<64>) : run(indexer_generic_kernel<128>);
}

}  // namespace csa
