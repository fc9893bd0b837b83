// k_indexer.cu -- lightning-indexer scoring, CUDA-core path.
//
// "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 2: Lightning Indexer
// Top-K 选择": a light indexer scores every compressed block per query.
// score_b = sum_h w_h * relu(q_h . k_b) over causally complete blocks
// (b*m + m - 1 <= i); other blocks get -inf so the selection skips them.
//
// This path serves every shape (fp32 and bf16, idx_dim 64 or 128).  The
// tensor-core path for bf16 / idx_dim 128 lives in k_indexer_tc.cu.
#include <limits.h>
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
                              int dI, const void* keys, const float* key_scales, int64_t n_cap, int B,
                              int Q, const int64_t* q_pos, uint32_t* status, float* scores, int64_t ld,
                              cudaStream_t st, bool* launched);

cudaError_t launch_indexer(const Geometry& g, const void* q_idx, const float* w_idx, int HI,
                           int dI, const void* keys, int64_t n_cap, int B, int Q,
                           const int64_t* q_pos, uint32_t* status, float* scores, int64_t ld,
                           cudaStream_t st) {
    if (Q == 0 || n_cap == 0) return cudaSuccess;
    bool launched = false;
    cudaError_t e = launch_indexer_tc(g, q_idx, w_idx, HI, dI, keys, nullptr, n_cap, B, Q, q_pos, status,
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
            cudaError_t a = set_smem_attr(reinterpret_cast<const void*>(kern), smem);
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

// ------------------------------------------------------------ E4M3 indexer rows
// One warp quantises a row of 128 values (4 per lane, lane l the dims
// 4l .. 4l+3): scale = amax/448 (1 for an all-zero row), code = E4M3 of
// x / scale, round to nearest even with saturation, both divisions in float32
// (the rule of the mixed cache rows, over the whole row).  The lane's four
// codes come back packed little-endian; the scale goes to every lane.
__device__ __forceinline__ float warp_quant_row128(const uint8_t* row, int act, int lane, uint32_t* codes4) {
    float x[4];
#pragma unroll
    for (int e = 0; e < 4; e++) x[e] = load_act(row, act, 4 * lane + e);
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    amax = warp_max(amax);
    const float scale = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
    uint32_t c = 0;
#pragma unroll
    for (int e = 0; e < 4; e++) c |= (uint32_t)f32_to_e4m3_sat(__fdiv_rn(x[e], scale)) << (8 * e);
    *codes4 = c;
    return scale;
}

// rows [n, 128] (act format) -> codes [n, 128], scales [n]; 8 rows a block.
__global__ void __launch_bounds__(256)
    pack_idx_keys_kernel(const uint8_t* __restrict__ rows, int act, int64_t n, uint8_t* __restrict__ codes,
                         float* __restrict__ scales) {
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= n) return;
    const int64_t rb = act == CSA_F32 ? 4 * 128 : 2 * 128;
    uint32_t c;
    const float sc = warp_quant_row128(rows + r * rb, act, lane, &c);
    reinterpret_cast<uint32_t*>(codes + r * 128)[lane] = c;
    if (lane == 0) scales[r] = sc;
}

// Query heads [Q*64, 128] -> E4M3 codes, and the head weights times the head
// scales: w_eff[q, h] = w_idx[q, h] * scale_qh (the score is
// sk * sum_h w_h * scale_qh * relu(q8_h . k8), every scale positive).
__global__ void __launch_bounds__(256)
    quant_idx_queries_kernel(const uint8_t* __restrict__ q, int act, const float* __restrict__ w_idx, int64_t rows,
                             uint8_t* __restrict__ q8, float* __restrict__ w_eff) {
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const int64_t rb = act == CSA_F32 ? 4 * 128 : 2 * 128;
    uint32_t c;
    const float sc = warp_quant_row128(q + r * rb, act, lane, &c);
    reinterpret_cast<uint32_t*>(q8 + r * 128)[lane] = c;
    if (lane == 0) w_eff[r] = w_idx[r] * sc;
}

cudaError_t launch_pack_idx_keys(const Geometry& g, const void* rows, int64_t n, uint8_t* codes, float* scales,
                                 cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    pack_idx_keys_kernel<<<(unsigned)((n + 7) / 8), 256, 0, st>>>(reinterpret_cast<const uint8_t*>(rows), g.act,
                                                                   n, codes, scales);
    note_launch();
    return cudaGetLastError();
}

// ------------------------------------------------------------ FP4 indexer keys
// floor(log2 a) of a positive float32, exactly (subnormals included).
__device__ __forceinline__ int floor_log2_pos(float a) {
    const uint32_t b = __float_as_uint(a);
    const int ex = (int)(b >> 23);
    if (ex != 0) return ex - 127;
    return (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
}

// E2M1 code of q: the nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6, ties to the even
// code, saturating at 6; sign in bit 3 (never on a zero code).
__device__ __forceinline__ uint32_t e2m1_code(float q) {
    const float a = fabsf(q);
    uint32_t c;
    if (a <= 0.25f) c = 0;        // tie 0.25 -> 0 (even)
    else if (a < 0.75f) c = 1;    // tie 0.75 -> 1.0 (even)
    else if (a <= 1.25f) c = 2;   // tie 1.25 -> 1.0
    else if (a < 1.75f) c = 3;    // tie 1.75 -> 2
    else if (a <= 2.5f) c = 4;    // tie 2.5 -> 2
    else if (a < 3.5f) c = 5;     // tie 3.5 -> 4
    else if (a <= 5.f) c = 6;     // tie 5 -> 4
    else c = 7;
    return (c != 0 && q < 0.f) ? (c | 8u) : c;
}

// keys [B, n_cap, 128] (act format) -> packed tiles [B, n_tiles] of 8704
// bytes: tile t holds keys 128t .. 128t+127, first their codes (64 bytes a
// key: dim 2i in the low nibble of byte i, dim 2i+1 in the high one), then
// their exponent bytes (4 a key, block j's scale 2^(byte - 127)); key slots
// past n_cap hold an all-zero key (codes 0, exponent bytes 127).  Block j: e_j = floor(log2 amax) - 2 (its largest value
// in [4, 8)), 0 for an all-zero block; a nonzero block more than 14 binades
// below the key's largest is raised to it minus 14 (the key then converts to
// E4M3 with one scale without loss); codes = E2M1 of x / 2^e_j.  One warp a
// key slot, lane l holding dims 4l .. 4l+3 (block l / 8).
__global__ void __launch_bounds__(256)
    pack_idx_keys_fp4_kernel(const uint8_t* __restrict__ keys, int act, int64_t n_cap, int n_tiles,
                             int64_t total_slots, uint8_t* __restrict__ pack) {
    const int64_t slot = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (slot >= total_slots) return;
    const int64_t per_seq = (int64_t)n_tiles * 128;
    const int64_t seq = slot / per_seq, r = slot - seq * per_seq;
    const int64_t t = r >> 7;
    const int k = (int)(r & 127);
    uint8_t* tile = pack + (seq * n_tiles + t) * 8704;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < n_cap) {
        const uint8_t* row = keys + (seq * n_cap + r) * (int64_t)(act == CSA_F32 ? 512 : 256);
#pragma unroll
        for (int e = 0; e < 4; e++) x[e] = load_act(row, act, 4 * lane + e);
    }
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const bool nz = amax > 0.f;
    int e = nz ? floor_log2_pos(amax) - 2 : 0;
    int E = nz ? e : INT_MIN;
    E = max(E, __shfl_xor_sync(0xffffffffu, E, 8));
    E = max(E, __shfl_xor_sync(0xffffffffu, E, 16));
    if (nz && e < E - 14) e = E - 14;
    e = min(127, max(-127, e));
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) c |= e2m1_code(ldexpf(x[i], -e)) << (4 * i);
    *reinterpret_cast<uint16_t*>(tile + k * 64 + 2 * lane) = (uint16_t)c;
    if ((lane & 7) == 0) tile[128 * 64 + k * 4 + (lane >> 3)] = (uint8_t)(e + 127);
}

cudaError_t launch_pack_idx_keys_fp4(const Geometry& g, const void* keys, int B, int64_t n_cap, uint8_t* pack,
                                     cudaStream_t st) {
    if (B == 0 || n_cap == 0) return cudaSuccess;
    const int n_tiles = (int)((n_cap + 127) / 128);
    const int64_t slots = (int64_t)B * n_tiles * 128;
    pack_idx_keys_fp4_kernel<<<(unsigned)((slots + 7) / 8), 256, 0, st>>>(reinterpret_cast<const uint8_t*>(keys),
                                                                          g.act, n_cap, n_tiles, slots, pack);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_indexer_tc_fp4(const Geometry& g, const uint8_t* q8, const float* w_eff, const uint8_t* key_pack,
                                  int64_t n_cap, int B, int Q, const int64_t* q_pos, uint32_t* status,
                                  float* scores, int64_t ld, cudaStream_t st, bool* launched);

// FP4 indexer: the queries are quantised as for E4M3 keys, then the tcgen05
// kernel expands the packed keys to E4M3 in shared memory and scores them.
cudaError_t launch_indexer_fp4(const Geometry& g, const void* q_idx, const float* w_idx, const uint8_t* key_pack,
                               int64_t n_cap, int B, int Q, const int64_t* q_pos, uint32_t* status, float* scores,
                               int64_t ld, uint8_t* q8, float* w_eff, cudaStream_t st) {
    if (Q == 0 || n_cap == 0) return cudaSuccess;
    const int64_t rows = (int64_t)Q * 64;
    quant_idx_queries_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(reinterpret_cast<const uint8_t*>(q_idx),
                                                                          g.act, w_idx, rows, q8, w_eff);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bool launched = false;
    e = launch_indexer_tc_fp4(g, q8, w_eff, key_pack, n_cap, B, Q, q_pos, status, scores, ld, st, &launched);
    if (e == cudaSuccess && !launched) return cudaErrorInvalidValue;  // shapes checked by the C ABI
    return e;
}

// E4M3 indexer: the queries are quantised into q8 / w_eff (workspace), then
// the tcgen05 kernel scores E4M3 keys against them.
cudaError_t launch_indexer_fp8(const Geometry& g, const void* q_idx, const float* w_idx, const uint8_t* key_codes,
                               const float* key_scales, int64_t n_cap, int B, int Q, const int64_t* q_pos,
                               uint32_t* status, float* scores, int64_t ld, uint8_t* q8, float* w_eff,
                               cudaStream_t st) {
    if (Q == 0 || n_cap == 0) return cudaSuccess;
    const int64_t rows = (int64_t)Q * 64;
    quant_idx_queries_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(reinterpret_cast<const uint8_t*>(q_idx),
                                                                          g.act, w_idx, rows, q8, w_eff);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bool launched = false;
    e = launch_indexer_tc(g, q8, w_eff, 64, 128, key_codes, key_scales, n_cap, B, Q, q_pos, status, scores, ld,
                          st, &launched);
    if (e == cudaSuccess && !launched) return cudaErrorInvalidValue;  // shapes checked by the C ABI
    return e;
}

}  // namespace csa
