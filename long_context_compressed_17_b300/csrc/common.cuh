// common.cuh -- device helpers shared by the kernels of libcsa (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa.h"

namespace csa {

constexpr int kRopeDims = 64;
constexpr uint32_t kStatusWordBytes = 256;  // head of every workspace

// ---------------------------------------------------------------- formats
__host__ __device__ inline int64_t fp8m_row_bytes(int D) {
    int64_t raw = (int64_t)(D - kRopeDims) + kRopeDims * 2 + 4 * (int64_t)((D - kRopeDims) / 64);
    return (raw + 15) / 16 * 16;
}

__host__ __device__ inline int64_t row_bytes(int fmt, int D) {
    if (fmt == CSA_F32) return 4 * (int64_t)D;
    if (fmt == CSA_BF16) return 2 * (int64_t)D;
    if (fmt == CSA_FP8_MIXED) return fp8m_row_bytes(D);
    return -1;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&b);
}

// E4M3 code -> float (exact); uses the hardware conversion.
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __half2float(*reinterpret_cast<__half*>(&hr));
}

// float -> E4M3, round to nearest even, saturating to +-448 (hardware conversion).
__device__ __forceinline__ uint8_t f32_to_e4m3_sat(float f) {
    return (uint8_t)__nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3);
}

// Read element d of a row in an activation format (F32 / BF16).
__device__ __forceinline__ float load_act(const void* row, int fmt, int d) {
    if (fmt == CSA_F32) return reinterpret_cast<const float*>(row)[d];
    return bf16_to_f32(reinterpret_cast<const uint16_t*>(row)[d]);
}

__device__ __forceinline__ void store_act(void* row, int fmt, int d, float v) {
    if (fmt == CSA_F32)
        reinterpret_cast<float*>(row)[d] = v;
    else
        reinterpret_cast<uint16_t*>(row)[d] = f32_to_bf16_rn(v);
}

// Decode element d of a stored cache row (F32 / BF16 / FP8_MIXED).
__device__ __forceinline__ float load_kv(const uint8_t* row, int fmt, int D, int d) {
    if (fmt == CSA_F32) return reinterpret_cast<const float*>(row)[d];
    if (fmt == CSA_BF16) return bf16_to_f32(reinterpret_cast<const uint16_t*>(row)[d]);
    int nf = D - kRopeDims;
    if (d >= nf) return bf16_to_f32(reinterpret_cast<const uint16_t*>(row + nf)[d - nf]);
    const float* scales = reinterpret_cast<const float*>(row + nf + 2 * kRopeDims);
    return e4m3_to_f32(row[d]) * scales[d >> 6];
}

// ---------------------------------------------------------------- RoPE
// cos/sin of pos * theta.  The angle (up to ~1e6 rad at 1M context) is formed
// and reduced modulo 2*pi in double, so the float sincos sees |r| <= pi and
// the result keeps full float accuracy at any position.
__device__ __forceinline__ void rope_cs(double pos, double theta, float* c, float* s) {
    const double kTwoPi = 6.283185307179586476925286766559;
    const double a = pos * theta;
    const double k = rint(a * (1.0 / kTwoPi));
    const float r = (float)fma(-k, kTwoPi, a);
    sincosf(r, s, c);
}

// Q queries' tile lists (T tiles each, total = Q*T) dealt to `grid` CTAs in
// contiguous ranges.  qcta == 0: balanced, n units over grid CTAs with the
// first n % grid CTAs taking one more (share / owner).  Every query counts
// as qc + T units, qc of them (the cost of preparing its q' and writing its
// partial, in tiles) before its first tile, and CTA c owns the tiles among
// its units of U = Q*(qc + T): a CTA that starts a second query takes qc
// fewer tiles (qc 0: the tiles themselves are the units).  qcta > 0,
// query-aligned: queries 0 .. qrem-1 get qcta+1 CTAs and the others qcta
// (grid = Q*qcta + qrem), each query's tiles split evenly over its CTAs, so
// that no CTA meets two queries (a CTA meeting two prepares two q' and
// writes two partials, and the slowest CTA sets the kernel's time).
// Unit, tile and CTA counts are below 2^31 (the host plans no more), so the
// divisions run in 32 bits.
struct TileDeal {
    int64_t total, T;
    int grid, qcta, qrem, qc;
    // first of n units that CTA c owns (c = grid: n)
    __host__ __device__ static int64_t share(int64_t c, int64_t n, int grid) {
        const uint32_t per = (uint32_t)n / (uint32_t)grid, rem = (uint32_t)n - per * (uint32_t)grid;
        return c * (int64_t)per + (c < (int64_t)rem ? c : (int64_t)rem);
    }
    // CTA owning unit u of n (n >= grid)
    __host__ __device__ static int64_t owner(int64_t u, int64_t n, int grid) {
        const uint32_t per = (uint32_t)n / (uint32_t)grid, rem = (uint32_t)n - per * (uint32_t)grid;
        const uint32_t big = rem * (per + 1);
        return (uint32_t)u < big ? (uint32_t)u / (per + 1) : rem + ((uint32_t)u - big) / per;
    }
    __host__ __device__ int64_t first_cta(int64_t qi) const { return qi * qcta + (qi < qrem ? qi : qrem); }
    __host__ __device__ int64_t ctas(int64_t qi) const { return qcta + (qi < qrem ? 1 : 0); }
    __host__ __device__ int64_t units() const { return (int64_t)((uint32_t)total / (uint32_t)T) * (T + qc); }
    // first tile of CTA c (c = grid: total)
    __host__ __device__ int64_t begin(int64_t c) const {
        if (qcta == 0) {
            if (qc == 0) return share(c, total, grid);
            const int64_t u = share(c, units(), grid);
            const int64_t qi = (uint32_t)u / (uint32_t)(T + qc), r = u - qi * (T + qc) - qc;
            return qi * T + (r > 0 ? r : 0);
        }
        const int64_t big = (int64_t)qrem * (qcta + 1);
        const int64_t qi = c < big ? (int64_t)((uint32_t)c / (uint32_t)(qcta + 1))
                                   : qrem + (int64_t)((uint32_t)(c - big) / (uint32_t)qcta);
        return qi * T + (uint32_t)((c - first_cta(qi)) * T) / (uint32_t)ctas(qi);
    }
    // CTA that owns tile g
    __host__ __device__ int64_t cta_of(int64_t g) const {
        const int64_t qi = (uint32_t)g / (uint32_t)T, t = g - qi * T;
        if (qcta == 0) {
            if (qc == 0) return owner(g, total, grid);
            return owner(qi * (T + qc) + qc + t, units(), grid);
        }
        return first_cta(qi) + (uint32_t)((t + 1) * ctas(qi) - 1) / (uint32_t)T;
    }
};

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Store one row held in shared memory (float32, D values) into a cache row
// format.  Executed by one full warp.  For FP8_MIXED every 64-dim group is
// quantised with scale = amax/448 (1 for an all-zero group).
__device__ inline void warp_pack_row(const float* __restrict__ src, int D, int fmt,
                                     uint8_t* __restrict__ dst) {
    const int lane = threadIdx.x & 31;
    if (fmt == CSA_F32) {
        float* o = reinterpret_cast<float*>(dst);
        for (int d = lane; d < D; d += 32) o[d] = src[d];
        return;
    }
    if (fmt == CSA_BF16) {
        uint16_t* o = reinterpret_cast<uint16_t*>(dst);
        for (int d = lane; d < D; d += 32) o[d] = f32_to_bf16_rn(src[d]);
        return;
    }
    const int nf = D - kRopeDims;
    float* scales = reinterpret_cast<float*>(dst + nf + 2 * kRopeDims);
    // chunks of 16 dims: four consecutive lanes cover one 64-dim group
    for (int c0 = 0; c0 < nf / 16; c0 += 32) {
        int c = c0 + lane;
        bool active = c < nf / 16;
        float amax = 0.f;
        if (active)
            for (int e = 0; e < 16; e++) amax = fmaxf(amax, fabsf(src[16 * c + e]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        float scale = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
        if (active) {
            uint32_t w[4];
            for (int e4 = 0; e4 < 4; e4++) {
                uint32_t v = 0;
                for (int b = 0; b < 4; b++) {
                    float x = __fdiv_rn(src[16 * c + 4 * e4 + b], scale);
                    v |= (uint32_t)f32_to_e4m3_sat(x) << (8 * b);
                }
                w[e4] = v;
            }
            *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
            if ((c & 3) == 0) scales[c >> 2] = scale;
        }
    }
    uint16_t* rope = reinterpret_cast<uint16_t*>(dst + nf);
    for (int j = lane; j < kRopeDims; j += 32) rope[j] = f32_to_bf16_rn(src[nf + j]);
    // zero padding after the scales
    int64_t used = nf + 2 * kRopeDims + 4 * (nf / 64);
    int64_t total = fp8m_row_bytes(D);
    for (int64_t b = used + lane; b < total; b += 32) dst[b] = 0;
}

}  // namespace csa
