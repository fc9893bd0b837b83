/*
 * oracle.c -- plain, slow CPU reference for the DeepSeek-V4 hybrid compressed
 * attention hot path (CSA + HCA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * with the CUDA library; both sides are written independently from the pages.
 *
 * Pages cited (title, site):
 *   [peacm]   "DeepSeek-V4百万上下文时代的开源宣言" (peacm.com)
 *   [gitcode] "DeepSeek-V4 技术报告深度解析" (gitcode.csdn.net)
 *   [wiki]    "DeepSeek V4 (Flash & Pro)：通往百万级上下文与万亿参数推理的新纪元"
 *
 * Arithmetic is double precision throughout, with the single exception of the
 * FP8 encoder, which decides an integer code and therefore takes that decision
 * in float32, the precision the kernels use (see oracle_pack_fp8_row).
 *
 * Storage formats accepted by the row readers (the oracle's own numbering):
 *   ORC_F64 = 0  plain double
 *   ORC_F32 = 1  IEEE float32
 *   ORC_BF16 = 2 bfloat16 bit patterns (uint16)
 *   ORC_FP8M = 3 mixed-precision cache row: for a row of D dims,
 *                (D-64) E4M3 bytes for dims 0..D-65, then 64 bfloat16 for the
 *                RoPE dims D-64..D-1, then (D-64)/64 float32 scales (one per
 *                64-dim group), zero padding to a multiple of 16 bytes.
 *
 * Parity pins for every function live in tests/test_oracle_*.py.
 */
#include <limits.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F64 0
#define ORC_F32 1
#define ORC_BF16 2
#define ORC_FP8M 3

#define ORC_OK 0
#define ORC_BAD_INDEX 1
#define ORC_BAD_WINDOW 2
#define ORC_BAD_ARG 3

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 -> double: a bfloat16 is the upper half of a float32. Exact. */
static double bf16_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* float32 -> bfloat16, round to nearest, ties to even (finite inputs). */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;
    return (uint16_t)upper;
}

/* OCP 8-bit floating point, E4M3 variant (bias 7, no infinities, the single
 * NaN pattern S.1111.111): value of a code, from the format's definition. */
double oracle_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, mt = c & 7;
    double v;
    if (e == 15 && mt == 7) return NAN;
    if (e == 0)
        v = ldexp((double)mt / 8.0, -6); /* subnormal: 0.mmm x 2^(1-7) */
    else
        v = ldexp(1.0 + (double)mt / 8.0, e - 7);
    return s ? -v : v;
}

/* E4M3 encoding of a float32, round to nearest with ties to even mantissa,
 * saturating to the largest finite magnitude (448).  The 127 finite
 * non-negative codes 0..126 decode to strictly increasing magnitudes, so the
 * nearest representable magnitude is found by bisection over the codes; on an
 * exact tie the code whose mantissa LSB is 0 wins. */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    double a = fabs((double)x);
    int lo = 0, hi = 126; /* invariant: value(lo) <= a or lo == 0; a <= value(hi) or hi == 126 */
    if (a >= oracle_e4m3_decode(126)) {
        lo = hi = 126; /* at or above 448: saturate */
    } else {
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (oracle_e4m3_decode((uint8_t)mid) <= a)
                lo = mid;
            else
                hi = mid;
        }
    }
    int best = lo;
    if (hi != lo) {
        double dl = a - oracle_e4m3_decode((uint8_t)lo);
        double dh = oracle_e4m3_decode((uint8_t)hi) - a;
        if (dh < dl || (dh == dl && (hi & 1) == 0)) best = hi;
    }
    uint8_t code = (uint8_t)best;
    if (signbit(x)) code |= 0x80; /* negative values, including -0, keep the sign bit */
    return code;
}

/* Bytes of one mixed-precision row of D dims (see the header comment). */
int64_t oracle_fp8m_row_bytes(int D) {
    int64_t raw = (int64_t)(D - 64) + 64 * 2 + 4 * (int64_t)((D - 64) / 64);
    return (raw + 15) / 16 * 16;
}

/* Quantise one float32 row into the mixed-precision cache format
 * [gitcode §2.1.4 "KV 缓存精度": RoPE dims in BF16, the other dims in FP8].
 * Per 64-dim group: scale = amax/448 in float32 (scale 1 for an all-zero
 * group); code = E4M3(x / scale) with the division in float32.  The RoPE dims
 * are rounded to bfloat16. */
void oracle_pack_fp8_row(const float* x, int D, uint8_t* row) {
    int ng = (D - 64) / 64;
    int64_t nb = oracle_fp8m_row_bytes(D);
    memset(row, 0, (size_t)nb);
    float* scales = (float*)malloc(sizeof(float) * (size_t)ng);
    for (int g = 0; g < ng; g++) {
        float amax = 0.0f;
        for (int d = 64 * g; d < 64 * g + 64; d++) {
            float a = fabsf(x[d]);
            if (a > amax) amax = a;
        }
        float scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;
        scales[g] = scale;
        for (int d = 64 * g; d < 64 * g + 64; d++) {
            volatile float q = x[d] / scale; /* float32 division, as stored */
            row[d] = oracle_e4m3_encode(q);
        }
    }
    uint16_t* rope = (uint16_t*)(row + (D - 64));
    for (int j = 0; j < 64; j++) rope[j] = oracle_f32_to_bf16(x[D - 64 + j]);
    memcpy(row + (D - 64) + 128, scales, sizeof(float) * (size_t)ng);
    free(scales);
}

int64_t oracle_row_bytes(int fmt, int D) {
    switch (fmt) {
        case ORC_F64: return 8 * (int64_t)D;
        case ORC_F32: return 4 * (int64_t)D;
        case ORC_BF16: return 2 * (int64_t)D;
        case ORC_FP8M: return oracle_fp8m_row_bytes(D);
    }
    return -1;
}

/* Read row r of a stored [rows, D] array into doubles ("read the inputs as
 * stored"; FP8 rows decode as E4M3 code value times the group scale). */
void oracle_read_row(const void* base, int fmt, int D, int64_t r, double* out) {
    const uint8_t* p = (const uint8_t*)base + r * oracle_row_bytes(fmt, D);
    if (fmt == ORC_F64) {
        memcpy(out, p, sizeof(double) * (size_t)D);
    } else if (fmt == ORC_F32) {
        const float* f = (const float*)p;
        for (int d = 0; d < D; d++) out[d] = (double)f[d];
    } else if (fmt == ORC_BF16) {
        const uint16_t* h = (const uint16_t*)p;
        for (int d = 0; d < D; d++) out[d] = bf16_to_double(h[d]);
    } else {
        const uint16_t* rope = (const uint16_t*)(p + (D - 64));
        const float* scales = (const float*)(p + (D - 64) + 128);
        for (int d = 0; d < D - 64; d++)
            out[d] = oracle_e4m3_decode(p[d]) * (double)scales[d / 64];
        for (int j = 0; j < 64; j++) out[D - 64 + j] = bf16_to_double(rope[j]);
    }
}

/* ------------------------------------------------------------------------ */
/* Q/KV RMSNorm and partial RoPE                                             */
/* ------------------------------------------------------------------------ */

/* RMSNorm with unit gain over all D dims [peacm §三.2 四项关键 Trick
 * "Q/KV Normalization"; gitcode §2.1.4 "查询归一化"]:
 *   out = x / sqrt(mean(x^2) + eps). */
void oracle_rmsnorm(const double* x, int D, double eps, double* out) {
    double ss = 0.0;
    for (int d = 0; d < D; d++) ss += x[d] * x[d];
    double r = 1.0 / sqrt(ss / (double)D + eps);
    for (int d = 0; d < D; d++) out[d] = x[d] * r;
}

/* Partial RoPE on the last R dims, in place [peacm §三.2 四项关键 Trick
 * "Partial RoPE仅对最后 64 维"; gitcode §2.1.4 "部分旋转位置编码"].
 * Pair j = (D-R+2j, D-R+2j+1) rotates by angle pos * base^(-2j/R). */
void oracle_rope(double* x, int D, int R, double base, double pos) {
    for (int j = 0; j < R / 2; j++) {
        double theta = pow(base, -2.0 * (double)j / (double)R);
        double ang = pos * theta;
        double c = cos(ang), s = sin(ang);
        int d0 = D - R + 2 * j;
        double x0 = x[d0], x1 = x[d0 + 1];
        x[d0] = x0 * c - x1 * s;
        x[d0 + 1] = x0 * s + x1 * c;
    }
}

/* ------------------------------------------------------------------------ */
/* a1: block compression                                                     */
/* ------------------------------------------------------------------------ */

/* Compress every m consecutive tokens into one KV entry [peacm §三.2 CSA
 * "Step 1: KV 压缩 每 m 个 token -> 1 个压缩 KV entry (attention-like 机制)";
 * HCA "压缩率 m' 128"; the CSA/HCA table "可学习权重"]:
 *   z_t   = kv_t . w_z + bias[t mod m]          (t = absolute position)
 *   alpha = softmax over the block of z
 *   c_b   = sum_t alpha_t kv_t
 *   e_b   = RoPE(RMSNorm(c_b), b*m + m - 1)      (position of the block's last token)
 * kv: [T, D] stored in kv_fmt, tokens at positions pos0 .. pos0+T-1; pos0 is a
 * multiple of m; a trailing partial block is not emitted.  out: [T/m, D]. */
int oracle_compress(const void* kv, int kv_fmt, int64_t T, int D, int64_t pos0, int m,
                    const double* w_z, const double* bias, int R, double base, double eps,
                    double* out) {
    if (m < 1 || pos0 % m != 0) return ORC_BAD_ARG;
    int64_t nb = T / m;
    double* rows = (double*)malloc(sizeof(double) * (size_t)m * (size_t)D);
    double* z = (double*)malloc(sizeof(double) * (size_t)m);
    double* c = (double*)malloc(sizeof(double) * (size_t)D);
    for (int64_t b = 0; b < nb; b++) {
        for (int t = 0; t < m; t++) oracle_read_row(kv, kv_fmt, D, b * m + t, rows + (size_t)t * D);
        double zmax = -INFINITY;
        for (int t = 0; t < m; t++) {
            double acc = 0.0;
            for (int d = 0; d < D; d++) acc += rows[(size_t)t * D + d] * w_z[d];
            int64_t pos = pos0 + b * m + t;
            z[t] = acc + bias[pos % m];
            if (z[t] > zmax) zmax = z[t];
        }
        double den = 0.0;
        for (int t = 0; t < m; t++) den += exp(z[t] - zmax);
        for (int d = 0; d < D; d++) c[d] = 0.0;
        for (int t = 0; t < m; t++) {
            double a = exp(z[t] - zmax) / den;
            for (int d = 0; d < D; d++) c[d] += a * rows[(size_t)t * D + d];
        }
        double* e = out + (size_t)b * D;
        oracle_rmsnorm(c, D, eps, e);
        oracle_rope(e, D, R, base, (double)(pos0 + b * m + m - 1));
    }
    free(rows);
    free(z);
    free(c);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* a2/a3: lightning indexer and top-k                                        */
/* ------------------------------------------------------------------------ */

/* Number of causally complete blocks seen by the query at position i: block b
 * is complete when its last token b*m+m-1 <= i. */
int64_t oracle_n_complete(int64_t i, int m) { return (i + 1) / m; }

/* Indexer score of every complete block for one query [peacm §三.2 CSA
 * "Step 2: Lightning Indexer Top-K 选择 轻量 indexer 对每个 query 打分";
 * gitcode §2.1.1 "Lightning Indexer"]:
 *   score_b = sum_h w_h * relu(q_h . k_b),  b < n
 * q: [HI, dI] (stored in q_fmt), w: [HI], keys: [n, dI] (stored in k_fmt). */
void oracle_index_scores(const void* q, int q_fmt, const double* w, int HI, int dI,
                         const void* keys, int k_fmt, int64_t n, double* scores) {
    double* qq = (double*)malloc(sizeof(double) * (size_t)HI * (size_t)dI);
    double* kk = (double*)malloc(sizeof(double) * (size_t)dI);
    for (int h = 0; h < HI; h++) oracle_read_row(q, q_fmt, dI, h, qq + (size_t)h * dI);
    for (int64_t b = 0; b < n; b++) {
        oracle_read_row(keys, k_fmt, dI, b, kk);
        double s = 0.0;
        for (int h = 0; h < HI; h++) {
            double dot = 0.0;
            for (int d = 0; d < dI; d++) dot += qq[(size_t)h * dI + d] * kk[d];
            double relu = dot > 0.0 ? dot : 0.0;
            s += w[h] * relu;
        }
        scores[b] = s;
    }
    free(qq);
    free(kk);
}

/* Indexer keys in 8-bit floating point (the pages' lightning indexer runs
 * in low precision [gitcode §2.1.1 "Lightning Indexer"]; this build's FP8
 * variant): one float32 scale per key row, scale = amax/448 (1 for an
 * all-zero row), code = E4M3(x / scale) with the division in float32 -- the
 * same rule as a 64-dim group of the mixed cache row, over the whole row.
 * x: [n, dI] float32 -> codes [n, dI], scales [n]. */
static float orc_fp8_row_quant(const float* x, int dI, uint8_t* codes) {
    float amax = 0.0f;
    for (int d = 0; d < dI; d++) {
        float a = fabsf(x[d]);
        if (a > amax) amax = a;
    }
    float scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    for (int d = 0; d < dI; d++) {
        volatile float q = x[d] / scale; /* float32 division, as stored */
        codes[d] = oracle_e4m3_encode(q);
    }
    return scale;
}

void oracle_pack_idx_keys_fp8(const float* x, int64_t n, int dI, uint8_t* codes, float* scales) {
    for (int64_t b = 0; b < n; b++) scales[b] = orc_fp8_row_quant(x + b * dI, dI, codes + b * dI);
}

/* Indexer score with FP8 keys; each query head row is quantised by the same
 * rule (its float32 values, one scale per head):
 *   score_b = sum_h w_h * relu(sum_d (q8_hd * sq_h) * (k8_bd * sk_b)),  b < n
 * every dequantised value and the sums in double.
 * q: [HI, dI] stored in q_fmt; w: [HI]; key_codes [n, dI]; key_scales [n]. */
void oracle_index_scores_fp8(const void* q, int q_fmt, const double* w, int HI, int dI,
                             const uint8_t* key_codes, const float* key_scales, int64_t n,
                             double* scores) {
    double* qq = (double*)malloc(sizeof(double) * (size_t)HI * (size_t)dI);
    double* kk = (double*)malloc(sizeof(double) * (size_t)dI);
    double* row = (double*)malloc(sizeof(double) * (size_t)dI);
    float* rowf = (float*)malloc(sizeof(float) * (size_t)dI);
    uint8_t* qc = (uint8_t*)malloc((size_t)dI);
    for (int h = 0; h < HI; h++) {
        oracle_read_row(q, q_fmt, dI, h, row);
        for (int d = 0; d < dI; d++) rowf[d] = (float)row[d]; /* exact for bf16 / f32 storage */
        float sq = orc_fp8_row_quant(rowf, dI, qc);
        for (int d = 0; d < dI; d++) qq[(size_t)h * dI + d] = oracle_e4m3_decode(qc[d]) * (double)sq;
    }
    for (int64_t b = 0; b < n; b++) {
        for (int d = 0; d < dI; d++)
            kk[d] = oracle_e4m3_decode(key_codes[b * dI + d]) * (double)key_scales[b];
        double s = 0.0;
        for (int h = 0; h < HI; h++) {
            double dot = 0.0;
            for (int d = 0; d < dI; d++) dot += qq[(size_t)h * dI + d] * kk[d];
            double relu = dot > 0.0 ? dot : 0.0;
            s += w[h] * relu;
        }
        scores[b] = s;
    }
    free(qq);
    free(kk);
    free(row);
    free(rowf);
    free(qc);
}

/* ------------------------------------------------------------------------ */
/* FP4 indexer keys                                                          */
/* ------------------------------------------------------------------------ */

/* [gitcode] §2.1.1 and §3.2: the indexer's QK path is quantised to FP4 in
 * 1 x 32 sub-blocks, which convert to E4M3 without loss when the sub-block
 * scales of a row stay within the range E4M3's two extra exponent bits
 * cover.  This oracle's reading of that format: every 32 consecutive dims of
 * a key share one power-of-two scale 2^e (stored as the byte e + 127), set
 * by the block's largest magnitude a as e = floor(log2 a) - 2 (so a / 2^e
 * lies in [4, 8): the E2M1 grid tops out at 6 = 1.5 * 2^2), e = 0 for an
 * all-zero block; each dim is the E2M1 code of x / 2^e, round to nearest,
 * ties to the even code, saturating at +-6. */

/* E2M1 code (4 bits: sign, two exponent bits with bias 1, one mantissa bit)
 * -> value.  Exponent field 0 holds the subnormals 0 and 0.5. */
double oracle_e2m1_decode(uint8_t code) {
    const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* value -> E2M1 code: the nearest of the fifteen values, ties to the even
 * code, magnitudes beyond 6 saturating (a plain search over the codes). */
uint8_t oracle_e2m1_encode(double x) {
    const int neg = x < 0.0 || (x == 0.0 && signbit(x));
    const double a = fabs(x);
    int best = 0;
    double bd = fabs(a - oracle_e2m1_decode(0));
    for (int c = 1; c < 8; c++) {
        const double d = fabs(a - oracle_e2m1_decode((uint8_t)c));
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bd = d;
        }
    }
    return (uint8_t)(best | (neg && best != 0 ? 8 : 0));
}

/* Keys x [n, dI] (dI a multiple of 32) -> codes [n, dI/2] (dim 2j in the low
 * nibble of byte j, dim 2j+1 in the high nibble) and scale bytes [n, dI/32]
 * (block scale 2^(byte - 127)).
 * Block j of a key: amax = its largest magnitude; exponent e_j =
 * floor(log2 amax) - 2 (the block's largest value lands in [4, 8)), 0 for an
 * all-zero block.  The pages convert FP4 keys to FP8 (E4M3) without loss as
 * long as the ratio of a key's largest to smallest sub-block scale stays
 * within a threshold [gitcode §3.2]; with one E4M3 scale per key, set six
 * binades below the key's largest block scale E (its largest value 6 then
 * lands on 6 * 2^6 = 384 <= 448), a block converts exactly when its smallest
 * step 0.5 * 2^(e_j - E + 6) is still an E4M3 value (>= 2^-9), i.e.
 * e_j >= E - 14.  The format keeps every key within that ratio: a nonzero
 * block's exponent below E - 14 is raised to E - 14 (its values then round
 * on that coarser grid). */
void oracle_pack_idx_keys_fp4(const float* x, int64_t n, int dI, uint8_t* codes, uint8_t* scales) {
    const int nb = dI / 32;
    int* ex = (int*)malloc(sizeof(int) * (size_t)nb);
    int* nz = (int*)malloc(sizeof(int) * (size_t)nb);
    for (int64_t b = 0; b < n; b++) {
        const float* row = x + b * dI;
        int emax = INT_MIN;
        for (int j = 0; j < nb; j++) {
            double amax = 0.0;
            for (int d = 0; d < 32; d++) {
                const double a = fabs((double)row[j * 32 + d]);
                if (a > amax) amax = a;
            }
            int e = 0;
            nz[j] = amax > 0.0;
            if (nz[j]) {
                int ef;
                frexp(amax, &ef); /* amax = f * 2^ef, f in [0.5, 1): floor(log2 amax) = ef - 1 */
                e = ef - 1 - 2;
                if (e > emax) emax = e;
            }
            ex[j] = e;
        }
        for (int j = 0; j < nb; j++) {
            int e = ex[j];
            if (nz[j] && e < emax - 14) e = emax - 14; /* the conversion threshold */
            if (e < -127) e = -127;
            if (e > 127) e = 127;
            scales[b * nb + j] = (uint8_t)(e + 127);
            for (int d = 0; d < 32; d++) {
                const int dim = j * 32 + d;
                const uint8_t c = oracle_e2m1_encode(ldexp((double)row[dim], -e)); /* exact: a power of two */
                uint8_t* byte = codes + b * (dI / 2) + dim / 2;
                if ((dim & 1) == 0)
                    *byte = c;
                else
                    *byte = (uint8_t)(*byte | (c << 4));
            }
        }
    }
    free(ex);
    free(nz);
}

/* Indexer score with FP4 keys (above) and each query head quantised to E4M3
 * with one float32 scale per head, as for FP8 keys:
 *   score_b = sum_h w_h * relu(sum_d (q8_hd * sq_h) * (k4_bd * 2^e_b,d/32)),  b < n
 * every dequantised value and the sums in double. */
void oracle_index_scores_fp4(const void* q, int q_fmt, const double* w, int HI, int dI,
                             const uint8_t* key_codes, const uint8_t* key_scales, int64_t n,
                             double* scores) {
    double* qq = (double*)malloc(sizeof(double) * (size_t)HI * (size_t)dI);
    double* kk = (double*)malloc(sizeof(double) * (size_t)dI);
    double* row = (double*)malloc(sizeof(double) * (size_t)dI);
    float* rowf = (float*)malloc(sizeof(float) * (size_t)dI);
    uint8_t* qc = (uint8_t*)malloc((size_t)dI);
    for (int h = 0; h < HI; h++) {
        oracle_read_row(q, q_fmt, dI, h, row);
        for (int d = 0; d < dI; d++) rowf[d] = (float)row[d];
        float sq = orc_fp8_row_quant(rowf, dI, qc);
        for (int d = 0; d < dI; d++) qq[(size_t)h * dI + d] = oracle_e4m3_decode(qc[d]) * (double)sq;
    }
    const int nb = dI / 32;
    for (int64_t b = 0; b < n; b++) {
        for (int d = 0; d < dI; d++) {
            const uint8_t byte = key_codes[b * (dI / 2) + d / 2];
            const uint8_t c = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
            kk[d] = ldexp(oracle_e2m1_decode(c), (int)key_scales[b * nb + d / 32] - 127);
        }
        double s = 0.0;
        for (int h = 0; h < HI; h++) {
            double dot = 0.0;
            for (int d = 0; d < dI; d++) dot += qq[(size_t)h * dI + d] * kk[d];
            double relu = dot > 0.0 ? dot : 0.0;
            s += w[h] * relu;
        }
        scores[b] = s;
    }
    free(qq);
    free(kk);
    free(row);
    free(rowf);
    free(qc);
}

typedef struct {
    double s;
    int64_t i;
} orc_cand;

/* higher score first; equal scores: lower index first */
static int cand_cmp(const void* a, const void* b) {
    const orc_cand* x = (const orc_cand*)a;
    const orc_cand* y = (const orc_cand*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

/* Keep the top min(k, n) blocks by (score descending, index ascending)
 * [peacm §三.2 CSA Step 2 "选出最相关的 Top-K 压缩块"; ties go to the lower
 * index].  Output in that rank order, padded with -1 to k entries.  Returns
 * the number selected. */
int64_t oracle_topk(const double* scores, int64_t n, int k, int32_t* idx, double* sel_scores) {
    orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(n > 0 ? n : 1));
    for (int64_t b = 0; b < n; b++) {
        c[b].s = scores[b];
        c[b].i = b;
    }
    qsort(c, (size_t)n, sizeof(orc_cand), cand_cmp);
    int64_t nsel = n < k ? n : k;
    for (int j = 0; j < k; j++) {
        idx[j] = (j < nsel) ? (int32_t)c[j].i : -1;
        if (sel_scores) sel_scores[j] = (j < nsel) ? c[j].s : -INFINITY;
    }
    free(c);
    return nsel;
}

/* ------------------------------------------------------------------------ */
/* a4-a7: core attention with window and sink                                */
/* ------------------------------------------------------------------------ */

/* Multi-query attention of one query token (H heads sharing one KV head) over
 * J given rows [peacm §三.2 CSA "Step 3: Core Attention Multi-Query
 * Attention"; 四项关键 Trick: Q/KV Normalization, Partial RoPE with output
 * RoPE at position -i, Attention Sink; gitcode §2.1.4]:
 *   q'_h  = RoPE(RMSNorm(q_h), i)
 *   l_hj  = scale * q'_h . e_j
 *   lse_h = log(exp(s_h) + sum_j exp(l_hj))        (sink logit in the denominator)
 *   o_h   = sum_j exp(l_hj - lse_h) e_j            (one KV entry serves as key and value)
 *   o_h   = RoPE(o_h, -i)  when derotate is set.
 * With no rows and a sink of -inf the weights are empty: o_h = 0, lse_h = -inf.
 * q: [H, D] stored in q_fmt; rows: [J, D] doubles; sink: [H].
 * weights (optional): [H, J] attention weights, for tests. */
void oracle_attend_rows(const void* q, int q_fmt, int H, int D, int64_t i, const double* rows,
                        int64_t J, const double* sink, double scale, int R, double base, double eps,
                        int derotate, double* out, double* lse, double* weights) {
    double* qh = (double*)malloc(sizeof(double) * (size_t)D);
    double* tmp = (double*)malloc(sizeof(double) * (size_t)D);
    double* l = (double*)malloc(sizeof(double) * (size_t)(J > 0 ? J : 1));
    for (int h = 0; h < H; h++) {
        oracle_read_row(q, q_fmt, D, h, tmp);
        oracle_rmsnorm(tmp, D, eps, qh);
        oracle_rope(qh, D, R, base, (double)i);
        double mx = sink[h];
        for (int64_t j = 0; j < J; j++) {
            double dot = 0.0;
            for (int d = 0; d < D; d++) dot += qh[d] * rows[(size_t)j * D + d];
            l[j] = scale * dot;
            if (l[j] > mx) mx = l[j];
        }
        double* o = out + (size_t)h * D;
        for (int d = 0; d < D; d++) o[d] = 0.0;
        if (mx == -INFINITY) { /* no rows and no sink mass */
            lse[h] = -INFINITY;
            if (weights)
                for (int64_t j = 0; j < J; j++) weights[(size_t)h * J + j] = 0.0;
            continue;
        }
        double den = exp(sink[h] - mx);
        for (int64_t j = 0; j < J; j++) den += exp(l[j] - mx);
        lse[h] = mx + log(den);
        for (int64_t j = 0; j < J; j++) {
            double wj = exp(l[j] - lse[h]);
            if (weights) weights[(size_t)h * J + j] = wj;
            for (int d = 0; d < D; d++) o[d] += wj * rows[(size_t)j * D + d];
        }
        if (derotate) oracle_rope(o, D, R, base, -(double)i);
    }
    free(qh);
    free(tmp);
    free(l);
}

/* Gather the rows one query attends to and run oracle_attend_rows.
 *   entries: idx != NULL -> the selected blocks idx[0..k) (entries of -1 are
 *            skipped) [CSA, peacm §三.2 Step 3 "对 Top-K 块做注意力计算"];
 *            idx == NULL -> every complete block 0..n_complete(i)-1 [HCA,
 *            peacm §三.2 "对所有压缩 KV 做 dense attention"].
 *   window:  raw tokens max(0, i-W+1) .. i [peacm 四项关键 Trick "Sliding
 *            Window 辅助分支 每个 query 额外可见最近 128 个 token 的原始 KV"];
 *            window row r holds position win_pos0 + r.
 * cache: [n_cap, D] in kv_fmt; window: [n_win, D] in kv_fmt.
 * Returns ORC_BAD_INDEX if a selected block is not causally complete or is
 * beyond n_cap, ORC_BAD_WINDOW if a window position is not in the buffer. */
int oracle_attend_query(const void* q, int q_fmt, int H, int D, int64_t i, int m,
                        const void* cache, int kv_fmt, int64_t n_cap, const int32_t* idx, int k,
                        const void* window, int64_t win_pos0, int64_t n_win, int W,
                        const double* sink, double scale, int R, double base, double eps,
                        int derotate, double* out, double* lse) {
    int64_t nc = oracle_n_complete(i, m);
    int64_t ne;
    if (idx) {
        ne = 0;
        for (int j = 0; j < k; j++)
            if (idx[j] >= 0) ne++;
    } else {
        ne = nc;
    }
    int64_t w_lo = i - W + 1 > 0 ? i - W + 1 : 0;
    int64_t nw = W > 0 ? i - w_lo + 1 : 0;
    int64_t J = ne + nw;
    double* rows = (double*)malloc(sizeof(double) * (size_t)(J > 0 ? J : 1) * (size_t)D);
    int64_t r = 0;
    int status = ORC_OK;
    if (idx) {
        for (int j = 0; j < k; j++) {
            if (idx[j] < 0) continue;
            if (idx[j] >= nc || idx[j] >= n_cap) {
                status = ORC_BAD_INDEX;
                goto done;
            }
            oracle_read_row(cache, kv_fmt, D, idx[j], rows + (size_t)r * D);
            r++;
        }
    } else {
        if (nc > n_cap) {
            status = ORC_BAD_INDEX;
            goto done;
        }
        for (int64_t b = 0; b < nc; b++, r++) oracle_read_row(cache, kv_fmt, D, b, rows + (size_t)r * D);
    }
    for (int64_t p = w_lo; p < w_lo + nw; p++, r++) {
        int64_t wr = p - win_pos0;
        if (wr < 0 || wr >= n_win) {
            status = ORC_BAD_WINDOW;
            goto done;
        }
        oracle_read_row(window, kv_fmt, D, wr, rows + (size_t)r * D);
    }
    oracle_attend_rows(q, q_fmt, H, D, i, rows, J, sink, scale, R, base, eps, derotate, out, lse, NULL);
done:
    free(rows);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Batched drivers (OpenMP over independent queries; used for the CPU        */
/* baseline timing and for large parity samples)                             */
/* ------------------------------------------------------------------------ */

/* Lightning indexer + top-k for Q queries.  Query qi belongs to sequence
 * seq[qi] and sits at position pos[qi]; keys of sequence b start at row
 * b*n_cap.  Only complete blocks (b < n_complete(pos)) are scored.
 * idx_out: [Q, k]; score_out (optional): [Q, k]. */
int oracle_index_topk_batch(int Q, const void* q, int q_fmt, const double* w, int HI, int dI,
                            const void* keys, int k_fmt, int64_t n_cap, const int32_t* seq,
                            const int64_t* pos, int m, int k, int32_t* idx_out, double* score_out) {
    int bad = 0;
    int64_t qstride = oracle_row_bytes(q_fmt, dI) * HI;
    int64_t kstride = oracle_row_bytes(k_fmt, dI) * n_cap;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int qi = 0; qi < Q; qi++) {
        int64_t n = oracle_n_complete(pos[qi], m);
        if (n > n_cap) {
            bad |= 1;
            continue;
        }
        double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        oracle_index_scores((const uint8_t*)q + qi * qstride, q_fmt, w + (size_t)qi * HI, HI, dI,
                            (const uint8_t*)keys + (int64_t)seq[qi] * kstride, k_fmt, n, s);
        oracle_topk(s, n, k, idx_out + (size_t)qi * k, score_out ? score_out + (size_t)qi * k : NULL);
        free(s);
    }
    return bad ? ORC_BAD_INDEX : ORC_OK;
}

/* Core attention for Q queries (CSA when idx != NULL, HCA otherwise).
 * cache rows of sequence b start at b*n_cap; window rows at b*n_win with the
 * first window row of sequence b at position win_pos0[b]. */
int oracle_attend_batch(int Q, const void* q, int q_fmt, int H, int D, const int32_t* seq,
                        const int64_t* pos, int m, const void* cache, int kv_fmt, int64_t n_cap,
                        const int32_t* idx, int k, const void* window, const int64_t* win_pos0,
                        int64_t n_win, int W, const double* sink, double scale, int R, double base,
                        double eps, int derotate, double* out, double* lse) {
    int status = ORC_OK;
    int64_t qstride = oracle_row_bytes(q_fmt, D) * H;
    int64_t rb = oracle_row_bytes(kv_fmt, D);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int qi = 0; qi < Q; qi++) {
        int b = seq[qi];
        status |= oracle_attend_query((const uint8_t*)q + qi * qstride, q_fmt, H, D, pos[qi], m,
                                      (const uint8_t*)cache + (int64_t)b * n_cap * rb, kv_fmt, n_cap,
                                      idx ? idx + (size_t)qi * k : NULL, k,
                                      (const uint8_t*)window + (int64_t)b * n_win * rb, win_pos0[b],
                                      n_win, W, sink, scale, R, base, eps, derotate,
                                      out + (size_t)qi * H * D, lse + (size_t)qi * H);
    }
    return status;
}

/* Quantise n float32 rows into the mixed-precision format (OpenMP over rows). */
void oracle_pack_fp8_rows(const float* x, int64_t n, int D, uint8_t* out) {
    int64_t rb = oracle_fp8m_row_bytes(D);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; r++) oracle_pack_fp8_row(x + r * D, D, out + r * rb);
}

/* Store n double rows in a row format (the cache keeps compressor outputs in
 * its storage format): float32 rounding first, then bfloat16 (RNE) or the
 * mixed FP8 row quantiser. */
void oracle_store_rows(const double* x, int64_t n, int D, int fmt, void* out) {
    int64_t rb = oracle_row_bytes(fmt, D);
    float* f = (float*)malloc(sizeof(float) * (size_t)D);
    for (int64_t r = 0; r < n; r++) {
        uint8_t* dst = (uint8_t*)out + r * rb;
        const double* src = x + r * D;
        if (fmt == ORC_F64) {
            memcpy(dst, src, sizeof(double) * (size_t)D);
            continue;
        }
        for (int d = 0; d < D; d++) f[d] = (float)src[d];
        if (fmt == ORC_F32)
            memcpy(dst, f, sizeof(float) * (size_t)D);
        else if (fmt == ORC_BF16)
            for (int d = 0; d < D; d++) ((uint16_t*)dst)[d] = oracle_f32_to_bf16(f[d]);
        else
            oracle_pack_fp8_row(f, D, dst);
    }
    free(f);
}
