// csa_capi.cu -- the extern "C" boundary of libcsa: argument validation,
// workspace planning and dispatch to the kernels.  No allocation, no
// synchronisation (except csa_check_status), launches on the caller's stream.
#include <math.h>

#include <atomic>
#include <mutex>
#include <unordered_map>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace csa {

static thread_local char g_err[512] = "";
static std::atomic<unsigned long long> g_launches{0};

void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
static thread_local uint32_t g_dev_bits = 0;

static csa_status fail(csa_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

csa_status set_error(csa_status s, const char* msg) { return fail(s, "%s", msg); }

static csa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(CSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Per-device host caches: the SM count and the largest dynamic shared memory
// set on each kernel.  A process may drive several devices (each call works
// on the current one), so nothing is cached process-wide.
constexpr int kMaxDev = 64;
static std::atomic<int> g_sms[kMaxDev];
static std::mutex g_attr_mu;
static std::unordered_map<const void*, size_t> g_attr[kMaxDev];

static int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    return dev;
}

int num_sms() {
    const int dev = current_device();
    int n = (dev >= 0 && dev < kMaxDev) ? g_sms[dev].load(std::memory_order_relaxed) : 0;
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        if (dev >= 0 && dev < kMaxDev) g_sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

cudaError_t set_smem_attr(const void* kernel, size_t bytes) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDev)
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    std::lock_guard<std::mutex> lock(g_attr_mu);
    size_t& have = g_attr[dev][kernel];
    if (bytes <= have) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

Geometry resolve(const csa_params* p) {
    Geometry g;
    g.D = p->head_dim;
    g.R = p->rope_dims;
    g.m = p->ratio;
    g.k = p->topk;
    g.W = p->window;
    g.base = p->rope_base;
    g.eps = p->norm_eps;
    g.scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.f / sqrtf((float)p->head_dim);
    g.derotate = p->derotate_output != 0;
    g.act = p->act_format;
    g.kv = p->kv_format;
    g.kv_row_bytes = row_bytes(p->kv_format, p->head_dim);
    g.inv = p->batch_invariant != 0;
    return g;
}

RopeTheta rope_theta(const Geometry& g) {
    RopeTheta t;
    for (int j = 0; j < 32; j++)
        t.t[j] = pow((double)g.base, -2.0 * (double)j / (double)g.R);
    return t;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

IndexTopkPlan plan_index_topk(const Geometry& g, int B, int Q, int HI, int64_t n_cap, bool fp8) {
    (void)g;
    (void)B;
    (void)HI;
    IndexTopkPlan pl;
    pl.n_cap_pad = (n_cap + 127) / 128 * 128;
    pl.scores_off = kStatusWordBytes;
    pl.scores_bytes = align256((size_t)Q * (size_t)pl.n_cap_pad * sizeof(float));
    pl.q8_off = pl.weff_off = pl.scores_off + pl.scores_bytes;
    pl.total = pl.scores_off + pl.scores_bytes;
    if (fp8) {
        pl.weff_off = pl.q8_off + align256((size_t)Q * 64 * 128);
        pl.total = pl.weff_off + align256((size_t)Q * 64 * sizeof(float));
    }
    return pl;
}

bool attend_tc_supported(const Geometry& g, bool sparse, int H, int64_t n_cap, int64_t n_win);
bool plan_attend_tc(const Geometry& g, bool sparse, int Q, int64_t n_cap, int64_t n_win, bool ring, AttendPlan* pl);
void plan_attend_tc_aligned(int Q, AttendPlan* pl);

AttendPlan plan_attend(const Geometry& g, bool sparse, int B, int Q, int H, int64_t n_cap,
                       int64_t n_win, bool ring) {
    (void)B;
    AttendPlan pl;
    pl.ring = ring ? 1 : 0;
    pl.list_len = (sparse ? (int64_t)g.k : n_cap) + g.W;
    pl.use_tc = attend_tc_supported(g, sparse, H, n_cap, n_win) ? 1 : 0;
    pl.tc_T_sel = pl.tc_T = pl.tc_grid = pl.tc_deq = pl.tc_seg = pl.tc_nseg = pl.tc_qcta = pl.tc_qrem = pl.tc_qc = 0;
    pl.tc_total = 0;
    if (pl.use_tc) {
        pl.head_group = H;
        pl.rows_per_split = 0;
        // more than 2^31 tiles go to the CUDA-core kernel
        if (!plan_attend_tc(g, sparse, Q, n_cap, n_win, ring, &pl)) {
            pl.use_tc = 0;
            pl.tc_T_sel = pl.tc_T = pl.tc_grid = pl.tc_seg = pl.tc_nseg = pl.tc_qcta = pl.tc_qrem = pl.tc_qc = 0;
            pl.tc_total = 0;
        }
    }
    if (!pl.use_tc) {
        pl.head_group = (H % 16 == 0) ? 16 : 8;
        const int hgs = H / pl.head_group;
        if (g.inv) {  // fixed splits: a function of the list length only
            pl.rows_per_split = 64LL * inv_split_tiles((pl.list_len + 63) / 64);
        } else {
            const int64_t target = 4LL * num_sms();
            int64_t s = (target + (int64_t)Q * hgs - 1) / ((int64_t)Q * hgs);
            int64_t max_s = (pl.list_len + 31) / 32;
            if (s > max_s) s = max_s;
            if (s < 1) s = 1;
            int64_t per = (pl.list_len + s - 1) / s;
            pl.rows_per_split = (per + 31) / 32 * 32;
        }
        pl.splits = (int)((pl.list_len + pl.rows_per_split - 1) / pl.rows_per_split);
        if (pl.splits < 1) pl.splits = 1;
    }
    size_t deq_rows = 0;
    if (pl.use_tc && g.kv == CSA_FP8_MIXED) {
        // dequantise whichever is fewer rows: the ones the queries read or all
        const size_t per_query = (size_t)Q * pl.tc_T * 64;
        const size_t stored = (size_t)B * (size_t)(n_cap + (g.W > 0 ? n_win : 0));
        pl.tc_deq = per_query <= stored ? 1 : 2;
        deq_rows = pl.tc_deq == 1 ? per_query : stored;
    }
    if (pl.use_tc && sparse && pl.tc_deq != 1) plan_attend_tc_aligned(Q, &pl);  // the rows are gathered
    pl.part_o_off = kStatusWordBytes;
    size_t o_bytes = align256((size_t)Q * pl.splits * H * g.D * sizeof(float));
    pl.part_ml_off = pl.part_o_off + o_bytes;
    size_t ml_bytes = align256((size_t)Q * pl.splits * H * 2 * sizeof(float));
    pl.nslots_off = 0;
    size_t ns_bytes = 0;
    if (pl.use_tc && pl.tc_seg == 0) {
        pl.nslots_off = pl.part_ml_off + ml_bytes;
        ns_bytes = align256((size_t)Q * sizeof(int32_t));
    }
    pl.deq_off = pl.part_ml_off + ml_bytes + ns_bytes;
    const size_t deq_bytes = align256(deq_rows * g.D * 2);
    pl.total = pl.deq_off + deq_bytes;
    return pl;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Checks shared by every entry point.
static csa_status check_params(const csa_params* p) {
    if (!p) return fail(CSA_ERR_INVALID_ARG, "params is NULL");
    if (p->head_dim < 64 || p->head_dim > 512 || p->head_dim % 64 != 0)
        return fail(CSA_ERR_UNSUPPORTED, "head_dim %d: must be a multiple of 64 in [64, 512]",
                    p->head_dim);
    if (p->head_dim != 128 && p->head_dim != 256 && p->head_dim != 512)
        return fail(CSA_ERR_UNSUPPORTED, "head_dim %d: this build runs 128, 256 or 512", p->head_dim);
    if (p->rope_dims != 64) return fail(CSA_ERR_UNSUPPORTED, "rope_dims %d: must be 64", p->rope_dims);
    if (!(p->rope_base > 1.f) || !isfinite(p->rope_base))
        return fail(CSA_ERR_INVALID_ARG, "rope_base must be finite and > 1");
    if (!(p->norm_eps >= 0.f) || !isfinite(p->norm_eps))
        return fail(CSA_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
    if (!isfinite(p->softmax_scale)) return fail(CSA_ERR_INVALID_ARG, "softmax_scale not finite");
    if (p->ratio < 1 || p->ratio > 1024) return fail(CSA_ERR_INVALID_ARG, "ratio %d not in [1, 1024]", p->ratio);
    if (p->window < 0 || p->window > 1024) return fail(CSA_ERR_INVALID_ARG, "window %d not in [0, 1024]", p->window);
    if (p->act_format != CSA_F32 && p->act_format != CSA_BF16)
        return fail(CSA_ERR_INVALID_ARG, "act_format %d", p->act_format);
    if (p->kv_format != CSA_F32 && p->kv_format != CSA_BF16 && p->kv_format != CSA_FP8_MIXED)
        return fail(CSA_ERR_INVALID_ARG, "kv_format %d", p->kv_format);
    if ((p->act_format == CSA_F32) != (p->kv_format == CSA_F32))
        return fail(CSA_ERR_UNSUPPORTED, "F32 activations pair with F32 rows only");
    return CSA_OK;
}

static csa_status check_ptr(const void* p, const char* name, bool nullable = false) {
    if (!p) return nullable ? CSA_OK : fail(CSA_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p)) return fail(CSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return CSA_OK;
}

#define CHECK(x)                       \
    do {                               \
        csa_status _s = (x);           \
        if (_s != CSA_OK) return _s;   \
    } while (0)

}  // namespace csa

using namespace csa;

extern "C" {

int64_t csa_row_bytes(int32_t kv_format, int32_t head_dim) {
    if (head_dim < 64 || head_dim % 64 != 0) return -1;
    return row_bytes(kv_format, head_dim);
}

const char* csa_status_string(csa_status s) {
    switch (s) {
        case CSA_OK: return "CSA_OK";
        case CSA_ERR_INVALID_ARG: return "CSA_ERR_INVALID_ARG";
        case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED";
        case CSA_ERR_CUDA: return "CSA_ERR_CUDA";
        case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE";
        case CSA_ERR_DEVICE: return "CSA_ERR_DEVICE";
    }
    return "unknown csa_status";
}

const char* csa_last_error(void) { return g_err; }
uint32_t csa_last_device_bits(void) { return g_dev_bits; }

csa_status csa_cache_pack(const csa_params* p, const float* src, int64_t n_rows, void* dst,
                          csa_stream_t stream) {
    CHECK(check_params(p));
    if (n_rows < 0) return fail(CSA_ERR_INVALID_ARG, "n_rows < 0");
    if (n_rows == 0) return CSA_OK;
    CHECK(check_ptr(src, "src"));
    CHECK(check_ptr(dst, "dst"));
    Geometry g = resolve(p);
    cudaError_t e = launch_cache_pack(g, src, n_rows, dst, (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_cache_pack");
}

csa_status csa_compress(const csa_params* p, const void* kv_raw, int32_t B, int64_t T,
                        int64_t kv_seq_stride, int64_t pos0, const float* w_z, const float* bias,
                        void* out, int64_t out_seq_stride, csa_stream_t stream) {
    CHECK(check_params(p));
    if (B < 0 || B > 65535 || T < 0) return fail(CSA_ERR_INVALID_ARG, "B %d / T %lld out of range", B, (long long)T);
    if (pos0 < 0 || pos0 % p->ratio != 0)
        return fail(CSA_ERR_INVALID_ARG, "pos0 %lld is not a non-negative multiple of ratio %d",
                    (long long)pos0, p->ratio);
    const int64_t nb = T / p->ratio;
    if (B == 0 || nb == 0) return CSA_OK;
    if (B > 1 && kv_seq_stride < T) return fail(CSA_ERR_INVALID_ARG, "kv_seq_stride < T");
    if (B > 1 && out_seq_stride < nb) return fail(CSA_ERR_INVALID_ARG, "out_seq_stride < T/ratio");
    if (nb > 0x7fffffffLL) return fail(CSA_ERR_INVALID_ARG, "too many blocks");
    CHECK(check_ptr(kv_raw, "kv_raw"));
    CHECK(check_ptr(w_z, "w_z"));
    if (!bias) return fail(CSA_ERR_INVALID_ARG, "bias is NULL");
    CHECK(check_ptr(out, "out"));
    Geometry g = resolve(p);
    cudaError_t e = launch_compress(g, kv_raw, B, T, kv_seq_stride, pos0, w_z, bias, out,
                                    out_seq_stride, nullptr, 0, (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_compress");
}

csa_status csa_append(const csa_params* p, const void* kv_new, int32_t B, int64_t kv_seq_stride,
                      int64_t pos0, const float* w_z, const float* bias, void* entry_out,
                      int64_t out_seq_stride, void* win_out, int64_t win_seq_stride,
                      csa_stream_t stream) {
    CHECK(check_params(p));
    if (B < 0 || B > 65535) return fail(CSA_ERR_INVALID_ARG, "B %d out of range", B);
    if (pos0 < 0 || pos0 % p->ratio != 0)
        return fail(CSA_ERR_INVALID_ARG, "pos0 %lld is not a non-negative multiple of ratio %d",
                    (long long)pos0, p->ratio);
    if (B == 0) return CSA_OK;
    if (B > 1 && kv_seq_stride < p->ratio) return fail(CSA_ERR_INVALID_ARG, "kv_seq_stride < ratio");
    if (B > 1 && (out_seq_stride < 1 || win_seq_stride < 1))
        return fail(CSA_ERR_INVALID_ARG, "out_seq_stride / win_seq_stride < 1");
    CHECK(check_ptr(kv_new, "kv_new"));
    CHECK(check_ptr(w_z, "w_z"));
    if (!bias) return fail(CSA_ERR_INVALID_ARG, "bias is NULL");
    CHECK(check_ptr(entry_out, "entry_out"));
    CHECK(check_ptr(win_out, "win_out"));
    Geometry g = resolve(p);
    cudaError_t e = launch_compress(g, kv_new, B, p->ratio, kv_seq_stride, pos0, w_z, bias, entry_out,
                                    out_seq_stride, win_out, win_seq_stride, (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_append");
}

csa_status csa_decode_append(const csa_params* p, const void* kv_tok, int32_t B, const int64_t* pos,
                             void* raw_ring, const float* w_z, const float* bias, void* cache, int64_t n_cap,
                             void* window, int64_t n_win, void* ws, size_t ws_bytes, csa_stream_t stream) {
    CHECK(check_params(p));
    if (B < 0 || B > 65535) return fail(CSA_ERR_INVALID_ARG, "B %d out of range", B);
    if (n_cap < 0 || n_cap > (1LL << 30) || n_win < 0 || n_win > (1LL << 30))
        return fail(CSA_ERR_INVALID_ARG, "n_cap / n_win out of range");
    if (B == 0) return CSA_OK;
    Geometry g = resolve(p);
    if (!decode_append_supported(g))
        return fail(CSA_ERR_UNSUPPORTED, "csa_decode_append: a block of %d tokens of %d dims does not fit the compressor",
                    p->ratio, p->head_dim);
    CHECK(check_ptr(kv_tok, "kv_tok"));
    CHECK(check_ptr(pos, "pos"));
    CHECK(check_ptr(raw_ring, "raw_ring", p->ratio == 1));
    CHECK(check_ptr(w_z, "w_z"));
    if (!bias) return fail(CSA_ERR_INVALID_ARG, "bias is NULL");
    CHECK(check_ptr(cache, "cache", n_cap == 0));
    const bool win = p->window > 0 && n_win > 0;
    CHECK(check_ptr(window, "window", !win));
    CHECK(check_ptr(ws, "ws"));
    if (ws_bytes < kStatusWordBytes) return fail(CSA_ERR_WORKSPACE, "workspace smaller than 256 bytes");
    cudaError_t e = launch_decode_append(g, kv_tok, B, pos, raw_ring, w_z, bias, cache, n_cap,
                                         win ? window : nullptr, n_win, reinterpret_cast<uint32_t*>(ws),
                                         (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_decode_append");
}

size_t csa_workspace_bytes(const csa_params* p, int32_t op, int32_t B, int32_t Q, int32_t H,
                           int32_t n_idx_heads, int64_t n_cap, int64_t n_win) {
    if (check_params(p) != CSA_OK || B <= 0 || Q < 0 || n_cap < 0 || n_win < 0) return 0;
    Geometry g = resolve(p);
    if (op == CSA_OP_INDEX_TOPK) return plan_index_topk(g, B, Q, n_idx_heads, n_cap).total;
    if (op == CSA_OP_INDEX_TOPK_FP8 || op == CSA_OP_INDEX_TOPK_FP4)
        return plan_index_topk(g, B, Q, n_idx_heads, n_cap, true).total;
    // one size serves both window layouts (linear or ring)
    if (op == CSA_OP_ATTEND || op == CSA_OP_HCA_ATTEND) {
        if (H <= 0) return 0;
        const bool sparse = op == CSA_OP_ATTEND;
        const size_t a = plan_attend(g, sparse, B, Q, H, n_cap, n_win, false).total;
        const size_t b = plan_attend(g, sparse, B, Q, H, n_cap, n_win, true).total;
        return a > b ? a : b;
    }
    return 0;
}

csa_status csa_workspace_init(void* ws, size_t ws_bytes, csa_stream_t stream) {
    CHECK(check_ptr(ws, "ws"));
    if (ws_bytes < kStatusWordBytes) return fail(CSA_ERR_WORKSPACE, "workspace smaller than 256 bytes");
    cudaError_t e = cudaMemsetAsync(ws, 0, kStatusWordBytes, (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_workspace_init");
}

csa_status csa_check_status(void* ws, csa_stream_t stream) {
    CHECK(check_ptr(ws, "ws"));
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "csa_check_status: stream");
    uint32_t bits = 0;
    e = cudaMemcpy(&bits, ws, sizeof(bits), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "csa_check_status: read");
    g_dev_bits = bits;
    if (bits == 0) return CSA_OK;
    e = cudaMemset(ws, 0, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "csa_check_status: clear");
    return fail(CSA_ERR_DEVICE, "device status 0x%x:%s%s%s%s", bits,
                (bits & CSA_DEV_BAD_TOPK_INDEX) ? " top-k index not a complete block;" : "",
                (bits & CSA_DEV_BAD_WINDOW) ? " window position missing from the buffer;" : "",
                (bits & CSA_DEV_BAD_POSITION) ? " query position beyond cache capacity;" : "",
                (bits & CSA_DEV_TIMEOUT) ? " bounded wait expired;" : "");
}

csa_status csa_index_topk(const csa_params* p, const void* q_idx, const float* w_idx,
                          int32_t n_idx_heads, int32_t idx_dim, const void* keys, int64_t n_cap,
                          int32_t B, int32_t Q, const int64_t* q_pos, int32_t* topk_idx,
                          float* topk_score, void* ws, size_t ws_bytes, csa_stream_t stream) {
    CHECK(check_params(p));
    if (p->topk < 1 || p->topk > 4096) return fail(CSA_ERR_INVALID_ARG, "topk %d not in [1, 4096]", p->topk);
    if (idx_dim != 64 && idx_dim != 128) return fail(CSA_ERR_UNSUPPORTED, "idx_dim %d: 64 or 128", idx_dim);
    if (n_idx_heads < 1 || n_idx_heads > 64) return fail(CSA_ERR_UNSUPPORTED, "n_idx_heads %d: 1..64", n_idx_heads);
    if (B < 1 || Q < 0 || Q % B != 0) return fail(CSA_ERR_INVALID_ARG, "Q %d must be a multiple of B %d", Q, B);
    if (n_cap < 0 || n_cap > (1LL << 30)) return fail(CSA_ERR_INVALID_ARG, "n_cap out of range");
    if (Q == 0) return CSA_OK;
    CHECK(check_ptr(q_idx, "q_idx"));
    CHECK(check_ptr(w_idx, "w_idx"));
    CHECK(check_ptr(keys, "keys", n_cap == 0));
    CHECK(check_ptr(q_pos, "q_pos"));
    CHECK(check_ptr(topk_idx, "topk_idx"));
    CHECK(check_ptr(topk_score, "topk_score", true));
    CHECK(check_ptr(ws, "ws"));
    if (topk_chunk(n_cap, Q, p->topk) == 0)
        return fail(CSA_ERR_UNSUPPORTED, "top-%d of %lld blocks does not fit the selection's shared memory",
                    p->topk, (long long)n_cap);
    Geometry g = resolve(p);
    IndexTopkPlan pl = plan_index_topk(g, B, Q, n_idx_heads, n_cap);
    if (ws_bytes < pl.total) return fail(CSA_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, pl.total);
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    uint32_t* status = reinterpret_cast<uint32_t*>(w);
    float* scores = reinterpret_cast<float*>(w + pl.scores_off);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = launch_indexer(g, q_idx, w_idx, n_idx_heads, idx_dim, keys, n_cap, B, Q,
                                   q_pos, status, scores, pl.n_cap_pad, st);
    if (e != cudaSuccess) return cuda_fail(e, "csa_index_topk: indexer");
    e = launch_topk(g, scores, pl.n_cap_pad, n_cap, Q, q_pos, topk_idx, topk_score, st);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_index_topk: top-k");
}

csa_status csa_index_score(const csa_params* p, const void* q_idx, const float* w_idx,
                           int32_t n_idx_heads, int32_t idx_dim, const void* keys, int64_t n_cap,
                           int32_t B, int32_t Q, const int64_t* q_pos, float* scores,
                           int64_t ld_scores, void* ws, size_t ws_bytes, csa_stream_t stream) {
    CHECK(check_params(p));
    if (idx_dim != 64 && idx_dim != 128) return fail(CSA_ERR_UNSUPPORTED, "idx_dim %d: 64 or 128", idx_dim);
    if (n_idx_heads < 1 || n_idx_heads > 64) return fail(CSA_ERR_UNSUPPORTED, "n_idx_heads %d: 1..64", n_idx_heads);
    if (B < 1 || Q < 0 || Q % B != 0) return fail(CSA_ERR_INVALID_ARG, "Q %d must be a multiple of B %d", Q, B);
    if (n_cap < 0 || n_cap > (1LL << 30)) return fail(CSA_ERR_INVALID_ARG, "n_cap out of range");
    if (ld_scores < n_cap || ld_scores % 4 != 0)
        return fail(CSA_ERR_INVALID_ARG, "ld_scores %lld must be >= n_cap and a multiple of 4", (long long)ld_scores);
    if (Q == 0) return CSA_OK;
    CHECK(check_ptr(q_idx, "q_idx"));
    CHECK(check_ptr(w_idx, "w_idx"));
    CHECK(check_ptr(keys, "keys", n_cap == 0));
    CHECK(check_ptr(q_pos, "q_pos"));
    CHECK(check_ptr(scores, "scores"));
    CHECK(check_ptr(ws, "ws"));
    if (ws_bytes < kStatusWordBytes) return fail(CSA_ERR_WORKSPACE, "workspace smaller than 256 bytes");
    Geometry g = resolve(p);
    cudaError_t e = launch_indexer(g, q_idx, w_idx, n_idx_heads, idx_dim, keys, n_cap, B, Q, q_pos,
                                   reinterpret_cast<uint32_t*>(ws), scores, ld_scores,
                                   (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_index_score");
}

csa_status csa_topk_select(const csa_params* p, float* scores, int64_t ld_scores,
                           int64_t n_cap, int32_t Q, const int64_t* q_pos, int32_t* topk_idx,
                           float* topk_score, csa_stream_t stream) {
    CHECK(check_params(p));
    if (p->topk < 1 || p->topk > 4096) return fail(CSA_ERR_INVALID_ARG, "topk %d not in [1, 4096]", p->topk);
    if (Q < 0 || n_cap < 0 || n_cap > (1LL << 30) || ld_scores < n_cap)
        return fail(CSA_ERR_INVALID_ARG, "bad Q / n_cap / ld_scores");
    if (Q == 0) return CSA_OK;
    if (topk_chunk(n_cap, Q, p->topk) == 0)
        return fail(CSA_ERR_UNSUPPORTED, "top-%d of %lld blocks does not fit the selection's shared memory",
                    p->topk, (long long)n_cap);
    CHECK(check_ptr(scores, "scores"));
    CHECK(check_ptr(q_pos, "q_pos"));
    CHECK(check_ptr(topk_idx, "topk_idx"));
    CHECK(check_ptr(topk_score, "topk_score", true));
    Geometry g = resolve(p);
    cudaError_t e = launch_topk(g, scores, ld_scores, n_cap, Q, q_pos, topk_idx, topk_score,
                                (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_topk_select");
}

csa_status csa_grouped_out_proj(const void* o, int32_t Q, int32_t H, int32_t D, int32_t G, const void* w,
                                int32_t d_g, void* out, void* ws, size_t ws_bytes, csa_stream_t stream) {
    if (Q < 0 || Q > (1 << 24) || H < 1 || D < 1 || G < 1 || d_g < 1)
        return fail(CSA_ERR_INVALID_ARG, "csa_grouped_out_proj: bad sizes");
    if (!out_proj_supported(H, D, G, d_g))
        return fail(CSA_ERR_UNSUPPORTED, "csa_grouped_out_proj: needs H %% G == 0, H/G*D and d_g multiples of 64");
    if (Q == 0) return CSA_OK;
    CHECK(check_ptr(o, "o"));
    CHECK(check_ptr(w, "w"));
    CHECK(check_ptr(out, "out"));
    CHECK(check_ptr(ws, "ws"));
    if (ws_bytes < kStatusWordBytes) return fail(CSA_ERR_WORKSPACE, "workspace smaller than 256 bytes");
    // decode-sized calls split K when the workspace holds the float32 sums
    float* acc = (Q <= 128 && ws_bytes >= csa_grouped_out_proj_ws_bytes(Q, G, d_g))
                     ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + kStatusWordBytes)
                     : nullptr;
    cudaError_t e = launch_out_proj(o, Q, H, D, G, w, d_g, out, acc, reinterpret_cast<uint32_t*>(ws),
                                    (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_grouped_out_proj");
}

size_t csa_grouped_out_proj_ws_bytes(int32_t Q, int32_t G, int32_t d_g) {
    if (Q < 0 || G < 1 || d_g < 1) return 0;
    size_t n = kStatusWordBytes;
    if (Q <= 128) n += (size_t)4 * (size_t)Q * (size_t)G * (size_t)d_g;
    return n;
}

uint64_t csa_launch_count(void) { return (uint64_t)g_launches.load(); }

csa_status csa_test_withhold_indexer_loads(int32_t on) {
    set_indexer_withhold(on);
    return CSA_OK;
}

static csa_status attend_common(const csa_params* p, bool sparse, const void* q, int32_t H,
                                int32_t B, int32_t Q, const int64_t* q_pos, const void* cache,
                                int64_t n_cap, const int32_t* topk_idx, const void* window,
                                int64_t n_win, const int64_t* win_pos0, const float* sink,
                                void* out, float* lse, void* ws, size_t ws_bytes,
                                csa_stream_t stream, const char* name) {
    CHECK(check_params(p));
    if (sparse && (p->topk < 1 || p->topk > 4096))
        return fail(CSA_ERR_INVALID_ARG, "%s: topk %d not in [1, 4096]", name, p->topk);
    if (H < 1 || H > 128 || H % 8 != 0)
        return fail(CSA_ERR_UNSUPPORTED, "%s: H %d must be a multiple of 8 up to 128", name, H);
    if (B < 1 || Q < 0 || Q % B != 0) return fail(CSA_ERR_INVALID_ARG, "%s: Q %d must be a multiple of B %d", name, Q, B);
    if (n_cap < 0 || n_cap > (1LL << 30) || n_win < 0 || n_win > (1LL << 30))
        return fail(CSA_ERR_INVALID_ARG, "%s: n_cap / n_win out of range", name);
    if (Q == 0) return CSA_OK;
    CHECK(check_ptr(q, "q"));
    CHECK(check_ptr(q_pos, "q_pos"));
    CHECK(check_ptr(cache, "cache", n_cap == 0));
    if (sparse) CHECK(check_ptr(topk_idx, "topk_idx"));
    CHECK(check_ptr(window, "window", n_win == 0 || p->window == 0));
    CHECK(check_ptr(win_pos0, "win_pos0", true));  // NULL: the window is a ring
    const bool ring = win_pos0 == nullptr;
    if (ring && p->window > 0 && n_win < p->window)
        return fail(CSA_ERR_INVALID_ARG, "%s: a ring window needs n_win (%lld) >= W (%d)", name, (long long)n_win,
                    p->window);
    CHECK(check_ptr(sink, "sink"));
    CHECK(check_ptr(out, "out"));
    CHECK(check_ptr(lse, "lse", true));
    CHECK(check_ptr(ws, "ws"));
    Geometry g = resolve(p);
    AttendPlan pl = plan_attend(g, sparse, B, Q, H, n_cap, n_win, ring);
    if (ws_bytes < pl.total) return fail(CSA_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", name, ws_bytes, pl.total);
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    cudaError_t e = launch_attend(g, pl, sparse, q, H, B, Q, q_pos, cache, n_cap, topk_idx, window,
                                  n_win, win_pos0, sink, out, lse, w,
                                  reinterpret_cast<uint32_t*>(w), (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, name);
}

csa_status csa_index_keys_pack(const csa_params* p, const void* keys, int64_t n_rows, int32_t idx_dim,
                               uint8_t* codes, float* scales, csa_stream_t stream) {
    CHECK(check_params(p));
    if (idx_dim != 128) return fail(CSA_ERR_UNSUPPORTED, "idx_dim %d: E4M3 keys take 128", idx_dim);
    if (n_rows < 0) return fail(CSA_ERR_INVALID_ARG, "n_rows < 0");
    if (n_rows == 0) return CSA_OK;
    CHECK(check_ptr(keys, "keys"));
    CHECK(check_ptr(codes, "codes"));
    CHECK(check_ptr(scales, "scales"));
    Geometry g = resolve(p);
    cudaError_t e = launch_pack_idx_keys(g, keys, n_rows, codes, scales, (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_index_keys_pack");
}

csa_status csa_index_score_fp8(const csa_params* p, const void* q_idx, const float* w_idx,
                               int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_codes,
                               const float* key_scales, int64_t n_cap, int32_t B, int32_t Q,
                               const int64_t* q_pos, float* scores, int64_t ld_scores, void* ws,
                               size_t ws_bytes, csa_stream_t stream) {
    CHECK(check_params(p));
    if (idx_dim != 128 || n_idx_heads != 64)
        return fail(CSA_ERR_UNSUPPORTED, "E4M3 keys take 64 heads of 128 dims (got %d x %d)", n_idx_heads, idx_dim);
    if (B < 1 || Q < 0 || Q % B != 0) return fail(CSA_ERR_INVALID_ARG, "Q %d must be a multiple of B %d", Q, B);
    if (n_cap < 0 || n_cap > (1LL << 30)) return fail(CSA_ERR_INVALID_ARG, "n_cap out of range");
    if (ld_scores < n_cap || ld_scores % 4 != 0)
        return fail(CSA_ERR_INVALID_ARG, "ld_scores %lld must be >= n_cap and a multiple of 4", (long long)ld_scores);
    if (Q == 0) return CSA_OK;
    if (n_cap > 0 && n_cap < 128) return fail(CSA_ERR_UNSUPPORTED, "E4M3 keys need n_cap >= 128");
    CHECK(check_ptr(q_idx, "q_idx"));
    CHECK(check_ptr(w_idx, "w_idx"));
    CHECK(check_ptr(key_codes, "key_codes", n_cap == 0));
    CHECK(check_ptr(key_scales, "key_scales", n_cap == 0));
    CHECK(check_ptr(q_pos, "q_pos"));
    CHECK(check_ptr(scores, "scores"));
    CHECK(check_ptr(ws, "ws"));
    // workspace: status word, then the query codes and weights
    const size_t q8_off = kStatusWordBytes;
    const size_t weff_off = q8_off + align256((size_t)Q * 64 * 128);
    const size_t need = weff_off + align256((size_t)Q * 64 * sizeof(float));
    if (ws_bytes < need) return fail(CSA_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
    Geometry g = resolve(p);
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    cudaError_t e = launch_indexer_fp8(g, q_idx, w_idx, key_codes, key_scales, n_cap, B, Q, q_pos,
                                       reinterpret_cast<uint32_t*>(w), scores, ld_scores, w + q8_off,
                                       reinterpret_cast<float*>(w + weff_off), (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_index_score_fp8");
}

csa_status csa_index_topk_fp8(const csa_params* p, const void* q_idx, const float* w_idx,
                              int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_codes,
                              const float* key_scales, int64_t n_cap, int32_t B, int32_t Q,
                              const int64_t* q_pos, int32_t* topk_idx, float* topk_score, void* ws,
                              size_t ws_bytes, csa_stream_t stream) {
    CHECK(check_params(p));
    if (p->topk < 1 || p->topk > 4096) return fail(CSA_ERR_INVALID_ARG, "topk %d not in [1, 4096]", p->topk);
    if (idx_dim != 128 || n_idx_heads != 64)
        return fail(CSA_ERR_UNSUPPORTED, "E4M3 keys take 64 heads of 128 dims (got %d x %d)", n_idx_heads, idx_dim);
    if (B < 1 || Q < 0 || Q % B != 0) return fail(CSA_ERR_INVALID_ARG, "Q %d must be a multiple of B %d", Q, B);
    if (n_cap < 0 || n_cap > (1LL << 30)) return fail(CSA_ERR_INVALID_ARG, "n_cap out of range");
    if (Q == 0) return CSA_OK;
    if (n_cap > 0 && n_cap < 128) return fail(CSA_ERR_UNSUPPORTED, "E4M3 keys need n_cap >= 128");
    CHECK(check_ptr(q_idx, "q_idx"));
    CHECK(check_ptr(w_idx, "w_idx"));
    CHECK(check_ptr(key_codes, "key_codes", n_cap == 0));
    CHECK(check_ptr(key_scales, "key_scales", n_cap == 0));
    CHECK(check_ptr(q_pos, "q_pos"));
    CHECK(check_ptr(topk_idx, "topk_idx"));
    CHECK(check_ptr(topk_score, "topk_score", true));
    CHECK(check_ptr(ws, "ws"));
    if (topk_chunk(n_cap, Q, p->topk) == 0)
        return fail(CSA_ERR_UNSUPPORTED, "top-%d of %lld blocks does not fit the selection's shared memory",
                    p->topk, (long long)n_cap);
    Geometry g = resolve(p);
    IndexTopkPlan pl = plan_index_topk(g, B, Q, n_idx_heads, n_cap, true);
    if (ws_bytes < pl.total) return fail(CSA_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, pl.total);
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    uint32_t* status = reinterpret_cast<uint32_t*>(w);
    float* scores = reinterpret_cast<float*>(w + pl.scores_off);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = launch_indexer_fp8(g, q_idx, w_idx, key_codes, key_scales, n_cap, B, Q, q_pos, status, scores,
                                       pl.n_cap_pad, w + pl.q8_off, reinterpret_cast<float*>(w + pl.weff_off), st);
    if (e != cudaSuccess) return cuda_fail(e, "csa_index_topk_fp8: indexer");
    e = launch_topk(g, scores, pl.n_cap_pad, n_cap, Q, q_pos, topk_idx, topk_score, st);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_index_topk_fp8: top-k");
}

int64_t csa_index_keys_fp4_bytes(int64_t n_cap) {
    if (n_cap < 0) return -1;
    return (n_cap + 127) / 128 * kFp4KeyTileBytes;
}

csa_status csa_index_keys_pack_fp4(const csa_params* p, const void* keys, int32_t B, int64_t n_cap,
                                   int32_t idx_dim, uint8_t* pack, csa_stream_t stream) {
    CHECK(check_params(p));
    if (idx_dim != 128) return fail(CSA_ERR_UNSUPPORTED, "idx_dim %d: FP4 keys take 128", idx_dim);
    if (B < 0 || n_cap < 0 || n_cap > (1LL << 30)) return fail(CSA_ERR_INVALID_ARG, "B / n_cap out of range");
    if (B == 0 || n_cap == 0) return CSA_OK;
    CHECK(check_ptr(keys, "keys"));
    CHECK(check_ptr(pack, "pack"));
    Geometry g = resolve(p);
    cudaError_t e = launch_pack_idx_keys_fp4(g, keys, B, n_cap, pack, (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_index_keys_pack_fp4");
}

// The checks shared by the FP4 scoring calls.
static csa_status check_fp4_index(const csa_params* p, int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_pack,
                                  int64_t n_cap, int32_t B, int32_t Q, const void* q_idx, const float* w_idx,
                                  const int64_t* q_pos) {
    CHECK(check_params(p));
    if (idx_dim != 128 || n_idx_heads != 64)
        return fail(CSA_ERR_UNSUPPORTED, "FP4 keys take 64 heads of 128 dims (got %d x %d)", n_idx_heads, idx_dim);
    if (B < 1 || Q < 0 || Q % B != 0) return fail(CSA_ERR_INVALID_ARG, "Q %d must be a multiple of B %d", Q, B);
    if (n_cap < 0 || n_cap > (1LL << 30)) return fail(CSA_ERR_INVALID_ARG, "n_cap out of range");
    if (Q == 0) return CSA_OK;
    if (n_cap > 0 && n_cap < 128) return fail(CSA_ERR_UNSUPPORTED, "FP4 keys need n_cap >= 128");
    CHECK(check_ptr(q_idx, "q_idx"));
    CHECK(check_ptr(w_idx, "w_idx"));
    CHECK(check_ptr(key_pack, "key_pack", n_cap == 0));
    CHECK(check_ptr(q_pos, "q_pos"));
    return CSA_OK;
}

csa_status csa_index_score_fp4(const csa_params* p, const void* q_idx, const float* w_idx,
                               int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_pack, int64_t n_cap,
                               int32_t B, int32_t Q, const int64_t* q_pos, float* scores, int64_t ld_scores,
                               void* ws, size_t ws_bytes, csa_stream_t stream) {
    CHECK(check_fp4_index(p, n_idx_heads, idx_dim, key_pack, n_cap, B, Q, q_idx, w_idx, q_pos));
    if (ld_scores < n_cap || ld_scores % 4 != 0)
        return fail(CSA_ERR_INVALID_ARG, "ld_scores %lld must be >= n_cap and a multiple of 4", (long long)ld_scores);
    if (Q == 0) return CSA_OK;
    CHECK(check_ptr(scores, "scores"));
    CHECK(check_ptr(ws, "ws"));
    const size_t q8_off = kStatusWordBytes;
    const size_t weff_off = q8_off + align256((size_t)Q * 64 * 128);
    const size_t need = weff_off + align256((size_t)Q * 64 * sizeof(float));
    if (ws_bytes < need) return fail(CSA_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
    Geometry g = resolve(p);
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    cudaError_t e = launch_indexer_fp4(g, q_idx, w_idx, key_pack, n_cap, B, Q, q_pos, reinterpret_cast<uint32_t*>(w),
                                       scores, ld_scores, w + q8_off, reinterpret_cast<float*>(w + weff_off),
                                       (cudaStream_t)stream);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_index_score_fp4");
}

csa_status csa_index_topk_fp4(const csa_params* p, const void* q_idx, const float* w_idx,
                              int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_pack, int64_t n_cap,
                              int32_t B, int32_t Q, const int64_t* q_pos, int32_t* topk_idx, float* topk_score,
                              void* ws, size_t ws_bytes, csa_stream_t stream) {
    CHECK(check_fp4_index(p, n_idx_heads, idx_dim, key_pack, n_cap, B, Q, q_idx, w_idx, q_pos));
    if (p->topk < 1 || p->topk > 4096) return fail(CSA_ERR_INVALID_ARG, "topk %d not in [1, 4096]", p->topk);
    if (Q == 0) return CSA_OK;
    CHECK(check_ptr(topk_idx, "topk_idx"));
    CHECK(check_ptr(topk_score, "topk_score", true));
    CHECK(check_ptr(ws, "ws"));
    if (topk_chunk(n_cap, Q, p->topk) == 0)
        return fail(CSA_ERR_UNSUPPORTED, "top-%d of %lld blocks does not fit the selection's shared memory",
                    p->topk, (long long)n_cap);
    Geometry g = resolve(p);
    IndexTopkPlan pl = plan_index_topk(g, B, Q, n_idx_heads, n_cap, true);
    if (ws_bytes < pl.total) return fail(CSA_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, pl.total);
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    float* scores = reinterpret_cast<float*>(w + pl.scores_off);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = launch_indexer_fp4(g, q_idx, w_idx, key_pack, n_cap, B, Q, q_pos, reinterpret_cast<uint32_t*>(w),
                                       scores, pl.n_cap_pad, w + pl.q8_off, reinterpret_cast<float*>(w + pl.weff_off),
                                       st);
    if (e != cudaSuccess) return cuda_fail(e, "csa_index_topk_fp4: indexer");
    e = launch_topk(g, scores, pl.n_cap_pad, n_cap, Q, q_pos, topk_idx, topk_score, st);
    return e == cudaSuccess ? CSA_OK : cuda_fail(e, "csa_index_topk_fp4: top-k");
}

csa_status csa_attend(const csa_params* p, const void* q, int32_t H, int32_t B, int32_t Q,
                      const int64_t* q_pos, const void* cache, int64_t n_cap,
                      const int32_t* topk_idx, const void* window, int64_t n_win,
                      const int64_t* win_pos0, const float* sink, void* out, float* lse,
                      void* ws, size_t ws_bytes, csa_stream_t stream) {
    return attend_common(p, true, q, H, B, Q, q_pos, cache, n_cap, topk_idx, window, n_win,
                         win_pos0, sink, out, lse, ws, ws_bytes, stream, "csa_attend");
}

csa_status hca_attend(const csa_params* p, const void* q, int32_t H, int32_t B, int32_t Q,
                      const int64_t* q_pos, const void* cache, int64_t n_cap, const void* window,
                      int64_t n_win, const int64_t* win_pos0, const float* sink, void* out,
                      float* lse, void* ws, size_t ws_bytes, csa_stream_t stream) {
    return attend_common(p, false, q, H, B, Q, q_pos, cache, n_cap, nullptr, window, n_win,
                         win_pos0, sink, out, lse, ws, ws_bytes, stream, "hca_attend");
}

}  // extern "C"
