// internal.h -- launchers behind the C ABI (host side, no validation here:
// csa_capi.cu validates every argument before calling these).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "csa.h"

namespace csa {

// RoPE frequencies theta_j = base^(-2j/R) of the 32 rotated pairs (R = 64),
// computed once per call in double on the host and passed by value to the
// kernels.
struct RopeTheta {
    double t[32];
};

struct Geometry {  // resolved layer constants
    int D, R, m, k, W;
    float base, eps, scale;
    int derotate;
    int act, kv;
    int64_t kv_row_bytes;
    int inv;  // batch-invariant attention splits
};

// Batch-invariant attention: split length, in tiles of 64 rows, of a row
// list of T tiles -- the largest power of two <= T/8, clamped to [2, 16]; a
// function of the list's length only.
inline int inv_split_tiles(int64_t T) {
    int s = 2;
    while (s < 16 && (int64_t)s * 16 <= T) s *= 2;
    return s;
}

Geometry resolve(const csa_params* p);

// theta_j = base^(-2j/R) for the RoPE pairs of the last R dims.
RopeTheta rope_theta(const Geometry& g);

// Workspace layout of an operation.  Offsets are in bytes from the start of
// the workspace; every region is 256-byte aligned.
struct IndexTopkPlan {
    size_t scores_off, scores_bytes;  // [Q, n_cap_pad] float32
    int64_t n_cap_pad;
    size_t q8_off, weff_off;          // E4M3 keys: query codes [Q, 64, 128], weights [Q, 64] float32
    size_t total;
};
IndexTopkPlan plan_index_topk(const Geometry& g, int B, int Q, int HI, int64_t n_cap, bool fp8 = false);

struct AttendPlan {
    int splits;           // split-K factor over the row list
    int64_t list_len;     // rows per query in the list (before masking)
    int64_t rows_per_split;
    int head_group;       // heads per CTA
    int use_tc;           // tensor-core kernel
    // tensor-core kernel: tiles of 64 rows per query (selected / cache part
    // and all), Q * tc_T tiles dealt to tc_grid persistent CTAs
    int tc_T_sel, tc_T, tc_grid;
    // window tiles: ceil(W / 64) tiles of positions (linear window), or
    // ceil(n_win / 64) tiles of ring rows (ring window: position p at row
    // p mod n_win, every row whose position is in the window valid)
    int ring;
    int64_t tc_total;
    // batch-invariant splits: tc_seg tiles each (0: balanced ranges), tc_nseg
    // per query
    int tc_seg, tc_nseg;
    // query-aligned ranges (see TileDeal): CTAs per query, and how many
    // queries get one more (tc_qcta 0: balanced over all tiles, each query
    // counted as tc_qc more tiles than it has)
    int tc_qcta, tc_qrem, tc_qc;
    // FP8 rows reach the tensor-core kernel dequantised to bf16 in the
    // workspace: 1 = the rows each query reads, [Q, tc_T * 64, D] in tile
    // order; 2 = every stored row, [B, n_cap, D] then [B, n_win, D]; 0 = the
    // stored rows are bf16 already
    int tc_deq;
    size_t part_o_off, part_ml_off;  // [Q, S, H, D] and [Q, S, H, 2] float32
    // [Q] int32 (tensor-core ranges only, else 0): how many CTAs left a
    // partial of each query (0: its only CTA finished it)
    size_t nslots_off;
    size_t deq_off;                  // bf16 rows of tc_deq
    size_t total;
};
AttendPlan plan_attend(const Geometry& g, bool sparse, int B, int Q, int H, int64_t n_cap,
                       int64_t n_win, bool ring);

cudaError_t launch_cache_pack(const Geometry& g, const float* src, int64_t n, void* dst,
                              cudaStream_t st);
// win_out (or nullptr): also the window row of every block's last token, at
// row b of sequence s's win_stride rows.
cudaError_t launch_compress(const Geometry& g, const void* kv, int B, int64_t T,
                            int64_t kv_stride, int64_t pos0, const float* w_z, const float* bias,
                            void* out, int64_t out_stride, void* win_out, int64_t win_stride,
                            cudaStream_t st);
// Ragged decode append (csa_decode_append): raw ring slot, window ring row
// and, for sequences whose newest token completes a block, the block's entry.
bool decode_append_supported(const Geometry& g);
cudaError_t launch_decode_append(const Geometry& g, const void* tok, int B, const int64_t* pos, void* ring,
                                 const float* w_z, const float* bias, void* cache, int64_t n_cap, void* window,
                                 int64_t n_win, uint32_t* status, cudaStream_t st);
cudaError_t launch_indexer(const Geometry& g, const void* q_idx, const float* w_idx, int HI,
                           int dI, const void* keys, int64_t n_cap, int B, int Q,
                           const int64_t* q_pos, uint32_t* status, float* scores, int64_t ld,
                           cudaStream_t st);
cudaError_t launch_indexer_fp8(const Geometry& g, const void* q_idx, const float* w_idx, const uint8_t* key_codes,
                               const float* key_scales, int64_t n_cap, int B, int Q, const int64_t* q_pos,
                               uint32_t* status, float* scores, int64_t ld, uint8_t* q8, float* w_eff,
                               cudaStream_t st);
// FP4 indexer keys: packed tiles of 8704 bytes (128 keys' E2M1 codes, then
// their block-exponent bytes), ceil(n_cap / 128) tiles a sequence.
constexpr int64_t kFp4KeyTileBytes = 8704;
cudaError_t launch_pack_idx_keys_fp4(const Geometry& g, const void* keys, int B, int64_t n_cap, uint8_t* pack,
                                     cudaStream_t st);
cudaError_t launch_indexer_fp4(const Geometry& g, const void* q_idx, const float* w_idx, const uint8_t* key_pack,
                               int64_t n_cap, int B, int Q, const int64_t* q_pos, uint32_t* status, float* scores,
                               int64_t ld, uint8_t* q8, float* w_eff, cudaStream_t st);
cudaError_t launch_pack_idx_keys(const Geometry& g, const void* rows, int64_t n, uint8_t* codes, float* scales,
                                 cudaStream_t st);
cudaError_t launch_topk(const Geometry& g, float* scores, int64_t ld, int64_t n_cap, int Q,
                        const int64_t* q_pos, int32_t* idx, float* sel, cudaStream_t st);
// Chunk size of the top-k selection for these sizes; 0: does not fit.
int64_t topk_chunk(int64_t n_cap, int Q, int k);
// Test hook of csa_test_withhold_indexer_loads.
void set_indexer_withhold(int on);
cudaError_t launch_attend(const Geometry& g, const AttendPlan& pl, bool sparse, const void* q,
                          int H, int B, int Q, const int64_t* q_pos, const void* cache,
                          int64_t n_cap, const int32_t* topk_idx, const void* window,
                          int64_t n_win, const int64_t* win_pos0, const float* sink, void* out,
                          float* lse, uint8_t* ws, uint32_t* status, cudaStream_t st);

// Grouped output projection (k_out_proj.cu).
bool out_proj_supported(int H, int D, int G, int d_g);
// acc: float32 [Q, G * d_g] scratch for split-K sums (decode-sized Q), or
// nullptr to run unsplit.
cudaError_t launch_out_proj(const void* o, int Q, int H, int D, int G, const void* w, int d_g, void* out,
                            float* acc, uint32_t* status, cudaStream_t st);

// SM count of the current device (cached per device).
int num_sms();

// Launch `kernel` as a programmatic dependent of the grid before it in the
// stream: its CTAs may be scheduled while that grid finishes, and every read
// of that grid's results comes after grid_dep_wait() in the kernel.
template <class... KArgs, class... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raise a kernel's dynamic shared memory limit to at least `bytes` on the
// current device (cached per device and kernel; thread-safe).
cudaError_t set_smem_attr(const void* kernel, size_t bytes);

// Kernel launch accounting (csa_launch_count).
void note_launch(int n = 1);

// Record a failure for csa_last_error() and return its status.
csa_status set_error(csa_status s, const char* msg);

}  // namespace csa
