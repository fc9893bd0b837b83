/*
 * csa.h -- C ABI of the B300 (sm_103a) library for the DeepSeek-V4 hybrid
 * compressed attention hot path: CSA (compressed sparse attention) and HCA
 * (heavily compressed attention).
 *
 * Pages defining the operations (title, site):
 *   [peacm]   "DeepSeek-V4百万上下文时代的开源宣言" (peacm.com), §三.2 混合注意力机制
 *   [gitcode] "DeepSeek-V4 技术报告深度解析" (gitcode.csdn.net), §2.1 混合注意力机制
 *   [wiki]    "DeepSeek V4 (Flash & Pro)：通往百万级上下文与万亿参数推理的新纪元",
 *             混合注意力机制：CSA 与 HCA 的协同逻辑
 *
 * Conventions common to every entry point
 *   - Every data pointer is a caller-owned DEVICE buffer unless stated.  The
 *     library never allocates or frees memory, never keeps pointers after a
 *     call returns, and launches all work on the given stream without
 *     synchronising (csa_check_status is the one call that synchronises).
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns CSA_ERR_INVALID_ARG or CSA_ERR_UNSUPPORTED, has no
 *     side effect and launches nothing.  A failed launch returns CSA_ERR_CUDA.
 *     csa_last_error() then holds a one-line reason (per host thread).
 *   - Data-dependent errors that only the device can see (a top-k index that
 *     is not a complete block, a window position missing from the window
 *     buffer, a query position beyond the cache capacity) never fault: the
 *     kernel skips the offending row and sets a bit in the status word at the
 *     start of the workspace.  csa_check_status() reports and clears it.
 *   - Row-major layouts; the last dimension is contiguous.  Every device
 *     pointer must be 16-byte aligned.
 *   - Positions are absolute token indices (int64).  A query at position i
 *     sees compressed block b when b*m + m - 1 <= i ("causally complete"),
 *     i.e. the first floor((i+1)/m) blocks, and the raw window tokens
 *     max(0, i-W+1) .. i.
 */
#ifndef CSA_B300_H
#define CSA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* csa_stream_t;

typedef enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or params     */
    CSA_ERR_UNSUPPORTED = 2, /* valid request outside the shapes this build runs */
    CSA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed              */
    CSA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required        */
    CSA_ERR_DEVICE = 5       /* csa_check_status: the device flagged bad data     */
} csa_status;

/* Storage formats.
 *   CSA_F32, CSA_BF16: D values per row.
 *   CSA_FP8_MIXED (cache/window rows only) [gitcode §2.1.4 "KV 缓存精度":
 *   RoPE dims in BF16, the other dims in FP8]: dims 0..D-65 as OCP E4M3 bytes,
 *   then the 64 RoPE dims D-64..D-1 as bfloat16, then (D-64)/64 float32
 *   scales, one per 64-dim group (value = code * scale; scale = group amax /
 *   448, or 1 for an all-zero group), zero padding to a multiple of 16 bytes
 *   (608 bytes for D = 512). */
typedef enum { CSA_F32 = 0, CSA_BF16 = 1, CSA_FP8_MIXED = 2 } csa_format;

/* Device status bits (csa_check_status). */
#define CSA_DEV_BAD_TOPK_INDEX 0x1u /* selected block not complete or >= n_cap */
#define CSA_DEV_BAD_WINDOW 0x2u     /* window position not in the window buffer */
#define CSA_DEV_BAD_POSITION 0x4u   /* floor((i+1)/m) exceeds the cache capacity */
#define CSA_DEV_TIMEOUT 0x8u        /* a bounded wait inside a kernel expired     */

/* Layer hyper-parameters, passed by pointer (read during the call only). */
typedef struct {
    int32_t head_dim;        /* D: 128 or 512 (any multiple of 64 up to 512)          */
    int32_t rope_dims;       /* rotated trailing dims; must be 64 [peacm 四项关键 Trick] */
    float rope_base;         /* theta_j = rope_base^(-2j/rope_dims); 10000              */
    float norm_eps;          /* RMSNorm epsilon (unit gain); 1e-6                       */
    float softmax_scale;     /* logit scale; <= 0 selects 1/sqrt(D)                     */
    int32_t ratio;           /* m: tokens per compressed block (CSA 4, HCA 128, 1 = window rows) */
    int32_t topk;            /* k: blocks kept per query (CSA), 1..4096                 */
    int32_t window;          /* W: raw sliding-window tokens per query, 0..1024         */
    int32_t derotate_output; /* nonzero: rotate the output by RoPE at position -i       */
    int32_t act_format;      /* CSA_F32 or CSA_BF16: q, raw kv, indexer q/keys, outputs */
    int32_t kv_format;       /* CSA_F32 (with F32 act), CSA_BF16 or CSA_FP8_MIXED      */
    int32_t batch_invariant; /* nonzero: attention outputs bit-identical in any batch  */
} csa_params;

/* Bytes of one stored cache/window row of `head_dim` dims in `kv_format`
 * (D*4, D*2, or the mixed layout above); -1 for an unsupported pair. */
int64_t csa_row_bytes(int32_t kv_format, int32_t head_dim);

/* Write float32 rows into the cache row format p->kv_format (the cache
 * writer).  For CSA_FP8_MIXED each 64-dim group is quantised with
 * scale = amax/448 (float32), code = E4M3 round-to-nearest-even of x/scale
 * with saturation [gitcode §2.1.4 "KV 缓存精度"].
 *   src: [n_rows, D] float32.  dst: [n_rows] rows of csa_row_bytes bytes. */
csa_status csa_cache_pack(const csa_params* p, const float* src, int64_t n_rows, void* dst,
                          csa_stream_t stream);

/* Block compressor [peacm §三.2 CSA "Step 1: KV 压缩 每 m 个 token -> 1 个压缩
 * KV entry" (attention-like pooling with learnable weights); HCA "压缩率 m'
 * 128"; 四项关键 Trick "Q/KV Normalization", "Partial RoPE"].  For every
 * complete block b of m = p->ratio tokens at positions pos0+b*m .. pos0+b*m+m-1:
 *   z_t = kv_t . w_z + bias[t mod m];  alpha = softmax_t(z);  c = sum alpha_t kv_t
 *   entry = RoPE(RMSNorm(c), pos0 + b*m + m - 1)
 * stored in p->kv_format.  m = 1 produces the window rows RoPE(RMSNorm(kv_t), t).
 *   kv_raw: B sequences of T raw tokens [.., D] in p->act_format; sequence s
 *           starts at row s*kv_seq_stride.
 *   pos0:   position of the first token (same for every sequence); must be a
 *           multiple of m.  T need not be: a trailing partial block is skipped.
 *   w_z: [D] float32; bias: [m] float32.
 *   out:    the T/m entries of sequence s start at row s*out_seq_stride. */
csa_status csa_compress(const csa_params* p, const void* kv_raw, int32_t B, int64_t T,
                        int64_t kv_seq_stride, int64_t pos0, const float* w_z, const float* bias,
                        void* out, int64_t out_seq_stride, csa_stream_t stream);

/* Decode append in one launch: the cache entry of one newly completed block
 * per sequence and the window row of its last token -- exactly what
 *   csa_compress(p, kv_new, B, m, kv_seq_stride, pos0, w_z, bias,
 *                entry_out, out_seq_stride)
 * and csa_compress with ratio 1 over the block's last token (position
 * pos0+m-1) into win_out write (same arithmetic, bit for bit).  This entry
 * point has no counterpart on the pages: it fuses the two steps of keeping a
 * decode cache current [peacm §三.2 CSA "Step 1"; 四项关键 Trick "滑动窗口"].
 *   kv_new: B blocks of m = p->ratio raw tokens [.., D] in p->act_format at
 *           positions pos0 .. pos0+m-1 (pos0 a multiple of m); sequence s
 *           starts at row s*kv_seq_stride.
 *   entry_out: sequence s's entry at row s*out_seq_stride (p->kv_format rows).
 *   win_out:   sequence s's window row at row s*win_seq_stride.
 *   w_z: [D] float32; bias: [m] float32.  All buffers device, 16-byte aligned. */
csa_status csa_append(const csa_params* p, const void* kv_new, int32_t B, int64_t kv_seq_stride,
                      int64_t pos0, const float* w_z, const float* bias, void* entry_out,
                      int64_t out_seq_stride, void* win_out, int64_t win_seq_stride,
                      csa_stream_t stream);

/* One decode step's cache maintenance for a ragged batch, in one launch
 * [peacm §三.2 CSA "Step 1: KV 压缩" (every m tokens pooled into one entry),
 * HCA (m' = 128); 四项关键 Trick "Sliding Window" (the most recent W raw
 * tokens)].  This entry point has no counterpart on the pages: it keeps the
 * decode state current one token at a time.  Sequence s's newest token is at
 * position t = pos[s]; every sequence has its own length.  The call
 *   - stores the token's raw row in slot t mod m of the sequence's raw ring
 *     (the raw tokens of its current block: position p sits in slot p mod m);
 *   - writes its window row RoPE(RMSNorm(kv_t), t) at row t mod n_win of the
 *     sequence's window ring (read by csa_attend / hca_attend with
 *     win_pos0 = NULL);
 *   - when t + 1 is a multiple of m, pools the completed block (positions
 *     t-m+1 .. t: ring slots 0 .. m-2 and the new token) into cache entry
 *     (t + 1)/m - 1, with the arithmetic of csa_compress.
 *   kv_tok:   [B, D] the newest raw token of each sequence, p->act_format
 *   pos:      [B] int64 (device)
 *   raw_ring: [B, m, D] in p->act_format: state kept by the caller between
 *             calls (zero-initialise it); may be NULL when m = 1
 *   cache:    [B, n_cap] rows in p->kv_format
 *   window:   [B, n_win] rows in p->kv_format, a ring; ignored (may be NULL)
 *             when p->window = 0 or n_win = 0
 *   ws:       at least 256 bytes; its status word receives
 *             CSA_DEV_BAD_POSITION for a negative position or an entry at or
 *             beyond n_cap, and that sequence's write is skipped.
 * Blocks that do not fit the compressor's shared-memory staging return
 * CSA_ERR_UNSUPPORTED. */
csa_status csa_decode_append(const csa_params* p, const void* kv_tok, int32_t B, const int64_t* pos,
                             void* raw_ring, const float* w_z, const float* bias, void* cache, int64_t n_cap,
                             void* window, int64_t n_win, void* ws, size_t ws_bytes, csa_stream_t stream);

/* Lightning indexer + top-k [peacm §三.2 CSA "Step 2: Lightning Indexer Top-K
 * 选择"; gitcode §2.1.1].  For query q at position i = q_pos[q] in sequence
 * s = q / (Q/B), over the complete blocks b < floor((i+1)/m):
 *   score_b = sum_h w_idx[q,h] * relu(q_idx[q,h,:] . keys[s,b,:])
 * and keeps the top min(k, floor((i+1)/m)) blocks, ties to the lower index.
 *   q_idx:  [Q, n_idx_heads, idx_dim] in p->act_format; w_idx: [Q, n_idx_heads] f32
 *   keys:   [B, n_cap, idx_dim] in p->act_format
 *   q_pos:  [Q] int64 (device)
 *   topk_idx:   [Q, k] int32, selected block indices in ascending index order,
 *               padded with -1 at the end
 *   topk_score: [Q, k] float32 scores in the same order (-inf padding) or NULL
 *   ws: workspace of at least csa_workspace_bytes(p, CSA_OP_INDEX_TOPK, ...).
 * Requires Q % B == 0, idx_dim in {64, 128}, n_idx_heads <= 64. */
csa_status csa_index_topk(const csa_params* p, const void* q_idx, const float* w_idx,
                          int32_t n_idx_heads, int32_t idx_dim, const void* keys, int64_t n_cap,
                          int32_t B, int32_t Q, const int64_t* q_pos, int32_t* topk_idx,
                          float* topk_score, void* ws, size_t ws_bytes, csa_stream_t stream);

/* The two halves of csa_index_topk, for callers that keep or inspect the
 * scores.  csa_index_score writes score_b for b < floor((i+1)/m) and -inf for
 * the other blocks b < n_cap into scores[q*ld_scores + b] (float32, device,
 * ld_scores >= n_cap, caller-owned); blocks are laid out as for keys.
 * ws: status word only (>= 256 bytes).
 * csa_topk_select reads such a score matrix and writes topk_idx/topk_score
 * exactly as csa_index_topk does; it flags nothing.  It CONSUMES the score
 * matrix: when a query's blocks are selected in several chunks, the chunks'
 * candidates are written over the scores (copy them first to keep them).
 * Sizes whose selection does not fit in shared memory (k * ceil(n_cap / 32768)
 * above 40960, e.g. k = 4096 with n_cap > 327680, or k above 8192) return
 * CSA_ERR_UNSUPPORTED, as csa_index_topk does. */
csa_status csa_index_score(const csa_params* p, const void* q_idx, const float* w_idx,
                           int32_t n_idx_heads, int32_t idx_dim, const void* keys, int64_t n_cap,
                           int32_t B, int32_t Q, const int64_t* q_pos, float* scores,
                           int64_t ld_scores, void* ws, size_t ws_bytes, csa_stream_t stream);
csa_status csa_topk_select(const csa_params* p, float* scores, int64_t ld_scores,
                           int64_t n_cap, int32_t Q, const int64_t* q_pos, int32_t* topk_idx,
                           float* topk_score, csa_stream_t stream);

/* The lightning indexer with 8-bit floating-point keys and queries (the
 * pages' indexer runs in low precision [gitcode §2.1.1]; this FP8 variant is
 * this library's).  Keys are stored as E4M3 codes with one float32 scale per
 * key row: scale = amax/448 (1 for an all-zero row), code = E4M3 of
 * x/scale (round to nearest even, saturating; both divisions in float32).
 * csa_index_keys_pack writes that form:
 *   keys: [n_rows, idx_dim] in p->act_format -> codes [n_rows, idx_dim] uint8,
 *   scales [n_rows] float32 (device, 16-byte aligned); idx_dim must be 128.
 * csa_index_topk_fp8 is csa_index_topk over such keys (key_codes
 * [B, n_cap, 128], key_scales [B, n_cap]); every query head row of q_idx is
 * quantised by the same rule inside the call, and
 *   score_b = sum_h w_idx[q,h] * relu((q8_h * sq_h) . (k8_b * sk_b))
 * with the E4M3 products accumulated in float32 on the tensor cores.
 * Requires n_idx_heads = 64, idx_dim = 128, n_cap >= 128 (or 0), and a
 * workspace of csa_workspace_bytes(p, CSA_OP_INDEX_TOPK_FP8, ...).
 * csa_index_score_fp8 is its scoring half, as csa_index_score is for bf16
 * keys (scores [Q, ld_scores] float32); its workspace needs 256 bytes plus
 * Q*64*128 bytes and Q*64 floats, each rounded up to 256 bytes (no more than
 * the CSA_OP_INDEX_TOPK_FP8 size for the same shapes). */
csa_status csa_index_keys_pack(const csa_params* p, const void* keys, int64_t n_rows, int32_t idx_dim,
                               uint8_t* codes, float* scales, csa_stream_t stream);
csa_status csa_index_score_fp8(const csa_params* p, const void* q_idx, const float* w_idx,
                               int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_codes,
                               const float* key_scales, int64_t n_cap, int32_t B, int32_t Q,
                               const int64_t* q_pos, float* scores, int64_t ld_scores, void* ws,
                               size_t ws_bytes, csa_stream_t stream);
csa_status csa_index_topk_fp8(const csa_params* p, const void* q_idx, const float* w_idx,
                              int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_codes,
                              const float* key_scales, int64_t n_cap, int32_t B, int32_t Q,
                              const int64_t* q_pos, int32_t* topk_idx, float* topk_score, void* ws,
                              size_t ws_bytes, csa_stream_t stream);

/* The lightning indexer with FP4 keys [gitcode §2.1.1: the indexer's QK path
 * in FP4; §3.2: FP4 with 1x32 sub-block scales, converted to FP8 (E4M3)
 * without loss for computation].  A key of 128 dims is stored as E2M1 codes
 * (dim 2i in the low nibble of byte i, dim 2i+1 in the high one) and four
 * block exponent bytes, block j (dims 32j .. 32j+31) scaled by
 * 2^(byte - 127): e_j = floor(log2 amax_j) - 2 (the block's largest value in
 * [4, 8); 0 for an all-zero block), a nonzero block more than 14 binades below
 * the key's largest raised to that largest minus 14 (the key then converts to
 * E4M3 codes with one power-of-two scale per key without loss), code = E2M1 of
 * x / 2^e_j, nearest with ties to the even code, saturating at 6.  68 bytes a
 * key (bf16 keys take 256, E4M3 keys 132).
 * Storage: per sequence, ceil(n_cap / 128) tiles of csa_index_keys_fp4_bytes(128)
 * = 8704 bytes, tile t holding keys 128t .. 128t+127: their 64-byte code rows,
 * then their 4 exponent bytes each (key slots past n_cap hold an all-zero
 * key: codes 0, exponent bytes 127).
 * csa_index_keys_pack_fp4 writes that form from keys [B, n_cap, 128] in
 * p->act_format; pack: B * csa_index_keys_fp4_bytes(n_cap) bytes (device).
 * csa_index_topk_fp4 / csa_index_score_fp4 are csa_index_topk_fp8 /
 * csa_index_score_fp8 over such keys: the query heads are quantised to E4M3
 * inside the call as for E4M3 keys, every key is expanded to E4M3 codes with
 * one power-of-two scale in shared memory, and
 *   score_b = sum_h w_idx[q,h] * relu((q8_h * sq_h) . k4_b)
 * with the products accumulated in float32 on the tensor cores.  Requires
 * n_idx_heads = 64, idx_dim = 128, n_cap >= 128 (or 0), and the workspace
 * of CSA_OP_INDEX_TOPK_FP4 (the scoring half: as csa_index_score_fp8's). */
int64_t csa_index_keys_fp4_bytes(int64_t n_cap);
csa_status csa_index_keys_pack_fp4(const csa_params* p, const void* keys, int32_t B, int64_t n_cap,
                                   int32_t idx_dim, uint8_t* pack, csa_stream_t stream);
csa_status csa_index_score_fp4(const csa_params* p, const void* q_idx, const float* w_idx,
                               int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_pack, int64_t n_cap,
                               int32_t B, int32_t Q, const int64_t* q_pos, float* scores, int64_t ld_scores,
                               void* ws, size_t ws_bytes, csa_stream_t stream);
csa_status csa_index_topk_fp4(const csa_params* p, const void* q_idx, const float* w_idx,
                              int32_t n_idx_heads, int32_t idx_dim, const uint8_t* key_pack, int64_t n_cap,
                              int32_t B, int32_t Q, const int64_t* q_pos, int32_t* topk_idx, float* topk_score,
                              void* ws, size_t ws_bytes, csa_stream_t stream);

/* csa_index_topk for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for integration only.
 *
 * Some callers cannot call cudaMalloc: a plug-in or custom operator whose
 * host framework owns every device allocation and hands it only its input and
 * output buffers, or a latency-critical path that cannot afford the implicit
 * device-wide synchronisation an allocation may cause.  This variant computes
 * exactly what csa_index_topk computes, with the same arguments minus the
 * workspace, and keeps its intermediate indexer scores in a scratch array
 * compiled into the library: CSA_NOALLOC_MAX_SCORES float32 values (16 MiB)
 * plus a 256-byte status header.  Every GPU that loads the library holds that
 * scratch until the process exits.
 *   - Q * ceil(n_cap / 128) * 128 must not exceed CSA_NOALLOC_MAX_SCORES;
 *     larger requests return CSA_ERR_INVALID_ARG and launch nothing.
 *   - Every call looks up the scratch's device address on the current
 *     device (a host-side query, no allocation).  The first call on a device
 *     loads the library's device code there if nothing has yet; make that
 *     first call before any stream capture.  Sizes the top-k selection cannot
 *     hold (as for csa_index_topk) return CSA_ERR_UNSUPPORTED, launching
 *     nothing.
 *   - All calls share the one scratch array, which keeps the last call's
 *     contents.  Calls whose work overlaps on the GPU (different streams or
 *     threads without ordering between them) race and give wrong results:
 *     order them on one stream.
 *   - status: optional device uint32 that receives the call's device status
 *     bits (CSA_DEV_*), cleared at the start of every call; NULL to ignore. */
#define CSA_NOALLOC_MAX_SCORES 4194304
csa_status csa_index_topk_noalloc(const csa_params* p, const void* q_idx, const float* w_idx,
                                  int32_t n_idx_heads, int32_t idx_dim, const void* keys,
                                  int64_t n_cap, int32_t B, int32_t Q, const int64_t* q_pos,
                                  int32_t* topk_idx, float* topk_score, uint32_t* status,
                                  csa_stream_t stream);

/* CSA core attention [peacm §三.2 CSA "Step 3: Core Attention Multi-Query
 * Attention" over the top-k blocks; 四项关键 Trick: Q/KV Normalization, Partial
 * RoPE and output RoPE at -i, Sliding Window (most recent W raw tokens),
 * Attention Sink; gitcode §2.1.4].  For query q (position i, sequence s):
 *   q'_h  = RoPE(RMSNorm(q[q,h,:]), i)
 *   J     = { cache[s, topk_idx[q,j]] : topk_idx != -1 } U { window rows of
 *           positions max(0, i-W+1) .. i }   (one KV head: key = value = row)
 *   l_hj  = scale * q'_h . row_j
 *   lse_h = log(exp(sink[h]) + sum_j exp(l_hj))
 *   out_h = sum_j exp(l_hj - lse_h) row_j, then RoPE(out_h, -i) when
 *           p->derotate_output is set.  Empty J with sink -inf gives out 0, lse -inf.
 *   q:      [Q, H, D] in p->act_format (raw: normalised and rotated here)
 *   cache:  [B, n_cap] rows in p->kv_format
 *   topk_idx: [Q, k] int32 (-1 entries skipped), e.g. from csa_index_topk
 *   window: [B, n_win] rows in p->kv_format; row r of sequence s holds
 *           position win_pos0[s] + r (win_pos0: [B] int64, device)
 *   sink:   [H] float32 (-inf allowed)
 *   out:    [Q, H, D] in p->act_format;  lse: [Q, H] float32 or NULL
 * Requires Q % B == 0, H <= 128.
 *
 * Batch invariance [gitcode §5.3 "批次不变且确定性内核": with split-KV a
 * query's output depends on where it sits in the batch].  By default the
 * row lists of all Q queries are dealt out to the SMs in balanced ranges, so
 * where a query's list is split, and hence the rounding of its result,
 * depends on the other queries.  With p->batch_invariant set, every query's
 * list is cut at fixed points that depend only on its length: with T the
 * list's tiles of 64 rows (tensor-core path: ceil(k/64) + ceil(W/64) tiles,
 * HCA ceil(n_cap/64) + ceil(W/64); CUDA-core path: ceil((k + W)/64), HCA
 * ceil((n_cap + W)/64)), one split every s tiles, s = the largest power of
 * two <= T/8 clamped to [2, 16].  Every split leaves a partial and the
 * partials are merged in split order, so a query's out and lse are
 * bit-identical for any Q, B, batch order and companion queries, and from
 * run to run.  The price is coarser load balance (whole splits) and one
 * partial per split. */
csa_status csa_attend(const csa_params* p, const void* q, int32_t H, int32_t B, int32_t Q,
                      const int64_t* q_pos, const void* cache, int64_t n_cap,
                      const int32_t* topk_idx, const void* window, int64_t n_win,
                      const int64_t* win_pos0, const float* sink, void* out, float* lse,
                      void* ws, size_t ws_bytes, csa_stream_t stream);

/* HCA core attention [peacm §三.2 HCA "无稀疏筛选 对所有压缩 KV 做 dense
 * attention"; wiki "128:1 的比例压缩为稠密的 MQA 流 并辅以一个 128 令牌的滑动
 * 窗口"]: as csa_attend with J = every complete block 0 .. floor((i+1)/m)-1
 * of the sequence plus the same window; m = p->ratio (128 for HCA). */
csa_status hca_attend(const csa_params* p, const void* q, int32_t H, int32_t B, int32_t Q,
                      const int64_t* q_pos, const void* cache, int64_t n_cap, const void* window,
                      int64_t n_win, const int64_t* win_pos0, const float* sink, void* out,
                      float* lse, void* ws, size_t ws_bytes, csa_stream_t stream);

/* Grouped output projection [peacm §三.2 CSA "Step 4: Grouped Output
 * Projection" (the heads of dim 512 are projected in groups, cutting the
 * cost)].  The H heads form G consecutive groups of H/G; group g's
 * concatenated head outputs x_g (K = H/G * D values a query) are projected by
 * its own matrix W_g [d_g, K]:
 *   out[q, g*d_g + n] = sum_k x_g[q, k] * W_g[n, k]
 * (block-diagonal: G times cheaper than one dense projection of the same
 * width), in bf16 on the tensor cores with float32 accumulation, rounded to
 * bf16 once.
 *   o:   [Q, H, D] bf16 (e.g. csa_attend's out)
 *   w:   [G, d_g, K] bf16 (row n of W_g: output n's weights over K)
 *   out: [Q, G * d_g] bf16
 *   ws:  at least 256 bytes (status word: CSA_DEV_TIMEOUT on an expired wait).
 *        With at least csa_grouped_out_proj_ws_bytes(Q, G, d_g) bytes, a
 *        decode-sized call (Q <= 128) splits K over several CTAs a group and
 *        sums their float32 products in the workspace (in no fixed order: the
 *        bits of an output may differ between calls within float32 rounding)
 *        before the one bf16 rounding; with less it runs unsplit.
 * Requires H % G == 0, K a multiple of 64, d_g a positive multiple of 64;
 * other shapes return CSA_ERR_UNSUPPORTED. */
csa_status csa_grouped_out_proj(const void* o, int32_t Q, int32_t H, int32_t D, int32_t G, const void* w,
                                int32_t d_g, void* out, void* ws, size_t ws_bytes, csa_stream_t stream);

/* Workspace bytes csa_grouped_out_proj uses at most for these sizes: 256, plus
 * 4 * Q * G * d_g when Q <= 128 (the split products' float32 sums). */
size_t csa_grouped_out_proj_ws_bytes(int32_t Q, int32_t G, int32_t d_g);

/* Workspace */
typedef enum {
    CSA_OP_INDEX_TOPK = 1,
    CSA_OP_ATTEND = 2,
    CSA_OP_HCA_ATTEND = 3,
    CSA_OP_INDEX_TOPK_FP8 = 4,
    CSA_OP_INDEX_TOPK_FP4 = 5
} csa_op;

/* Bytes of workspace an operation needs for these sizes (0 on invalid input).
 * The first 256 bytes of every workspace hold the device status word; one
 * workspace may serve several operations in stream order. */
size_t csa_workspace_bytes(const csa_params* p, int32_t op, int32_t B, int32_t Q, int32_t H,
                           int32_t n_idx_heads, int64_t n_cap, int64_t n_win);

/* Zero the status word (asynchronous; call once after allocating a workspace). */
csa_status csa_workspace_init(void* ws, size_t ws_bytes, csa_stream_t stream);

/* Synchronise `stream`, read and clear the status word.  Returns CSA_OK, or
 * CSA_ERR_DEVICE with the CSA_DEV_* bits described by csa_last_error(). */
csa_status csa_check_status(void* ws, csa_stream_t stream);

/* Raw status bits of the last csa_check_status on this thread. */
uint32_t csa_last_device_bits(void);

/* Number of kernels this library has launched in this process (all
 * threads), for launch accounting in benchmarks. */
uint64_t csa_launch_count(void);

/* Test hook for failure detection (the pages have no counterpart; off by
 * default, process-wide).  While on, every launch of the tensor-core lightning
 * indexer (csa_index_score / csa_index_topk with bf16 keys of 128 dims, 64
 * heads, n_cap >= 128) has its TMA producer issue no copy at all, so the MMA
 * warps' bounded waits for the query and key tiles expire after 2 s of wall
 * time: the kernel sets CSA_DEV_TIMEOUT in the caller's status word, every
 * role leaves its loop (nothing is in flight), TMEM is freed, and the
 * context stays usable.  csa_check_status then reports CSA_ERR_DEVICE.  Scores
 * written under the hook are meaningless.  Pass 0 to turn it off. */
csa_status csa_test_withhold_indexer_loads(int32_t on);

const char* csa_status_string(csa_status s);
const char* csa_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA_B300_H */
