// csa_noalloc.cu -- csa_index_topk_noalloc: the indexer + top-k step for
// callers that cannot allocate device memory.
//
// Such callers (a plug-in whose host framework owns all device memory, or a
// latency-critical path that cannot risk the device-wide synchronisation an
// allocation may cause) still pass their inputs and outputs; the intermediate
// indexer scores live in the file-scope scratch array below instead of a
// caller-provided workspace.  The scratch is a fixed 16 MiB of float32 scores
// behind a 256-byte status header, held by every device that loads the library
// until the process exits.  All calls share it, so calls that overlap on the
// GPU race; the status header is cleared at the start of every call and the
// scores are fully rewritten before they are read.
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr size_t kNoallocHeader = kStatusWordBytes;
constexpr size_t kNoallocScratchBytes = kNoallocHeader + (size_t)CSA_NOALLOC_MAX_SCORES * sizeof(float);

// Host code must not use this name as an address: it is a host-side stand-in.
// The device address comes from cudaGetSymbolAddress on the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch on the current device.  It is looked up on
// every call rather than cached: the lookup is a host-side table read once
// the library's module is loaded on the device, and a cached address would go
// stale if the device's primary context were reset and the module reloaded
// elsewhere.
static csa_status scratch_address(void** out) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        char msg[160];
        snprintf(msg, sizeof(msg), "csa_index_topk_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return set_error(CSA_ERR_CUDA, msg);
    }
    *out = p;
    return CSA_OK;
}

}  // namespace csa

using namespace csa;

extern "C" csa_status csa_index_topk_noalloc(const csa_params* p, const void* q_idx,
                                             const float* w_idx, int32_t n_idx_heads,
                                             int32_t idx_dim, const void* keys, int64_t n_cap,
                                             int32_t B, int32_t Q, const int64_t* q_pos,
                                             int32_t* topk_idx, float* topk_score,
                                             uint32_t* status, csa_stream_t stream) {
    if (n_cap < 0 || Q < 0) return set_error(CSA_ERR_INVALID_ARG, "csa_index_topk_noalloc: negative size");
    const int64_t ld = (n_cap + 127) / 128 * 128;
    if ((int64_t)Q * ld > (int64_t)CSA_NOALLOC_MAX_SCORES) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "csa_index_topk_noalloc: Q * ceil128(n_cap) = %lld scores exceed the static "
                 "scratch of %d; use csa_index_topk with a workspace",
                 (long long)Q * ld, CSA_NOALLOC_MAX_SCORES);
        return set_error(CSA_ERR_INVALID_ARG, msg);
    }
    if (status && ((uintptr_t)status & 3u))
        return set_error(CSA_ERR_INVALID_ARG, "csa_index_topk_noalloc: status is not 4-byte aligned");
    // every check csa_index_score / csa_topk_select apply, made before anything is launched
    if (!p || csa_workspace_bytes(p, CSA_OP_INDEX_TOPK, B > 0 ? B : 1, Q, 1, n_idx_heads, n_cap, 0) == 0)
        return set_error(CSA_ERR_INVALID_ARG, "csa_index_topk_noalloc: invalid params or sizes");
    if (p->topk < 1 || p->topk > 4096)
        return set_error(CSA_ERR_INVALID_ARG, "csa_index_topk_noalloc: topk not in [1, 4096]");
    if ((idx_dim != 64 && idx_dim != 128) || n_idx_heads < 1 || n_idx_heads > 64)
        return set_error(CSA_ERR_UNSUPPORTED, "csa_index_topk_noalloc: idx_dim 64/128, 1..64 heads");
    if (B < 1 || Q % B != 0)
        return set_error(CSA_ERR_INVALID_ARG, "csa_index_topk_noalloc: Q must be a multiple of B");
    if (Q == 0) return CSA_OK;
    if (topk_chunk(n_cap, Q, p->topk) == 0)
        return set_error(CSA_ERR_UNSUPPORTED,
                         "csa_index_topk_noalloc: the top-k selection of these sizes does not fit in shared memory");
    const void* ptrs[] = {q_idx, w_idx, q_pos, topk_idx};
    for (const void* ptr : ptrs)
        if (!ptr || ((uintptr_t)ptr & 15u))
            return set_error(CSA_ERR_INVALID_ARG, "csa_index_topk_noalloc: NULL or misaligned pointer");
    if ((n_cap > 0 && (!keys || ((uintptr_t)keys & 15u))) || ((uintptr_t)topk_score & 15u))
        return set_error(CSA_ERR_INVALID_ARG, "csa_index_topk_noalloc: NULL or misaligned pointer");
    void* scratch = nullptr;
    csa_status s = scratch_address(&scratch);
    if (s != CSA_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* base = reinterpret_cast<uint8_t*>(scratch);
    float* scores = reinterpret_cast<float*>(base + kNoallocHeader);
    cudaError_t e = cudaMemsetAsync(base, 0, kNoallocHeader, st);  // status word starts at zero
    if (e != cudaSuccess) return set_error(CSA_ERR_CUDA, "csa_index_topk_noalloc: clearing the status word failed");
    s = csa_index_score(p, q_idx, w_idx, n_idx_heads, idx_dim, keys, n_cap, B, Q, q_pos, scores, ld,
                        base, kNoallocHeader, stream);
    if (s != CSA_OK) return s;
    s = csa_topk_select(p, scores, ld, n_cap, Q, q_pos, topk_idx, topk_score, stream);
    if (s != CSA_OK) return s;
    if (status) {
        e = cudaMemcpyAsync(status, base, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return set_error(CSA_ERR_CUDA, "csa_index_topk_noalloc: status copy failed");
    }
    return CSA_OK;
}
