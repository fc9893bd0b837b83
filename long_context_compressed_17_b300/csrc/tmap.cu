// tmap.cu -- TMA tensor maps (host side).  The driver entry point is fetched
// through the runtime once, so the library does not link libcuda directly.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace csa {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor of `rank` dims (dims[0] innermost), 128-byte swizzled boxes (or,
// linear, boxes stored row after row), zero fill outside the tensor.  Returns
// false if the map cannot be built.
static bool make_tmap(CUtensorMapDataType dt, CUtensorMap* map, const void* base, int rank,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      bool linear = false) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bd[5], es[5];
    for (int i = 0; i < rank; i++) {
        gd[i] = dims[i];
        bd[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides_bytes[i];
    }
    CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void*>(base), gd,
                    gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    linear ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box) {
    return make_tmap(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, base, rank, dims, strides_bytes, box);
}

// The same for a tensor of bytes (E4M3 codes).
bool make_tmap_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box) {
    return make_tmap(CU_TENSOR_MAP_DATA_TYPE_UINT8, map, base, rank, dims, strides_bytes, box);
}

// Bytes, boxes stored linearly (packed FP4 key tiles, copied as they are).
bool make_tmap_u8_linear(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides_bytes, const uint32_t* box) {
    return make_tmap(CU_TENSOR_MAP_DATA_TYPE_UINT8, map, base, rank, dims, strides_bytes, box, true);
}

}  // namespace csa
