// k_indexer_tc.cu -- tensor-core (tcgen05) lightning indexer: not yet built.
#include "common.cuh"
#include "internal.h"

namespace csa {

cudaError_t launch_indexer_tc(const Geometry&, const IndexTopkPlan&, const void*, const float*, int,
                              int, const void*, int64_t, int, int, const int64_t*, uint32_t*,
                              float*, cudaStream_t, bool* launched) {
    *launched = false;
    return cudaSuccess;
}

}  // namespace csa
