// k_attend_tc.cu -- tensor-core (tcgen05) core attention: not yet built.
#include "common.cuh"
#include "internal.h"

namespace csa {

bool attend_tc_supported(const Geometry&, int) { return false; }
int attend_tc_splits(const Geometry&, bool, int, int64_t) { return 1; }

cudaError_t launch_attend_tc(const Geometry&, const AttendPlan&, bool, const void*, int, int, int,
                             const int64_t*, const void*, int64_t, const int32_t*, const void*,
                             int64_t, const int64_t*, uint8_t*, uint32_t*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace csa
