// tcgen05 grouped GEMM (tensor-core path) -- not built yet.
#include "common.cuh"

namespace moe {

bool tc_available() { return false; }

moe_status_t tc_qmm(const void*, int, const int32_t*, const int32_t*, int, int, int, int, int,
                    bool, const uint32_t*, const uint16_t*, const uint16_t*, int, void*, int,
                    cudaStream_t) {
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
