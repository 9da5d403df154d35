// Stages 4 and 6 on the tensor cores (tcgen05): not yet enabled.
#include "mmq.cuh"

namespace moe {

bool mmq_tc_supported(int, bool, int, int) { return false; }

int launch_mmq_tc(int, bool, const uint8_t*, size_t, const int32_t*, const int32_t*, const int32_t*,
                  int, const int8_t*, const uint16_t*, int, int, int, float*, uint8_t*,
                  const WsLayout&, cudaStream_t) {
    return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
