// prefill_tc.cu -- tcgen05 causal prefill (bf16, d = 64).
#include "common.cuh"
#include "internal.h"

namespace gqa {

bool prefill_tc_supported(int, int, int) { return false; }

cudaError_t launch_prefill_tc(const void*, const void*, const void*, void*, int, int, int, const int32_t*, int, int,
                              int, int, float, unsigned*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace gqa
