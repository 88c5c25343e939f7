// ra_bwd_tc.cu — tcgen05 tensor-core backward (bf16, D = 128).
#include "ra_common.cuh"
#include "ra_kernels.h"

namespace ra {

bool bwd_tc_supported(int64_t, int64_t, int32_t) { return false; }

cudaError_t launch_bwd_tc(const AttnArgs&, const float*, const void*, const float*, float*, void*,
                          void*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ra
