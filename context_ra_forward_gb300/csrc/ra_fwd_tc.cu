// ra_fwd_tc.cu — tcgen05 tensor-core forward (bf16, D = 128).
#include "ra_common.cuh"
#include "ra_kernels.h"

namespace ra {

bool fwd_tc_supported(int64_t, int64_t, int32_t) { return false; }

cudaError_t launch_fwd_tc(const AttnArgs&, void*, float*, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ra
