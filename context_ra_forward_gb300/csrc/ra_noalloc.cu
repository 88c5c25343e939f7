// ra_noalloc.cu — ra_backward_noalloc: the backward pass with library-owned scratch.
//
// ra_backward needs a device workspace (the per-row term D_i and the fp32 dQ
// accumulator) that the caller allocates.  Some callers cannot do that at the
// point where they run the backward: plug-ins inside a host framework that owns
// every device allocation and forbids allocating on its behalf, programs whose
// device memory is laid out once at start-up, and latency-critical loops where an
// allocation's implicit device synchronisation is not acceptable.  For them this
// file keeps a fixed scratch buffer in device memory, sized at build time, that
// every call reuses.
//
// The buffer is a file-scope __device__ array, so every GPU that loads the
// library holds kScratchBytes of it until the process exits.  In host code the
// array's name is only a host-side stand-in, so its device address is looked up
// (cudaGetSymbolAddress) once per device, with that device current, the first
// time this entry point runs on the device; that first call should therefore
// come before any stream capture.
#include <mutex>

#include "ra_common.cuh"
#include "ra_kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // RA_NOALLOC_SCRATCH_BYTES

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

ra_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return RA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RA_OK;
}

}  // namespace

extern "C" {

size_t ra_noalloc_scratch_bytes(void) { return kScratchBytes; }

ra_status ra_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dtype,
                              int32_t causal, const float* alibi_slopes, float softmax_scale,
                              int32_t N, ra_layout layout, void* stream) {
  // The arguments are checked exactly as ra_backward checks them, so an invalid
  // call gets the error ra_backward would give; only then is the (now bounded)
  // scratch requirement compared with the buffer.
  ra_status s = ra::backward_precheck(q, k, v, o, lse, dout, dq, dk, dv, B, H, S, D, dtype, alibi_slopes,
                                      softmax_scale, N, layout);
  if (s != RA_OK) return s;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  if (ra_backward_workspace_bytes(B, H, S, D) > kScratchBytes) return RA_ERR_WORKSPACE;
  void* scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != RA_OK) return s;
  // The backward's pre-pass writes every D_i and zeroes the dQ accumulator before
  // the main kernel reads them, so whatever an earlier call left in the buffer
  // does not matter.  Nothing here allocates.
  return ra_backward(q, k, v, o, lse, dout, dq, dk, dv, scratch, kScratchBytes, B, H, S, D, dtype,
                     causal, alibi_slopes, softmax_scale, N, layout, stream);
}

}  // extern "C"
