// ra_kernels.h — launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ra_common.cuh"

namespace ra {

struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  int64_t B, H, S, D;
  int32_t dtype;
  int32_t causal;
  const float* slopes;  // device [H] or nullptr
  float scale;          // resolved softmax scale (> 0)
  SeqMap map;
  int32_t* status;      // device status word
  int32_t t_begin;      // ring steps [t_begin, t_end) are visited (all: 0, N)
  int32_t t_end;
  float* o_f32;         // forward: when set, O goes here as fp32 (a ring-step partial)
  float qk_scale;       // e4m3 forward: product of the Q and K scales (1 otherwise)
  float v_scale;        // e4m3 forward: V scale (1 otherwise)
};

// ra_api.cu — counts every kernel launch the library makes (host side).
void note_launch();
// ra_api.cu — every check ra_backward makes before it looks at its workspace, in
// the same order (sizes, dtype, scale, pointers, alignment): RA_OK or the error.
ra_status backward_precheck(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S,
                            int64_t D, ra_dtype dt, const float* slopes, float scale, int32_t N,
                            ra_layout layout);

// ra_permute.cu
cudaError_t launch_permute(const void* x, void* y, int64_t BH, int64_t S, int64_t row_bytes,
                           const SeqMap& m, bool inverse, cudaStream_t st);

// ra_permute.cu — the same map with a rotary position embedding applied on the way.
// F_i = theta_i / (2 pi) as a 64-bit binary fraction (turns per position), i < D/2.
struct RopeTurns {
  uint64_t f[128];
};
// inverse = false: y[slot] = R(pos0 + g(slot)) x[g(slot)]   (original -> shard-major)
// inverse = true:  y[g] = R(pos0 + g)^T x[inv(g)]            (shard-major -> original)
cudaError_t launch_rope_permute(const void* x, void* y, int64_t B, int64_t H, int64_t S, int64_t D,
                                int32_t dtype, const SeqMap& m, bool inverse, int64_t pos0,
                                const RopeTurns& turns, cudaStream_t st);

// ra_simt.cu — CUDA-core kernels (exact fp32 arithmetic)
cudaError_t launch_fwd_simt(const AttnArgs& a, void* o, float* lse, cudaStream_t st);
// D_i = dO_i . O_i into dvec; also zeroes dq_acc ([B,H,S,D] fp32) when it is not null.
cudaError_t launch_bwd_rowdot(const AttnArgs& a, const void* o, const void* dout, float* dvec,
                              float* dq_acc, cudaStream_t st);
cudaError_t launch_bwd_simt(const AttnArgs& a, const float* lse, const void* dout,
                            const float* dvec, void* dq, void* dk, void* dv, cudaStream_t st);

// ra_fwd_tc.cu — tcgen05 tensor-core forward (bf16 or e4m3, D = 128)
bool fwd_tc_supported(int64_t S, int64_t D, int32_t dtype);
cudaError_t launch_fwd_tc(const AttnArgs& a, void* o, float* lse, cudaStream_t st);

// ra_bwd_tc.cu — tcgen05 tensor-core backward (bf16, D = 128)
bool bwd_tc_supported(int64_t S, int64_t D, int32_t dtype, const SeqMap& m);
cudaError_t launch_bwd_tc(const AttnArgs& a, const float* lse, const void* dout,
                          const float* dvec, float* dq_acc, void* dq, void* dk, void* dv,
                          cudaStream_t st);

// ra_merge.cu — (o_acc, lse_acc) <- LSE merge with (o_t, lse_t); optional converted copy
cudaError_t launch_lse_merge(float* o_acc, float* lse_acc, const float* o_t, const float* lse_t, void* out,
                             int32_t out_dtype, int64_t rows, int64_t D, cudaStream_t st);

// ra_debug.cu
cudaError_t launch_debug_wait(int32_t limit_us, int32_t* status, cudaStream_t st);

}  // namespace ra
