// ra_merge.cu — merge of two ring-step partial results through their log-sum-exp.
//
// [ZZ] "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" §Zig Zag Ring
// Attention: each shard's queries meet one K/V block per ring step; the partial
// results of the steps combine into exact attention.  For one query row with
// partials (O_a, LSE_a) and (O_b, LSE_b) over disjoint key sets:
//   LSE = log(e^LSE_a + e^LSE_b),  O = e^(LSE_a - LSE) O_a + e^(LSE_b - LSE) O_b,
// and two empty partials (LSE = -inf) merge to (O = 0, LSE = -inf).
//
// HBM-bound: one warp per row (D = 128: 32 lanes x 4 floats; D = 64: 16 lanes,
// two rows per warp), 16-byte loads and stores, grid-stride over rows.
#include "ra_common.cuh"
#include "ra_kernels.h"

namespace ra {

namespace {

template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(float* __restrict__ o_acc, float* __restrict__ lse_acc,
                                                        const float* __restrict__ o_t,
                                                        const float* __restrict__ lse_t, void* __restrict__ out,
                                                        int32_t out_dtype, int64_t rows) {
  constexpr int kLanesPerRow = D / 4;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t base = warp * kRowsPerWarp; base < rows; base += nwarps * kRowsPerWarp) {
    const int64_t row = base + lane / kLanesPerRow;
    if (row >= rows) continue;
    const int col = 4 * (lane % kLanesPerRow);
    const float la = lse_acc[row], lb = lse_t[row];
    const float mx = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f, l = -INFINITY;
    if (mx != -INFINITY) {
      const float ea = exp2f((la - mx) * kLog2e), eb = exp2f((lb - mx) * kLog2e);
      const float sum = ea + eb;
      wa = ea / sum;
      wb = eb / sum;
      l = mx + log2f(sum) * kLn2;
    }
    const float4 a = *reinterpret_cast<const float4*>(o_acc + row * D + col);
    const float4 b = *reinterpret_cast<const float4*>(o_t + row * D + col);
    // an empty side contributes nothing (its O is zero, never scaled NaN)
    float4 r;
    r.x = (wa != 0.f ? wa * a.x : 0.f) + (wb != 0.f ? wb * b.x : 0.f);
    r.y = (wa != 0.f ? wa * a.y : 0.f) + (wb != 0.f ? wb * b.y : 0.f);
    r.z = (wa != 0.f ? wa * a.z : 0.f) + (wb != 0.f ? wb * b.z : 0.f);
    r.w = (wa != 0.f ? wa * a.w : 0.f) + (wb != 0.f ? wb * b.w : 0.f);
    *reinterpret_cast<float4*>(o_acc + row * D + col) = r;
    if (lane % kLanesPerRow == 0) lse_acc[row] = l;
    if (out != nullptr) {
      if (out_dtype == RA_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + row * D + col) = r;
      } else {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(r.x, r.y), p1 = __floats2bfloat162_rn(r.z, r.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&p0);
        u.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + row * D + col) = u;
      }
    }
  }
}

}  // namespace

cudaError_t launch_lse_merge(float* o_acc, float* lse_acc, const float* o_t, const float* lse_t, void* out,
                             int32_t out_dtype, int64_t rows, int64_t D, cudaStream_t st) {
  const int64_t rows_per_block = 8 * (D == 64 ? 2 : 1);
  int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (D == 64)
    lse_merge_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(o_acc, lse_acc, o_t, lse_t, out, out_dtype, rows);
  else
    lse_merge_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(o_acc, lse_acc, o_t, lse_t, out, out_dtype, rows);
  note_launch();
  return cudaGetLastError();
}

}  // namespace ra
