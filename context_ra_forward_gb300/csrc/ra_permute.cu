// ra_permute.cu — original order <-> shard-major order, a bit-exact row gather.
//
// [ZZ] "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" §Zig Zag Ring
// Attention (interleaved assignment; "the index logic is slightly more involved")
// and [CP] "百万Token上下文训练的挑战与突破" §2.1 (contiguous split); the token-strided
// assignment is the one [ZZ] §Zig Zag prints ("GPU 0 gets tokens [0, 4, 8...]").
//
// Design: HBM-bound copy.  Every thread moves 16-byte chunks; consecutive threads
// write consecutive chunks of the output (coalesced stores), reading the matching
// chunks of the source row given by the closed-form map (coalesced within a row).
// Each thread keeps kUnroll loads in flight before storing, and both directions
// use streaming cache hints (data is touched once).  blockIdx.y walks (b, h).
#include "ra_common.cuh"
#include "ra_kernels.h"

namespace ra {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(int4* p, int4 v) {
  asm volatile("st.global.cs.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// 32-bit closed forms (the host checks S * chunks_per_row < 2^31).
struct Map32 {
  uint32_t c, h, N;
  int32_t layout;
  __device__ __forceinline__ uint32_t g(uint32_t p) const {
    if (layout == RA_LAYOUT_ZIGZAG) {
      const uint32_t r = p / c, u = p - r * c;
      return u < h ? r * h + u : (2 * N - 1 - r) * h + (u - h);
    }
    if (layout == RA_LAYOUT_STRIDED) {
      const uint32_t r = p / c, u = p - r * c;
      return u * N + r;
    }
    return p;
  }
  __device__ __forceinline__ uint32_t inv(uint32_t gp) const {
    if (layout == RA_LAYOUT_ZIGZAG) {
      const uint32_t k = gp / h, u = gp - k * h;
      return k < N ? k * c + u : (2 * N - 1 - k) * c + h + u;
    }
    if (layout == RA_LAYOUT_STRIDED) {
      const uint32_t u = gp / N, r = gp - u * N;
      return r * c + u;
    }
    return gp;
  }
};

template <int kLogCpr>  // log2 of 16-byte chunks per row
__global__ void __launch_bounds__(kThreads) permute_rows_kernel(const int4* __restrict__ x,
                                                                int4* __restrict__ y, uint32_t S,
                                                                Map32 m, int32_t inverse,
                                                                int64_t n_heads) {
  constexpr uint32_t kCpr = 1u << kLogCpr;
  const uint32_t per_head = S << kLogCpr;  // chunks in one (b, h) slice
  const uint32_t base = blockIdx.x * (uint32_t)(kThreads * kUnroll) + threadIdx.x;
  for (int64_t bh = blockIdx.y; bh < n_heads; bh += gridDim.y) {
    const int4* xs = x + bh * (int64_t)per_head;
    int4* ys = y + bh * (int64_t)per_head;
    int4 val[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t idx = base + u * kThreads;
      if (idx < per_head) {
        const uint32_t row = idx >> kLogCpr;
        const uint32_t src_row = inverse ? m.inv(row) : m.g(row);
        val[u] = ld_stream(xs + ((src_row << kLogCpr) | (idx & (kCpr - 1))));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t idx = base + u * kThreads;
      if (idx < per_head) st_stream(ys + idx, val[u]);
    }
  }
}

}  // namespace

cudaError_t launch_permute(const void* x, void* y, int64_t BH, int64_t S, int64_t row_bytes,
                           const SeqMap& sm, bool inverse, cudaStream_t st) {
  Map32 m;
  m.c = (uint32_t)sm.c;
  m.h = (uint32_t)sm.h;
  m.N = (uint32_t)sm.N;
  m.layout = sm.layout;
  const int64_t cpr = row_bytes / 16;
  const int64_t per_head = S * cpr;
  const int64_t per_block = kThreads * kUnroll;
  dim3 grid((unsigned)((per_head + per_block - 1) / per_block), (unsigned)(BH < 65535 ? BH : 65535));
  const int4* xi = static_cast<const int4*>(x);
  int4* yi = static_cast<int4*>(y);
  switch (cpr) {
    case 4:  permute_rows_kernel<2><<<grid, kThreads, 0, st>>>(xi, yi, (uint32_t)S, m, inverse, BH); note_launch(); break;
    case 8:  permute_rows_kernel<3><<<grid, kThreads, 0, st>>>(xi, yi, (uint32_t)S, m, inverse, BH); note_launch(); break;
    case 16: permute_rows_kernel<4><<<grid, kThreads, 0, st>>>(xi, yi, (uint32_t)S, m, inverse, BH); note_launch(); break;
    case 32: permute_rows_kernel<5><<<grid, kThreads, 0, st>>>(xi, yi, (uint32_t)S, m, inverse, BH); note_launch(); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ra
