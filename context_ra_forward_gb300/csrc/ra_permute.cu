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
//
// The same map with a rotary position embedding applied on the way (a fused RoPE
// prologue for Q and K, and its transpose for their gradients): [LC] "超长上下文技术"
// §2.1.3 RoPE.  Feature i and feature i + D/2 of a row at position t are rotated
// by the angle t * theta_i, theta_i = 1 / base^(2i/D).
//
// Angles: the fp32 product t * theta_i is off by up to ulp(2^18) / 2 = 2^-6 rad at
// the positions of a 256K-token sequence, so the angle is reduced exactly instead.
// The host stores theta_i / (2 pi) as a 64-bit binary fraction F_i (turns per
// position); the top 32 bits of t * F_i mod 2^64 are the angle's fractional turn
// (two 32-bit integer multiplies), which sincospif evaluates as a signed fraction
// of a half-turn.  Absolute error of cos / sin: a few 1e-7.
#include <math.h>

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

// ---------------------------------------------------------------------------
// Fused RoPE + permute.  One warp per output row index (b, o), all H heads: the
// angles of a position are evaluated once and reused for every head.  A lane owns
// kE consecutive pairs (i, i + D/2); the two half-warps take alternate heads, so
// each head row moves as two coalesced 16-lane accesses (first and second half).
// ---------------------------------------------------------------------------
constexpr int kRopeThreads = 256;
constexpr int kRopeHeads = 8;  // heads in flight per half-warp (16 per warp)

template <int kBytes> struct VecT;
template <> struct VecT<4> { using type = unsigned int; };
template <> struct VecT<8> { using type = uint2; };
template <> struct VecT<16> { using type = uint4; };

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float get(const float* p, int i) { return p[i]; }
  static __device__ __forceinline__ void put(float* p, int i, float v) { p[i] = v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float get(const __nv_bfloat16* p, int i) { return __bfloat162float(p[i]); }
  static __device__ __forceinline__ void put(__nv_bfloat16* p, int i, float v) { p[i] = __float2bfloat16_rn(v); }
};

template <typename T, int kE> struct Lanes {
  using V = typename VecT<kE * (int)sizeof(T)>::type;
  union U {
    V v;
    T e[kE];
  };
};

template <typename T, int kD>
__global__ void __launch_bounds__(kRopeThreads) rope_rows_kernel(const T* __restrict__ x, T* __restrict__ y,
                                                                 int64_t B, int64_t H, uint32_t S, Map32 m,
                                                                 int32_t inverse, uint32_t pos0,
                                                                 const __grid_constant__ RopeTurns turns) {
  constexpr int kE = kD / 32;  // pairs per lane
  constexpr int kHalfE = kE / 2;  // pairs whose angle this lane evaluates (its partner lane the rest)
  using L = Lanes<T, kE>;
  using V = typename L::V;
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 4, li = lane & 15;
  uint32_t flo[kHalfE], fhi[kHalfE];
#pragma unroll
  for (int j = 0; j < kHalfE; ++j) {
    const uint64_t f = turns.f[li * kE + sub * kHalfE + j];
    flo[j] = (uint32_t)f;
    fhi[j] = (uint32_t)(f >> 32);
  }
  const int64_t head_stride = (int64_t)S * kD;
  const uint32_t nwarps = (gridDim.x * kRopeThreads) >> 5;
  const uint32_t warp0 = (blockIdx.x * kRopeThreads + threadIdx.x) >> 5;
  for (int64_t b = 0; b < B; ++b) {
    const T* xb = x + b * H * head_stride;
    T* yb = y + b * H * head_stride;
    for (uint32_t o = warp0; o < S; o += nwarps) {
      const uint32_t gpos = inverse ? o : m.g(o);      // position of the row (original index)
      const uint32_t src = inverse ? m.inv(o) : gpos;  // source row in x
      const uint32_t t = pos0 + gpos;
      float c[kE], sn[kE];
      for (int64_t h0 = 0; h0 < H; h0 += 2 * kRopeHeads) {
        typename L::U a[kRopeHeads], z[kRopeHeads];
#pragma unroll
        for (int j = 0; j < kRopeHeads; ++j) {
          const int64_t h = h0 + sub + 2 * j;
          if (h < H) {
            const V* row = reinterpret_cast<const V*>(xb + h * head_stride + (int64_t)src * kD);
            a[j].v = __ldcs(row + li);
            z[j].v = __ldcs(row + 16 + li);
          }
        }
        if (h0 == 0) {
          // fractional turn of t * theta_i: bits 32..63 of t * F_i mod 2^64; each
          // lane evaluates half of its pairs' angles and swaps with lane ^ 16
          float cm[kHalfE], sm[kHalfE];
#pragma unroll
          for (int j = 0; j < kHalfE; ++j) {
            const uint32_t turn = t * fhi[j] + __umulhi(t, flo[j]);
            sincospif((float)(int32_t)turn * 0x1p-31f, &sm[j], &cm[j]);
            if (inverse) sm[j] = -sm[j];
          }
#pragma unroll
          for (int j = 0; j < kHalfE; ++j) {
            const float co = __shfl_xor_sync(0xffffffffu, cm[j], 16);
            const float so = __shfl_xor_sync(0xffffffffu, sm[j], 16);
            c[j] = sub ? co : cm[j];
            sn[j] = sub ? so : sm[j];
            c[kHalfE + j] = sub ? cm[j] : co;
            sn[kHalfE + j] = sub ? sm[j] : so;
          }
        }
#pragma unroll
        for (int j = 0; j < kRopeHeads; ++j) {
          const int64_t h = h0 + sub + 2 * j;
          if (h < H) {
            typename L::U ra, rz;
#pragma unroll
            for (int e = 0; e < kE; ++e) {
              const float x1 = Elem<T>::get(a[j].e, e), x2 = Elem<T>::get(z[j].e, e);
              Elem<T>::put(ra.e, e, x1 * c[e] - x2 * sn[e]);
              Elem<T>::put(rz.e, e, x1 * sn[e] + x2 * c[e]);
            }
            V* row = reinterpret_cast<V*>(yb + h * head_stride + (int64_t)o * kD);
            __stcs(row + li, ra.v);
            __stcs(row + 16 + li, rz.v);
          }
        }
      }
    }
  }
}

// One wave of resident blocks (occupancy of this instantiation), or fewer when the
// rows run out; the warps stride over the remaining rows.
template <typename T, int kD>
int rope_grid(int64_t units) {
  static int per_dev[64] = {};  // resident blocks on the whole device, per device
  int dev = 0;
  cudaGetDevice(&dev);
  int cap = (dev >= 0 && dev < 64) ? per_dev[dev] : 0;
  if (cap == 0) {
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rope_rows_kernel<T, kD>, kRopeThreads, 0) !=
            cudaSuccess ||
        per_sm <= 0)
      per_sm = 1;
    cap = sms * per_sm;
    if (dev >= 0 && dev < 64) per_dev[dev] = cap;
  }
  constexpr int kWarps = kRopeThreads / 32;
  const int64_t need = (units + kWarps - 1) / kWarps;  // one row index per warp
  return (int)(need < cap ? need : cap);
}

}  // namespace

cudaError_t launch_rope_permute(const void* x, void* y, int64_t B, int64_t H, int64_t S, int64_t D,
                                int32_t dtype, const SeqMap& sm, bool inverse, int64_t pos0,
                                const RopeTurns& turns, cudaStream_t st) {
  Map32 m;
  m.c = (uint32_t)sm.c;
  m.h = (uint32_t)sm.h;
  m.N = (uint32_t)sm.N;
  m.layout = sm.layout;
  const int32_t inv = inverse ? 1 : 0;
  const uint32_t p0 = (uint32_t)pos0, s32 = (uint32_t)S;
  if (dtype == RA_BF16 && D == 128)
    rope_rows_kernel<__nv_bfloat16, 128><<<rope_grid<__nv_bfloat16, 128>(S), kRopeThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), B, H, s32, m, inv, p0, turns);
  else if (dtype == RA_BF16 && D == 64)
    rope_rows_kernel<__nv_bfloat16, 64><<<rope_grid<__nv_bfloat16, 64>(S), kRopeThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), B, H, s32, m, inv, p0, turns);
  else if (dtype == RA_F32 && D == 128)
    rope_rows_kernel<float, 128><<<rope_grid<float, 128>(S), kRopeThreads, 0, st>>>(static_cast<const float*>(x),
                                                                static_cast<float*>(y), B, H, s32, m, inv, p0, turns);
  else if (dtype == RA_F32 && D == 64)
    rope_rows_kernel<float, 64><<<rope_grid<float, 64>(S), kRopeThreads, 0, st>>>(static_cast<const float*>(x),
                                                               static_cast<float*>(y), B, H, s32, m, inv, p0, turns);
  else
    return cudaErrorInvalidValue;
  note_launch();
  return cudaGetLastError();
}

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
