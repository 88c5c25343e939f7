// ra_simt.cu — CUDA-core kernels: the exact-fp32 forward, and a backward that
// serves fp32 and every shape the tensor-core kernels do not take.
//
// Pages cited:
//   [ZZ] "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" §Zig Zag Ring
//        Attention: the queries of shard r meet, at ring step t, the K/V of shard
//        (r - t) mod N, until every Q has met every K/V block.
//   [LC] "超长上下文技术" survey §2.1.2 (scale 1/sqrt(head dim), ALiBi bias
//        -|i-j| * slope after scaling), §3.1.2 (running max m and sum l per row,
//        output rescaled when m grows; recompute in backward).
//
// Layout: four lanes ("a quad") own one row; lane ql holds the 16-byte chunks
// ql, ql+4, ql+8, ... of the D-wide row, so a quad's four loads from a staged
// K/V row hit four consecutive 16-byte chunks (no bank conflict) and all rows of
// a warp read the same staged row (broadcast).  Dot products are reduced over the
// quad with two xor-shuffles, which leaves the same value in all four lanes.
// K/V (forward, dQ) or Q/dO (dK/dV) are staged 64 rows at a time as fp32.
#include <math.h>

#include "ra_common.cuh"
#include "ra_kernels.h"

namespace ra {

namespace {

constexpr int kRowsPerBlock = 32;
constexpr int kThreads = 128;
constexpr int kTile = 64;

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  float4 f;
  f.x = __uint_as_float(u.x << 16);
  f.y = __uint_as_float(u.x & 0xffff0000u);
  f.z = __uint_as_float(u.y << 16);
  f.w = __uint_as_float(u.y & 0xffff0000u);
  return f;
}
template <typename T>
__device__ __forceinline__ void store4(T* p, float4 f);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 f) {
  *reinterpret_cast<float4*>(p) = f;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 f) {
  __nv_bfloat162 a = __floats2bfloat162_rn(f.x, f.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(f.z, f.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// Stage rows [r0, r0 + kTile) of a [S, D] slice into fp32 shared memory
// (rows past S are zero) and record their global positions (-1 past S).
template <typename T, int D>
__device__ __forceinline__ void stage_rows(float* dst, const T* src, int64_t r0, int64_t S) {
  constexpr int kChunks = kTile * D / 4;
  for (int idx = threadIdx.x; idx < kChunks; idx += kThreads) {
    const int row = idx / (D / 4), col = (idx % (D / 4)) * 4;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 + row < S) f = load4<T>(src + (r0 + row) * D + col);
    *reinterpret_cast<float4*>(dst + row * D + col) = f;
  }
}

// First and one-past-last kv tile (kTile rows, aligned to the buffer) whose first
// row lies in shard s: the tile-level ring order visits those with shard s.
__device__ __forceinline__ void shard_tiles(const SeqMap& m, int32_t s, int64_t& t0, int64_t& t1) {
  t0 = (s * m.c + kTile - 1) / kTile;
  t1 = ((s + 1) * m.c + kTile - 1) / kTile;
}

// ----------------------------------------------------------------------------
// Forward: one quad per query row, 32 rows per block.
// ----------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(AttnArgs a, T* __restrict__ o,
                                                            float* __restrict__ lse) {
  constexpr int kC = D / 16;  // float4 chunks per lane
  extern __shared__ __align__(16) float smem[];
  float* Ks = smem;
  float* Vs = smem + kTile * D;
  int64_t* gk = reinterpret_cast<int64_t*>(smem + 2 * kTile * D);

  const SeqMap& m = a.map;
  const int64_t S = a.S;
  const int64_t bh = blockIdx.y;
  const int hh = (int)(bh % a.H);
  const T* q = static_cast<const T*>(a.q) + bh * S * D;
  const T* k = static_cast<const T*>(a.k) + bh * S * D;
  const T* v = static_cast<const T*>(a.v) + bh * S * D;

  const int r = threadIdx.x >> 2, ql = threadIdx.x & 3;
  const int64_t p_lo = (int64_t)blockIdx.x * kRowsPerBlock;
  const int64_t p_hi = (p_lo + kRowsPerBlock < S) ? p_lo + kRowsPerBlock : S;
  const int64_t pi = p_lo + r;
  const bool row_ok = pi < S;
  const int64_t gi = row_ok ? m.g(pi) : 0;
  const float c2 = a.scale * kLog2e;  // scores are kept in the log2 domain
  const float slope2 = a.slopes ? a.slopes[hh] * kLog2e : 0.f;

  float qf[4 * kC], acc[4 * kC];
#pragma unroll
  for (int t = 0; t < kC; ++t) {
    float4 f = row_ok ? load4<T>(q + pi * D + 4 * (ql + 4 * t)) : make_float4(0.f, 0.f, 0.f, 0.f);
    qf[4 * t + 0] = f.x * c2;
    qf[4 * t + 1] = f.y * c2;
    qf[4 * t + 2] = f.z * c2;
    qf[4 * t + 3] = f.w * c2;
    acc[4 * t + 0] = acc[4 * t + 1] = acc[4 * t + 2] = acc[4 * t + 3] = 0.f;
  }
  float mrun = -INFINITY, l = 0.f;

  int64_t qgmin, qgmax;
  m.grange(p_lo, p_hi, qgmin, qgmax);
  const int32_t r0 = m.shard(p_lo);

  for (int32_t t = a.t_begin; t < a.t_end; ++t) {
    const int32_t s = (r0 - t + m.N) % m.N;  // ring step t meets shard (r0 - t) mod N
    int64_t t0, t1;
    shard_tiles(m, s, t0, t1);
    for (int64_t ti = t0; ti < t1; ++ti) {
      const int64_t k0 = ti * kTile;
      const int64_t k1 = (k0 + kTile < S) ? k0 + kTile : S;
      if (a.causal) {
        int64_t kgmin, kgmax;
        m.grange(k0, k1, kgmin, kgmax);
        if (kgmin > qgmax) continue;  // every key of the tile is in every row's future
      }
      __syncthreads();
      stage_rows<T, D>(Ks, k, k0, S);
      stage_rows<T, D>(Vs, v, k0, S);
      for (int j = threadIdx.x; j < kTile; j += kThreads) gk[j] = (k0 + j < S) ? m.g(k0 + j) : -1;
      __syncthreads();

#pragma unroll 1
      for (int jc = 0; jc < kTile; jc += 16) {
        float sc[16];
        float cmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float* kr = Ks + (jc + u) * D;
          float d = 0.f;
#pragma unroll
          for (int t = 0; t < kC; ++t) {
            const float4 kv = *reinterpret_cast<const float4*>(kr + 4 * (ql + 4 * t));
            d = fmaf(qf[4 * t + 0], kv.x, d);
            d = fmaf(qf[4 * t + 1], kv.y, d);
            d = fmaf(qf[4 * t + 2], kv.z, d);
            d = fmaf(qf[4 * t + 3], kv.w, d);
          }
          d = quad_sum(d);
          const int64_t gj = gk[jc + u];
          const bool vis = row_ok && gj >= 0 && (!a.causal || gj <= gi);
          if (a.slopes) d -= slope2 * (float)(gi > gj ? gi - gj : gj - gi);
          sc[u] = vis ? d : -INFINITY;
          cmax = fmaxf(cmax, sc[u]);
        }
        const float m_new = fmaxf(mrun, cmax);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = mrun == -INFINITY ? 0.f : exp2f(mrun - m_use);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < 4 * kC; ++e) acc[e] *= alpha;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float p = exp2f(sc[u] - m_use);
          l += p;
          const float* vr = Vs + (jc + u) * D;
#pragma unroll
          for (int t = 0; t < kC; ++t) {
            const float4 vv = *reinterpret_cast<const float4*>(vr + 4 * (ql + 4 * t));
            acc[4 * t + 0] = fmaf(p, vv.x, acc[4 * t + 0]);
            acc[4 * t + 1] = fmaf(p, vv.y, acc[4 * t + 1]);
            acc[4 * t + 2] = fmaf(p, vv.z, acc[4 * t + 2]);
            acc[4 * t + 3] = fmaf(p, vv.w, acc[4 * t + 3]);
          }
        }
        mrun = m_new;
      }
    }
  }

  if (row_ok) {
    const float inv_l = l == 0.f ? 0.f : 1.f / l;  // only l == 0 means "no visible key"; NaN inputs keep l (and O) NaN
    T* orow = o + (bh * S + pi) * D;
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      const float4 f = make_float4(acc[4 * t] * inv_l, acc[4 * t + 1] * inv_l, acc[4 * t + 2] * inv_l,
                                   acc[4 * t + 3] * inv_l);
      if (a.o_f32 != nullptr)  // ring-step partial: fp32 rows
        store4<float>(a.o_f32 + (bh * S + pi) * D + 4 * (ql + 4 * t), f);
      else
        store4<T>(orow + 4 * (ql + 4 * t), f);
    }
    if (ql == 0) lse[bh * S + pi] = l != 0.f ? (mrun + log2f(l)) * kLn2 : -INFINITY;
  }
}

// ----------------------------------------------------------------------------
// Backward row term D_i = dO_i . O_i (fp32), one warp per row.
// ----------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const T* __restrict__ o,
                                                         const T* __restrict__ dout,
                                                         float* __restrict__ dvec,
                                                         float* __restrict__ dq_acc, int64_t rows) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  if (dq_acc != nullptr) {
    for (int d = lane * 4; d < D; d += 128)
      *reinterpret_cast<float4*>(dq_acc + row * D + d) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float s = 0.f;
  for (int d = lane * 2; d < D; d += 64) {
    s = fmaf(to_f32<T>(o[row * D + d]), to_f32<T>(dout[row * D + d]), s);
    s = fmaf(to_f32<T>(o[row * D + d + 1]), to_f32<T>(dout[row * D + d + 1]), s);
  }
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
  if (lane == 0) dvec[row] = s;
}

// ----------------------------------------------------------------------------
// Backward dK/dV: one quad per key row; query tiles visited in ring order (the
// K/V block of shard s meets, at step t, the queries of shard (s + t) mod N).
// ----------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_dkdv_simt_kernel(AttnArgs a,
                                                                 const float* __restrict__ lse,
                                                                 const T* __restrict__ dout,
                                                                 const float* __restrict__ dvec,
                                                                 T* __restrict__ dk,
                                                                 T* __restrict__ dv) {
  constexpr int kC = D / 16;
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;
  float* Os = smem + kTile * D;  // dO rows
  float* Ls = smem + 2 * kTile * D;
  float* Ds = Ls + kTile;
  int64_t* gq = reinterpret_cast<int64_t*>(Ds + kTile);

  const SeqMap& m = a.map;
  const int64_t S = a.S;
  const int64_t bh = blockIdx.y;
  const int hh = (int)(bh % a.H);
  const T* q = static_cast<const T*>(a.q) + bh * S * D;
  const T* k = static_cast<const T*>(a.k) + bh * S * D;
  const T* v = static_cast<const T*>(a.v) + bh * S * D;
  const T* go = dout + bh * S * D;

  const int r = threadIdx.x >> 2, ql = threadIdx.x & 3;
  const int64_t p_lo = (int64_t)blockIdx.x * kRowsPerBlock;
  const int64_t p_hi = (p_lo + kRowsPerBlock < S) ? p_lo + kRowsPerBlock : S;
  const int64_t pj = p_lo + r;
  const bool row_ok = pj < S;
  const int64_t gj = row_ok ? m.g(pj) : 0;
  const float slope = a.slopes ? a.slopes[hh] : 0.f;

  float kf[4 * kC], vf[4 * kC], dka[4 * kC], dva[4 * kC];
#pragma unroll
  for (int t = 0; t < kC; ++t) {
    const float4 kk = row_ok ? load4<T>(k + pj * D + 4 * (ql + 4 * t)) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 vv = row_ok ? load4<T>(v + pj * D + 4 * (ql + 4 * t)) : make_float4(0.f, 0.f, 0.f, 0.f);
    kf[4 * t] = kk.x; kf[4 * t + 1] = kk.y; kf[4 * t + 2] = kk.z; kf[4 * t + 3] = kk.w;
    vf[4 * t] = vv.x; vf[4 * t + 1] = vv.y; vf[4 * t + 2] = vv.z; vf[4 * t + 3] = vv.w;
#pragma unroll
    for (int e = 0; e < 4; ++e) dka[4 * t + e] = dva[4 * t + e] = 0.f;
  }

  int64_t kgmin, kgmax;
  m.grange(p_lo, p_hi, kgmin, kgmax);
  const int32_t s0 = m.shard(p_lo);

  for (int32_t t = 0; t < m.N; ++t) {
    const int32_t s = (s0 + t) % m.N;
    int64_t t0, t1;
    shard_tiles(m, s, t0, t1);
    for (int64_t ti = t0; ti < t1; ++ti) {
      const int64_t q0 = ti * kTile;
      const int64_t q1 = (q0 + kTile < S) ? q0 + kTile : S;
      if (a.causal) {
        int64_t qgmin, qgmax;
        m.grange(q0, q1, qgmin, qgmax);
        if (qgmax < kgmin) continue;  // these queries see none of the block's keys
      }
      __syncthreads();
      stage_rows<T, D>(Qs, q, q0, S);
      stage_rows<T, D>(Os, go, q0, S);
      for (int i = threadIdx.x; i < kTile; i += kThreads) {
        const bool ok = q0 + i < S;
        gq[i] = ok ? m.g(q0 + i) : -1;
        Ls[i] = ok ? lse[bh * S + q0 + i] : -INFINITY;
        Ds[i] = ok ? dvec[bh * S + q0 + i] : 0.f;
      }
      __syncthreads();
#pragma unroll 1
      for (int i = 0; i < kTile; ++i) {
        const float* qr = Qs + i * D;
        const float* dr = Os + i * D;
        float sd = 0.f, dp = 0.f;
#pragma unroll
        for (int t = 0; t < kC; ++t) {
          const float4 qq = *reinterpret_cast<const float4*>(qr + 4 * (ql + 4 * t));
          const float4 dd = *reinterpret_cast<const float4*>(dr + 4 * (ql + 4 * t));
          sd = fmaf(qq.x, kf[4 * t], sd); sd = fmaf(qq.y, kf[4 * t + 1], sd);
          sd = fmaf(qq.z, kf[4 * t + 2], sd); sd = fmaf(qq.w, kf[4 * t + 3], sd);
          dp = fmaf(dd.x, vf[4 * t], dp); dp = fmaf(dd.y, vf[4 * t + 1], dp);
          dp = fmaf(dd.z, vf[4 * t + 2], dp); dp = fmaf(dd.w, vf[4 * t + 3], dp);
        }
        sd = quad_sum(sd);
        dp = quad_sum(dp);
        const int64_t gi = gq[i];
        const float li = Ls[i];
        const bool vis = row_ok && gi >= 0 && (!a.causal || gj <= gi) && li != -INFINITY;
        float sc = sd * a.scale;
        if (a.slopes) sc -= slope * (float)(gi > gj ? gi - gj : gj - gi);
        const float p = vis ? exp2f((sc - li) * kLog2e) : 0.f;
        const float ds = p * (dp - Ds[i]) * a.scale;
#pragma unroll
        for (int t = 0; t < kC; ++t) {
          const float4 qq = *reinterpret_cast<const float4*>(qr + 4 * (ql + 4 * t));
          const float4 dd = *reinterpret_cast<const float4*>(dr + 4 * (ql + 4 * t));
          dva[4 * t] = fmaf(p, dd.x, dva[4 * t]); dva[4 * t + 1] = fmaf(p, dd.y, dva[4 * t + 1]);
          dva[4 * t + 2] = fmaf(p, dd.z, dva[4 * t + 2]); dva[4 * t + 3] = fmaf(p, dd.w, dva[4 * t + 3]);
          dka[4 * t] = fmaf(ds, qq.x, dka[4 * t]); dka[4 * t + 1] = fmaf(ds, qq.y, dka[4 * t + 1]);
          dka[4 * t + 2] = fmaf(ds, qq.z, dka[4 * t + 2]); dka[4 * t + 3] = fmaf(ds, qq.w, dka[4 * t + 3]);
        }
      }
    }
  }
  if (row_ok) {
    T* dkr = dk + (bh * S + pj) * D;
    T* dvr = dv + (bh * S + pj) * D;
#pragma unroll
    for (int t = 0; t < kC; ++t) {
      store4<T>(dkr + 4 * (ql + 4 * t), make_float4(dka[4 * t], dka[4 * t + 1], dka[4 * t + 2], dka[4 * t + 3]));
      store4<T>(dvr + 4 * (ql + 4 * t), make_float4(dva[4 * t], dva[4 * t + 1], dva[4 * t + 2], dva[4 * t + 3]));
    }
  }
}

// ----------------------------------------------------------------------------
// Backward dQ: one quad per query row, key tiles in the forward's ring order.
// ----------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_dq_simt_kernel(AttnArgs a,
                                                               const float* __restrict__ lse,
                                                               const T* __restrict__ dout,
                                                               const float* __restrict__ dvec,
                                                               T* __restrict__ dq) {
  constexpr int kC = D / 16;
  extern __shared__ __align__(16) float smem[];
  float* Ks = smem;
  float* Vs = smem + kTile * D;
  int64_t* gk = reinterpret_cast<int64_t*>(smem + 2 * kTile * D);

  const SeqMap& m = a.map;
  const int64_t S = a.S;
  const int64_t bh = blockIdx.y;
  const int hh = (int)(bh % a.H);
  const T* q = static_cast<const T*>(a.q) + bh * S * D;
  const T* k = static_cast<const T*>(a.k) + bh * S * D;
  const T* v = static_cast<const T*>(a.v) + bh * S * D;
  const T* go = dout + bh * S * D;

  const int r = threadIdx.x >> 2, ql = threadIdx.x & 3;
  const int64_t p_lo = (int64_t)blockIdx.x * kRowsPerBlock;
  const int64_t p_hi = (p_lo + kRowsPerBlock < S) ? p_lo + kRowsPerBlock : S;
  const int64_t pi = p_lo + r;
  const bool row_ok = pi < S;
  const int64_t gi = row_ok ? m.g(pi) : 0;
  const float slope = a.slopes ? a.slopes[hh] : 0.f;
  const float li = row_ok ? lse[bh * S + pi] : -INFINITY;
  const float Di = row_ok ? dvec[bh * S + pi] : 0.f;

  float qf[4 * kC], df[4 * kC], acc[4 * kC];
#pragma unroll
  for (int t = 0; t < kC; ++t) {
    const float4 qq = row_ok ? load4<T>(q + pi * D + 4 * (ql + 4 * t)) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 dd = row_ok ? load4<T>(go + pi * D + 4 * (ql + 4 * t)) : make_float4(0.f, 0.f, 0.f, 0.f);
    qf[4 * t] = qq.x; qf[4 * t + 1] = qq.y; qf[4 * t + 2] = qq.z; qf[4 * t + 3] = qq.w;
    df[4 * t] = dd.x; df[4 * t + 1] = dd.y; df[4 * t + 2] = dd.z; df[4 * t + 3] = dd.w;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[4 * t + e] = 0.f;
  }

  int64_t qgmin, qgmax;
  m.grange(p_lo, p_hi, qgmin, qgmax);
  const int32_t r0 = m.shard(p_lo);

  for (int32_t t = 0; t < m.N; ++t) {
    const int32_t s = (r0 - t + m.N) % m.N;
    int64_t t0, t1;
    shard_tiles(m, s, t0, t1);
    for (int64_t ti = t0; ti < t1; ++ti) {
      const int64_t k0 = ti * kTile;
      const int64_t k1 = (k0 + kTile < S) ? k0 + kTile : S;
      if (a.causal) {
        int64_t kgmin, kgmax;
        m.grange(k0, k1, kgmin, kgmax);
        if (kgmin > qgmax) continue;
      }
      __syncthreads();
      stage_rows<T, D>(Ks, k, k0, S);
      stage_rows<T, D>(Vs, v, k0, S);
      for (int j = threadIdx.x; j < kTile; j += kThreads) gk[j] = (k0 + j < S) ? m.g(k0 + j) : -1;
      __syncthreads();
#pragma unroll 1
      for (int j = 0; j < kTile; ++j) {
        const float* kr = Ks + j * D;
        const float* vr = Vs + j * D;
        float sd = 0.f, dp = 0.f;
#pragma unroll
        for (int t = 0; t < kC; ++t) {
          const float4 kk = *reinterpret_cast<const float4*>(kr + 4 * (ql + 4 * t));
          const float4 vv = *reinterpret_cast<const float4*>(vr + 4 * (ql + 4 * t));
          sd = fmaf(qf[4 * t], kk.x, sd); sd = fmaf(qf[4 * t + 1], kk.y, sd);
          sd = fmaf(qf[4 * t + 2], kk.z, sd); sd = fmaf(qf[4 * t + 3], kk.w, sd);
          dp = fmaf(df[4 * t], vv.x, dp); dp = fmaf(df[4 * t + 1], vv.y, dp);
          dp = fmaf(df[4 * t + 2], vv.z, dp); dp = fmaf(df[4 * t + 3], vv.w, dp);
        }
        sd = quad_sum(sd);
        dp = quad_sum(dp);
        const int64_t gj = gk[j];
        const bool vis = row_ok && gj >= 0 && (!a.causal || gj <= gi) && li != -INFINITY;
        float sc = sd * a.scale;
        if (a.slopes) sc -= slope * (float)(gi > gj ? gi - gj : gj - gi);
        const float p = vis ? exp2f((sc - li) * kLog2e) : 0.f;
        const float ds = p * (dp - Di) * a.scale;
#pragma unroll
        for (int t = 0; t < kC; ++t) {
          const float4 kk = *reinterpret_cast<const float4*>(kr + 4 * (ql + 4 * t));
          acc[4 * t] = fmaf(ds, kk.x, acc[4 * t]); acc[4 * t + 1] = fmaf(ds, kk.y, acc[4 * t + 1]);
          acc[4 * t + 2] = fmaf(ds, kk.z, acc[4 * t + 2]); acc[4 * t + 3] = fmaf(ds, kk.w, acc[4 * t + 3]);
        }
      }
    }
  }
  if (row_ok) {
    T* dqr = dq + (bh * S + pi) * D;
#pragma unroll
    for (int t = 0; t < kC; ++t)
      store4<T>(dqr + 4 * (ql + 4 * t), make_float4(acc[4 * t], acc[4 * t + 1], acc[4 * t + 2], acc[4 * t + 3]));
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
cudaError_t fwd_simt_t(const AttnArgs& a, void* o, float* lse, cudaStream_t st) {
  const size_t smem = 2 * kTile * D * sizeof(float) + kTile * sizeof(int64_t);
  cudaError_t e = set_smem(fwd_simt_kernel<T, D>, smem);
  if (e != cudaSuccess) return e;
  const int64_t BH = a.B * a.H;
  // (b, h) slices beyond the grid's y range are launched in pieces of whole batches,
  // so that blockIdx.y % H still names the head.
  const int64_t step = (65535 / a.H) * a.H;
  for (int64_t b0 = 0; b0 < BH; b0 += step) {
    AttnArgs sub = a;
    const int64_t nb = (BH - b0 < step) ? BH - b0 : step;
    sub.q = static_cast<const T*>(a.q) + b0 * a.S * D;
    sub.k = static_cast<const T*>(a.k) + b0 * a.S * D;
    sub.v = static_cast<const T*>(a.v) + b0 * a.S * D;
    dim3 grid((unsigned)((a.S + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)nb);
    if (a.o_f32 != nullptr) sub.o_f32 = a.o_f32 + b0 * a.S * D;
    fwd_simt_kernel<T, D><<<grid, kThreads, smem, st>>>(sub, static_cast<T*>(o) + b0 * a.S * D,
                                                        lse + b0 * a.S);
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename T, int D>
cudaError_t bwd_simt_t(const AttnArgs& a, const float* lse, const void* dout, const float* dvec,
                       void* dq, void* dk, void* dv, cudaStream_t st) {
  const size_t smem_kv = 2 * kTile * D * sizeof(float) + kTile * sizeof(int64_t);
  const size_t smem_q = 2 * kTile * D * sizeof(float) + 2 * kTile * sizeof(float) + kTile * sizeof(int64_t);
  cudaError_t e = set_smem(bwd_dq_simt_kernel<T, D>, smem_kv);
  if (e != cudaSuccess) return e;
  e = set_smem(bwd_dkdv_simt_kernel<T, D>, smem_q);
  if (e != cudaSuccess) return e;
  const int64_t BH = a.B * a.H;
  // (b, h) slices beyond the grid's y range are launched in pieces of whole batches,
  // so that blockIdx.y % H still names the head.
  const int64_t step = (65535 / a.H) * a.H;
  for (int64_t b0 = 0; b0 < BH; b0 += step) {
    const int64_t nb = (BH - b0 < step) ? BH - b0 : step;
    const int64_t off = b0 * a.S * D;
    AttnArgs sub = a;
    sub.q = static_cast<const T*>(a.q) + off;
    sub.k = static_cast<const T*>(a.k) + off;
    sub.v = static_cast<const T*>(a.v) + off;
    dim3 grid((unsigned)((a.S + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)nb);
    bwd_dq_simt_kernel<T, D><<<grid, kThreads, smem_kv, st>>>(
        sub, lse + b0 * a.S, static_cast<const T*>(dout) + off, dvec + b0 * a.S, static_cast<T*>(dq) + off);
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dkdv_simt_kernel<T, D><<<grid, kThreads, smem_q, st>>>(
        sub, lse + b0 * a.S, static_cast<const T*>(dout) + off, dvec + b0 * a.S,
        static_cast<T*>(dk) + off, static_cast<T*>(dv) + off);
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename T, int D>
cudaError_t rowdot_t(const AttnArgs& a, const void* o, const void* dout, float* dvec, float* dq_acc,
                     cudaStream_t st) {
  const int64_t rows = a.B * a.H * a.S;
  const int64_t blocks = (rows + 7) / 8;
  bwd_rowdot_kernel<T, D><<<(unsigned)blocks, 256, 0, st>>>(static_cast<const T*>(o),
                                                          static_cast<const T*>(dout), dvec, dq_acc, rows);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const AttnArgs& a, void* o, float* lse, cudaStream_t st) {
  if (a.dtype == RA_F32) return a.D == 64 ? fwd_simt_t<float, 64>(a, o, lse, st) : fwd_simt_t<float, 128>(a, o, lse, st);
  return a.D == 64 ? fwd_simt_t<__nv_bfloat16, 64>(a, o, lse, st) : fwd_simt_t<__nv_bfloat16, 128>(a, o, lse, st);
}

cudaError_t launch_bwd_rowdot(const AttnArgs& a, const void* o, const void* dout, float* dvec, float* dq_acc,
                              cudaStream_t st) {
  if (a.dtype == RA_F32)
    return a.D == 64 ? rowdot_t<float, 64>(a, o, dout, dvec, dq_acc, st)
                     : rowdot_t<float, 128>(a, o, dout, dvec, dq_acc, st);
  return a.D == 64 ? rowdot_t<__nv_bfloat16, 64>(a, o, dout, dvec, dq_acc, st)
                   : rowdot_t<__nv_bfloat16, 128>(a, o, dout, dvec, dq_acc, st);
}

cudaError_t launch_bwd_simt(const AttnArgs& a, const float* lse, const void* dout, const float* dvec,
                            void* dq, void* dk, void* dv, cudaStream_t st) {
  if (a.dtype == RA_F32)
    return a.D == 64 ? bwd_simt_t<float, 64>(a, lse, dout, dvec, dq, dk, dv, st)
                     : bwd_simt_t<float, 128>(a, lse, dout, dvec, dq, dk, dv, st);
  return a.D == 64 ? bwd_simt_t<__nv_bfloat16, 64>(a, lse, dout, dvec, dq, dk, dv, st)
                   : bwd_simt_t<__nv_bfloat16, 128>(a, lse, dout, dvec, dq, dk, dv, st);
}

}  // namespace ra
