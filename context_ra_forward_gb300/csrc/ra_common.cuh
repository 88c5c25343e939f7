// ra_common.cuh — pieces shared by every kernel of the library: the closed-form
// sequence -> shard maps, tile position ranges, bounded waits and the status word.
//
// Pages cited:
//   [CP] "百万Token上下文训练的挑战与突破" §2.1 (contiguous split into N pieces)
//   [ZZ] "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" §Zig Zag Ring
//        Attention (interleaved assignment; each shard's Q meets every K/V block)
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ra.h"

namespace ra {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Wait sites recorded in the status word when a bounded wait gives up.
enum WaitSite : int32_t {
  kSiteQFull = 1, kSiteKFull, kSiteKEmpty, kSiteVFull, kSiteVEmpty, kSiteSFull,
  kSitePFull, kSiteODone, kSiteDebug, kSiteBwd
};
enum KernelId : int32_t { kKernFwdTc = 1, kKernBwdTc = 2, kKernDebug = 3 };

// Limit of every in-kernel wait (nanoseconds of %globaltimer).  Work between two
// waits is one tile (microseconds), so two seconds only expires on a lost signal.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// Below this a wait does not look at the status word (see mbar_wait).
constexpr uint64_t kStatusCheckNs = 50000ull;

// ----------------------------------------------------------------------------
// Sequence -> shard-major slot maps ([CP] §2.1, [ZZ] §Zig Zag)
//   contiguous: slot p holds global position p.
//   zigzag:     c = S/N slots per shard, h = c/2 per chunk; slot p of shard
//               r = p div c, offset u = p mod c, holds global position
//               r*h + u (first chunk, u < h) or (2N-1-r)*h + (u-h) (second).
//   strided:    shard r holds tokens r, r+N, r+2N, ... ("GPU 0 gets tokens
//               [0, 4, 8...], GPU 1 gets [1, 5, 9...]"): slot p holds u*N + r.
// Within one chunk (zigzag), one shard (strided) or anywhere (contiguous) the
// global positions of consecutive slots form an arithmetic sequence.
// ----------------------------------------------------------------------------
struct SeqMap {
  int64_t S;
  int64_t c;   // slots per shard
  int64_t h;   // tokens per chunk (zigzag) / c (otherwise)
  int32_t N;
  int32_t layout;

  __host__ __device__ static SeqMap make(int64_t S_, int32_t N_, int32_t layout_) {
    SeqMap m;
    m.S = S_;
    m.N = N_;
    m.layout = layout_;
    m.c = N_ > 0 ? S_ / N_ : 0;
    m.h = layout_ == RA_LAYOUT_ZIGZAG ? m.c / 2 : m.c;
    return m;
  }
  // slot -> global position
  __host__ __device__ __forceinline__ int64_t g(int64_t p) const {
    if (layout == RA_LAYOUT_ZIGZAG) {
      const int64_t r = p / c, u = p - r * c;
      return u < h ? r * h + u : (2 * (int64_t)N - 1 - r) * h + (u - h);
    }
    if (layout == RA_LAYOUT_STRIDED) {
      const int64_t r = p / c, u = p - r * c;
      return u * N + r;
    }
    return p;
  }
  // global position -> slot
  __host__ __device__ __forceinline__ int64_t inv(int64_t gp) const {
    if (layout == RA_LAYOUT_ZIGZAG) {
      const int64_t k = gp / h, u = gp - k * h;
      return k < N ? k * c + u : (2 * (int64_t)N - 1 - k) * c + h + u;
    }
    if (layout == RA_LAYOUT_STRIDED) {
      const int64_t u = gp / N, r = gp - u * N;
      return r * c + u;
    }
    return gp;
  }
  __host__ __device__ __forceinline__ int32_t shard(int64_t p) const { return (int32_t)(p / c); }
  // Slots per run of arithmetic global positions (a chunk or a shard).
  __host__ __device__ __forceinline__ int64_t run() const { return layout == RA_LAYOUT_ZIGZAG ? h : c; }
  // Step of the global positions within a run.
  __host__ __device__ __forceinline__ int64_t run_step() const { return layout == RA_LAYOUT_STRIDED ? N : 1; }
  // Smallest and largest global position held by the slots [p0, p1) (p0 < p1 <= S).
  // Walks the runs the range touches; each run is increasing.
  __host__ __device__ void grange(int64_t p0, int64_t p1, int64_t& gmin, int64_t& gmax) const {
    if (layout == RA_LAYOUT_CONTIGUOUS) { gmin = p0; gmax = p1 - 1; return; }
    const int64_t L = run();
    gmin = INT64_MAX;
    gmax = -1;
    int64_t a = p0;
    while (a < p1) {
      const int64_t seg_end = (a / L + 1) * L;
      const int64_t b = seg_end < p1 ? seg_end : p1;
      const int64_t ga = g(a), gb = g(b - 1);
      gmin = ga < gmin ? ga : gmin;
      gmax = gb > gmax ? gb : gmax;
      a = b;
    }
  }
  // Step of the global positions over the slots [p0, p1) when they form one
  // arithmetic sequence (1 = consecutive positions), 0 when they do not.
  __host__ __device__ int64_t gstep(int64_t p0, int64_t p1) const {
    if (layout == RA_LAYOUT_CONTIGUOUS || p1 - p0 <= 1) return 1;
    return (p0 / run()) == ((p1 - 1) / run()) ? run_step() : 0;
  }
  // True when the slots [p0, p1) hold consecutive global positions.
  __host__ __device__ bool contiguous_range(int64_t p0, int64_t p1) const { return gstep(p0, p1) == 1; }
};

// ----------------------------------------------------------------------------
// Status word: [0] code, [1] kernel id, [2] block, [3] wait site.  The first
// failure wins; the host reads and clears it in ra_check_device_status.
// Words [4, 4 + kStatusWarps) record, for the block that failed first, what each
// warp was waiting on when its wait gave up: site << 24 | parity << 16 | the low
// 16 bits of the barrier's shared address (0 = that warp did not give up).
// ----------------------------------------------------------------------------
constexpr int kStatusWarps = 32;
constexpr int kStatusWords = 4 + kStatusWarps;
__device__ __forceinline__ void record_failure(int32_t* status, int32_t code, int32_t kernel,
                                               int32_t site) {
  if (status == nullptr) return;
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = kernel;
    status[2] = (int32_t)(blockIdx.x + gridDim.x * blockIdx.y);
    status[3] = site;
    __threadfence();
  }
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// mbarrier helpers (shared::cta addresses as 32-bit)
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete, at most `limit_ns`.
// On expiry records RA_ERR_TIMEOUT and returns false; the caller then stops its
// work and falls through to the kernel's teardown (no trap, no endless loop).
// A wait also gives up as soon as the status word holds a failure, so one lost
// signal ends the whole launch quickly; the word stays set (and later waits keep
// giving up) until the host reads and clears it.
__device__ __forceinline__ void record_wait_site(int32_t* status, uint32_t bar, uint32_t parity, int32_t site) {
  if (status == nullptr) return;
  const int32_t me = (int32_t)(blockIdx.x + gridDim.x * blockIdx.y);
  const int w = (int)(threadIdx.x >> 5);
  if (*reinterpret_cast<volatile int32_t*>(status + 2) == me && w < kStatusWarps)
    status[4 + w] = (site << 24) | (int32_t)((parity & 1u) << 16) | (int32_t)(bar & 0xffffu);
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status,
                                          int32_t kernel, int32_t site,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    // The status word (a global load, slow under load) is consulted only once a
    // wait has lasted longer than any wait of a healthy pipeline, so that an
    // ordinary wait wakes as soon as its phase completes.
    const uint64_t dt = globaltimer_ns() - t0;
    if (dt < kStatusCheckNs) continue;
    if (status != nullptr && *reinterpret_cast<volatile int32_t*>(status) != 0) {
      record_wait_site(status, bar, parity, site);
      return false;
    }
    if (dt > limit_ns) {
      record_failure(status, RA_ERR_TIMEOUT, kernel, site);
      record_wait_site(status, bar, parity, site);
      return false;
    }
  }
}

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

}  // namespace ra
