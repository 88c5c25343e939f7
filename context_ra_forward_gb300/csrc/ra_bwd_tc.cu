// ra_bwd_tc.cu — tcgen05 tensor-core backward for bf16, head dim 128.
//
// Pages cited:
//   [LC] "超长上下文技术" survey §3.1.2: backward recomputes intermediates (the
//        block probabilities) instead of storing them; §2.1.2 scale and ALiBi.
//   [ZZ] "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" §Zig Zag Ring
//        Attention: every K/V block meets every Q block, one ring step at a time.
// The gradient itself is the analytic derivative of the forward (the pages give
// none): with P = exp(s - LSE) and D_i = dO_i.O_i,
//   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i.V_j - D_i),
//   dK_j = scale sum_i dS_ij Q_i,  dQ_i = scale sum_j dS_ij K_j.
//
// One CTA owns one 128-row K/V tile of one (batch, head) and walks the 128-row Q
// tiles that see it in ring order (the queries of shard (s + t) mod N at step t),
// skipping tiles every query of which lies before every key (causal).
//
// Warp roles (384 threads, three warpgroups; setmaxnreg gives the two softmax
// warpgroups 200 registers and the third 104):
//   warps 0-7  "softmax": warp w owns K/V rows 32*(w%4).. (its TMEM lane quarter)
//              and Q columns 64*(w/4)..: P^T, dS^T, the dQ drain, the dK/dV epilogue
//   warp  8    TMA producer: K and V once, then Q and dO tiles into a 2-stage ring
//              (aligned shapes: with each tile's LSE and D rows, so that no softmax
//              warp waits on a global load); it also issues the bulk reduce-adds of
//              each Q tile's dQ partial
//   warp  9    TMEM allocation and MMA issue (one thread); warps 10-11 idle
// TMEM (512 columns): S^T [0,128), dP^T [128,256), dK [256,384), dV [384,512);
// all fp32 with K/V row r in lane r.  Each softmax warp writes P^T (bf16 pairs)
// over the first half of its 64 S^T columns (Q columns 0..63 -> TMEM columns
// 0..31, 64..127 -> 64..95) and dS^T over the second half (-> 32..63, 96..127):
// the A operands of dV += P^T dO and dK += dS^T Q.  dS^T also goes to shared
// memory in the 128-byte-swizzled layout, the MN-major A operand of dQ = dS K,
// whose result (row = query) takes the dP^T region once the dS pass has read it.
//
// MMA order per Q tile i:  [P^T_i] dV_i  [dS^T_i] dQ_i, dK_i -> S^T_{i+1}
//                          [dQ_i drained] dP^T_{i+1}
// (the pipe runs in order, so S^T_{i+1} follows the reads of P^T_i and dS^T_i).
// dQ partials are staged in shared memory and added into an fp32 workspace
// (zeroed by the row-term pre-pass) with TMA reduce-adds issued by the TMA warp:
// columns 0..63 over the dS^T tile (which dQ_i has read), 64..127 over the dO
// half of the tile's stage (which dV_i has read), both as soon as dQ_i is
// complete.  The next tile's dS pass waits for the first reduce to have read the
// dS^T tile; the Q half is refilled once dK_i has read it.  A post-pass scales
// and converts the sums.  The LSE and D rows of a Q tile reach shared memory by
// bulk copies (ragged shapes: the softmax warps load them from global memory
// before the waits they would otherwise follow).
#include <cuda.h>
#include <math.h>
#include <mutex>
#include <type_traits>

#include "ra_common.cuh"
#include "ra_kernels.h"
#include "ra_tc.cuh"

namespace ra {

namespace {

constexpr int kBM = 128;
constexpr int kD = 128;
constexpr int kTileBytes = kBM * kD * 2;   // 32 KB
constexpr int kBoxBytes = kTileBytes / 2;  // 16 KB
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 384;  // 3 warpgroups: softmax x2, then producer, MMA and two idle warps
// Register split (setmaxnreg, per warpgroup): the block launches with 168 per
// thread (65536 / 384, rounded down to 8); the third warpgroup gives back to 104
// and the softmax warpgroups take 200: 2 x 128 x 200 + 128 x 104 = 64512 = 384 x 168.
// (ptxas still reports a few tens of bytes of spill traffic here, fewer than at
// 192/120 or 208/88.)
constexpr uint32_t kRegsSoftmax = 200, kRegsOther = 104;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 384;

// Shared memory (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffQ = kOffV + kTileBytes;        // 2 stages of [Q | dO]
constexpr uint32_t kStageBytes = 2 * kTileBytes;
constexpr uint32_t kOffDS = kOffQ + 2 * kStageBytes;  // dS^T, 32 KB
// LSE rows of the Q tiles of both stages (512 B each), then one D row (the dS pass
// of a tile reads it; each half is refilled once its four warps have drained)
constexpr uint32_t kRowBytes = kBM * 4;
constexpr uint32_t kOffLse = kOffDS + kTileBytes;
constexpr uint32_t kOffDrow = kOffLse + 2 * kRowBytes;
constexpr uint32_t kOffBar = kOffDrow + kRowBytes;
enum Bar {
  kBarKV = 0,
  kBarQFull = 1,    // + stage: the Q half of the stage is loaded
  kBarDOFull = 3,   // + stage: the dO half of the stage is loaded
  // + stage: dQ columns 0..63 of tile i are staged over the dS^T tile (DrainQ),
  // 64..127 over the dO half of its stage (DrainDO).  One barrier per stage: the
  // producer waits for tile i after it has refilled tile i-1's stage, and tile i+1
  // may finish before that; only tile i+2, which needs this stage refilled, could
  // complete the next phase of the barrier.
  kBarDrainQ = 5,
  kBarDrainDO = 7,
  // + stage: dK_i is complete, so the Q half of tile i's stage may be refilled.
  // Per stage for the same reason: the producer waits for it after letting the
  // next tile's dS pass go on (kBarDPFull); only tile i+2, whose Q it has yet to
  // load, could complete the next phase of the same barrier.
  kBarKDone = 9,
  kBarSFull = 11,
  // dP^T_i is in TMEM and the reduce-add has read tile i-1's dQ columns staged over
  // the dS^T tile (count 2: the MMA commit and the producer's arrive)
  kBarDPFull,
  kBarPReady,
  kBarDSReady,
  kBarDQFull,
  kBarDQEmpty,
  kBarFinal,
  kBarEpiDone,  // every softmax warp has finished reading TMEM (count 8)
  kBarDRow,     // + half: the D row of the next tile's columns 64*half.. is loaded
  kNumBars = kBarDRow + 2
};
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffTmemSlot + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kIdescKK = tc::idesc_bf16(128, 128, 0, 0);  // A K-major, B K-major
constexpr uint32_t kIdescKM = tc::idesc_bf16(128, 128, 0, 1);  // A K-major (or TMEM), B MN-major
constexpr uint32_t kIdescMM = tc::idesc_bf16(128, 128, 1, 1);  // A MN-major, B MN-major

struct BwdParams {
  SeqMap map;
  int64_t S;
  int32_t H;
  int32_t BH;
  int32_t causal;
  const float* slopes;
  float c2;      // scale * log2(e)
  float scale;
  const float* lse;
  const float* dvec;
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t* status;
};

struct QTile {
  int64_t p0;      // first shard-major slot
  int64_t g0;      // its global position
  int64_t g1;      // global position of column cb (when cb < valid)
  int64_t gmin, gmax;
  int32_t valid;   // columns below S
  int32_t cb;      // columns 0..cb-1 are g0 + step*col, columns cb.. are g1 + step*(col - cb)
};

// Q tiles that see a K/V tile, in ring order.  Aligned shapes (every run a whole
// number of 128-row tiles): every tile lies inside one run (a zig-zag chunk, or a
// shard otherwise), so its global positions are g0, g0 + step, ... (step 1, or N
// when strided).  Ragged shapes (kRagged: runs of at least 128 slots that are not
// a multiple of 128): the tiles are the 128-slot tiles of the buffer owned by the
// shard of their first row; such a tile holds at most one run boundary (two
// arithmetic pieces), and the last one ends at S.
template <bool kStrided, bool kRagged>
struct QWalk {
  const BwdParams* P;
  int64_t kgmin;
  int32_t s0, t, seg;
  int64_t ti, tend, seg_p0, seg_g0;
  int64_t step;  // global-position step inside a run: N when strided, else 1

  __device__ void init(const BwdParams* p, int64_t kgmin_, int32_t s0_) {
    P = p;
    step = kStrided ? p->map.N : 1;
    kgmin = kgmin_;
    s0 = s0_;
    t = -1;
    seg = 1;
    ti = tend = 0;
    seg_p0 = seg_g0 = 0;
  }
  __device__ bool next(QTile& out) {
    const SeqMap& m = P->map;
    if constexpr (kRagged) {
      while (true) {
        while (ti >= tend) {
          if (++t >= m.N) {
            t = m.N;
            return false;
          }
          const int32_t s = (s0 + t) % m.N;
          ti = (s * m.c + kBM - 1) / kBM;
          tend = ((s + 1) * m.c + kBM - 1) / kBM;
        }
        const int64_t p0 = ti * kBM;
        ++ti;
        const int64_t p1 = p0 + kBM < P->S ? p0 + kBM : P->S;
        int64_t gmin, gmax;
        m.grange(p0, p1, gmin, gmax);
        if (P->causal && gmax < kgmin) continue;  // every query before every key
        out.p0 = p0;
        out.g0 = m.g(p0);
        out.gmin = gmin;
        out.gmax = gmax;
        out.valid = (int32_t)(p1 - p0);
        const int64_t run_end = (p0 / m.run() + 1) * m.run();
        out.cb = m.layout != RA_LAYOUT_CONTIGUOUS && run_end - p0 < out.valid ? (int32_t)(run_end - p0)
                                                                            : out.valid;
        out.g1 = out.cb < out.valid ? m.g(p0 + out.cb) : 0;
        return true;
      }
    }
    const int32_t nseg = m.layout == RA_LAYOUT_ZIGZAG ? 2 : 1;
    while (ti >= tend) {
      if (++seg >= nseg) {
        seg = 0;
        if (++t >= m.N) {
          t = m.N;  // exhausted: every later call returns false too
          seg = nseg;
          return false;
        }
      }
      const int32_t s = (s0 + t) % m.N;  // step t: the queries of shard (s0 + t) mod N
      int64_t len;
      if (m.layout == RA_LAYOUT_ZIGZAG) {
        len = m.h;
        seg_p0 = s * m.c + seg * m.h;
        seg_g0 = seg == 0 ? s * m.h : (2 * (int64_t)m.N - 1 - s) * m.h;
      } else {
        len = m.c;
        seg_p0 = s * m.c;
        seg_g0 = m.g(seg_p0);  // s for strided, s*c for contiguous
      }
      tend = len / kBM;
      ti = 0;
      if (P->causal) {
        // tile ti covers seg_g0 + 128*step*ti .. + 127*step; it is visible if its
        // last query is not before the K/V tile's first key
        if (seg_g0 + (len - 1) * step < kgmin) {
          tend = 0;
        } else if (kgmin > seg_g0 + (kBM - 1) * step) {
          ti = (kgmin - seg_g0 - (kBM - 1) * step + kBM * step - 1) / (kBM * step);
        }
      }
    }
    out.p0 = seg_p0 + ti * kBM;
    out.g0 = seg_g0 + ti * kBM * step;
    out.gmin = out.g0;
    out.gmax = out.g0 + (kBM - 1) * step;
    out.valid = kBM;
    out.cb = kBM;
    out.g1 = 0;
    ++ti;
    return true;
  }
};

enum TileKind { kPlain = 0, kLinear = 1, kGeneral = 2 };

// Probability P^T of K/V row gj against query column col (global position
// q0g + step*col), log2 domain.
struct ColCtx {
  float c2, slope2, lin_base, lin_sl;
  int64_t gj, q0g, q1g, step;
  int32_t cb, valid;  // the tile's column pieces and columns below S (as QTile)
  bool causal, alibi, row_ok;
};

// col: query column within the tile; colh: the same within this warp's 64-column
// half (a compile-time constant in the unrolled loops; the half's offset is folded
// into lin_base, so the ALiBi term needs no per-element int -> float conversion).
template <int kKind>
__device__ __forceinline__ float prob(float s, float lse2, int col, int colh, const ColCtx& c) {
  if constexpr (kKind == kPlain) {
    return tc::ex2(fmaf(s, c.c2, -lse2));
  } else if constexpr (kKind == kLinear) {
    return tc::ex2(fmaf(s, c.c2, fmaf(c.lin_sl, (float)colh, c.lin_base) - lse2));
  } else {
    const int64_t gi = col < c.cb ? c.q0g + c.step * col : c.q1g + c.step * (col - c.cb);
    const bool vis = c.row_ok && col < c.valid && (!c.causal || c.gj <= gi);
    float v = s * c.c2 - lse2;
    if (c.alibi) v -= c.slope2 * (float)(gi > c.gj ? gi - c.gj : c.gj - gi);
    return vis ? tc::ex2(v) : 0.f;
  }
}

// P^T for this warp's 64 query columns: from S^T in TMEM into registers (fp32)
// and back into TMEM as bf16 pairs for the dV product.
// Row values (LSE or D) of this warp's 64 query columns, four at a time: held in
// registers (loaded from global memory ahead of use), or read from the shared-memory
// row where each is needed.
struct RowsInRegs {
  float4 v[16];
  __device__ __forceinline__ float4 operator()(int q) const { return v[q]; }
};
struct RowsInSmem {
  const float4* s;
  __device__ __forceinline__ float4 operator()(int q) const { return s[q]; }
};

template <int kKind, typename Rows>
// lse4(q): the LSE values of columns 4q..4q+3 of this warp's half.
__device__ __forceinline__ void compute_p(uint32_t t_row, int h, const Rows& lse4, const ColCtx& c,
                                          float (&p)[64]) {
  uint32_t rr[2][32];
  tc::tmem_ld64(t_row + kColS + 64 * h, rr);
  tc::tmem_wait_ld();
#pragma unroll
  for (int ci = 0; ci < 2; ++ci) {
    const uint32_t (&r)[32] = rr[ci];
#pragma unroll
    for (int u = 0; u < 32; u += 2) {
      const float4 lq = lse4(8 * ci + (u >> 2));
      const float l4[4] = {lq.x, lq.y, lq.z, lq.w};
      if constexpr (kKind == kGeneral) {
        p[32 * ci + u] = prob<kKind>(__uint_as_float(r[u]), l4[u & 3] * kLog2e, 64 * h + 32 * ci + u, 32 * ci + u, c);
        p[32 * ci + u + 1] = prob<kKind>(__uint_as_float(r[u + 1]), l4[(u + 1) & 3] * kLog2e,
                                         64 * h + 32 * ci + u + 1, 32 * ci + u + 1, c);
      } else {
        // exponent arguments of the column pair in packed fp32 pairs: s * c2 (+ ALiBi) - LSE * log2(e)
        float2 off = tc::mul2(make_float2(l4[u & 3], l4[(u + 1) & 3]), make_float2(-kLog2e, -kLog2e));
        if constexpr (kKind == kLinear)
          off = tc::add2(off, tc::fma2(make_float2(c.lin_sl, c.lin_sl),
                                       make_float2((float)(32 * ci + u), (float)(32 * ci + u + 1)),
                                       make_float2(c.lin_base, c.lin_base)));
        const float2 x = tc::fma2(make_float2(__uint_as_float(r[u]), __uint_as_float(r[u + 1])),
                                  make_float2(c.c2, c.c2), off);
        p[32 * ci + u] = tc::ex2(x.x);
        p[32 * ci + u + 1] = tc::ex2(x.y);
      }
    }
  }
  uint32_t pk[32];
#pragma unroll
  for (int u = 0; u < 32; ++u) pk[u] = tc::pack_bf16(p[2 * u], p[2 * u + 1]);
  tc::tmem_st32(t_row + kColS + 64 * h, pk);
}

// Bulk copy without a tensor map: `bytes` (a multiple of 16) from 16-byte aligned
// global memory into 16-byte aligned shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <bool kStrided, bool kRagged>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ BwdParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kOffTmemSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqMap& m = P.map;
  const int64_t S = P.S;

  // Work item: (b, h) major, then the K/V tile (lowest global positions first
  // under causal: they are seen by the most queries).  Resident CTAs then belong
  // to one or two heads and share that head's Q/dO tiles and dQ rows in L2 (with
  // heads minor they spanned every head and the kernel ran at the DRAM roofline).
  const int64_t L = blockIdx.x;
  const int64_t ntiles = (S + kBM - 1) / kBM;
  const int64_t bh = L / ntiles;
  const int64_t tile = L - bh * ntiles;
  const int hh = (int)(bh % P.H);
  // (heaviest first under causal where tiles hold consecutive positions; strided
  // shards are balanced already)
  const int64_t kp0 = P.causal && !kStrided && !kRagged ? m.inv(tile * kBM) : tile * kBM;
  const int64_t kg0 = m.g(kp0);
  const int32_t s0 = m.shard(kp0);
  // ragged: K/V rows below S, and the smallest and largest key position of the tile
  const int32_t kvalid = kRagged ? (int32_t)(S - kp0 < kBM ? S - kp0 : kBM) : kBM;
  int64_t kgmin_t = kg0, kgmax_t = kg0 + (kBM - 1) * (kStrided ? (int64_t)m.N : 1);
  if constexpr (kRagged) m.grange(kp0, kp0 + kvalid, kgmin_t, kgmax_t);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kBarPReady || i == kBarDSReady || i == kBarDQEmpty || i == kBarEpiDone) cnt = 8;
      if (i == kBarDPFull) cnt = 2;
      if (i == kBarDrainQ || i == kBarDrainQ + 1 || i == kBarDrainDO || i == kBarDrainDO + 1) cnt = 4;
      mbar_init(bar(i), cnt);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // The roles never meet again after this point (each register budget holds for
  // the rest of its warps' code): the MMA warp frees TMEM once the softmax warps
  // have signalled the end of their TMEM reads.
  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
  if (warp == kProducerWarp) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::tma_prefetch_desc(&tm_do);
      tc::tma_prefetch_desc(&tm_dq);
      const int32_t z = (int32_t)bh;
      mbar_arrive_expect_tx(bar(kBarKV), 2 * kTileBytes);
      for (int hf = 0; hf < 2; ++hf) {
        tc::tma_load_3d(sbase + kOffK + hf * kBoxBytes, &tm_k, hf * 64, (int32_t)kp0, z, bar(kBarKV));
        tc::tma_load_3d(sbase + kOffV + hf * kBoxBytes, &tm_v, hf * 64, (int32_t)kp0, z, bar(kBarKV));
      }
      // Stage s holds Q and dO of Q tile i (s = i & 1).  Once dQ_i is complete its
      // columns 0..63 are staged over the dS^T tile and 64..127 over the dO half;
      // each part is added to the accumulator with its own bulk reduce as soon as
      // the softmax warps have staged it.  The stage is refilled once both
      // reduces have read their sources and dK_i has read Q_i (Q first).
      QWalk<kStrided, kRagged> walk;
      walk.init(&P, kgmin_t, s0);
      QTile qt;
      int64_t stage_p0[2] = {0, 0};
      int loaded = 0;
      // Aligned shapes: the tile's LSE row comes with its Q tile (same barrier), and
      // its D row into the one D buffer by halves, each once the four warps that
      // read that half for the previous tile have drained it.
      const float* lse_bh = P.lse + bh * S;
      const float* dvec_bh = P.dvec + bh * S;
      int drows[2] = {0, 0};  // D row halves loaded
      auto load_half = [&](const CUtensorMap* tm, int st, uint32_t off, int b, int64_t p0) {
        const uint32_t dst = sbase + kOffQ + st * kStageBytes + off;
        const bool lse_row = !kRagged && b == kBarQFull;
        mbar_arrive_expect_tx(bar(b + st), kTileBytes + (lse_row ? kRowBytes : 0));
        for (int hf = 0; hf < 2; ++hf)
          tc::tma_load_3d(dst + hf * kBoxBytes, tm, hf * 64, (int32_t)p0, z, bar(b + st));
        if (lse_row) bulk_load(sbase + kOffLse + st * kRowBytes, lse_bh + p0, kRowBytes, bar(b + st));
      };
      auto load_drow = [&](int half, int64_t p0) {
        mbar_arrive_expect_tx(bar(kBarDRow + half), kRowBytes / 2);
        bulk_load(sbase + kOffDrow + half * (kRowBytes / 2), dvec_bh + p0 + 64 * half, kRowBytes / 2,
                  bar(kBarDRow + half));
        ++drows[half];
      };
      mbar_arrive(bar(kBarDPFull));  // tile 0 has no predecessor
      for (int st = 0; st < 2 && walk.next(qt); ++st) {
        load_half(&tm_q, st, 0, kBarQFull, qt.p0);
        load_half(&tm_do, st, kTileBytes, kBarDOFull, qt.p0);
        stage_p0[st] = qt.p0;
        ++loaded;
      }
      if (!kRagged && loaded > 0) {
        load_drow(0, stage_p0[0]);
        load_drow(1, stage_p0[0]);
      }
      for (int i = 0; i < loaded; ++i) {
        const int st = i & 1;
        const uint32_t src = sbase + kOffQ + st * kStageBytes;
        // dQ columns 0..63 from the dS^T tile first (the next tile's dS pass waits
        // for that read), then 64..127 from the dO half; Q_{i+2} once dK_i has read Q_i
        if (!mbar_wait(bar(kBarDrainQ + st), (i >> 1) & 1, P.status, kKernBwdTc, kSiteBwd)) break;
        if (!kRagged && i + 1 < loaded) load_drow(0, stage_p0[(i + 1) & 1]);
        for (int b = 0; b < 2; ++b)  // 128-row x 32-column fp32 boxes
          tc::tma_reduce_add_3d(&tm_dq, sbase + kOffDS + b * kBoxBytes, 32 * b, (int32_t)stage_p0[st], z);
        tc::bulk_commit();
        if (!mbar_wait(bar(kBarDrainDO + st), (i >> 1) & 1, P.status, kKernBwdTc, kSiteBwd)) break;
        if (!kRagged && i + 1 < loaded) load_drow(1, stage_p0[(i + 1) & 1]);
        for (int b = 2; b < 4; ++b)
          tc::tma_reduce_add_3d(&tm_dq, src + b * kBoxBytes, 32 * b, (int32_t)stage_p0[st], z);
        tc::bulk_commit();
        tc::bulk_wait_read1();
        mbar_arrive(bar(kBarDPFull));  // for tile i+1
        const bool next = walk.next(qt);
        if (!mbar_wait(bar(kBarKDone + st), (i >> 1) & 1, P.status, kKernBwdTc, kSiteBwd)) break;
        if (next) load_half(&tm_q, st, 0, kBarQFull, qt.p0);
        tc::bulk_wait_read0();
        if (next) {
          load_half(&tm_do, st, kTileBytes, kBarDOFull, qt.p0);
          stage_p0[st] = qt.p0;
          ++loaded;
        }
      }
      tc::bulk_wait_all0();
      // Let every load this warp issued land before the CTA can exit.
      mbar_wait(bar(kBarKV), 0, P.status, kKernBwdTc, kSiteKFull);
      for (int back = 1; back <= 2 && back <= loaded; ++back) {
        const int ii = loaded - back;
        mbar_wait(bar(kBarQFull + (ii & 1)), (ii >> 1) & 1, P.status, kKernBwdTc, kSiteQFull);
        mbar_wait(bar(kBarDOFull + (ii & 1)), (ii >> 1) & 1, P.status, kKernBwdTc, kSiteQFull);
      }
      for (int hf = 0; hf < 2; ++hf)
        if (drows[hf] > 0) mbar_wait(bar(kBarDRow + hf), (drows[hf] - 1) & 1, P.status, kKernBwdTc, kSiteQFull);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t kb = sbase + kOffK, vb = sbase + kOffV, dsb = sbase + kOffDS;
      QWalk<kStrided, kRagged> walk;
      walk.init(&P, kgmin_t, s0);
      QTile qt;
      bool ok = mbar_wait(bar(kBarKV), 0, P.status, kKernBwdTc, kSiteKFull);
      bool more = ok && walk.next(qt);
      if (more) {
        ok = mbar_wait(bar(kBarQFull + 0), 0, P.status, kKernBwdTc, kSiteQFull);
        if (ok) {
          tc::fence_after_sync();
          const uint32_t qb = sbase + kOffQ;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // S^T = K Q^T
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            tc::mma_ss(tmem + kColS, tc::smem_desc(kb + off, 16, 1024), tc::smem_desc(qb + off, 16, 1024),
                       kIdescKK, kk > 0);
          }
          tc::mma_commit(bar(kBarSFull));
          ok = mbar_wait(bar(kBarDOFull + 0), 0, P.status, kKernBwdTc, kSiteQFull);
        }
        if (ok) {
          tc::fence_after_sync();
          const uint32_t dob = sbase + kOffQ + kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dP^T = V dO^T
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            tc::mma_ss(tmem + kColDP, tc::smem_desc(vb + off, 16, 1024), tc::smem_desc(dob + off, 16, 1024),
                       kIdescKK, kk > 0);
          }
          tc::mma_commit(bar(kBarDPFull));
        }
      }
      int i = 0;
      while (ok && more) {
        const int st = i & 1;
        const uint32_t qb = sbase + kOffQ + st * kStageBytes, dob = qb + kTileBytes;
        ok = mbar_wait(bar(kBarPReady), i & 1, P.status, kKernBwdTc, kSitePFull);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // dV += P^T dO   (A from TMEM)
          const uint32_t acol = kColS + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
          tc::mma_ts(tmem + kColDV, tmem + acol, tc::smem_desc(dob + kk * 2048, kBoxBytes, 1024), kIdescKM,
                     (i > 0 || kk > 0) ? 1u : 0u);
        }
        ok = mbar_wait(bar(kBarDSReady), i & 1, P.status, kKernBwdTc, kSiteBwd);
        if (!ok) break;
        tc::fence_after_sync();
        // dQ_i = dS K (A = dS^T MN-major, B = K MN-major) into the dP^T region, which
        // the dS pass has read
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          tc::mma_ss(tmem + kColDP, tc::smem_desc(dsb + kk * 2048, kBoxBytes, 1024),
                     tc::smem_desc(kb + kk * 2048, kBoxBytes, 1024), kIdescMM, kk > 0);
        }
        tc::mma_commit(bar(kBarDQFull));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // dK += dS^T Q   (A = dS^T from TMEM, B MN-major)
          const uint32_t acol = kColS + 32 + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
          tc::mma_ts(tmem + kColDK, tmem + acol, tc::smem_desc(qb + kk * 2048, kBoxBytes, 1024), kIdescKM,
                     (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(bar(kBarKDone + st));
        more = walk.next(qt);
        if (!more) break;
        const int nst = (i + 1) & 1;
        const uint32_t nqb = sbase + kOffQ + nst * kStageBytes, ndob = nqb + kTileBytes;
        // S^T_{i+1} over P^T_i and dS^T_i, which dV_i and dK_i (issued before it) read
        ok = mbar_wait(bar(kBarQFull + nst), ((i + 1) >> 1) & 1, P.status, kKernBwdTc, kSiteQFull);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          tc::mma_ss(tmem + kColS, tc::smem_desc(kb + off, 16, 1024), tc::smem_desc(nqb + off, 16, 1024),
                     kIdescKK, kk > 0);
        }
        tc::mma_commit(bar(kBarSFull));
        // dP^T_{i+1} over dQ_i once the softmax warps have read it
        ok = mbar_wait(bar(kBarDQEmpty), i & 1, P.status, kKernBwdTc, kSiteODone) &&
             mbar_wait(bar(kBarDOFull + nst), ((i + 1) >> 1) & 1, P.status, kKernBwdTc, kSiteQFull);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          tc::mma_ss(tmem + kColDP, tc::smem_desc(vb + off, 16, 1024), tc::smem_desc(ndob + off, 16, 1024),
                     kIdescKK, kk > 0);
        }
        tc::mma_commit(bar(kBarDPFull));
        ++i;
      }
      // dK/dV complete (and every MMA issued) before the epilogue and TMEM release.
      tc::mma_commit(bar(kBarFinal));
      mbar_wait(bar(kBarFinal), 0, P.status, kKernBwdTc, kSiteODone);
      tc::fence_before_sync();
    }
    __syncwarp();
    mbar_wait(bar(kBarEpiDone), 0, P.status, kKernBwdTc, kSiteODone);
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------- softmax warps
    const int qd = warp & 3;   // TMEM lane quarter: K/V rows 32*qd ..
    const int h = warp >> 2;   // Q column half: 64*h ..
    const int krow = qd * 32 + lane;
    const uint32_t t_row = tmem + ((uint32_t)(qd * 32) << 16);
    const int64_t gstep = kStrided ? m.N : 1;  // compile-time 1 unless strided
    // aligned: K/V tiles are arithmetic runs; ragged: this row's own position
    const bool krow_ok = krow < kvalid;
    const int64_t gj = kRagged ? (krow_ok ? m.g(kp0 + krow) : 0) : kg0 + gstep * krow;
    const bool alibi = P.slopes != nullptr;
    const float slope2 = alibi ? P.slopes[hh] * kLog2e : 0.f;
    ColCtx cc;
    cc.c2 = P.c2;
    cc.slope2 = slope2;
    cc.gj = gj;
    cc.step = gstep;
    cc.causal = P.causal != 0;
    cc.alibi = alibi;
    cc.row_ok = krow_ok;
    uint8_t* ds_tile = sgen + kOffDS + h * kBoxBytes;
    const float* lse_bh = P.lse + bh * S;
    const float* dvec_bh = P.dvec + bh * S;
    // 16-byte row loads need 16-byte aligned rows: always when S is a multiple of
    // 128 (aligned shapes); ragged shapes check the head's offset
    const bool rows16 = !kRagged || ((bh * S) & 3) == 0;

    QWalk<kStrided, kRagged> walk;
    walk.init(&P, kgmin_t, s0);
    QTile qt;
    int i = 0;
    bool ok = true;
    while (walk.next(qt)) {
      // Tile kind for this K/V row block against this Q tile.
      const int64_t qgmin = qt.gmin, qgmax = qt.gmax;
      const int64_t kgmin = kgmin_t, kgmax = kgmax_t;
      const bool below = kgmax <= qgmin;                 // every key at or before every query
      const bool above = !cc.causal && kgmin >= qgmax;   // every key at or after every query
      // (ragged: partial tiles and tiles with two position pieces take the per-element path)
      const bool whole = !kRagged || (kvalid == kBM && qt.valid == kBM && qt.cb == kBM);
      const bool full = whole && (cc.causal ? below : (!alibi || below || above));
      const int kind = full ? (alibi ? kLinear : kPlain) : kGeneral;
      cc.q0g = qt.g0;
      cc.q1g = qt.g1;
      cc.cb = qt.cb;
      cc.valid = qt.valid;
      // bias of column col: below: -slope (q0g + col - gj); above: -slope (gj - q0g - col)
      cc.lin_sl = (below ? -slope2 : slope2) * (float)gstep;
      cc.lin_base = (below ? -slope2 * (float)(qt.g0 - gj) : -slope2 * (float)(gj - qt.g0)) +
                    cc.lin_sl * (float)(64 * h);  // this warp's first column

      // the LSE row: aligned shapes read it from shared memory as it is needed (the
      // producer loaded it with the Q tile); ragged ones load it into registers from
      // global memory while S^T is computed
      std::conditional_t<kRagged, RowsInRegs, RowsInSmem> lse4;
      if constexpr (!kRagged) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarQFull + (i & 1)), (i >> 1) & 1, P.status, kKernBwdTc,
                                               kSiteQFull));
        if (!ok) break;
        lse4.s = reinterpret_cast<const float4*>(sgen + kOffLse + (i & 1) * kRowBytes) + 16 * h;
      } else if (qt.valid == kBM && rows16) {
        const float4* lse_q = reinterpret_cast<const float4*>(lse_bh + qt.p0 + 64 * h);
#pragma unroll
        for (int u = 0; u < 16; ++u) lse4.v[u] = __ldg(lse_q + u);
      } else {
        // one column at a time; columns at or past S: an infinite LSE makes their
        // probabilities 0
        float lv[64];
#pragma unroll
        for (int u = 0; u < 64; ++u) {
          const int col = 64 * h + u;
          lv[u] = col < qt.valid ? __ldg(lse_bh + qt.p0 + col) : INFINITY;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) lse4.v[u] = make_float4(lv[4 * u], lv[4 * u + 1], lv[4 * u + 2], lv[4 * u + 3]);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull), i & 1, P.status, kKernBwdTc, kSiteSFull));
      if (!ok) break;
      tc::fence_after_sync();
      float p[64];
      if (kind == kPlain) compute_p<kPlain>(t_row, h, lse4, cc, p);
      else if (kind == kLinear) compute_p<kLinear>(t_row, h, lse4, cc, p);
      else compute_p<kGeneral>(t_row, h, lse4, cc, p);
      // the D row (ragged shapes: from global memory, loaded while dP^T is computed)
      std::conditional_t<kRagged, RowsInRegs, RowsInSmem> d4;
      if constexpr (kRagged) {
        if (qt.valid == kBM && rows16) {
          const float4* dv_q = reinterpret_cast<const float4*>(dvec_bh + qt.p0 + 64 * h);
#pragma unroll
          for (int u = 0; u < 16; ++u) d4.v[u] = __ldg(dv_q + u);
        } else {
          float dl[64];
#pragma unroll
          for (int u = 0; u < 64; ++u) {
            const int col = 64 * h + u;
            dl[u] = col < qt.valid ? __ldg(dvec_bh + qt.p0 + col) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < 16; ++u) d4.v[u] = make_float4(dl[4 * u], dl[4 * u + 1], dl[4 * u + 2], dl[4 * u + 3]);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPReady));
      if constexpr (!kRagged) {
        // aligned shapes: from shared memory, loaded by the producer once the previous
        // tile's dS pass had read the buffer
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarDRow + h), i & 1, P.status, kKernBwdTc, kSiteQFull));
        if (!ok) break;
        d4.s = reinterpret_cast<const float4*>(sgen + kOffDrow) + 16 * h;
      }

      // dS^T = P^T o (dP^T - D) into TMEM and shared memory (bf16, 128-byte
      // swizzle), once dP^T_i is complete and the reduce-add has read the previous
      // tile's dQ columns from the dS^T tile.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarDPFull), i & 1, P.status, kKernBwdTc, kSiteSFull));
      if (!ok) break;
      tc::fence_after_sync();
#pragma unroll
      for (int ci = 0; ci < 2; ++ci) {
        uint32_t r[32];
        tc::tmem_ld32(t_row + kColDP + 64 * h + 32 * ci, r);
        tc::tmem_wait_ld();
        uint32_t dsk[16];  // dS^T of these 32 columns as bf16 pairs
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int u = 2 * e;
          const float4 dq = d4(8 * ci + (u >> 2));
          const float d0[4] = {dq.x, dq.y, dq.z, dq.w};
          // P o (dP - D) for the column pair, in packed fp32 pairs
          const float2 diff = tc::fma2(make_float2(d0[u & 3], d0[(u + 1) & 3]), make_float2(-1.f, -1.f),
                                       make_float2(__uint_as_float(r[u]), __uint_as_float(r[u + 1])));
          const float2 ab = tc::mul2(make_float2(p[32 * ci + u], p[32 * ci + u + 1]), diff);
          dsk[e] = tc::pack_bf16(ab.x, ab.y);
        }
        // into TMEM first (the A operand of dK, in the half of this warp's S^T columns
        // that P^T left free: query columns 64h + 32ci.. -> TMEM columns
        // kColS + 64h + 32 + 16ci ..), then the 128-byte-swizzled shared-memory copy
        // while that store completes
        tc::tmem_st16(t_row + kColS + 64 * h + 32 + 16 * ci, dsk);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {  // four 16-byte chunks of 8 columns
          const int chunk = 4 * ci + c8;  // 16-byte chunk within the 128-byte row
          const uint32_t off = (uint32_t)krow * 128u + ((uint32_t)(chunk ^ (krow & 7)) << 4);
          *reinterpret_cast<uint4*>(ds_tile + off) =
              make_uint4(dsk[4 * c8], dsk[4 * c8 + 1], dsk[4 * c8 + 2], dsk[4 * c8 + 3]);
        }
      }
      tc::tmem_wait_st();
      fence_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarDSReady));

      // Drain this Q tile's dQ partial (TMEM lane = query row): into registers, free
      // the TMEM region, then stage it in shared memory that the tile's finished
      // MMAs no longer read, for the TMA warp's reduce-add.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarDQFull), i & 1, P.status, kKernBwdTc, kSiteODone));
      if (!ok) break;
      tc::fence_after_sync();
      {
        uint32_t rr[2][32];
        tc::tmem_ld64(t_row + kColDP + 64 * h, rr);
        tc::tmem_wait_ld();
        const uint32_t (&r0)[32] = rr[0];
        const uint32_t (&r1)[32] = rr[1];
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarDQEmpty));
        // fp32 boxes of 128 rows x 32 columns (128-byte rows, 128-byte swizzle), two
        // per warp: columns 0..63 over the dS^T tile (free since dQ_i has read it),
        // 64..127 over the dO half of the tile's stage (dV_i, before dQ_i, read it)
        uint8_t* box0 = (h == 0 ? sgen + kOffDS : sgen + kOffQ + (i & 1) * kStageBytes + kTileBytes) + krow * 128;
        uint8_t* box1 = box0 + kBoxBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t off = (uint32_t)((c ^ (krow & 7)) << 4);
          *reinterpret_cast<uint4*>(box0 + off) = make_uint4(r0[4 * c], r0[4 * c + 1], r0[4 * c + 2], r0[4 * c + 3]);
          *reinterpret_cast<uint4*>(box1 + off) = make_uint4(r1[4 * c], r1[4 * c + 1], r1[4 * c + 2], r1[4 * c + 3]);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar((h == 0 ? kBarDrainQ : kBarDrainDO) + (i & 1)));
      ++i;
    }
    // ------------------------------------------------------------- epilogue: dK (scaled), dV
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarFinal), 0, P.status, kKernBwdTc, kSiteODone));
    if (ok) {
      tc::fence_after_sync();
      // warps 0-3 write dK, warps 4-7 write dV; thread = K/V row, 128 columns.  A
      // tile that no query sees (none: the walk was empty) gets zero gradients.
      const uint32_t col0 = h == 0 ? kColDK : kColDV;
      const float mul = i == 0 ? 0.f : (h == 0 ? P.scale : 1.f);
      __nv_bfloat16* dst = (h == 0 ? P.dk : P.dv) + (bh * S + kp0 + krow) * kD;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(t_row + col0 + 32 * c, r);
        tc::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = tc::pack_bf16(__uint_as_float(r[2 * u]) * mul, __uint_as_float(r[2 * u + 1]) * mul);
        if (krow_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarEpiDone));
  }
}

// dq = scale * dq_acc, fp32 -> bf16, 8 elements per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         __nv_bfloat16* __restrict__ dq, float scale,
                                                         int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 o;
    o.x = tc::pack_bf16(a.x * scale, a.y * scale);
    o.y = tc::pack_bf16(a.z * scale, a.w * scale);
    o.z = tc::pack_bf16(b.x * scale, b.y * scale);
    o.w = tc::pack_bf16(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = o;
  }
}

}  // namespace

bool bwd_tc_supported(int64_t S, int64_t D, int32_t dtype, const SeqMap& m) {
  // aligned runs, or runs of at least one tile (a 128-slot tile then meets at most
  // one run boundary); the contiguous layout is a single run of positions
  const bool runs_ok = m.layout == RA_LAYOUT_CONTIGUOUS || m.run() >= kBM;
  return dtype == RA_BF16 && D == kD && S >= kBM && runs_ok;
}

cudaError_t launch_bwd_tc(const AttnArgs& a, const float* lse, const void* dout, const float* dvec,
                          float* dq_acc, void* dq, void* dk, void* dv, cudaStream_t st) {
  const int64_t BH = a.B * a.H;
  if (BH > INT32_MAX) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!tc::make_tmap_bhsd(&tq, a.q, BH, a.S, a.D, kBM) || !tc::make_tmap_bhsd(&tk, a.k, BH, a.S, a.D, kBM) ||
      !tc::make_tmap_bhsd(&tv, a.v, BH, a.S, a.D, kBM) || !tc::make_tmap_bhsd(&tdo, dout, BH, a.S, a.D, kBM) ||
      !tc::make_tmap_bhsd_f32(&tdq, dq_acc, BH, a.S, a.D, kBM))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.map = a.map;
  p.S = a.S;
  p.H = (int32_t)a.H;
  p.BH = (int32_t)BH;
  p.causal = a.causal;
  p.slopes = a.slopes;
  p.c2 = a.scale * kLog2e;
  p.scale = a.scale;
  p.lse = lse;
  p.dvec = dvec;
  p.dq_acc = dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.status = a.status;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    const void* kernels[] = {(const void*)bwd_tc_kernel<false, false>, (const void*)bwd_tc_kernel<true, false>,
                             (const void*)bwd_tc_kernel<false, true>, (const void*)bwd_tc_kernel<true, true>};
    for (const void* k : kernels)
      if (attr_err == cudaSuccess)
        attr_err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t tiles = (a.S + kBM - 1) / kBM;
  const int64_t blocks = tiles * BH;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  const bool strided = a.map.layout == RA_LAYOUT_STRIDED;
  const bool ragged = a.map.run() % kBM != 0;
  if (!ragged && strided)
    bwd_tc_kernel<true, false><<<(unsigned)blocks, kThreads, kSmemBytes, st>>>(tq, tk, tv, tdo, tdq, p);
  else if (!ragged)
    bwd_tc_kernel<false, false><<<(unsigned)blocks, kThreads, kSmemBytes, st>>>(tq, tk, tv, tdo, tdq, p);
  else if (strided)
    bwd_tc_kernel<true, true><<<(unsigned)blocks, kThreads, kSmemBytes, st>>>(tq, tk, tv, tdo, tdq, p);
  else
    bwd_tc_kernel<false, true><<<(unsigned)blocks, kThreads, kSmemBytes, st>>>(tq, tk, tv, tdo, tdq, p);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n8 = BH * a.S * a.D / 8;
  const int64_t grid = (n8 + 255) / 256 < 152 * 16 ? (n8 + 255) / 256 : 152 * 16;
  dq_convert_kernel<<<(unsigned)grid, 256, 0, st>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), a.scale, n8);
  note_launch();
  return cudaGetLastError();
}

}  // namespace ra
