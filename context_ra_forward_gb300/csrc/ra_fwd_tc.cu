// ra_fwd_tc.cu — tcgen05 tensor-core forward for bf16 (kind::f16) and e4m3
// (kind::f8f6f4, per-tensor scales), head dim 128.
//
// Pages cited:
//   [ZZ] "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" §Zig Zag Ring
//        Attention: the Q block of shard r meets the K/V of shard (r - t) mod N at
//        ring step t until it has met every K/V block; zig-zag assignment balances
//        causal work, fully masked blocks need not be computed.
//   [LC] "超长上下文技术" survey §3.1.2 (blockwise attention with a running row max
//        m and sum l; output rescaled when m grows) and §2.1.2 (scale 1/sqrt(d),
//        ALiBi bias -|i-j| * slope after scaling).
//
// One CTA owns 256 consecutive shard-major query rows (two 128-row Q tiles A, B)
// of one (batch, head) and walks the K/V tiles in ring order, skipping tiles that
// are fully masked for both Q tiles.  The (m, l, O) state carries across ring
// steps, which is the online log-sum-exp merge of the per-step partial results.
//
// Warp roles (384 threads, three warpgroups; setmaxnreg gives the two softmax
// warpgroups 200 registers and the third 104):
//   warps 0-3  softmax for Q tile A (thread = row; TMEM lanes 0..127)
//   warps 4-7  softmax for Q tile B
//   warp  8    TMA producer: Q once, then K and V tiles into 2-stage rings
//   warp  9    TMEM allocation and MMA issue (one thread); warps 10-11 idle
// On tiles that are unmasked, or whose visible keys are a prefix of the columns
// (a causal diagonal, a ragged tile), a row's 128 scores are read from TMEM once
// and both softmax passes run from registers.
// Causal ALiBi (bf16): every visible key lies at or before its query, so the bias
// -slope*(g_i - g_j) is linear in the key: a per-row constant plus slope*step*u
// for column u of the tile.  The column term is added to the scores by the
// tensor core (one more K = 16 step of the Q K^T product against a fixed block:
// ones for Q, the column term split into four bf16 parts for K), and the row
// constant is an offset of the row's reference; the tiles then take the register
// path of unbiased tiles.  Heads whose slope makes that term too large for the
// fp32 accumulator run in a second launch with the bias added per element.
// The kernel is a template over the element type, the bias mode (none, tensor
// core, per element) and whether every tile lies in one run of arithmetic
// positions (aligned); each instantiation holds only the tile paths it can meet.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512),
// all fp32 with row i in lane i.  The softmax writes P (bf16 pairs) over the
// first 64 columns of its S tile, and the PV product reads it from there.
//
// MMA issue order per K/V tile j (ping-pong, so one softmax warpgroup always has
// its scores while the tensor core works for the other):
//   PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
// Each S(j+1) commit therefore also certifies PV(j) complete, which is what lets
// the softmax rescale O in TMEM right after it sees S(j+1).
//
// The running max is only moved when a tile's max exceeds it by more than 8 (log2
// units); otherwise probabilities are taken against the stale max (<= 2^8).  O and
// l use the same reference, so the final O / l and LSE are exact.
#include <cuda.h>
#include <math.h>
#include <mutex>

#include "ra_common.cuh"
#include "ra_kernels.h"
#include "ra_tc.cuh"

namespace ra {

namespace {

constexpr int kBM = 128;
constexpr int kD = 128;
constexpr int kStages = 2;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 384;  // 3 warpgroups: softmax x2, then producer, MMA and two idle warps
// Register split (setmaxnreg, per warpgroup): the block launches with 168 per
// thread (65536 / 384, rounded down to 8); the third warpgroup gives back to 104
// and the softmax warpgroups take 200: 2 x 128 x 200 + 128 x 104 = 64512 = 384 x 168.
constexpr uint32_t kRegsSoftmax = 200, kRegsOther = 104;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;

enum Bar {
  kBarQFull = 0,
  kBarKFull = 1,                  // + stage
  kBarKEmpty = kBarKFull + kStages,
  kBarVFull = kBarKEmpty + kStages,
  kBarVEmpty = kBarVFull + kStages,
  kBarSFull = kBarVEmpty + kStages,  // + Q tile
  kBarPFull = kBarSFull + 2,
  kBarODone = kBarPFull + 2,
  kBarFinal = kBarODone + 2,
  kBarEpiDone = kBarFinal + 1,  // every softmax thread has finished reading TMEM
  kNumBars = kBarEpiDone + 1
};

// Element-type dependent layout.  Shared-memory rows are 128 bytes either way
// (64 bf16 or 128 e4m3 per box row, 128-byte swizzle); one MMA consumes 32 bytes
// of K per row (16 bf16 or 32 e4m3).
template <bool kFp8>
struct FwdCfg {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kTileBytes = kBM * kD * kElem;     // 32 KB bf16, 16 KB e4m3
  static constexpr int kBoxCols = 128 / kElem;            // elements in a 128-byte row
  static constexpr int kBoxes = kD / kBoxCols;            // boxes per 128-wide head dim
  static constexpr int kBoxBytes = kTileBytes / kBoxes;   // 16 KB
  static constexpr int kKStep = 32 / kElem;               // K per MMA
  static constexpr int kSteps = kD / kKStep;              // MMAs per Q K^T tile
  static constexpr int kPvSteps = kBM / kKStep;           // MMAs per P V tile
  // Shared memory map (offsets from a 1024-byte aligned base).
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + 2 * kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;
  static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffGtab = kOffTmemSlot + 16;             // 8 warps x 128 int32 key positions
  // ALiBi column-term blocks (bf16 only), 128-byte swizzled like the tiles, of
  // which the MMA reads the first 32 bytes (K = 16) of every row: one 8-row atom
  // of ones for Q (read with an 8-row-group stride of 0), 128 rows for K.
  static constexpr uint32_t kOffQext = (kOffGtab + 8 * kBM * 4 + 1023u) & ~1023u;
  static constexpr uint32_t kOffKext = kOffQext + 1024;
  static constexpr uint32_t kSmemBytes = kOffKext + kBM * 128 + 1024;  // + alignment slack
  // Q (K-major) x K (K-major); P (TMEM) x V (MN-major)
  static constexpr uint32_t kIdescS = kFp8 ? tc::idesc_e4m3(128, 128, 0, 0) : tc::idesc_bf16(128, 128, 0, 0);
  static constexpr uint32_t kIdescPV = kFp8 ? tc::idesc_e4m3(128, 128, 0, 1) : tc::idesc_bf16(128, 128, 0, 1);
};

struct FwdParams {
  SeqMap map;
  int64_t S;
  int32_t H;
  int32_t BH;
  int32_t causal;
  int32_t aligned;      // every 256-row query pair and 128-row tile lies in one run
  int32_t heavy_first;  // causal + aligned: CTAs ordered by decreasing work (1: by position, 2: strided)
  int32_t head_filter;  // 0: every head; 1: only heads whose column term fits the tensor core; 2: only the others
  const float* slopes;
  float c2;             // softmax scale * log2(e) (for e4m3: times the Q and K scales)
  float o_scale;        // V scale (1 for bf16)
  __nv_bfloat16* o;
  float* o_f32;         // when set: O as fp32 (a ring-step partial) instead of o
  float* lse;
  int32_t* status;
  int32_t t_begin, t_end;  // ring steps visited
};

struct TileInfo {
  int64_t p0;    // first shard-major slot of the K/V tile
  int64_t gk0;   // global position of p0 when the tile's positions are arithmetic
  int64_t step;  // their step (1 = consecutive; N inside a strided shard); 0 = irregular
  int64_t gmin, gmax;
  int32_t valid; // rows of the tile below S
};

// Walks the K/V tiles of one query pair in ring order, skipping tiles every key
// of which lies in the future of every query of the pair.  Every role of the CTA
// runs its own copy in lockstep.
// kStatic: every 256-row query pair and 128-row tile lies in one run (aligned),
// known at compile time, so only the run-by-run walk is compiled.
template <bool kStatic>
struct KvWalk {
  const FwdParams* P;
  int64_t qgmax;
  int32_t r0;
  int32_t t;
  int32_t seg;
  int64_t ti, tend;
  int64_t seg_p0, seg_g0;

  __device__ void init(const FwdParams* p, int64_t qgmax_, int32_t r0_) {
    P = p;
    qgmax = qgmax_;
    r0 = r0_;
    t = p->t_begin - 1;
    seg = 1;  // forces a step to (t = 0, seg = 0)
    ti = tend = 0;
    seg_p0 = seg_g0 = 0;
  }

  __device__ bool next(TileInfo& out) {
    const SeqMap& m = P->map;
    if (kStatic || P->aligned) {
      const int32_t nseg = m.layout == RA_LAYOUT_ZIGZAG ? 2 : 1;
      while (ti >= tend) {
        if (++seg >= nseg) {
          seg = 0;
          if (++t >= P->t_end) {
            t = P->t_end;  // exhausted: every later call returns false too
            seg = nseg;
            return false;
          }
        }
        const int32_t s = (r0 - t + m.N) % m.N;  // ring step t meets shard (r0 - t) mod N
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
        const int64_t span = kBM * m.run_step();  // global positions one tile covers
        int64_t cnt = len / kBM;
        if (P->causal) {
          const int64_t vis = qgmax < seg_g0 ? 0 : (qgmax - seg_g0) / span + 1;
          cnt = vis < cnt ? vis : cnt;
        }
        ti = 0;
        tend = cnt;
      }
      const int64_t step = m.run_step();
      out.p0 = seg_p0 + ti * kBM;
      out.gk0 = seg_g0 + ti * kBM * step;
      out.step = step;
      out.gmin = out.gk0;
      out.gmax = out.gk0 + (kBM - 1) * step;
      out.valid = kBM;
      ++ti;
      return true;
    }
    // General shapes: tiles aligned to the buffer, owned by the shard of their first row.
    while (true) {
      while (ti >= tend) {
        if (++t >= P->t_end) return false;
        const int32_t s = (r0 - t + m.N) % m.N;
        ti = (s * m.c + kBM - 1) / kBM;
        tend = ((s + 1) * m.c + kBM - 1) / kBM;
      }
      const int64_t p0 = ti * kBM;
      ++ti;
      const int64_t p1 = p0 + kBM < P->S ? p0 + kBM : P->S;
      int64_t gmin, gmax;
      m.grange(p0, p1, gmin, gmax);
      if (P->causal && gmin > qgmax) continue;
      out.p0 = p0;
      out.step = m.gstep(p0, p1);
      out.gk0 = out.step ? m.g(p0) : -1;
      out.gmin = gmin;
      out.gmax = gmax;
      out.valid = (int32_t)(p1 - p0);
      return true;
    }
  }
};

// Per-row context of one K/V tile for the softmax.
struct RowCtx {
  float c2, sl, base, slope2;
  int64_t gi, gk0, step;
  int32_t valid;
  bool causal, row_ok, alibi;
  const volatile int32_t* gtab;
};

enum TileKind { kPlain = 0, kLinear = 1, kGeneral = 2, kMasked = 3 };

// Score of column u in the log2 domain.  kPlain keeps the raw score (scaled
// inside the exponent); kLinear adds the ALiBi bias of a tile that lies wholly
// on one side of every query; kGeneral masks and biases element by element.
// kMasked (no bias; the visible keys of each row are the columns up to a row
// limit, as on a causal diagonal or a ragged tile) takes the kPlain path with the
// columns past the limit set to -inf.
// `lin` is the ALiBi term of this column for kLinear (c.base + c.sl * u), else unused.
template <int kKind>
__device__ __forceinline__ float tile_score(int u, float raw, float lin, const RowCtx& c) {
  if constexpr (kKind == kPlain) {
    return raw;
  } else if constexpr (kKind == kLinear) {
    return fmaf(raw, c.c2, lin);
  } else {
    const int64_t gj = c.step ? c.gk0 + c.step * u : (int64_t)c.gtab[u];
    const bool vis = c.row_ok && u < c.valid && (!c.causal || gj <= c.gi);
    float v = raw * c.c2;
    if (c.alibi) v -= c.slope2 * (float)(c.gi > gj ? c.gi - gj : gj - c.gi);
    return vis ? v : -INFINITY;
  }
}

// kPlain and kMasked tiles: the row's 128 scores are read from TMEM once and both
// passes run from registers.  kLinear and kGeneral tiles keep the two rolled TMEM
// passes (their per-column bias terms or per-element positions would not fit
// beside 128 held scores without spilling).
using SRow = uint32_t[4][32];

// Columns u > lim of a row are not visible: their scores become -inf.
__device__ __forceinline__ void mask_after(SRow& sr, int lim) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch)
#pragma unroll
    for (int u = 0; u < 32; ++u)
      if (32 * ch + u > lim) sr[ch][u] = 0xff800000u;  // -inf
}

__device__ __forceinline__ float plain_max(const SRow& sr, float c2) {
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int ch = 0; ch < 4; ++ch)
#pragma unroll
    for (int u = 0; u < 32; u += 2)
      mx[(u >> 1) & 3] = tc::max3(mx[(u >> 1) & 3], __uint_as_float(sr[ch][u]), __uint_as_float(sr[ch][u + 1]));
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2;
}

template <bool kFp8>
__device__ __forceinline__ float plain_probs(uint32_t t_s, const SRow& sr, float mu, float c2) {
  if constexpr (!kFp8) {
    float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t pk[32];
#pragma unroll
      for (int ci = 0; ci < 2; ++ci)
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const uint32_t* r = sr[2 * hf + ci];
          const float2 x = tc::fma2(make_float2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])),
                                    make_float2(c2, c2), make_float2(-mu, -mu));
          const float pa = tc::ex2(x.x), pb = tc::ex2(x.y);
          ls2[u & 1] = tc::add2(ls2[u & 1], make_float2(pa, pb));
          pk[16 * ci + u] = tc::pack_bf16(pa, pb);
        }
      tc::tmem_st32(t_s + 32 * hf, pk);
    }
    return (ls2[0].x + ls2[1].x) + (ls2[0].y + ls2[1].y);
  } else {
    float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t pk[16];
#pragma unroll
      for (int ci = 0; ci < 2; ++ci)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t* r = sr[2 * hf + ci];
          const float2 x0 = tc::fma2(make_float2(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1])),
                                     make_float2(c2, c2), make_float2(-mu, -mu));
          const float2 x1 = tc::fma2(make_float2(__uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])),
                                     make_float2(c2, c2), make_float2(-mu, -mu));
          const float2 p0 = make_float2(tc::ex2(x0.x), tc::ex2(x0.y));
          const float2 p1 = make_float2(tc::ex2(x1.x), tc::ex2(x1.y));
          ls2[u & 1] = tc::add2(ls2[u & 1], tc::add2(p0, p1));
          pk[8 * ci + u] = tc::pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
        }
      tc::tmem_st16(t_s + 16 * hf, pk);
    }
    return (ls2[0].x + ls2[1].x) + (ls2[0].y + ls2[1].y);
  }
}

template <int kKind>
__device__ __forceinline__ float tile_max(uint32_t t_s, const RowCtx& c) {
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t r[32];
    tc::tmem_ld32(t_s + 32 * ch, r);
    // ALiBi term of column 32ch + u is lb + sl*u: the chunk's part once, the
    // column's part an immediate (no per-element int -> float conversion)
    const float lb = fmaf(c.sl, (float)(32 * ch), c.base);
    tc::tmem_wait_ld();
#pragma unroll
    for (int u = 0; u < 32; u += 2)
      mx[(u >> 1) & 3] =
          tc::max3(mx[(u >> 1) & 3], tile_score<kKind>(32 * ch + u, __uint_as_float(r[u]), fmaf(c.sl, (float)u, lb), c),
                   tile_score<kKind>(32 * ch + u + 1, __uint_as_float(r[u + 1]), fmaf(c.sl, (float)(u + 1), lb), c));
  }
  const float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
  return kKind == kPlain ? m * c.c2 : m;
}

template <int kKind, bool kFp8>
__device__ __forceinline__ float tile_probs(uint32_t t_s, float mu, const RowCtx& c) {
  float ls[4] = {0.f, 0.f, 0.f, 0.f};
  float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // bf16 path: pairs of partial sums
  auto prob = [&](float s) -> float {
    if constexpr (kKind == kPlain) return tc::ex2(fmaf(s, c.c2, -mu));
    else return tc::ex2(s - mu);
  };
  if constexpr (!kFp8) {
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t pk[32];
      // kLinear: the row's reference folded into the bias base first, so the
      // exponent is formed from small numbers even where the bias is large
      const float lbm = fmaf(c.sl, (float)(64 * hf), c.base - mu);
#pragma unroll
      for (int ci = 0; ci < 2; ++ci) {
        uint32_t r[32];
        tc::tmem_ld32(t_s + 64 * hf + 32 * ci, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int col = 64 * hf + 32 * ci + 2 * u;
          float2 x;  // exponent arguments of the column pair, scaled to the log2 domain
          if constexpr (kKind == kPlain) {
            x = tc::fma2(make_float2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])),
                         make_float2(c.c2, c.c2), make_float2(-mu, -mu));
          } else if constexpr (kKind == kLinear) {
            // raw * c2 + (ALiBi term of the column - mu)
            const float2 lin = tc::fma2(make_float2(c.sl, c.sl),
                                        make_float2((float)(32 * ci + 2 * u), (float)(32 * ci + 2 * u + 1)),
                                        make_float2(lbm, lbm));
            x = tc::fma2(make_float2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])),
                         make_float2(c.c2, c.c2), lin);
          } else {
            x = make_float2(tile_score<kKind>(col, __uint_as_float(r[2 * u]), 0.f, c) - mu,
                            tile_score<kKind>(col + 1, __uint_as_float(r[2 * u + 1]), 0.f, c) - mu);
          }
          const float pa = tc::ex2(x.x), pb = tc::ex2(x.y);
          ls2[u & 1] = tc::add2(ls2[u & 1], make_float2(pa, pb));
          pk[16 * ci + u] = tc::pack_bf16(pa, pb);
        }
      }
      tc::tmem_st32(t_s + 32 * hf, pk);
    }
  } else {
    // e4m3: four probabilities per TMEM column; columns 64hf.. of S become P
    // columns 16hf.. (all inside the S columns read in the first half).
#pragma unroll 1
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t pk[16];
      const float lbm = fmaf(c.sl, (float)(64 * hf), c.base - mu);  // kLinear, as above
#pragma unroll
      for (int ci = 0; ci < 2; ++ci) {
        uint32_t r[32];
        tc::tmem_ld32(t_s + 64 * hf + 32 * ci, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float pv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cc = 32 * ci + 4 * u + e;
            const float raw = __uint_as_float(r[4 * u + e]);
            if constexpr (kKind == kLinear) pv[e] = tc::ex2(fmaf(raw, c.c2, fmaf(c.sl, (float)cc, lbm)));
            else pv[e] = prob(tile_score<kKind>(64 * hf + cc, raw, 0.f, c));
          }
          ls[u & 3] += (pv[0] + pv[1]) + (pv[2] + pv[3]);
          pk[8 * ci + u] = tc::pack_e4m3x4(pv[0], pv[1], pv[2], pv[3]);
        }
      }
      tc::tmem_st16(t_s + 16 * hf, pk);
    }
  }
  if constexpr (!kFp8) return (ls2[0].x + ls2[1].x) + (ls2[0].y + ls2[1].y);
  return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// The column term is taken relative to the tile's middle column (kBiasMid), which
// halves its largest magnitude, slope2 * step * 64 in log2 units.  The fp32 score
// accumulator holds the term to about 2^-24 of that; up to kMaxMmaColumnTerm
// (≈ 1.2e-4 in the exponent, far below the bf16 rounding of P) the tensor core
// carries it.  Heads with steeper slopes run in a second launch of the
// per-element form (launch_fwd_tc).
constexpr int kBiasMid = 64;
constexpr float kMaxMmaColumnTerm = 2048.0f;

// Whether head hh's ALiBi column term can ride on the Q K^T product (every CTA of
// both launches of a causal ALiBi forward evaluates the same expression).
__device__ __forceinline__ bool column_term_fits(const FwdParams& P, int hh) {
  const float t = fabsf(P.slopes[hh] * kLog2e) * (float)P.map.run_step() * (float)kBiasMid;
  return t <= kMaxMmaColumnTerm;  // false for NaN slopes too
}

// Fills the column-term blocks: K row u holds the four bf16 parts of
// w_u = slope2 * step * (u - 64) / c2 (the term in raw-score units, so that
// c2 * w_u is the log2-domain bias of column u relative to column 64) in columns
// 0..3 and zeros in 4..15; every Q row holds ones in columns 0..3.  Row r of an
// 8-row atom keeps its 16-byte chunk c at chunk c ^ r (the 128-byte swizzle).
// Called by threads 0..135 before the block-wide barrier that precedes the first MMA.
__device__ __forceinline__ void fill_bias_blocks(uint8_t* qext, uint8_t* kext, float slope2, float step,
                                                 float c2) {
  const int t = threadIdx.x;
  uint32_t w[4] = {0u, 0u, 0u, 0u};  // chunk 0 of the row: 8 bf16 as 4 pairs
  uint8_t* row;
  int r;
  if (t < kBM) {
    // the exact term in fp64, then four successive bf16 roundings of what is left
    double rest = (double)slope2 * (double)step * (double)(t - kBiasMid) / (double)c2;
    __nv_bfloat16 part[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      part[i] = __double2bfloat16(rest);
      rest -= (double)__bfloat162float(part[i]);
    }
    w[0] = (uint32_t)__bfloat16_as_ushort(part[0]) | ((uint32_t)__bfloat16_as_ushort(part[1]) << 16);
    w[1] = (uint32_t)__bfloat16_as_ushort(part[2]) | ((uint32_t)__bfloat16_as_ushort(part[3]) << 16);
    row = kext + (t >> 3) * 1024;
    r = t & 7;
  } else if (t < kBM + 8) {
    const uint32_t one = (uint32_t)__bfloat16_as_ushort(__float2bfloat16(1.0f));
    w[0] = w[1] = one | (one << 16);
    row = qext;
    r = t - kBM;
  } else {
    return;
  }
  uint4* chunk0 = reinterpret_cast<uint4*>(row + r * 128 + ((0 ^ r) << 4));
  uint4* chunk1 = reinterpret_cast<uint4*>(row + r * 128 + ((1 ^ r) << 4));
  *chunk0 = make_uint4(w[0], w[1], w[2], w[3]);
  *chunk1 = make_uint4(0u, 0u, 0u, 0u);
  // make the generic-proxy stores visible to the tensor core's reads
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <bool kFp8>
__device__ __forceinline__ void issue_s(uint32_t tmem, uint32_t sbase, int X, int ks, bool bias_mma) {
  using C = FwdCfg<kFp8>;
  const uint32_t qa = sbase + C::kOffQ + X * C::kTileBytes;
  const uint32_t kb = sbase + C::kOffK + ks * C::kTileBytes;
#pragma unroll
  for (int kk = 0; kk < C::kSteps; ++kk) {
    // four 32-byte K steps per 128-byte swizzle row, then the next box
    const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
    const uint64_t a = tc::smem_desc(qa + off, 16, 1024);
    const uint64_t b = tc::smem_desc(kb + off, 16, 1024);
    if constexpr (kFp8) tc::mma_ss_f8(tmem + X * 128, a, b, C::kIdescS, kk > 0 ? 1u : 0u);
    else tc::mma_ss(tmem + X * 128, a, b, C::kIdescS, kk > 0 ? 1u : 0u);
  }
  if constexpr (!kFp8) {
    if (bias_mma) {
      // + ones . (column term): the 8-row Q atom serves all 16 row groups (stride 0)
      const uint64_t a = tc::smem_desc(sbase + C::kOffQext, 16, 0);
      const uint64_t b = tc::smem_desc(sbase + C::kOffKext, 16, 1024);
      tc::mma_ss(tmem + X * 128, a, b, C::kIdescS, 1u);
    }
  }
}

template <bool kFp8>
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t sbase, int X, int vs, bool acc) {
  using C = FwdCfg<kFp8>;
  const uint32_t vb = sbase + C::kOffV + vs * C::kTileBytes;
#pragma unroll
  for (int kk = 0; kk < C::kPvSteps; ++kk) {
    // V is [kv rows, d] with d contiguous: MN-major B.  kKStep kv rows per step
    // (128 bytes each); the 64-wide d halves of bf16 are one box (16 KB) apart.
    const uint64_t b = tc::smem_desc(vb + kk * C::kKStep * 128, C::kBoxBytes, 1024);
    if constexpr (kFp8)
      tc::mma_ts_f8(tmem + 256 + X * 128, tmem + X * 128 + kk * 8, b, C::kIdescPV, (acc || kk > 0) ? 1u : 0u);
    else
      tc::mma_ts(tmem + 256 + X * 128, tmem + X * 128 + kk * 8, b, C::kIdescPV, (acc || kk > 0) ? 1u : 0u);
  }
}

// How a kernel instantiation adds the ALiBi bias: not at all (no slopes), on the
// tensor core (causal, aligned, bf16: see the header), or per element in the
// softmax (every other case).  kAligned (every 256-row query pair and 128-row tile
// in one run of arithmetic positions) drops the per-element path from the
// unbiased instantiation.  Each instantiation holds only the tile paths its case
// uses, which keeps the softmax warps' registers and code within their budget.
enum BiasMode { kBiasNone = 0, kBiasMma = 1, kBiasElem = 2 };

template <bool kFp8, int kBias, bool kAligned>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FwdParams P) {
  using C = FwdCfg<kFp8>;
  // aligned bf16: the tile walk and the row checks known at compile time (measured
  // faster for bf16 and slower for e4m3, whose instantiations keep the run-time form)
  constexpr bool kStaticWalk = kAligned && !kFp8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + C::kOffTmemSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SeqMap& m = P.map;
  const int64_t S = P.S;

  // Work item: (b, h) major, then the pair index (heaviest first when causal and
  // aligned).  Resident CTAs then belong to one or two heads and share that
  // head's K/V tiles in L2 (with heads minor, the resident CTAs spanned every head,
  // whose tensors sit at power-of-two strides, and nearly every K/V tile load
  // went to DRAM).
  const int64_t L = blockIdx.x;
  const int64_t npairs = (S + 255) / 256;
  const int64_t bh = L / npairs;
  const int64_t pair = L - bh * npairs;
  const int hh = (int)(bh % P.H);
  // Heaviest pairs first under causal.  Consecutive positions (zig-zag, contiguous):
  // the pair holding the latest 256 positions first.  Token-strided: every shard's
  // slots hold increasing positions, so pair k takes shard k mod N's (k div N)-th
  // pair from the end.
  int64_t P0 = 256 * pair;
  if (P.heavy_first == 1) P0 = m.inv(S - 256 * (pair + 1));
  else if (P.heavy_first == 2) P0 = (pair % m.N) * m.c + m.c - 256 * (pair / m.N + 1);
  const int64_t qend = P0 + 256 < S ? P0 + 256 : S;
  int64_t pair_gmin, pair_gmax;
  m.grange(P0, qend, pair_gmin, pair_gmax);
  const int32_t r0 = m.shard(P0);
  // A causal ALiBi forward runs as two launches: the tensor-core form for the heads
  // whose column term fits, the per-element form for the rest; each CTA of the
  // other launch's heads returns at once (the whole block, before any barrier).
  if (P.head_filter != 0 && (P.head_filter == 1) != column_term_fits(P, hh)) return;
  const bool bias_mma = kBias == kBiasMma;
  if constexpr (!kFp8 && kBias == kBiasMma) {
    if (bias_mma)
      fill_bias_blocks(sgen + C::kOffQext, sgen + C::kOffKext, P.slopes[hh] * kLog2e, (float)m.run_step(), P.c2);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kBarPFull || i == kBarPFull + 1) cnt = 128;
      if (i == kBarEpiDone) cnt = 8;
      mbar_init(bar(i), cnt);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(sbase + C::kOffTmemSlot, kTmemCols);
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
      const int32_t z = (int32_t)bh;
      mbar_arrive_expect_tx(bar(kBarQFull), 2 * C::kTileBytes);
      for (int X = 0; X < 2; ++X)
        for (int hf = 0; hf < C::kBoxes; ++hf)
          tc::tma_load_3d(sbase + C::kOffQ + X * C::kTileBytes + hf * C::kBoxBytes, &tm_q, hf * C::kBoxCols,
                          (int32_t)(P0 + X * kBM), z, bar(kBarQFull));
      KvWalk<kStaticWalk> walk;
      walk.init(&P, pair_gmax, r0);
      TileInfo tile;
      int j = 0;          // tiles whose K load was issued
      bool last_v = true; // whether the V load of tile j-1 was issued too
      bool ok = true;
      while (ok && walk.next(tile)) {
        const int st = j % kStages;
        const uint32_t par = ((j / kStages) & 1) ^ 1;
        ok = mbar_wait(bar(kBarKEmpty + st), par, P.status, kKernFwdTc, kSiteKEmpty);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(kBarKFull + st), C::kTileBytes);
        for (int hf = 0; hf < C::kBoxes; ++hf)
          tc::tma_load_3d(sbase + C::kOffK + st * C::kTileBytes + hf * C::kBoxBytes, &tm_k, hf * C::kBoxCols,
                          (int32_t)tile.p0, z, bar(kBarKFull + st));
        ok = mbar_wait(bar(kBarVEmpty + st), par, P.status, kKernFwdTc, kSiteVEmpty);
        if (!ok) {
          ++j;  // the K load of this tile is in flight, its V load is not
          last_v = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarVFull + st), C::kTileBytes);
        for (int hf = 0; hf < C::kBoxes; ++hf)
          tc::tma_load_3d(sbase + C::kOffV + st * C::kTileBytes + hf * C::kBoxBytes, &tm_v, hf * C::kBoxCols,
                          (int32_t)tile.p0, z, bar(kBarVFull + st));
        ++j;
      }
      // Let every load this warp issued land before the CTA can exit.
      mbar_wait(bar(kBarQFull), 0, P.status, kKernFwdTc, kSiteQFull);
      for (int back = 1; back <= kStages && back <= j; ++back) {
        const int jj = j - back;
        const int st = jj % kStages;
        const uint32_t par = (jj / kStages) & 1;
        mbar_wait(bar(kBarKFull + st), par, P.status, kKernFwdTc, kSiteKFull);
        if (last_v || back > 1) mbar_wait(bar(kBarVFull + st), par, P.status, kKernFwdTc, kSiteVFull);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      KvWalk<kStaticWalk> walk;
      walk.init(&P, pair_gmax, r0);
      TileInfo tile;
      bool ok = mbar_wait(bar(kBarQFull), 0, P.status, kKernFwdTc, kSiteQFull);
      if (ok && walk.next(tile)) {
        ok = mbar_wait(bar(kBarKFull + 0), 0, P.status, kKernFwdTc, kSiteKFull);
        if (ok) {
          tc::fence_after_sync();
          issue_s<kFp8>(tmem, sbase, 0, 0, bias_mma);
          tc::mma_commit(bar(kBarSFull + 0));
          issue_s<kFp8>(tmem, sbase, 1, 0, bias_mma);
          tc::mma_commit(bar(kBarSFull + 1));
          tc::mma_commit(bar(kBarKEmpty + 0));
        }
        int j = 0;
        while (ok) {
          const bool more = walk.next(tile);
          const int vs = j % kStages;
          const int ks = (j + 1) % kStages;
          ok = mbar_wait(bar(kBarVFull + vs), (j / kStages) & 1, P.status, kKernFwdTc, kSiteVFull) &&
               mbar_wait(bar(kBarPFull + 0), j & 1, P.status, kKernFwdTc, kSitePFull);
          if (!ok) break;
          tc::fence_after_sync();
          issue_pv<kFp8>(tmem, sbase, 0, vs, j > 0);
          if (more) {
            ok = mbar_wait(bar(kBarKFull + ks), ((j + 1) / kStages) & 1, P.status, kKernFwdTc, kSiteKFull);
            if (!ok) break;
            tc::fence_after_sync();
            issue_s<kFp8>(tmem, sbase, 0, ks, bias_mma);
            tc::mma_commit(bar(kBarSFull + 0));
          } else {
            tc::mma_commit(bar(kBarODone + 0));
          }
          ok = mbar_wait(bar(kBarPFull + 1), j & 1, P.status, kKernFwdTc, kSitePFull);
          if (!ok) break;
          tc::fence_after_sync();
          issue_pv<kFp8>(tmem, sbase, 1, vs, j > 0);
          tc::mma_commit(bar(kBarVEmpty + vs));
          if (more) {
            issue_s<kFp8>(tmem, sbase, 1, ks, bias_mma);
            tc::mma_commit(bar(kBarSFull + 1));
            tc::mma_commit(bar(kBarKEmpty + ks));
          } else {
            tc::mma_commit(bar(kBarODone + 1));
            break;
          }
          ++j;
        }
      } else if (ok) {
        tc::mma_commit(bar(kBarODone + 0));
        tc::mma_commit(bar(kBarODone + 1));
      }
      // Every MMA this thread issued completes before TMEM is released.
      tc::mma_commit(bar(kBarFinal));
      mbar_wait(bar(kBarFinal), 0, P.status, kKernFwdTc, kSiteODone);
      tc::fence_before_sync();
    }
    __syncwarp();
    mbar_wait(bar(kBarEpiDone), 0, P.status, kKernFwdTc, kSiteODone);
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------- softmax
    const int X = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int64_t qp0 = P0 + X * kBM;
    const int64_t slot = qp0 + row;
    const bool row_ok = kStaticWalk || slot < S;
    const int64_t gi = row_ok ? m.g(slot) : 0;
    const bool tile_has_rows = kStaticWalk || qp0 < S;
    int64_t qgmin = 0, qgmax = -1;
    if (tile_has_rows) m.grange(qp0, qp0 + kBM < S ? qp0 + kBM : S, qgmin, qgmax);
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + X * 128;
    const uint32_t t_o = tmem + lane_off + 256 + X * 128;
    const float c2 = P.c2;
    const bool alibi = kBias != kBiasNone;
    const float slope2 = alibi ? P.slopes[hh] * kLog2e : 0.f;
    volatile int32_t* gtab = reinterpret_cast<volatile int32_t*>(sgen + C::kOffGtab) + warp * kBM;

    float m_ref = -INFINITY, l = 0.f;
    KvWalk<kStaticWalk> walk;
    walk.init(&P, pair_gmax, r0);
    TileInfo tile;
    int j = 0;
    bool ok = true;
    while (walk.next(tile)) {
      // Classify the tile for this Q tile (before waiting for its scores).
      const bool below = tile.gmax <= qgmin;              // every key at or before every query
      const bool above = !P.causal && tile.gmin >= qgmax; // every key at or after every query
      // kPlain: every key visible to every row, no bias; kLinear: the same with an
      // ALiBi bias linear in the column (tile on one side of every query and its
      // positions arithmetic); kMasked: no bias, visible keys a prefix of the
      // columns; kGeneral: element by element.
      // With the ALiBi column term on the tensor core the tile's scores already
      // carry it, and the row part is an offset of the reference (below).
      const bool visible_all = tile_has_rows && tile.valid == kBM && (P.causal ? below : true);
      int kind;
      if constexpr (kBias == kBiasNone)
        kind = visible_all ? kPlain : (kAligned || tile.step != 0 || !P.causal ? kMasked : kGeneral);
      else if constexpr (kBias == kBiasMma)
        kind = visible_all ? kPlain : kMasked;  // (aligned: every step != 0)
      else
        kind = visible_all && (below || above) && tile.step != 0 ? kLinear : kGeneral;

      // kMasked: key u of the tile is visible to this row iff u <= lim (u < valid,
      // and under causal gk0 + step * u <= gi)
      int lim = -1;
      if (kind == kMasked && row_ok) {
        lim = tile.valid - 1;
        if (P.causal) {
          const int64_t dlt = gi - tile.gk0;
          if (dlt < 0) lim = -1;
          else if (dlt < (int64_t)lim * tile.step) lim = (int)(dlt / tile.step);
        }
      }
      if (kind == kGeneral && tile.step == 0) {
        // Keys of this tile come from several chunks: the warp maps the 128 slots
        // (four per lane) into its own table.
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int u = lane + 32 * e;
          gtab[u] = u < tile.valid ? (int32_t)m.g(tile.p0 + u) : 0;
        }
        __syncwarp();
      }
      RowCtx rc;
      rc.c2 = c2;
      rc.sl = (below ? slope2 : -slope2) * (float)tile.step;
      rc.base = below ? slope2 * (float)(tile.gk0 - gi) : slope2 * (float)(gi - tile.gk0);
      rc.slope2 = slope2;
      rc.gi = gi;
      rc.gk0 = tile.gk0;
      rc.valid = tile.valid;
      rc.step = tile.step;
      rc.causal = P.causal != 0;
      rc.row_ok = row_ok;
      rc.alibi = alibi;
      rc.gtab = gtab;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + X), j & 1, P.status, kKernFwdTc, kSiteSFull));
      if (!ok) break;
      tc::fence_after_sync();
      // Move the reference max only when the tile's max exceeds it by > 8; returns
      // the offset the probabilities are taken against.
      auto move_max = [&](float mt) -> float {
        const bool need = mt > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mt : m_ref;
          const float alpha = need ? (m_ref == -INFINITY ? 0.f : tc::ex2(m_ref - m_new)) : 1.f;
          if (j > 0) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t r[32];
              tc::tmem_ld32(t_o + 32 * c, r);
              tc::tmem_wait_ld();
#pragma unroll
              for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * alpha);
              tc::tmem_st32(t_o + 32 * c, r);
            }
          }
          l *= alpha;
          m_ref = m_new;
        }
        return m_ref == -INFINITY ? 0.f : m_ref;
      };
      // Pass 1: the row max of this tile (log2 domain); pass 2: probabilities,
      // packed to bf16 pairs and stored over S columns that have already been read
      // (P column k holds scores 2k, 2k+1).
      if (kBias != kBiasElem && (kind == kPlain || kind == kMasked)) {
        SRow sr;
        tc::tmem_ld128(t_s, sr);
        tc::tmem_wait_ld();
        if (kind == kMasked) mask_after(sr, lim);
        const float pm = plain_max(sr, c2);
        if constexpr (kBias == kBiasMma) {
          // the row part slope2 * (g(column 64) - g_i) as an unevaluated sum (exact product)
          const float dk = (float)(tile.gk0 + kBiasMid * tile.step - gi);
          const float bhi = slope2 * dk;
          const float blo = fmaf(slope2, dk, -bhi);
          const float mu = move_max(pm + bhi);
          l += plain_probs<kFp8>(t_s, sr, (mu - bhi) - blo, c2);
        } else {
          const float mu = move_max(pm);
          l += plain_probs<kFp8>(t_s, sr, mu, c2);
        }
      } else if (kBias == kBiasElem && kind == kLinear) {
        const float mu = move_max(tile_max<kLinear>(t_s, rc));
        l += tile_probs<kLinear, kFp8>(t_s, mu, rc);
      } else if constexpr (kBias != kBiasMma && !(kBias == kBiasNone && kAligned)) {
        const float mu = move_max(tile_max<kGeneral>(t_s, rc));
        l += tile_probs<kGeneral, kFp8>(t_s, mu, rc);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(bar(kBarPFull + X));
      ++j;
    }
    // ------------------------------------------------------------- epilogue
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarODone + X), 0, P.status, kKernFwdTc, kSiteODone));
    if (ok) {
      tc::fence_after_sync();
      // only l == 0 means "no visible key"; NaN inputs keep l (and O) NaN
      const float inv_l = l == 0.f ? 0.f : P.o_scale / l;
      const int64_t orow_off = (bh * S + (row_ok ? slot : 0)) * kD;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(t_o + 32 * c, r);
        tc::tmem_wait_ld();
        if (P.o_f32 != nullptr) {  // ring-step partial: fp32 rows
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(P.o_f32 + orow_off + 32 * c);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              dst[u] = l != 0.f ? make_float4(__uint_as_float(r[4 * u]) * inv_l, __uint_as_float(r[4 * u + 1]) * inv_l,
                                              __uint_as_float(r[4 * u + 2]) * inv_l, __uint_as_float(r[4 * u + 3]) * inv_l)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          continue;
        }
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = l != 0.f ? tc::pack_bf16(__uint_as_float(r[2 * u]) * inv_l, __uint_as_float(r[2 * u + 1]) * inv_l)
                          : 0u;
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(P.o + orow_off + 32 * c);
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      if (row_ok) P.lse[bh * S + slot] = l != 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarEpiDone));
  }
}

}  // namespace

bool fwd_tc_supported(int64_t S, int64_t D, int32_t dtype) {
  return (dtype == RA_BF16 || dtype == RA_E4M3) && D == kD && S >= kBM;
}

namespace {

template <bool kFp8, int kBias, bool kAligned>
cudaError_t launch_fwd_tc_t(const AttnArgs& a, void* o, float* lse, cudaStream_t st, int32_t head_filter = 0) {
  using C = FwdCfg<kFp8>;
  const int64_t BH = a.B * a.H;
  if (BH > INT32_MAX) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  auto make = [&](CUtensorMap* m, const void* base) {
    return kFp8 ? tc::make_tmap_bhsd_u8(m, base, BH, a.S, a.D, kBM) : tc::make_tmap_bhsd(m, base, BH, a.S, a.D, kBM);
  };
  if (!make(&tq, a.q) || !make(&tk, a.k) || !make(&tv, a.v)) return cudaErrorInvalidValue;
  FwdParams p;
  p.map = a.map;
  p.S = a.S;
  p.H = (int32_t)a.H;
  p.BH = (int32_t)BH;
  p.causal = a.causal;
  // aligned: every 256-row query pair and 128-row tile lies in one run of
  // arithmetic positions (a zig-zag chunk, or a shard otherwise).
  p.aligned = (a.map.run() % 256) == 0;
  // Heaviest pairs first under causal, where pairs hold consecutive positions (in
  // the strided layout every pair already has about the same work).
  p.heavy_first = !(p.aligned && a.causal) ? 0 : (a.map.layout == RA_LAYOUT_STRIDED ? 2 : 1);
  p.head_filter = head_filter;
  p.slopes = a.slopes;
  p.c2 = a.scale * a.qk_scale * kLog2e;
  p.o_scale = a.v_scale;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.o_f32 = a.o_f32;
  p.t_begin = a.t_begin;
  p.t_end = a.t_end;
  p.lse = lse;
  p.status = a.status;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(fwd_tc_kernel<kFp8, kBias, kAligned>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t pairs = (a.S + 255) / 256;
  const int64_t blocks = pairs * BH;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  fwd_tc_kernel<kFp8, kBias, kAligned><<<(unsigned)blocks, kThreads, C::kSmemBytes, st>>>(tq, tk, tv, p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const AttnArgs& a, void* o, float* lse, cudaStream_t st) {
  // aligned: every 256-row query pair and 128-row tile lies in one run of arithmetic
  // positions, so the unbiased instantiation needs no per-element path
  const bool aligned = (a.map.run() % 256) == 0;
  if (a.slopes == nullptr) {
    if (a.dtype == RA_E4M3)
      return aligned ? launch_fwd_tc_t<true, kBiasNone, true>(a, o, lse, st)
                     : launch_fwd_tc_t<true, kBiasNone, false>(a, o, lse, st);
    return aligned ? launch_fwd_tc_t<false, kBiasNone, true>(a, o, lse, st)
                   : launch_fwd_tc_t<false, kBiasNone, false>(a, o, lse, st);
  }
  if (a.dtype == RA_E4M3) return launch_fwd_tc_t<true, kBiasElem, false>(a, o, lse, st);
  // the tensor core takes the column term when every visible key lies at or
  // before its query (causal) and every tile's positions are arithmetic (aligned)
  if (!(a.causal && aligned)) return launch_fwd_tc_t<false, kBiasElem, false>(a, o, lse, st);
  // heads whose column term fits the tensor core, then (per element) the others
  const cudaError_t e = launch_fwd_tc_t<false, kBiasMma, true>(a, o, lse, st, 1);
  return e != cudaSuccess ? e : launch_fwd_tc_t<false, kBiasElem, false>(a, o, lse, st, 2);
}

}  // namespace ra
