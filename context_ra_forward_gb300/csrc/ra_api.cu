// ra_api.cu — the C ABI of include/ra.h: argument validation, dispatch to the
// kernels on the caller's stream, and the device status word.
//
// Nothing here allocates device memory at call time.  The status word is a
// file-scope __device__ array that exists from library load; its device address
// is looked up once per device and handed to kernels that have bounded waits.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>

#include "ra_common.cuh"
#include "ra_kernels.h"

namespace {

__device__ int32_t g_status_word[ra::kStatusWords];

constexpr int kMaxDevices = 64;
int32_t* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

// Device address of the status word for the current device (looked up once).
ra_status status_word(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return RA_ERR_CUDA;
    g_status_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_status_ptr[dev];
  return RA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t elem_bytes(ra_dtype dt) { return dt == RA_F32 ? 4 : (dt == RA_E4M3 ? 1 : 2); }

// Shared scalar checks; returns RA_OK or the first error.
ra_status check_sizes(int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dt, int32_t N,
                      ra_layout layout) {
  if (B < 0 || H < 0 || S < 0) return RA_ERR_INVALID_ARG;
  if (dt != RA_F32 && dt != RA_BF16 && dt != RA_E4M3) return RA_ERR_UNSUPPORTED;
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIDED)
    return RA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return RA_ERR_UNSUPPORTED;
  if (N < 1) return RA_ERR_INVALID_ARG;
  const int64_t parts = layout == RA_LAYOUT_ZIGZAG ? 2 * (int64_t)N : (int64_t)N;
  if (S % parts) return RA_ERR_INVALID_ARG;
  // row index arithmetic in the kernels: S * D 16-byte chunks per head must stay
  // below 2^31, and B*H*S*D elements below 2^62.
  if (S > 0 && (S * D * elem_bytes(dt) / 16) >= (int64_t(1) << 31)) return RA_ERR_UNSUPPORTED;
  if (B > 0 && H > 0 && S > 0 && (double)B * H * S * D >= 4.0e18) return RA_ERR_UNSUPPORTED;
  return RA_OK;
}

bool overlaps(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bytes && y < x + bytes;
}

// [a, a + na) and [b, b + nb) intersect
bool overlaps2(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

ra_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return RA_OK;
  g_last_cuda_error = e;
  return RA_ERR_CUDA;
}

float resolve_scale(float s, int64_t D) { return s > 0.f ? s : 1.0f / sqrtf((float)D); }

ra_status permute_common(const void* x, void* y, int64_t B, int64_t H, int64_t S, int64_t D,
                         ra_dtype dt, int32_t N, ra_layout layout, void* stream, bool inverse) {
  ra_status s = check_sizes(B, H, S, D, dt, N, layout);
  if (s != RA_OK) return s;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  if (!x || !y) return RA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return RA_ERR_MISALIGNED;
  const int64_t row_bytes = D * elem_bytes(dt);
  if (overlaps(x, y, (size_t)(B * H * S * row_bytes))) return RA_ERR_INVALID_ARG;
  const ra::SeqMap m = ra::SeqMap::make(S, N, layout);
  return from_cuda(ra::launch_permute(x, y, B * H, S, row_bytes, m, inverse,
                                      static_cast<cudaStream_t>(stream)));
}

ra_status rope_common(const void* x, void* y, int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dt,
                      int32_t N, ra_layout layout, double base, int64_t pos0, void* stream, bool inverse) {
  ra_status s = check_sizes(B, H, S, D, dt, N, layout);
  if (s != RA_OK) return s;
  if (dt == RA_E4M3) return RA_ERR_UNSUPPORTED;
  if (!(base > 1.0) || !isfinite(base)) return RA_ERR_INVALID_ARG;
  if (pos0 < 0 || pos0 + S > (int64_t(1) << 31)) return RA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  if (!x || !y) return RA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return RA_ERR_MISALIGNED;
  if (overlaps(x, y, (size_t)(B * H * S * D * elem_bytes(dt)))) return RA_ERR_INVALID_ARG;
  // theta_i / (2 pi) as a 64-bit binary fraction: below 1/(2 pi) since base > 1
  ra::RopeTurns turns;
  memset(&turns, 0, sizeof(turns));
  const double inv_two_pi = 0.15915494309189535;
  for (int64_t i = 0; i < D / 2; ++i) {
    const double theta = 1.0 / pow(base, (double)(2 * i) / (double)D);
    turns.f[i] = (uint64_t)llrint(ldexp(theta * inv_two_pi, 64));
  }
  const ra::SeqMap m = ra::SeqMap::make(S, N, layout);
  return from_cuda(ra::launch_rope_permute(x, y, B, H, S, D, dt, m, inverse, pos0, turns,
                                           static_cast<cudaStream_t>(stream)));
}

bool is_sm103() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
  return major == 10 && minor == 3;
}

ra_status attn_args(const void* q, const void* k, const void* v, int64_t B, int64_t H, int64_t S,
                    int64_t D, ra_dtype dt, int32_t causal, const float* slopes, float scale,
                    int32_t N, ra_layout layout, ra::AttnArgs* a) {
  a->q = q;
  a->k = k;
  a->v = v;
  a->B = B;
  a->H = H;
  a->S = S;
  a->D = D;
  a->dtype = dt;
  a->causal = causal ? 1 : 0;
  a->slopes = slopes;
  a->scale = resolve_scale(scale, D);
  if (!(a->scale > 0.f) || !isfinite(a->scale)) return RA_ERR_INVALID_ARG;
  a->map = ra::SeqMap::make(S, N, layout);
  a->t_begin = 0;
  a->t_end = N;
  a->o_f32 = nullptr;
  a->qk_scale = 1.f;
  a->v_scale = 1.f;
  return status_word(&a->status);
}

std::atomic<int64_t> g_launches{0};
int32_t g_last_sites[ra::kStatusWarps] = {};

}  // namespace

namespace ra {
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace ra

extern "C" {

int64_t ra_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* ra_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "cudaSuccess" : cudaGetErrorName(g_last_cuda_error);
}


const char* ra_status_string(ra_status s) {
  switch (s) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
    case RA_ERR_MISALIGNED: return "RA_ERR_MISALIGNED";
    case RA_ERR_CUDA: return "RA_ERR_CUDA";
    case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT";
    case RA_ERR_WORKSPACE: return "RA_ERR_WORKSPACE";
    default: return "RA_ERR_UNKNOWN";
  }
}

ra_status ra_index_map(int64_t S, int32_t N, ra_layout layout, int64_t* perm_host, int64_t* inv_host) {
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIDED)
    return RA_ERR_UNSUPPORTED;
  if (S < 0 || N < 1) return RA_ERR_INVALID_ARG;
  const int64_t parts = layout == RA_LAYOUT_ZIGZAG ? 2 * (int64_t)N : (int64_t)N;
  if (S % parts) return RA_ERR_INVALID_ARG;
  const ra::SeqMap m = ra::SeqMap::make(S, N, layout);
  for (int64_t p = 0; p < S; ++p) {
    if (perm_host) perm_host[p] = m.g(p);
    if (inv_host) inv_host[p] = m.inv(p);
  }
  return RA_OK;
}

ra_status ra_shard_work(int64_t S, int32_t N, ra_layout layout, int32_t causal, int64_t* pairs_host,
                        int64_t* tiles_full_host, int64_t* tiles_partial_host) {
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_ZIGZAG && layout != RA_LAYOUT_STRIDED)
    return RA_ERR_UNSUPPORTED;
  if (S < 0 || N < 1) return RA_ERR_INVALID_ARG;
  const int64_t parts = layout == RA_LAYOUT_ZIGZAG ? 2 * (int64_t)N : (int64_t)N;
  if (S % parts) return RA_ERR_INVALID_ARG;
  if (S > (int64_t(1) << 22)) return RA_ERR_UNSUPPORTED;  // the tile count is quadratic in S
  const ra::SeqMap m = ra::SeqMap::make(S, N, layout);
  const int64_t c = m.c;
  constexpr int64_t T = 128;
  // global position ranges of the K/V tiles (128 slots of the shard-major buffer)
  const int64_t nk = (S + T - 1) / T;
  int64_t* kmin = new (std::nothrow) int64_t[nk > 0 ? nk : 1];
  int64_t* kmax = new (std::nothrow) int64_t[nk > 0 ? nk : 1];
  if (!kmin || !kmax) {
    delete[] kmin;
    delete[] kmax;
    return RA_ERR_UNSUPPORTED;
  }
  for (int64_t b = 0; b < nk; ++b) m.grange(b * T, (b + 1) * T < S ? (b + 1) * T : S, kmin[b], kmax[b]);
  for (int32_t r = 0; r < N; ++r) {
    int64_t pairs = 0, full = 0, partial = 0;
    for (int64_t p = r * c; p < (r + 1) * c; ++p) pairs += causal ? m.g(p) + 1 : S;
    for (int64_t a = r * c; a < (r + 1) * c; a += T) {  // the shard's query tiles
      int64_t qmin, qmax;
      m.grange(a, a + T < (r + 1) * c ? a + T : (r + 1) * c, qmin, qmax);
      for (int64_t b = 0; b < nk; ++b) {
        if (!causal || kmax[b] <= qmin) ++full;
        else if (kmin[b] <= qmax) ++partial;
      }
    }
    if (pairs_host) pairs_host[r] = pairs;
    if (tiles_full_host) tiles_full_host[r] = full;
    if (tiles_partial_host) tiles_partial_host[r] = partial;
  }
  delete[] kmin;
  delete[] kmax;
  return RA_OK;
}

ra_status ra_zigzag_permute(const void* x, void* y, int64_t B, int64_t H, int64_t S, int64_t D,
                            ra_dtype dt, int32_t N, ra_layout layout, void* stream) {
  return permute_common(x, y, B, H, S, D, dt, N, layout, stream, false);
}

ra_status ra_unpermute(const void* x, void* y, int64_t B, int64_t H, int64_t S, int64_t D,
                       ra_dtype dt, int32_t N, ra_layout layout, void* stream) {
  return permute_common(x, y, B, H, S, D, dt, N, layout, stream, true);
}

ra_status ra_rope_permute(const void* x, void* y, int64_t B, int64_t H, int64_t S, int64_t D,
                          ra_dtype dt, int32_t N, ra_layout layout, double base, int64_t pos0, void* stream) {
  return rope_common(x, y, B, H, S, D, dt, N, layout, base, pos0, stream, false);
}

ra_status ra_rope_unpermute(const void* x, void* y, int64_t B, int64_t H, int64_t S, int64_t D,
                            ra_dtype dt, int32_t N, ra_layout layout, double base, int64_t pos0,
                            void* stream) {
  return rope_common(x, y, B, H, S, D, dt, N, layout, base, pos0, stream, true);
}

int32_t ra_forward_path(int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dt, int32_t N,
                        ra_layout layout) {
  const ra_status s = check_sizes(B, H, S, D, dt, N, layout);
  if (s != RA_OK) return s;
  if (dt == RA_E4M3 && (D != 128 || S < 128) && B > 0 && H > 0 && S > 0) return RA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || S == 0) return 0;
  return ra::fwd_tc_supported(S, D, dt) ? 1 : 2;
}

int32_t ra_backward_path(int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dt, int32_t N,
                         ra_layout layout) {
  const ra_status s = check_sizes(B, H, S, D, dt, N, layout);
  if (s != RA_OK) return s;
  if (dt == RA_E4M3) return RA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || S == 0) return 0;
  return ra::bwd_tc_supported(S, D, dt, ra::SeqMap::make(S, N, layout)) ? 1 : 2;
}

ra_status ra_forward(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                     int64_t H, int64_t S, int64_t D, ra_dtype dt, int32_t causal,
                     const float* slopes, float scale, int32_t N, ra_layout layout, void* stream) {
  ra_status s = check_sizes(B, H, S, D, dt, N, layout);
  if (s != RA_OK) return s;
  if (dt == RA_E4M3) return RA_ERR_UNSUPPORTED;  // 8-bit inputs need scales: ra_forward_fp8
  if (!(scale <= 0.f || isfinite(scale))) return RA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  if (!q || !k || !v || !o || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return RA_ERR_MISALIGNED;
  if (!aligned(lse, 4) || (slopes && !aligned(slopes, 4))) return RA_ERR_MISALIGNED;
  const size_t bytes = (size_t)(B * H * S * D * elem_bytes(dt));
  if (overlaps(o, q, bytes) || overlaps(o, k, bytes) || overlaps(o, v, bytes)) return RA_ERR_INVALID_ARG;
  if (!is_sm103()) return RA_ERR_UNSUPPORTED;
  ra::AttnArgs a;
  s = attn_args(q, k, v, B, H, S, D, dt, causal, slopes, scale, N, layout, &a);
  if (s != RA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (ra::fwd_tc_supported(S, D, dt)) return from_cuda(ra::launch_fwd_tc(a, o, lse, st));
  return from_cuda(ra::launch_fwd_simt(a, o, lse, st));
}

ra_status ra_forward_fp8(const void* q, const void* k, const void* v, float q_scale, float k_scale,
                         float v_scale, void* o, float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                         int32_t causal, const float* slopes, float scale, int32_t N, ra_layout layout,
                         void* stream) {
  ra_status s = check_sizes(B, H, S, D, RA_E4M3, N, layout);
  if (s != RA_OK) return s;
  if (!(scale <= 0.f || isfinite(scale))) return RA_ERR_INVALID_ARG;
  if (!(q_scale > 0.f) || !(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(q_scale) || !isfinite(k_scale) ||
      !isfinite(v_scale))
    return RA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  if (!ra::fwd_tc_supported(S, D, RA_E4M3)) return RA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return RA_ERR_MISALIGNED;
  if (!aligned(lse, 4) || (slopes && !aligned(slopes, 4))) return RA_ERR_MISALIGNED;
  const size_t in_bytes = (size_t)(B * H * S * D), out_bytes = 2 * in_bytes;
  if (overlaps2(o, out_bytes, q, in_bytes) || overlaps2(o, out_bytes, k, in_bytes) || overlaps2(o, out_bytes, v, in_bytes))
    return RA_ERR_INVALID_ARG;
  if (!is_sm103()) return RA_ERR_UNSUPPORTED;
  ra::AttnArgs a;
  s = attn_args(q, k, v, B, H, S, D, RA_E4M3, causal, slopes, scale, N, layout, &a);
  if (s != RA_OK) return s;
  a.qk_scale = q_scale * k_scale;
  a.v_scale = v_scale;
  return from_cuda(ra::launch_fwd_tc(a, o, lse, static_cast<cudaStream_t>(stream)));
}

ra_status ra_forward_ring_step(const void* q, const void* k, const void* v, float* o_step, float* lse_step,
                               int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dt, int32_t causal,
                               const float* slopes, float scale, int32_t N, ra_layout layout, int32_t step,
                               void* stream) {
  ra_status s = check_sizes(B, H, S, D, dt, N, layout);
  if (s != RA_OK) return s;
  if (dt == RA_E4M3) return RA_ERR_UNSUPPORTED;  // 8-bit inputs need scales: ra_forward_fp8
  if (!(scale <= 0.f || isfinite(scale))) return RA_ERR_INVALID_ARG;
  if (step < 0 || step >= N) return RA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  const ra::SeqMap m = ra::SeqMap::make(S, N, layout);
  // every 256-row query block and 128-row key tile must lie inside one shard run
  if (m.run() % 256 != 0) return RA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o_step || !lse_step) return RA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o_step, 16)) return RA_ERR_MISALIGNED;
  if (!aligned(lse_step, 4) || (slopes && !aligned(slopes, 4))) return RA_ERR_MISALIGNED;
  const size_t in_bytes = (size_t)(B * H * S * D * elem_bytes(dt));
  const size_t out_bytes = (size_t)(B * H * S * D * 4);
  if (overlaps2(o_step, out_bytes, q, in_bytes) || overlaps2(o_step, out_bytes, k, in_bytes) ||
      overlaps2(o_step, out_bytes, v, in_bytes))
    return RA_ERR_INVALID_ARG;
  if (!is_sm103()) return RA_ERR_UNSUPPORTED;
  ra::AttnArgs a;
  s = attn_args(q, k, v, B, H, S, D, dt, causal, slopes, scale, N, layout, &a);
  if (s != RA_OK) return s;
  a.t_begin = step;
  a.t_end = step + 1;
  a.o_f32 = o_step;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (ra::fwd_tc_supported(S, D, dt)) return from_cuda(ra::launch_fwd_tc(a, nullptr, lse_step, st));
  return from_cuda(ra::launch_fwd_simt(a, nullptr, lse_step, st));
}

ra_status ra_lse_merge(float* o_acc, float* lse_acc, const float* o_step, const float* lse_step, void* out,
                       ra_dtype out_dtype, int64_t B, int64_t H, int64_t S, int64_t D, void* stream) {
  if (B < 0 || H < 0 || S < 0) return RA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return RA_ERR_UNSUPPORTED;
  if (out && out_dtype != RA_F32 && out_dtype != RA_BF16) return RA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  if (!o_acc || !lse_acc || !o_step || !lse_step) return RA_ERR_INVALID_ARG;
  if (!aligned(o_acc, 16) || !aligned(o_step, 16) || (out && !aligned(out, 16))) return RA_ERR_MISALIGNED;
  if (!aligned(lse_acc, 4) || !aligned(lse_step, 4)) return RA_ERR_MISALIGNED;
  const int64_t rows = B * H * S;
  if (overlaps(o_acc, o_step, (size_t)(rows * D * 4)) || overlaps(lse_acc, lse_step, (size_t)(rows * 4)))
    return RA_ERR_INVALID_ARG;
  return from_cuda(ra::launch_lse_merge(o_acc, lse_acc, o_step, lse_step, out, out_dtype, rows, D,
                                        static_cast<cudaStream_t>(stream)));
}

size_t ra_backward_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D) {
  if (B <= 0 || H <= 0 || S <= 0 || D <= 0) return 0;
  const size_t rows = (size_t)(B * H * S);
  const size_t dvec = (rows * 4 + 255) / 256 * 256;
  const size_t dq = (rows * (size_t)D * 4 + 255) / 256 * 256;
  return dvec + dq;
}

}  // extern "C"

namespace ra {

ra_status backward_precheck(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S,
                            int64_t D, ra_dtype dt, const float* slopes, float scale, int32_t N,
                            ra_layout layout) {
  ra_status s = check_sizes(B, H, S, D, dt, N, layout);
  if (s != RA_OK) return s;
  if (dt == RA_E4M3) return RA_ERR_UNSUPPORTED;  // 8-bit inputs need scales: ra_forward_fp8
  if (!(scale <= 0.f || isfinite(scale))) return RA_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return RA_ERR_INVALID_ARG;
  const void* in16[] = {q, k, v, o, dout, dq, dk, dv};
  for (const void* p : in16)
    if (!aligned(p, 16)) return RA_ERR_MISALIGNED;
  if (!aligned(lse, 4) || (slopes && !aligned(slopes, 4))) return RA_ERR_MISALIGNED;
  return RA_OK;
}

}  // namespace ra

extern "C" {

ra_status ra_backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, void* workspace,
                      size_t ws_bytes, int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dt,
                      int32_t causal, const float* slopes, float scale, int32_t N,
                      ra_layout layout, void* stream) {
  ra_status s = ra::backward_precheck(q, k, v, o, lse, dout, dq, dk, dv, B, H, S, D, dt, slopes, scale, N, layout);
  if (s != RA_OK) return s;
  if (B == 0 || H == 0 || S == 0) return RA_OK;
  const size_t need = ra_backward_workspace_bytes(B, H, S, D);
  if (!workspace || ws_bytes < need) return RA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return RA_ERR_MISALIGNED;
  const size_t bytes = (size_t)(B * H * S * D * elem_bytes(dt));
  const void* outs[] = {dq, dk, dv};
  const void* ins[] = {q, k, v, o, dout};
  for (const void* x : outs) {
    for (const void* y : ins)
      if (overlaps(x, y, bytes)) return RA_ERR_INVALID_ARG;
    if (overlaps2(x, bytes, workspace, ws_bytes) || (x != dq && overlaps(x, dq, bytes))) return RA_ERR_INVALID_ARG;
  }
  if (overlaps(dk, dv, bytes)) return RA_ERR_INVALID_ARG;
  if (!is_sm103()) return RA_ERR_UNSUPPORTED;
  ra::AttnArgs a;
  s = attn_args(q, k, v, B, H, S, D, dt, causal, slopes, scale, N, layout, &a);
  if (s != RA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)(B * H * S);
  float* dvec = static_cast<float*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + (rows * 4 + 255) / 256 * 256);
  const bool tc = ra::bwd_tc_supported(S, D, dt, a.map) && aligned(lse, 16);
  cudaError_t e = ra::launch_bwd_rowdot(a, o, dout, dvec, tc ? dq_acc : nullptr, st);
  if (e != cudaSuccess) return from_cuda(e);
  if (tc) return from_cuda(ra::launch_bwd_tc(a, lse, dout, dvec, dq_acc, dq, dk, dv, st));
  return from_cuda(ra::launch_bwd_simt(a, lse, dout, dvec, dq, dk, dv, st));
}

ra_status ra_check_device_status(void* stream, int32_t* detail_host) {
  int32_t* word = nullptr;
  if (status_word(&word) != RA_OK) return RA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return RA_ERR_CUDA;
  int32_t h[ra::kStatusWords] = {};
  if (cudaMemcpy(h, word, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return RA_ERR_CUDA;
  if (h[0] != 0) {
    memcpy(g_last_sites, h + 4, sizeof(g_last_sites));
    const int32_t zero[ra::kStatusWords] = {};
    if (cudaMemcpy(word, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return RA_ERR_CUDA;
  }
  if (detail_host) memcpy(detail_host, h, 4 * sizeof(int32_t));
  if (h[0] == RA_ERR_TIMEOUT) return RA_ERR_TIMEOUT;
  return h[0] == 0 ? RA_OK : RA_ERR_CUDA;
}

int32_t ra_debug_wait_sites(int32_t* host, int32_t n) {
  const int32_t m = n < ra::kStatusWarps ? n : ra::kStatusWarps;
  if (host) memcpy(host, g_last_sites, (size_t)(m > 0 ? m : 0) * sizeof(int32_t));
  return ra::kStatusWarps;
}

ra_status ra_debug_wait_timeout(int32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 2000000) return RA_ERR_INVALID_ARG;
  int32_t* word = nullptr;
  if (status_word(&word) != RA_OK) return RA_ERR_CUDA;
  return from_cuda(ra::launch_debug_wait(limit_us, word, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
