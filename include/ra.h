/*
 * ra.h — ring / zig-zag blockwise exact attention on one GPU (sm_103a): C ABI.
 *
 * Pages cited (titles as printed):
 *   [CP] "百万Token上下文训练的挑战与突破" — §2.1 序列切分策略对比 (split the
 *        sequence into N equal pieces along the sequence dimension), §3.1 环形通信拓扑
 *        (device i receives the K/V of device i-1, combines, passes on).
 *   [ZZ] "大模型如何訓練百萬 Token 上下文：上下文并行與 Ring Attention" — §Zig Zag Ring
 *        Attention (every shard's Q meets every K/V block, one ring step at a time;
 *        interleaved assignment balances causal work; indexing is more involved).
 *   [LC] "超长上下文技术" survey (intelliparadigm.com 2061774) — §2.1.2 ALiBi (scores
 *        scaled by 1/sqrt(head dim), bias -|i-j|*slope added), §3.1.2 FlashAttention
 *        (blockwise evaluation with a running max and sum; recompute in backward).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are [B, H, S, D] (batch, heads, sequence, head dim), contiguous, D
 *    innermost.  Q/K/V/O/dO/dQ/dK/dV of one call share one dtype: RA_F32 (fp32) or
 *    RA_BF16 (bf16) (ra_forward_fp8 and the permutes also take RA_E4M3).  LSE is
 *    always fp32 [B, H, S].  D must be 64 or 128.
 *  - Sequence order.  Attention calls take and return tensors in SHARD-MAJOR order:
 *    the N shards' token sequences concatenated, shard 0 first, which is what
 *    ra_zigzag_permute produces.  Global token positions (for the causal mask and
 *    ALiBi) are recovered from the slot index by the layout's closed form.
 *  - Layouts.  RA_LAYOUT_CONTIGUOUS: shard r holds tokens [r*S/N, (r+1)*S/N)
 *    ([CP] §2.1), needs S % N == 0.  RA_LAYOUT_ZIGZAG: the sequence is cut into 2N
 *    chunks of h = S/(2N) tokens; shard r holds chunk r followed by chunk 2N-1-r
 *    ([ZZ] §Zig Zag, 2N-chunk form), needs S % (2N) == 0.  RA_LAYOUT_STRIDED: shard r
 *    holds tokens r, r+N, r+2N, ... ([ZZ] §Zig Zag as printed: "GPU 0 gets tokens
 *    [0, 4, 8...], GPU 1 gets [1, 5, 9...]"), needs S % N == 0.
 *  - Pointers named "device" are CUDA device pointers (e.g. from PyTorch) and must
 *    be 16-byte aligned (LSE and the slopes: 4-byte aligned).  The caller owns every
 *    buffer; the library allocates no memory at call time and keeps no per-call
 *    state.  (A device status word, created when the library is loaded, records
 *    the first bounded-wait timeout a kernel hits; see ra_check_device_status.)
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All compute
 *    calls are asynchronous on it; arguments are validated on the host before any
 *    launch and a failed validation launches nothing.  No C++ exception crosses
 *    this interface.
 *  - Zero-size problems (B, H or S == 0) validate their scalar arguments and
 *    return RA_OK without launching.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ra_status;
#define RA_OK                 0
#define RA_ERR_INVALID_ARG   -1  /* NULL pointer, bad size, S not divisible, N < 1, aliasing */
#define RA_ERR_UNSUPPORTED   -2  /* D not 64/128, unknown dtype/layout, not an sm_103 device */
#define RA_ERR_MISALIGNED    -3  /* a pointer not aligned as stated above */
#define RA_ERR_CUDA          -4  /* a CUDA runtime/driver call or launch failed */
#define RA_ERR_TIMEOUT       -5  /* a bounded in-kernel wait expired (ra_check_device_status) */
#define RA_ERR_WORKSPACE     -6  /* backward workspace missing or too small */

typedef int32_t ra_dtype;
#define RA_F32   0
#define RA_BF16  1
#define RA_E4M3  2   /* 8-bit float (4 exponent, 3 mantissa bits): ra_forward_fp8 and the permutes */

typedef int32_t ra_layout;
#define RA_LAYOUT_CONTIGUOUS 0
#define RA_LAYOUT_ZIGZAG     1
#define RA_LAYOUT_STRIDED    2

/*
 * ra_index_map — the sequence -> shard assignment as explicit tables (host only).
 * [CP] §2.1 (contiguous), [ZZ] §Zig Zag (2N-chunk interleave; token-strided).
 *   perm_host[p] = global token position held at shard-major slot p;
 *   inv_host[g]  = shard-major slot of global position g.
 * Both are caller-owned host arrays of S int64 (either may be NULL to skip it).
 * Errors: RA_ERR_INVALID_ARG (S < 0, N < 1, S not divisible), RA_ERR_UNSUPPORTED
 * (unknown layout).
 */
ra_status ra_index_map(int64_t S, int32_t N, ra_layout layout,
                       int64_t* perm_host, int64_t* inv_host);

/*
 * ra_shard_work — how the attention work of one head splits over the shards (host
 * only): the balance the 2N-chunk assignment is for ([ZZ] §Zig Zag: under a
 * causal mask the contiguous split leaves the last shard with far more visible
 * pairs than the first; the interleaved one gives every shard the same work).
 * For each shard r (arrays of N int64, caller-owned host memory; any may be NULL):
 *   pairs_host[r]:         (query, key) pairs visible to the shard's queries
 *                          (causal: sum over its queries of g + 1; else S per query);
 *   tiles_full_host[r]:    128 x 128 tiles (the shard's 128-slot query tiles against
 *                          the 128-slot key tiles of the shard-major buffer) whose
 *                          every pair is visible;
 *   tiles_partial_host[r]: tiles with some but not all pairs visible (the causal
 *                          diagonals the kernels mask); fully masked tiles are skipped.
 * Multiply by B*H for a whole problem.  Errors: as ra_index_map, plus
 * RA_ERR_UNSUPPORTED for S > 2^22 (the tile count is quadratic in S).
 */
ra_status ra_shard_work(int64_t S, int32_t N, ra_layout layout, int32_t causal, int64_t* pairs_host,
                        int64_t* tiles_full_host, int64_t* tiles_partial_host);

/*
 * ra_zigzag_permute — y[b,h,p,:] = x[b,h,perm(p),:]: original order -> shard-major.
 * [ZZ] §Zig Zag ("the index logic is slightly more involved"), [CP] §2.1.
 *   x, y: device, [B,H,S,D] of `dtype`; must not overlap.  A bit-exact row copy.
 * The name is kept for both layouts; with RA_LAYOUT_CONTIGUOUS it is a plain copy.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_MISALIGNED, RA_ERR_CUDA.
 */
ra_status ra_zigzag_permute(const void* x, void* y, int64_t B, int64_t H, int64_t S,
                            int64_t D, ra_dtype dtype, int32_t N, ra_layout layout,
                            void* stream);

/*
 * ra_unpermute — the inverse: y[b,h,g,:] = x[b,h,inv(g),:] (shard-major -> original).
 * Same arguments, layout and errors as ra_zigzag_permute.
 */
ra_status ra_unpermute(const void* x, void* y, int64_t B, int64_t H, int64_t S,
                       int64_t D, ra_dtype dtype, int32_t N, ra_layout layout,
                       void* stream);

/*
 * ra_rope_permute — rotary position embedding fused with the permute:
 *   y[b,h,p,:] = R(pos0 + g) x[b,h,g,:],  g = perm(p)   (original -> shard-major).
 * [LC] §2.1.3 RoPE: the position enters Q and K through a rotation.  For a row at
 * position t and each i in [0, D/2), with theta_i = 1 / base^(2i/D):
 *   y[i]       = x[i] cos(t theta_i) - x[i + D/2] sin(t theta_i)
 *   y[i + D/2] = x[i] sin(t theta_i) + x[i + D/2] cos(t theta_i)
 * The position is the row's GLOBAL index g in the original sequence plus pos0
 * (pos0 = 0 for a sequence that starts at position 0), so every shard's rows are
 * rotated by their true positions whatever the layout.  Apply it to Q and K (not V,
 * not dO) in place of ra_zigzag_permute.
 *   x: device [B,H,S,D] `dtype`, original order; y: device, same shape, shard-major.
 *   dtype: RA_F32 or RA_BF16 (the rotation runs in fp32, y is rounded once).
 *   base: > 1 (the page's value is 10000).  pos0 >= 0 with pos0 + S <= 2^31.
 * The angle t * theta_i is reduced to a fraction of a turn exactly (64-bit
 * fixed-point turns per position): cos and sin carry an absolute error of a few
 * 1e-7 at every position, where an fp32 angle product is off by up to 2^-6 rad
 * near position 2^18 (its rounding bound; 7.8e-3 rad measured at t = 2^18).
 * Errors: as ra_zigzag_permute; RA_ERR_UNSUPPORTED for RA_E4M3; RA_ERR_INVALID_ARG
 * for base <= 1 or not finite, pos0 out of range, x and y overlapping.
 */
ra_status ra_rope_permute(const void* x, void* y, int64_t B, int64_t H, int64_t S,
                          int64_t D, ra_dtype dtype, int32_t N, ra_layout layout,
                          double base, int64_t pos0, void* stream);

/*
 * ra_rope_unpermute — the transpose of ra_rope_permute:
 *   y[b,h,g,:] = R(pos0 + g)^T x[b,h,inv(g),:]   (shard-major -> original).
 * R^T is the rotation by the negated angle, so this is both the inverse of
 * ra_rope_permute (up to rounding) and the map that takes the gradients dQ and dK
 * of the rotated, shard-major Q and K back to gradients of the caller's original
 * Q and K.  Same arguments, layout and errors as ra_rope_permute.
 */
ra_status ra_rope_unpermute(const void* x, void* y, int64_t B, int64_t H, int64_t S,
                            int64_t D, ra_dtype dtype, int32_t N, ra_layout layout,
                            double base, int64_t pos0, void* stream);

/*
 * ra_forward — exact softmax attention over N virtual ring shards.
 * [ZZ] §Zig Zag (each shard's Q meets every K/V block in ring-step order: at step
 * t shard r meets the K/V of shard (r-t) mod N), [CP] §3.1, [LC] §3.1.2 (blockwise
 * evaluation with running max m and running sum l; partials across ring steps are
 * merged through the log-sum-exp), [LC] §2.1.2 (scale and ALiBi).
 *   q, k, v:  device, [B,H,S,D] `dtype`, shard-major order.
 *   o:        device, [B,H,S,D] `dtype`, shard-major order (written).
 *   lse:      device, fp32 [B,H,S], shard-major (written): natural-log
 *             log-sum-exp of each row's scaled, biased, visible scores.
 *   causal:   nonzero -> key j is visible to query i iff g(j) <= g(i), g = global
 *             position (diagonal visible).
 *   alibi_slopes: device fp32 [H] or NULL; adds -|g(i)-g(j)| * slopes[h] to the
 *             scaled score.
 *   softmax_scale: <= 0 selects 1/sqrt(D).
 * bf16 runs on the tensor cores (fp32 accumulation, P rounded to bf16 for the PV
 * product); fp32 runs in exact fp32 arithmetic on the CUDA cores.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_MISALIGNED, RA_ERR_CUDA.
 */
ra_status ra_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dtype,
                     int32_t causal, const float* alibi_slopes, float softmax_scale,
                     int32_t N, ra_layout layout, void* stream);

/*
 * ra_forward_fp8 — ra_forward with e4m3 (8-bit float) Q, K, V and per-tensor
 * scales: the value of an element is its e4m3 number times the tensor's scale.
 * Same method and ring order as ra_forward ([ZZ] §Zig Zag, [LC] §3.1.2, §2.1.2);
 * the products run on the tensor cores at the 8-bit rate (kind::f8f6f4, fp32
 * accumulation) and the probabilities are rounded to e4m3 for the PV product
 * (relative rounding error <= 2^-4 per probability), so O carries a relative RMS
 * error of a few percent; LSE comes from fp32 sums.
 *   q, k, v: device, [B,H,S,D] e4m3 bytes (RA_E4M3), shard-major.
 *   q_scale, k_scale, v_scale: > 0, finite.
 *   o: device bf16 [B,H,S,D] (written); lse: device fp32 [B,H,S] (written).
 *   D must be 128 and S >= 128 (else RA_ERR_UNSUPPORTED).  Other arguments and
 *   errors as ra_forward.
 */
ra_status ra_forward_fp8(const void* q, const void* k, const void* v, float q_scale, float k_scale,
                         float v_scale, void* o, float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                         int32_t causal, const float* alibi_slopes, float softmax_scale, int32_t N,
                         ra_layout layout, void* stream);

/*
 * ra_forward_ring_step — one ring step of the forward as a separate partial result:
 * the queries of every shard r against the K/V of shard (r - step) mod N only
 * ([ZZ] §Zig Zag, one ring step; [CP] §3.1: device i works on the K/V received
 * from device i-1).  This is the dataflow of a multi-device ring, where each
 * step's partial is merged as the next K/V block arrives (ra_lse_merge).
 *   q, k, v: as ra_forward (device, [B,H,S,D] `dtype`, shard-major).
 *   o_step:  device fp32 [B,H,S,D] (written): the partial output, normalised over
 *            the step's visible keys; 0 for a row that sees none of them.
 *   lse_step: device fp32 [B,H,S] (written): the step's log-sum-exp (-inf: none).
 *   step: 0 <= step < N.  Other arguments as ra_forward.
 * Needs every shard run (S/N slots, or the S/(2N)-token chunks of RA_LAYOUT_ZIGZAG)
 * to be a multiple of 256 slots, else RA_ERR_UNSUPPORTED.  Errors as ra_forward.
 */
ra_status ra_forward_ring_step(const void* q, const void* k, const void* v, float* o_step, float* lse_step,
                               int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dtype, int32_t causal,
                               const float* alibi_slopes, float softmax_scale, int32_t N, ra_layout layout,
                               int32_t step, void* stream);

/*
 * ra_lse_merge — merges a partial result into an accumulated one through their
 * log-sum-exp ([ZZ] §Zig Zag: the partials of the ring steps combine into exact
 * attention): per row,
 *   LSE = log(e^lse_acc + e^lse_step),
 *   O   = e^(lse_acc - LSE) o_acc + e^(lse_step - LSE) o_step,
 * written back into (o_acc, lse_acc); a side with LSE = -inf contributes nothing.
 *   o_acc, o_step: device fp32 [B,H,S,D]; lse_acc, lse_step: device fp32 [B,H,S].
 *   Start the accumulation from the first step's partial (its buffers).
 *   out: device [B,H,S,D] of `out_dtype` (RA_F32 or RA_BF16) or NULL; when given,
 *   also receives the merged O (e.g. on the last step).
 *   D must be 64 or 128.  Any row order works (the merge is per row).
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_MISALIGNED, RA_ERR_CUDA.
 */
ra_status ra_lse_merge(float* o_acc, float* lse_acc, const float* o_step, const float* lse_step, void* out,
                       ra_dtype out_dtype, int64_t B, int64_t H, int64_t S, int64_t D, void* stream);

/*
 * ra_backward_workspace_bytes — device scratch ra_backward needs for these sizes:
 * an fp32 [B,H,S] row term D_i = dO_i . O_i and an fp32 [B,H,S,D] dQ accumulator,
 * each 256-byte aligned.  Returns 0 for an empty problem.
 */
size_t ra_backward_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D);

/*
 * ra_backward — dQ, dK, dV of ra_forward, recomputing each block's probabilities
 * from the saved LSE ([LC] §3.1.2 recompute strategy).  The gradient equations are
 * the analytic derivative of the forward (the pages give none):
 *   D_i = dO_i.O_i;  P_ij = exp(s_ij - LSE_i);  dS_ij = P_ij (dO_i.V_j - D_i);
 *   dV_j = sum_i P_ij dO_i;  dQ_i = scale sum_j dS_ij K_j;  dK_j = scale sum_i dS_ij Q_i.
 *   q, k, v, o, dout: device [B,H,S,D] `dtype`, shard-major; lse: device fp32
 *   [B,H,S] from ra_forward with the same arguments.  The tensor-core kernel (see
 *   ra_backward_path) reads LSE rows 16 bytes at a time: an LSE that is only
 *   4-byte aligned is accepted, and such a call runs the CUDA-core kernel.
 *   dq, dk, dv: device [B,H,S,D] `dtype`, shard-major (written).
 *   workspace: device, >= ra_backward_workspace_bytes(B,H,S,D) bytes, 256-byte
 *   aligned, caller-owned; its contents on entry do not matter.
 * Other arguments as ra_forward.  ALiBi slopes and the mask get no gradient.
 * Errors: as ra_forward, plus RA_ERR_WORKSPACE.
 */
ra_status ra_backward(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      void* workspace, size_t workspace_bytes,
                      int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dtype,
                      int32_t causal, const float* alibi_slopes, float softmax_scale,
                      int32_t N, ra_layout layout, void* stream);

/*
 * ra_backward_noalloc — ra_backward for callers that cannot allocate device memory
 * when they run the backward: a plug-in inside a host framework that owns every
 * device allocation and lets no library allocate on its behalf, a program whose
 * device memory is fixed once at start-up, or a latency-bound loop that cannot
 * take an allocation's implicit device synchronisation.  The pages have no
 * counterpart to this call: it only changes where the backward's scratch lives.
 *   Instead of a caller-provided workspace it uses a fixed scratch buffer inside
 * the library: RA_NOALLOC_SCRATCH_BYTES (32 MiB) of device memory that every GPU
 * which loads the library holds until the process exits.  Problems whose
 * ra_backward_workspace_bytes(B,H,S,D) exceeds that are rejected with
 * RA_ERR_WORKSPACE before anything is launched (use ra_backward for them).
 *   All other arguments, layouts, results and errors are those of ra_backward.
 * The call allocates nothing.  Its first call on a device looks up the buffer's
 * device address (once per device, with that device current), so make that first
 * call before any stream capture.  Argument errors are found before the size
 * check, so an invalid call gets exactly the error ra_backward would give it.  Every call reuses the same buffer: calls that
 * may overlap on the GPU (different streams without ordering, or several host
 * threads) race on it and must be serialised by the caller.  The buffer keeps the
 * last call's contents; each call clears what it needs before using it.
 */
#define RA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
ra_status ra_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dtype,
                              int32_t causal, const float* alibi_slopes, float softmax_scale,
                              int32_t N, ra_layout layout, void* stream);

/* ra_noalloc_scratch_bytes — size of the buffer ra_backward_noalloc uses (bytes). */
size_t ra_noalloc_scratch_bytes(void);

/* ra_status_string — a static, human-readable name for a status code. */
const char* ra_status_string(ra_status status);

/*
 * ra_check_device_status — synchronises `stream`, then reads and clears the device
 * status word.  Returns RA_ERR_TIMEOUT if a kernel gave up on a bounded wait since
 * the last check (its outputs are then not valid), RA_ERR_CUDA on a CUDA error,
 * RA_OK otherwise.  While the word holds a failure, kernels with bounded waits
 * give up at their first wait that does not succeed at once (fail-stop), so
 * check the status after a timeout before trusting further results.  `detail_host` (may be NULL) receives 4 int32: code, kernel id,
 * block index, wait site.
 */
ra_status ra_check_device_status(void* stream, int32_t* detail_host);

/*
 * ra_forward_path — which kernel ra_forward would run for these arguments:
 * 1 = tensor-core (tcgen05) kernel, 2 = CUDA-core fp32 kernel, 0 = nothing to do,
 * a negative ra_status if the arguments would be rejected.  Host only, no launch.
 */
int32_t ra_forward_path(int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dtype,
                        int32_t N, ra_layout layout);

/*
 * ra_backward_path — which kernel ra_backward would run for these arguments, given
 * a 16-byte aligned LSE (the tensor-core kernel reads LSE and D rows 16 bytes at a
 * time): 1 = tensor-core (tcgen05) kernel, 2 = CUDA-core fp32 kernel, 0 = nothing
 * to do, a negative ra_status if the arguments would be rejected.  The tensor-core
 * kernel takes bf16 with D = 128 and S >= 128 when each run of consecutive
 * positions (a zig-zag chunk or a strided shard) is at least 128 slots long, so a
 * 128-slot tile meets at most one run boundary; the contiguous layout is one run.
 * Host only, no launch.
 */
int32_t ra_backward_path(int64_t B, int64_t H, int64_t S, int64_t D, ra_dtype dtype,
                         int32_t N, ra_layout layout);

/*
 * ra_debug_wait_sites — after ra_check_device_status reported a failure: for the
 * block that failed first, what each of its warps was waiting on when its wait
 * gave up, one int32 per warp (site << 24 | parity << 16 | low 16 bits of the
 * barrier's shared-memory address; 0 = the warp did not give up).  Copies up to n
 * entries to `host` (may be NULL) and returns how many entries exist.  Host only.
 */
int32_t ra_debug_wait_sites(int32_t* host, int32_t n);

/*
 * ra_debug_wait_timeout — failure-detection self test.  Launches one block whose
 * warp waits on an mbarrier that nothing ever arrives on, with a limit of
 * `limit_us` microseconds; the wait gives up, records RA_ERR_TIMEOUT in the device
 * status word and the kernel returns normally (no trap, no fault).  A following
 * ra_check_device_status must report RA_ERR_TIMEOUT.
 */
ra_status ra_debug_wait_timeout(int32_t limit_us, void* stream);

/*
 * ra_last_cuda_error — name of the CUDA error behind this thread's most recent
 * RA_ERR_CUDA (a static string; "cudaSuccess" if there was none).
 */
const char* ra_last_cuda_error(void);

/*
 * ra_kernel_launch_count — number of kernels this library has launched in this
 * process so far (a host-side counter, incremented at each launch).  Lets a caller
 * count the library's launches inside a timed region.
 */
int64_t ra_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* RA_H_ */
