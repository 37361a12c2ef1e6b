/*
 * fp8rl.h -- C ABI of the GB300 (sm_103a) FP8 rollout hot path.
 *
 * The operations are those of "FP8-RL: A Practical and Stable Low-Precision
 * Stack for LLM Reinforcement Learning" (arXiv 2601.18150), as described by
 * its long-form summary page (sections 3.4.1-3.4.4) and abstract:
 *   - per-step blockwise re-quantization of BF16 policy weights into E4M3
 *     with one FP32 scale per 128x128 block,
 *   - per-token 1x128-group dynamic activation quantization,
 *   - a blockwise-scaled FP8 W8A8 GEMM with FP32 accumulation and BF16
 *     output, plus a grouped variant for MoE experts,
 *   - FP8 E4M3 KV-cache quantization with per-head scales,
 *   - token-level truncated importance-sampling (TIS) weights.
 *
 * Conventions shared by every call
 * --------------------------------
 * Numerics.  scale = fl32(amax / 448) (IEEE binary32 division), and a value
 *   x is stored as code = E4M3(fl32(x / scale)): the binary32 quotient
 *   rounded to nearest-even into E4M3 (OCP "e4m3fn": bias 7, max 448, no
 *   infinities), saturating at +-448, keeping the sign of zero.  A block,
 *   group or head whose amax is 0 gets scale 0 and codes +-0.  Results are
 *   bit-identical to that definition for every finite input.
 * BF16 inputs are raw bfloat16 bit patterns (2 bytes each); E4M3 codes are
 *   bytes.  All sizes are in elements unless the name says bytes.
 * Memory.  Every pointer argument is DEVICE memory on the current CUDA
 *   device unless the comment says HOST.  The caller owns every buffer.  The
 *   library owns one small per-device workspace (a status word and
 *   calibration slots), allocated by the first call that needs it on that
 *   device and kept until process exit; make that first call outside CUDA
 *   graph capture.
 * Streams.  Every compute call is asynchronous and stream-ordered on
 *   `stream` (0 = legacy default stream); it returns after launching.
 *   Argument errors are detected on the host before anything is launched.
 * Errors.  Calls return fp8rl_status; on failure fp8rl_last_error() gives a
 *   human-readable message (thread-local, valid until the next call on that
 *   thread).  No call throws, aborts or traps.  Kernels never fault on
 *   purpose: a device-side wait that exceeds its time limit sets a bit in
 *   the device status word and the kernel returns early; read it with
 *   fp8rl_device_status().
 */
#ifndef FP8RL_H_
#define FP8RL_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8RL_VERSION 100

typedef enum fp8rl_status {
  FP8RL_OK = 0,
  FP8RL_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad mode */
  FP8RL_ERR_ALIGNMENT = 2,          /* pointer or leading dimension misaligned */
  FP8RL_ERR_UNSUPPORTED_SHAPE = 3,  /* shape outside what a kernel supports */
  FP8RL_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed */
  FP8RL_ERR_TIMEOUT = 5,            /* a device-side wait hit its time limit */
  FP8RL_ERR_UNSUPPORTED_DEVICE = 6  /* current device is not sm_103 */
} fp8rl_status;

typedef enum fp8rl_kv_mode {
  FP8RL_KV_GIVEN = 0,      /* quantize with the caller's scales[heads] */
  FP8RL_KV_CALIBRATE = 1   /* compute scales[h] = amax_h/448 from x, write them, quantize */
} fp8rl_kv_mode;

/* One tensor of a multi-tensor weight re-quantization (see
 * fp8rl_quantize_weights_blockwise for the meaning of each field). */
typedef struct fp8rl_wdesc {
  const void* w;   /* BF16 [n, k], row stride ldw elements */
  uint8_t* q;      /* E4M3 [n, k], row stride ldq bytes */
  float* scales;   /* FP32 [ceil(n/128), ceil(k/128)], row-major */
  int64_t n, k, ldw, ldq;
} fp8rl_wdesc;

/* Library version (FP8RL_VERSION of the build). */
int32_t fp8rl_version(void);

/* Message of the last failed call on this thread ("" if none). */
const char* fp8rl_last_error(void);

/* Blockwise weight re-quantization.
 * Summary page section 3.4.1, equation W_hat_ij = round(W_ij / scale_ij) with
 * scale_ij from the max-abs of the 128x128 block holding (i, j); section 3.4.2
 * Phase 2 step 2 (runs every RL step on every quantized linear).
 *   w       BF16 [n, k] row-major with row stride ldw (elements), 16-byte aligned
 *   q       E4M3 codes [n, k], row stride ldq (bytes), 8-byte aligned
 *   scales  FP32 [ceil(n/128), ceil(k/128)] row-major; scales[bi][bj] belongs to
 *           rows [128 bi, 128 bi + 128) x cols [128 bj, 128 bj + 128)
 * Edge blocks (n or k not a multiple of 128) take amax over their valid
 * elements only.  Requires n, k >= 1, k % 8 == 0, ldw % 8 == 0, ldq % 8 == 0,
 * ldw >= k, ldq >= k.  One read of w and one write of q. */
fp8rl_status fp8rl_quantize_weights_blockwise(const void* w, int64_t n, int64_t k, int64_t ldw,
                                              uint8_t* q, int64_t ldq, float* scales,
                                              cudaStream_t stream);

/* The same operation over `count` tensors in one pass (the per-step sync of
 * a whole model; section 3.4.2 notes it is parallel across blocks and layers).
 *   descs   HOST array of `count` descriptors (read during the call only);
 *           each obeys the requirements above; tensors must not overlap.
 * Tensors are processed in launches of up to 160 descriptors. */
fp8rl_status fp8rl_quantize_weights_blockwise_multi(const fp8rl_wdesc* descs, int32_t count,
                                                    cudaStream_t stream);

/* Per-token 1x128-group activation quantization (dynamic quantization of
 * section 3.4.1 "Static vs. Dynamic Quantization" and section 3.4.2 Phase 3;
 * 1x128 tiles as in section 3.4.1).
 *   a       BF16 [m, k], row stride lda (elements), 16-byte aligned
 *   q       E4M3 codes [m, k] dense (row stride k bytes), 8-byte aligned
 *   scales  FP32 [ceil(k/128), m]: GROUP-MAJOR, scales[g * m + r] is the scale
 *           of row r, columns [128 g, 128 g + 128).  This is the layout the
 *           GEMMs read (one contiguous vector of m-scales per k-block).
 * Requires m, k >= 1, k % 8 == 0, lda % 8 == 0, lda >= k. */
fp8rl_status fp8rl_quantize_act_groupwise(const void* a, int64_t m, int64_t k, int64_t lda,
                                          uint8_t* q, float* scales, cudaStream_t stream);

/* Blockwise-scaled W8A8 GEMM, Y = A W^T.
 * Section 3.4.2 Phase 3 (FP8 x FP8 matmul on tensor cores, FP32 accumulation,
 * BF16 result) with the scales of sections 3.4.1 (weights 128x128) and the
 * activation groups above:
 *   Y[i, j] = bf16( sum_kb sa[kb, i] * sw[j/128, kb] * sum_{k in kb} dec(qa[i,k]) dec(qw[j,k]) )
 *   qa  E4M3 [m, k] dense;    sa  FP32 [k/128, m] (group-major, as above)
 *   qw  E4M3 [n, k] dense;    sw  FP32 [ceil(n/128), k/128] row-major
 *   y   BF16 [m, n], row stride ldy (elements)
 * Requires m >= 0, n >= 16, k >= 128, k % 128 == 0, n % 16 == 0, ldy % 8 == 0,
 * ldy >= n; qa, qw 16-byte aligned; y 16-byte aligned.  m = 0 is a no-op.
 * Accuracy: FP32 accumulation of per-128-k partial sums, each promoted with
 * its scale pair; one final BF16 rounding. */
fp8rl_status fp8rl_gemm_w8a8_blockwise(const uint8_t* qa, const float* sa, const uint8_t* qw,
                                       const float* sw, int64_t m, int64_t n, int64_t k,
                                       void* y, int64_t ldy, cudaStream_t stream);

/* Decode-sized linear layer: the 1x128 activation quantization fused with
 * the blockwise W8A8 GEMM, for m <= 256 rows (a decode batch).  Section 3.4.2
 * Phase 3: each decode step quantizes its activations dynamically and
 * multiplies them by the per-step FP8 weights on FP8 tensor cores, FP32
 * accumulation, BF16 output.  Results:
 *   qa, sa   exactly fp8rl_quantize_act_groupwise(a) (bit for bit)
 *   y        Y = A W^T as fp8rl_gemm_w8a8_blockwise defines it, to the same
 *            accuracy (the FP32 partial sums of a tile may be added in another
 *            order; the order is fixed, so results repeat bit for bit).
 * One cooperative launch over every SM: the CTAs quantize A together, meet at
 * a grid barrier, then split the (128-column tile, 128-deep k-block) units of
 * the GEMM evenly ("stream-K"); a tile shared by several CTAs is reduced by
 * the last one to finish it, in k order, through `workspace`.
 *   a        BF16 [m, k], row stride lda (>= k, multiple of 8), 16-byte
 *            aligned; NULL: qa and sa are inputs (already quantized A) and
 *            the call is the stream-K GEMM alone
 *   qa       E4M3 [m, k] dense, 16-byte aligned (written when a != NULL)
 *   sa       FP32 [k/128, m] group-major (written when a != NULL)
 *   qw, sw   E4M3 [n, k] and FP32 [n/128, k/128], as in the dense GEMM
 *   y        BF16 [m, n], row stride ldy (>= n, multiple of 8), 16-byte aligned
 *   workspace  DEVICE memory owned by the caller, 256-byte aligned, at least
 *            fp8rl_linear_w8a8_decode_workspace_bytes(n) bytes, ZERO-FILLED
 *            before its first use.  The call leaves its counters at zero
 *            again, so a workspace can be reused by later calls; calls that
 *            overlap on the GPU need separate workspaces.  After a call that
 *            reported FP8RL_ERR_TIMEOUT, zero it again.
 * Requires 0 <= m <= 256, n a positive multiple of 128, k a positive
 * multiple of 128; m = 0 is a no-op. */
size_t fp8rl_linear_w8a8_decode_workspace_bytes(int64_t n);
fp8rl_status fp8rl_linear_w8a8_decode(const void* a, int64_t lda, uint8_t* qa, float* sa,
                                      const uint8_t* qw, const float* sw, int64_t m, int64_t n,
                                      int64_t k, void* y, int64_t ldy, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream);

/* Grouped (MoE expert) variant: rows [offsets[e], offsets[e+1]) of A are the
 * tokens routed to expert e (section 3.4.1 "MoE expert layers: fc1, fc2") and
 * are multiplied by expert e's weights.
 *   qa       E4M3 [m_total, k] dense;  sa FP32 [k/128, m_total] group-major
 *   qw       E4M3 [e, n, k];           sw FP32 [e, n/128, k/128]
 *   offsets  int32 [e + 1] DEVICE, non-decreasing, offsets[0] = 0,
 *            offsets[e] <= m_total; read by the kernel (no host sync)
 *   y        BF16 [m_total, n] dense; rows outside every segment are not written
 * Requires 1 <= e <= 1024, n % 128 == 0, k % 128 == 0, alignment as above.
 * Empty segments are allowed. */
fp8rl_status fp8rl_grouped_gemm_w8a8_blockwise(const uint8_t* qa, const float* sa,
                                               const uint8_t* qw, const float* sw,
                                               const int32_t* offsets, int32_t num_experts,
                                               int64_t m_total, int64_t n, int64_t k,
                                               void* y, cudaStream_t stream);

/* FP8 E4M3 KV-cache quantization with per-head scales (section 3.4.4: K and V
 * stored as E4M3 with per-layer or per-head scales computed from the K/V the
 * first rollout forward observes).  Call once for K and once for V.
 *   x        BF16 [rows, heads, head_dim] dense (rows = sequences x tokens), 16-byte aligned
 *   mode     FP8RL_KV_GIVEN: scales[heads] is an input;
 *            FP8RL_KV_CALIBRATE: scales[h] = fl32(amax_h / 448) over all rows
 *            and dims of head h is computed from x and written, then used
 *   scales   FP32 [heads] (input or output per mode)
 *   q        E4M3 [rows, heads, head_dim] dense, 8-byte aligned
 * Requires head_dim % 8 == 0, heads * head_dim <= 2048, heads <= 256.
 * CALIBRATE uses the library workspace: do not overlap two CALIBRATE calls on
 * one device (different streams) -- they share the calibration slots. */
fp8rl_status fp8rl_quantize_kv_fp8(const void* x, int64_t rows, int32_t heads, int32_t head_dim,
                                   int32_t mode, float* scales, uint8_t* q, cudaStream_t stream);

/* Allocation-free variant of fp8rl_quantize_kv_fp8(..., FP8RL_KV_CALIBRATE, ...):
 * the same arguments (minus mode) and bit-identical results.  The paper has
 * no counterpart for this call; it is an engineering addition.
 * Some callers cannot let a library allocate device memory: an inference
 * engine that reserves nearly all of the GPU's memory for its own pools up
 * front (so a cudaMalloc by a library would fail or fragment that pool),
 * or a caller that must not risk the implicit device synchronization that
 * cudaMalloc/cudaFree may cause.  This call uses no cudaMalloc, cudaFree or
 * other allocating routine: its only scratch (the per-head running maxima)
 * is a fixed 256-entry (1 KB) array compiled into the library, which each
 * device that loads the library keeps until the process exits.
 *   heads    at most 256 (larger values fail with FP8RL_ERR_UNSUPPORTED_SHAPE
 *            before anything is launched); other requirements as above.
 * The first call on a device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * Every call on a device shares the one array and clears the slots it uses
 * at its start, so calls whose executions overlap on the GPU (for instance
 * on two streams) race and may produce wrong scales: serialize them. */
fp8rl_status fp8rl_quantize_kv_fp8_calibrate_noalloc(const void* x, int64_t rows, int32_t heads,
                                                     int32_t head_dim, float* scales, uint8_t* q,
                                                     cudaStream_t stream);

/* Token-level truncated importance-sampling weights (section 3.4.3):
 *   w[i] = pi_theta / pi_fp8 = exp(logp_train[i] - logp_rollout[i]), truncated:
 *   d = fl32(logp_train - logp_rollout); e = RN32(e^d), the correctly rounded
 *   binary32 exponential; w = min(e, c_hi), then max(w, c_lo) if c_lo > 0;
 *   NaN stays NaN; w = 0 where mask[i] == 0.
 *   logp_train, logp_rollout  FP32 [n], 16-byte aligned
 *   mask     uint8 [n] or NULL (all tokens valid)
 *   c_hi     truncation C (2 in the pages' experiments), finite, > 0
 *   c_lo     0 for the one-sided min(w, C); 1/C for the two-sided [1/C, C]
 *   w        FP32 [n], 16-byte aligned */
fp8rl_status fp8rl_tis_weights(const float* logp_train, const float* logp_rollout,
                               const uint8_t* mask, int64_t n, float c_hi, float c_lo, float* w,
                               cudaStream_t stream);

/* Per-step re-quantization from and to HOST memory (section 3.4.2, Phase 2:
 * the BF16 weights come from the training side, the E4M3 codes and scales go
 * to the inference engine, every RL step).  Same results as
 * fp8rl_quantize_weights_blockwise_multi, but each descriptor's w, q and
 * scales are HOST pointers (page-locked memory lets the copies run
 * asynchronously and overlap; pageable memory works but serializes them).
 * The tensors stream through `workspace` (DEVICE, 256-byte aligned, owned by
 * the caller, at least 2 x the bytes of 128 rows of the widest tensor,
 * 3 bytes per element plus scales; tens to hundreds of MB keep the copies
 * and the kernels overlapped): the host-to-device copy of one chunk, the
 * quantization of the previous one and the device-to-host copy of the one
 * before run together on internal streams; tensors larger than half the
 * workspace are split at 128-row boundaries.  Nothing is allocated.
 * Stream-ordered: starts after earlier work on `stream`, and `stream` waits
 * for the last copy; the host buffers must stay valid until then.  Calls on
 * one device are serialized on the library's internal streams.
 *   descs    HOST array of count descriptors (w, q, scales in host memory;
 *            k a multiple of 8, ldw >= k, ldq >= k)
 *   workspace, workspace_bytes  the device staging buffer */
fp8rl_status fp8rl_quantize_weights_blockwise_multi_host(const fp8rl_wdesc* descs, int32_t count,
                                                         void* workspace, size_t workspace_bytes,
                                                         cudaStream_t stream);

/* MoE glue before the expert GEMMs: permute + quantize.  The expert-sorted
 * activation matrix is the token matrix's rows a[rows[r]] (a token appears
 * once per expert it is routed to; section 3.4.1 names the MoE expert layers
 * among the quantized ones); each gathered row is quantized in 1x128 groups
 * exactly as fp8rl_quantize_act_groupwise does.
 *   a        BF16 [m_src, k] token matrix, row stride lda (>= k); k, lda
 *            multiples of 8; 16-byte aligned
 *   rows     int32 [m] (device), source row of each output row.  An index
 *            outside [0, m_src) leaves that row's codes and scales zero and
 *            sets a bit that fp8rl_device_status reports; nothing faults.
 *   q        E4M3 [m, k] (row stride k), 8-byte aligned
 *   scales   FP32 [ceil(k/128), m] group-major */
fp8rl_status fp8rl_quantize_act_gather(const void* a, int64_t m_src, int64_t k, int64_t lda,
                                       const int32_t* rows, int64_t m, uint8_t* q, float* scales,
                                       cudaStream_t stream);

/* MoE glue between the expert GEMMs: gated activation + quantize.  h holds
 * the gate_up projection's output, gate in columns [0, inter) and up in
 * [inter, 2*inter); y = BF16_RNE(silu(gate) * up) is quantized in 1x128
 * groups as fp8rl_quantize_act_groupwise does (the down projection's input).
 * The pages fix no activation arithmetic (section 3.4.1 names the expert
 * layers fc1/fc2 among the quantized linears); y is the plain definition,
 * the real product silu(g) * u with silu(g) = g / (1 + e^-g), rounded once
 * to the nearest BF16 (ties to even, overflow to +-inf, underflow to a
 * subnormal or a signed zero).  Special values follow the IEEE evaluation
 * of g * sigma(g) * u: a NaN input gives NaN, silu(+inf) = +inf,
 * silu(-inf) = NaN, silu(+-0) = +-0, and 0 * inf = NaN.  Bit-identical to
 * that definition (fp8rl_silu_mul_bf16 returns y itself).
 *   h        BF16 [m, 2*inter], row stride ldh (>= 2*inter); inter, ldh
 *            multiples of 8; 16-byte aligned
 *   q        E4M3 [m, inter] (row stride inter), 8-byte aligned
 *   scales   FP32 [ceil(inter/128), m] group-major */
fp8rl_status fp8rl_silu_mul_quantize(const void* h, int64_t m, int64_t inter, int64_t ldh,
                                     uint8_t* q, float* scales, cudaStream_t stream);

/* The gated activation of fp8rl_silu_mul_quantize without the quantization:
 * y[r, c] = BF16_RNE(silu(h[r, c]) * h[r, inter + c]) (same definition and
 * special values), for a BF16 down projection or for inspecting y.
 *   h        BF16 [m, 2*inter], row stride ldh (>= 2*inter)
 *   y        BF16 [m, inter], row stride ldy (>= inter)
 * Requires inter, ldh, ldy multiples of 8 and h, y 16-byte aligned; m = 0
 * is a no-op. */
fp8rl_status fp8rl_silu_mul_bf16(const void* h, int64_t m, int64_t inter, int64_t ldh, void* y,
                                 int64_t ldy, cudaStream_t stream);

/* Decode attention over an FP8 E4M3 KV cache (section 3.4.4: K and V are
 * stored in E4M3 with per-head scales recalibrated every step; the decode
 * step attends over that cache).  For every sequence s and query head hq,
 * with KV head h = hq / (q_heads / kv_heads):
 *   score_t = sm_scale * <q[s,hq], k_scale[h] * dec(K[s,t,h])>, t < seq_lens[s]
 *   out[s,hq] = BF16(sum_t softmax(score)_t * v_scale[h] * dec(V[s,t,h]))
 * computed in FP32 (an empty context gives zeros).  Token t of sequence s is
 * slot t % page of page block_table[s * max_pages + t / page]; with
 * block_table NULL, sequence s owns pages s*max_pages ... (a contiguous
 * [num_seqs, max_pages*page, kv_heads, 128] cache, as fp8rl_quantize_kv_fp8
 * writes it with rows = num_seqs * tokens).  Page indices outside
 * [0, num_pages) are skipped and lengths above max_pages*page are clamped;
 * both set the bit fp8rl_device_status reports.  Parity is within FP32
 * rounding (accumulation order is the kernel's).
 *   q          BF16 [num_seqs, q_heads, 128], 16-byte aligned
 *   k_cache, v_cache  E4M3 [num_pages, page, kv_heads, 128], 16-byte aligned
 *   k_scale, v_scale  FP32 [kv_heads] (device), the quantizer's scales
 *   block_table int32 [num_seqs, max_pages] (device) or NULL
 *   seq_lens   int32 [num_seqs] (device)
 *   head_dim   must be 128; q_heads / kv_heads in {1, 2, 4, 8}
 *   num_pages  pages in the pool (ignored when block_table is NULL)
 *   sm_scale   softmax scale, typically 1/sqrt(128)
 *   out        BF16 [num_seqs, q_heads, 128] */
fp8rl_status fp8rl_decode_attention_fp8kv(const void* q, const uint8_t* k_cache,
                                          const uint8_t* v_cache, const float* k_scale,
                                          const float* v_scale, const int32_t* block_table,
                                          const int32_t* seq_lens, int32_t num_seqs,
                                          int32_t q_heads, int32_t kv_heads, int32_t head_dim,
                                          int32_t page, int32_t max_pages, int32_t num_pages,
                                          float sm_scale, void* out, cudaStream_t stream);

typedef enum fp8rl_is_mode {
  FP8RL_IS_TRUNCATE = 0,   /* TIS: w = min(e, c_hi), then max(w, c_lo) if c_lo > 0 */
  FP8RL_IS_MASK = 1        /* MIS: w = e if c_lo <= e <= c_hi, else 0 (NaN e: 0) */
} fp8rl_is_mode;

/* Importance weights and the batch's mismatch statistics in one pass
 * (section 3.4.3: the weight pi_theta / pi_fp8, its truncation at C and
 * masked importance sampling as the stronger correction; the experiments'
 * metrics: the mismatch KL D_KL(pi_fp8 || pi_theta) and the sampling
 * importance ratio).  Per token d = fl32(logp_train - logp_rollout) and
 * e = RN32(e^d) as in fp8rl_tis_weights; w by `mode`; w = 0 where
 * mask[i] == 0.  Over the valid tokens (mask != 0, all if mask is NULL):
 *   stats[0]  number of valid tokens
 *   stats[1]  sum of fl32(logp_rollout - logp_train)  (k1 estimator of the KL:
 *             tokens are drawn from pi_fp8; divide by stats[0] for the mean)
 *   stats[2]  sum of fl32(fl32(e - 1) - d)          (k3 estimator, (r-1) - log r)
 *   stats[3]  sum of e                               (mean: sampling IS ratio)
 *   stats[4]  valid tokens whose weight was clipped (TIS) or masked (MIS)
 * The per-token terms are exact binary32 values; the sums are accumulated in
 * FP32 over 8 tokens at a time, then in float-float and FP64, in an order that can
 * change from call to call: each sum is within 2^-20 * (sum of |terms|) of
 * the exact sum of the terms.  Counts are exact.
 *   logp_train, logp_rollout, mask, c_hi, c_lo  as in fp8rl_tis_weights (the
 *            arrays may be NULL when n == 0; the statistics are then zeros)
 *   mode     fp8rl_is_mode
 *   w        FP32 [n], 16-byte aligned, or NULL (statistics only)
 *   stats    FP64 [5], 8-byte aligned, overwritten (cleared on `stream`
 *            first), complete when the call's work on `stream` is. */
fp8rl_status fp8rl_is_weights_stats(const float* logp_train, const float* logp_rollout,
                                    const uint8_t* mask, int64_t n, float c_hi, float c_lo,
                                    int32_t mode, float* w, double* stats, cudaStream_t stream);

/* fp8rl_is_weights_stats plus the importance-weighted token loss (section
 * 3.4.3: token-level TIS multiplies each token's policy-gradient loss by its
 * truncated weight).  With loss[i] the caller's per-token loss, stats[0..4]
 * are as above and
 *   stats[5]  sum over the valid tokens of fl32(w * loss)  (divide by
 *             stats[0] for the token mean)
 * accumulated like the other sums (within 2^-20 * sum of |terms|).
 *   loss     FP32 [n] (device), 16-byte aligned; may be NULL only when n == 0
 *   stats    FP64 [6], 8-byte aligned, overwritten (cleared on `stream` first)
 * Other arguments and errors as in fp8rl_is_weights_stats. */
fp8rl_status fp8rl_is_weights_stats_loss(const float* logp_train, const float* logp_rollout,
                                         const uint8_t* mask, const float* loss, int64_t n,
                                         float c_hi, float c_lo, int32_t mode, float* w,
                                         double* stats, cudaStream_t stream);

/* Synchronizes the device and returns FP8RL_ERR_TIMEOUT if any kernel since
 * the last clear hit a device-side wait limit, FP8RL_ERR_INVALID_ARG if a
 * kernel met an out-of-range device-side index (fp8rl_quantize_act_gather,
 * fp8rl_decode_attention_fp8kv),
 * FP8RL_OK otherwise; clears the word when clear != 0.  device = CUDA
 * ordinal. */
fp8rl_status fp8rl_device_status(int32_t device, int32_t clear);

/* Shard plan of the sharded weight synchronization (section 3.4.2 Phase 2:
 * the trainer's FSDP shards are gathered and quantized before they reach the
 * engine).  Here each rank quantizes its own rows first and the ranks then
 * all-gather the E4M3 codes and FP32 scales, about half the bytes of a BF16
 * gather.  Rank `rank` of `world` owns rows [*row_begin, *row_end) of an
 * n-row weight: a contiguous run of whole 128-row block bands (the bands are
 * dealt as evenly as possible, in rank order), so no 128 x 128 block crosses
 * two ranks and the gathered codes and scales equal those of the whole
 * tensor bit for bit.  A rank may own no rows (begin == end).  Host-only: no
 * device is touched. */
fp8rl_status fp8rl_weight_shard_rows(int64_t n, int32_t world, int32_t rank, int64_t* row_begin,
                                     int64_t* row_end);

/* Error-path support (no counterpart in the pages): lets a caller's tests
 * exercise its handling of fp8rl_device_status without faulting a GPU.
 * fp8rl_inject_device_status synchronizes `device` and overwrites its status
 * word with `flags` (a combination of 1 = wait timeout, 2 = out-of-range
 * device index; anything else is FP8RL_ERR_INVALID_ARG) and `site` (reported
 * in the timeout message).  Not stream-ordered; do not call it while a
 * capture is in progress. */
fp8rl_status fp8rl_inject_device_status(int32_t device, uint32_t flags, uint32_t site);

/* Launches on `stream` one small kernel that waits on a device-side barrier
 * nothing will complete, through the same bounded wait the pipelined kernels
 * use but with a limit of `limit_us` microseconds (1 .. 1000000).  The wait
 * gives up, sets the timeout flag with site 90 in the status word and the
 * kernel returns; the next fp8rl_device_status reports FP8RL_ERR_TIMEOUT and
 * the CUDA context stays usable. */
fp8rl_status fp8rl_selftest_bounded_wait(int32_t limit_us, cudaStream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* FP8RL_H_ */
