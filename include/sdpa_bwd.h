/*
 * sdpa_bwd.h -- C ABI of the GB300 (sm_103a) scaled-dot-product-attention
 * backward library, libsdpa_bwd.so.
 *
 * Operation (cuDNN frontend docs, "SDPA Backward (SM120)": Overview, API
 * Usage, and "Main-kernel pipeline: KV-stationary, five chained GEMMs"):
 * given the forward activations Q, K, V, the forward output O, the loss
 * gradient dO and the natural-log forward row statistic LSE, compute
 *     P     = exp(scale * Q K^T - LSE)       (masked entries and LSE = -inf rows: 0)
 *     delta = rowsum(dO * O)
 *     dP    = dO V^T
 *     dS    = P * (dP - delta)
 *     dV    = P^T dO,   dQ = scale * dS K,   dK = scale * dS^T Q
 * with the causal / sliding-window / padding masks of the page's "Causal,
 * sliding-window, and padding masks" section and GQA/MQA (section "GQA/MQA
 * group reduction": query head h reads KV head h / (H_q / H_kv); dK and dV of
 * a KV head sum over its group of query heads, in ascending head order).
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense, contiguous, row-major (B, H, S, D) bf16 device
 *     buffers (fp16 through sdpa_bwd_typed / sdpa_fwd_typed), D innermost;
 *     every tensor pointer must be 16-byte aligned.
 *     Q, O, dO, dQ have H_q heads; K, V, dK, dV have H_kv heads.
 *     Q, K, dQ, dK have D_qk columns; V, O, dO, dV have D_v columns.
 *   - lse is fp32 (B, H_q, S_q), natural log; -inf marks a row with no key.
 *   - The caller owns every buffer. The library writes only dq, dk, dv and the
 *     workspace; every element of dq, dk, dv is overwritten (masked or padded
 *     rows get exact zeros), so outputs need no clearing.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous with respect to the host.
 *   - Functions return an sdpa_status code and never abort the process. Errors
 *     found while validating arguments are returned before anything is
 *     launched. Errors that kernels detect while running (a bounded wait that
 *     ran out) are recorded in a per-device status word that
 *     sdpa_bwd_check_device_status() reads.
 */
#ifndef SDPA_BWD_H_
#define SDPA_BWD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID = 1,     /* null pointer, bad size (a tensor of 2^31 elements or
                               more), H_kv not dividing H_q                          */
  SDPA_ERR_UNSUPPORTED = 2, /* head dims / mask combination / device not served     */
  SDPA_ERR_ALIGN = 3,       /* a tensor pointer is not 16-byte aligned              */
  SDPA_ERR_WORKSPACE = 4,   /* workspace smaller than sdpa_bwd_workspace_size()     */
  SDPA_ERR_CUDA = 5,        /* a CUDA runtime call failed                           */
  SDPA_ERR_TIMEOUT = 6,     /* a device-side bounded wait ran out (reported later)  */
  SDPA_ERR_BOUNDS = 7       /* debug-bounds build only (libsdpa_bwd_debug.so, built
                               with SDPA_DEBUG_BOUNDS): a kernel found a global
                               access outside its region and skipped it (reported
                               later, results invalid)                               */
} sdpa_status;

/* Element types: of an optional additive bias (BF16, F16 or F32) and of the
 * io tensors (sdpa_bwd_typed, sdpa_fwd_typed: BF16 or F16). */
typedef enum {
  SDPA_DTYPE_BF16 = 0,
  SDPA_DTYPE_F32 = 1,
  SDPA_DTYPE_F16 = 2
} sdpa_dtype;

/*
 * Bytes of device workspace sdpa_bwd() (and sdpa_bwd_sink, sdpa_bwd_bias,
 * sdpa_bwd_typed) needs for this problem and mask (0 when none). The mask
 * arguments are those of the call (padded: 1 when seq_q_lens or seq_kv_lens
 * will be given). The workspace holds, each region 256-byte aligned:
 * per-query-tile fp32 row statistics (LSE * log2(e) and delta); either the
 * fp32 dQ accumulator (rows of 64 columns for D_qk up to 64, else 128) or, on
 * the routes that store dS (deterministic D_qk = 128, every D_qk = 192 or 256), the
 * 16-bit dS tiles of the band of query tiles each 128-key tile visits (the
 * whole rectangle when a bottom-right mask meets per-batch lengths) plus one
 * zero tile; the deterministic-mode turn counters (one int per query tile)
 * and a work ticket; one fp32 sink-token partial per query tile
 * (sdpa_bwd_sink); and, when H_kv < H_q, the per-query-head 16-bit dK/dV
 * partials of the GQA reduction. The size does not depend on the io type.
 * Returns 0 for arguments sdpa_bwd() would reject.
 */
size_t sdpa_bwd_workspace_size(int B, int H_q, int H_kv, int S_q, int S_kv, int D_qk, int D_v,
                               int causal, int bottom_right, int window_left, int window_right,
                               int deterministic, int padded);

/*
 * SDPA backward. Arguments:
 *   q, k, v, o, d_o   device bf16 inputs, layouts above.
 *   lse               device fp32 (B, H_q, S_q) natural-log LSE of the forward.
 *   dq, dk, dv        device bf16 outputs (same shapes as q, k, v).
 *   B, H_q, H_kv      batch and head counts; H_kv must divide H_q.
 *   S_q, S_kv         sequence lengths (>= 0; a zero length gives zero gradients).
 *   D_qk, D_v         head dims; served: D_qk = D_v, any multiple of 8 from 8 to
 *                     128 (up to 64 on the 64-column kernels, above on the
 *                     128-column ones, the columns past D zero-filled by TMA),
 *                     (192, 128), and (256, 256) (cuDNN frontend docs, "SDPA
 *                     Backward (SM120)", "Head-size support and tile configs":
 *                     two work units per key tile, each accumulating half of
 *                     the dK/dV columns; dS stored as for 192).
 *   scale             softmax scale applied to Q K^T; <= 0 or NaN selects 1/sqrt(D_qk).
 *   causal            1: keep key k for query q only if k <= q + diag + max(window_right, 0).
 *   bottom_right      1: diag = L_kv - L_q (the actual lengths of the batch row);
 *                     0: diag = 0. Applies to the causal and the window masks.
 *   window_left       W >= 0: mask keys k < q + diag - W; < 0: no left window.
 *   window_right      R >= 0 widens the causal diagonal by R keys; requires causal.
 *                     < 0: no widening.
 *   deterministic     1: repeated calls give bitwise-identical dQ. For D_qk =
 *                     128 the main kernel stores dS and a second kernel forms
 *                     dQ = scale * dS K over an ascending key walk (larger
 *                     workspace: 2 bytes per visited (query, key) position);
 *                     for other D_qk up to 128 the dQ partials of the KV tiles
 *                     are added in ascending KV-tile order. D_qk = 192 and 256
 *                     always take the stored-dS route, so their dQ is
 *                     reproducible in both modes. dK and dV are bitwise reproducible in both
 *                     modes.
 *   seq_q_lens,       device int32 (B,) per-batch valid lengths, or NULL for
 *   seq_kv_lens       "the full S". Queries at or past seq_q_lens[b] and keys
 *                     at or past seq_kv_lens[b] are masked; their gradient
 *                     rows are exact zeros.
 *   workspace         device buffer of >= sdpa_bwd_workspace_size() bytes,
 *                     256-byte aligned, used only for the duration of the call
 *                     on `stream`; NULL makes the library take one from the
 *                     stream-ordered allocator (cudaMallocAsync) and release
 *                     it after the last kernel.
 *   workspace_bytes   size of `workspace` (ignored when it is NULL).
 *   stream            cudaStream_t on which every kernel is enqueued.
 * Returns SDPA_OK once every kernel is enqueued, else an error code (nothing
 * enqueued). Calls that share a workspace must not overlap on the device.
 */
int sdpa_bwd(const void* q, const void* k, const void* v, const void* o, const void* d_o,
             const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int S_q,
             int S_kv, int D_qk, int D_v, float scale, int causal, int bottom_right,
             int window_left, int window_right, int deterministic, const int32_t* seq_q_lens,
             const int32_t* seq_kv_lens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * SDPA backward with sink tokens (cuDNN frontend docs, "SDPA Backward (SM120)":
 * the sink-token capability and the `dsink` step of the kernel chain). A sink
 * logit per query head joins every row's softmax denominator without a value
 * row. The forward's LSE already includes it, so dQ, dK and dV are exactly
 * those of sdpa_bwd() with the same lse; this call also writes
 *     dsink[h] = -sum_{b, q < L_q} exp(sink[h] - LSE[b,h,q]) * delta[b,h,q]
 * (terms with LSE = -inf count as 0). The sum runs in a fixed order (one
 * fp32 partial per 64-row query tile, then the tiles of a head in a fixed
 * tree), so dsink is bitwise reproducible in both modes.
 * Arguments: those of sdpa_bwd(), then
 *   sink      device fp32 (H_q,) sink logits (4-byte aligned).
 *   dsink     device fp32 (H_q,) output (4-byte aligned).
 * Returns SDPA_ERR_INVALID when sink or dsink is NULL; otherwise as sdpa_bwd().
 * The workspace size is sdpa_bwd_workspace_size() (it includes the partials).
 */
int sdpa_bwd_sink(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                  const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv,
                  int S_q, int S_kv, int D_qk, int D_v, float scale, int causal, int bottom_right,
                  int window_left, int window_right, int deterministic,
                  const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* workspace,
                  size_t workspace_bytes, const float* sink, float* dsink, void* stream);

/*
 * SDPA backward with an additive bias (cuDNN frontend docs, "SDPA Backward
 * (SM120)": the bias capability). A (bias_batch, H_q, S_q, S_kv) tensor is
 * added to the scaled scores before the softmax,
 *     P = exp(scale * Q K^T + bias - LSE),
 * where lse is the forward's LSE of the same biased scores. dQ, dK and dV keep
 * their formulas with this P; the gradient of the bias is
 *     dBias = dS = P * (dP - delta)     (fp32, 0 at masked pairs),
 * summed over the batch rows when bias_batch = 1 and B > 1.
 * Arguments: those of sdpa_bwd_sink(), where sink and dsink may both be NULL
 * (no sink) or dsink alone NULL (a sink in the forward's LSE, no dsink), then
 *   bias        device (bias_batch, H_q, S_q, S_kv) tensor, contiguous, S_kv
 *               innermost; bf16 or fp16 (2-byte aligned), or fp32 (4-byte aligned).
 *   bias_dtype  SDPA_DTYPE_BF16, SDPA_DTYPE_F16 or SDPA_DTYPE_F32.
 *   bias_batch  1 (one bias shared by every batch row) or B.
 *   dbias       device fp32 output shaped like bias (4-byte aligned), or NULL.
 *               Every element is overwritten. With bias_batch = B, or B = 1,
 *               each element is written once and the result is bitwise
 *               reproducible; with bias_batch = 1 and B > 1 the batch rows
 *               add into it atomically (not reproducible), which deterministic
 *               mode rejects.
 * Served for every head-dim pair of sdpa_bwd(). Returns SDPA_ERR_INVALID for a
 * NULL bias, an unknown dtype, bias_batch not 1 or B, or the deterministic case
 * above; otherwise as sdpa_bwd(). Workspace as sdpa_bwd_workspace_size().
 */
int sdpa_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                  const float* lse, void* dq, void* dk, void* dv, int B, int H_q, int H_kv,
                  int S_q, int S_kv, int D_qk, int D_v, float scale, int causal, int bottom_right,
                  int window_left, int window_right, int deterministic,
                  const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* workspace,
                  size_t workspace_bytes, const float* sink, float* dsink, const void* bias,
                  int bias_dtype, int bias_batch, float* dbias, void* stream);

/*
 * SDPA forward: the O and natural-log LSE that sdpa_bwd() takes (cuDNN frontend
 * docs, "SDPA Backward (SM120)": the forward statistics of "API Usage", the
 * masks of "Causal, sliding-window, and padding masks", GQA/MQA, and sink
 * tokens), so that a forward and a backward form a training step:
 *     S   = scale * Q K^T over the visible keys,
 *     LSE = log( sum_k exp(S) [+ exp(sink[h])] ),   O = sum_k exp(S - LSE) V.
 * A row with no visible key (queries at or past seq_q_lens[b] included) gets
 * O = 0 and LSE = -inf, or LSE = sink[h] with a sink.
 * Arguments are those of sdpa_bwd() with:
 *   D_qk, D_v  as sdpa_bwd(). D_qk = D_v up to 128 run on a kernel that keeps an
 *          O accumulator per half of each row's keys; (192, 128) and (256, 256)
 *          on kernels with one O whose softmax reference the two halves agree
 *          on every key tile (three score slots at 192/128; K and V in 16 KB
 *          pieces at 256).
 *   o      device bf16 (B, H_q, S_q, D_v) output, 16-byte aligned.
 *   lse    device fp32 (B, H_q, S_q) output, 4-byte aligned.
 *   sink   device fp32 (H_q,) sink logits, or NULL.
 * No workspace. The kernels are persistent (one CTA per SM) and take their work
 * items from a counter in the library's device memory; the library hands out
 * 64 such counters in turn, so more than 64 forward launches running at once on
 * one device (on different streams) could share one and must not be issued; a
 * CUDA graph that captured a forward launch reuses its counter on every replay,
 * so two replays of that graph must not run at the same time.
 * Returns SDPA_OK once the kernel is enqueued on `stream`, else an error code
 * (nothing enqueued); a device-side timeout is reported by
 * sdpa_bwd_check_device_status().
 */
int sdpa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
             int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale, int causal,
             int bottom_right, int window_left, int window_right, const int32_t* seq_q_lens,
             const int32_t* seq_kv_lens, const float* sink, void* stream);

/*
 * SDPA forward with an additive bias (cuDNN frontend docs, "SDPA Backward
 * (SM120)": the bias capability): as sdpa_fwd() with the scores
 *     S = scale * Q K^T + bias      (before the masks and the softmax),
 * so that O and LSE are the inputs sdpa_bwd_bias() takes with the same bias.
 * A visible key whose bias is -inf contributes nothing; a row whose visible
 * keys all have a -inf bias gets O = 0 and LSE = -inf (or the sink).
 * Arguments: those of sdpa_fwd(), then
 *   bias        device (bias_batch, H_q, S_q, S_kv) tensor, contiguous, S_kv
 *               innermost; bf16 or fp16 (2-byte aligned), or fp32 (4-byte aligned).
 *               Rows are read with 16-byte loads when S_kv times the element
 *               size is a multiple of 16 and bias is 16-byte aligned.
 *   bias_dtype  SDPA_DTYPE_BF16, SDPA_DTYPE_F16 or SDPA_DTYPE_F32.
 *   bias_batch  1 (one bias for every batch row) or B.
 * Returns SDPA_ERR_INVALID for a NULL bias, an unknown dtype or bias_batch
 * not 1 or B; otherwise as sdpa_fwd().
 */
int sdpa_fwd_bias(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                  int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale, int causal,
                  int bottom_right, int window_left, int window_right, const int32_t* seq_q_lens,
                  const int32_t* seq_kv_lens, const float* sink, const void* bias, int bias_dtype,
                  int bias_batch, void* stream);

/*
 * The general SDPA backward: the io element type as an argument ("SDPA
 * Backward (SM120)", support surface: FP16 / BF16, LSE fp32) and every optional
 * input of the other entry points. io_dtype is SDPA_DTYPE_BF16 or
 * SDPA_DTYPE_F16: with F16, q, k, v, o, d_o, dq, dk and dv are fp16, the GEMMs
 * take fp16 operands (P and dS rounded to fp16), and every accumulation stays
 * fp32. sink/dsink are as in sdpa_bwd_sink() and bias/bias_dtype/bias_batch/
 * dbias as in sdpa_bwd_bias(), each optional (NULL: absent); bias_dtype may
 * also be SDPA_DTYPE_F16 (the io type of an fp16 call, or any call).
 * dbias_dtype is the element type of dbias: SDPA_DTYPE_F32 (as sdpa_bwd_bias),
 * or SDPA_DTYPE_BF16 / SDPA_DTYPE_F16 (the page's io-dtype dBias, rounded to
 * nearest even; written directly, at half the bytes, for a per-batch bias; a
 * shared bias with B > 1 is summed in a temporary fp32 buffer, taken from the
 * stream-ordered allocator, and cast at the end). dbias then needs 2-byte
 * alignment.
 * With io_dtype BF16 and no bias this is sdpa_bwd_sink() / sdpa_bwd().
 * Returns SDPA_ERR_INVALID for another io_dtype or dbias_dtype, or dsink
 * without sink, or dbias without bias; otherwise as sdpa_bwd_bias(). The workspace size does
 * not depend on the io type.
 */
int sdpa_bwd_typed(int io_dtype, const void* q, const void* k, const void* v, const void* o,
                   const void* d_o, const float* lse, void* dq, void* dk, void* dv, int B, int H_q,
                   int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale, int causal,
                   int bottom_right, int window_left, int window_right, int deterministic,
                   const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* workspace,
                   size_t workspace_bytes, const float* sink, float* dsink, const void* bias,
                   int bias_dtype, int bias_batch, void* dbias, int dbias_dtype, void* stream);

/*
 * The general SDPA forward: sdpa_fwd() / sdpa_fwd_bias() with the io element
 * type as an argument (SDPA_DTYPE_BF16, or SDPA_DTYPE_F16: fp16 q, k, v and o,
 * P rounded to fp16 for the PV GEMM) and an optional bias (NULL: none; bf16,
 * fp16 or fp32). Returns SDPA_ERR_INVALID for another io_dtype; otherwise as
 * sdpa_fwd_bias().
 */
int sdpa_fwd_typed(int io_dtype, const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H_q, int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale,
                   int causal, int bottom_right, int window_left, int window_right,
                   const int32_t* seq_q_lens, const int32_t* seq_kv_lens, const float* sink,
                   const void* bias, int bias_dtype, int bias_batch, void* stream);

/*
 * NVFP4 fake quantization ("NVFP4 Attention QAT Backward" page, Overview):
 * y = fake_nvfp4(x) for n contiguous bf16 values, in blocks of 16 consecutive
 * values. A block's local scale is s = E4M3(amax / 6), amax its largest
 * magnitude; each value becomes E2M1(x / s) * s (0 when s is 0). Both
 * divisions are correctly rounded fp32 divisions; E4M3 and E2M1 roundings go to
 * the nearest value, ties to even, saturating at 448 and 6. Every result is
 * exact in bf16. For a (..., D) tensor with D a multiple of 16 the blocks run
 * along D.
 *   x, y    device bf16 buffers of n values, 16-byte aligned (may be equal).
 *   n       a multiple of 16 (>= 0).
 * Returns SDPA_ERR_INVALID for NULL pointers or n not a multiple of 16,
 * SDPA_ERR_ALIGN for misaligned pointers; enqueued on `stream`.
 */
int sdpa_nvfp4_fake_quant(const void* x, void* y, long long n, void* stream);

/*
 * Bytes of workspace sdpa_bwd_nvfp4_qat() needs: sdpa_bwd_workspace_size()'s
 * regions (non-deterministic route) plus bf16 copies of the fake-quantized Q,
 * K and V. Returns 0 for arguments sdpa_bwd_nvfp4_qat() would reject.
 */
size_t sdpa_bwd_nvfp4_qat_workspace_size(int B, int H_q, int H_kv, int S_q, int S_kv, int D_qk,
                                         int D_v);

/*
 * NVFP4 QAT backward ("NVFP4 Attention QAT Backward" page, Overview): with
 * Q^, K^, V^ the fake-quantized Q, K, V (sdpa_nvfp4_fake_quant),
 *     P  = exp(scale * Q^ K^^T - LSE),   dS = P * (dO V^^T - rowsum(O_hp * dO)),
 *     dQ = scale * dS K^,   dK = scale * dS^T Q^,   dV = fake_nvfp4(P)^T dO,
 * where dQ and dK use P itself (straight-through estimator) and dV uses P
 * fake-quantized in blocks of 16 consecutive keys of each query row (blocks
 * start at key 0; masked entries count as 0).
 * Arguments as sdpa_bwd() (no deterministic flag: the dQ-reduction route), with
 *   q, k, v   the unquantized bf16 activations (the library quantizes them
 *             into the workspace first).
 *   o_hp      the high-precision forward output softmax(scale Q^ K^^T) V^,
 *             i.e. sdpa_fwd() of the fake-quantized inputs, and lse its LSE.
 *   workspace >= sdpa_bwd_nvfp4_qat_workspace_size() bytes, or NULL.
 * Served for D_qk = D_v = 128 (SDPA_ERR_UNSUPPORTED otherwise), with every
 * mask, padding and GQA of sdpa_bwd(). Returns as sdpa_bwd().
 */
int sdpa_bwd_nvfp4_qat(const void* q, const void* k, const void* v, const void* o_hp,
                       const void* d_o, const float* lse, void* dq, void* dk, void* dv, int B,
                       int H_q, int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale,
                       int causal, int bottom_right, int window_left, int window_right,
                       const int32_t* seq_q_lens, const int32_t* seq_kv_lens, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* sdpa_status_string(int status);

/*
 * Synchronizes `stream`, then reads and clears the current device's status
 * word. Returns SDPA_OK, SDPA_ERR_TIMEOUT if any kernel gave up on a bounded
 * wait since the last check (its results are then invalid), or SDPA_ERR_CUDA
 * if the synchronization itself failed.
 */
int sdpa_bwd_check_device_status(void* stream);  /* SDPA_ERR_BOUNDS takes precedence */

/*
 * Failure detection of the ordered relay (deterministic mode for D_qk other
 * than 128 and 192; cuDNN frontend docs, "SDPA Backward (SM120)", section
 * "Deterministic vs. non-deterministic dQ": the relay can stall if its
 * ordering assumption fails). Each key tile waits for its turn on a query
 * tile at most `wait_limit_ns` nanoseconds (0 restores the default, 4 s);
 * then it adds out of order, the call's results are not reproducible, and the
 * next sdpa_bwd_check_device_status() returns SDPA_ERR_TIMEOUT. `turn_skew`
 * (0 in normal use) is added to every expected turn: a nonzero skew makes the
 * first key tile of each query tile wait for a turn that no tile releases,
 * which exercises the bounded wait without any fault. Process-wide; applies
 * to calls made afterwards. Returns SDPA_OK.
 */
int sdpa_bwd_debug_relay(unsigned long long wait_limit_ns, int turn_skew);

/*
 * Per-kernel timing for benchmarks. While enabled, sdpa_bwd() records CUDA
 * events around each launch and synchronizes the stream before returning, so
 * it is for measurement only. sdpa_bwd_profile_read() fills up to n entries of
 * ms[] (total milliseconds) and launches[] (count) per kernel in the order
 * preprocess (with, for sdpa_bwd_nvfp4_qat(), the fake quantization of Q, K
 * and V before it), main, dq (the dQ convert, or on the two-kernel route the
 * dQ = scale * dS K kernel; under GQA it also runs the dK/dV group
 * reduction), and returns the number of entries (3). sdpa_bwd_sink(),
 * sdpa_bwd_bias() and sdpa_bwd_nvfp4_qat() are timed the same way.
 * Enabling resets the totals.
 */
int sdpa_bwd_profile_enable(int on);
int sdpa_bwd_profile_read(float* ms, int* launches, int n);

/*
 * Allocation-free SDPA backward. The SDPA backward pages have no counterpart
 * to this entry point; it exists for callers that cannot allocate device
 * memory where they run the backward (plugins or foreign-function hooks of a
 * framework that already owns the whole device memory pool, where cudaMalloc
 * fails or fragments the pool, and latency-critical code that cannot accept
 * cudaMalloc's implicit synchronization).
 *
 * Same arguments and results as sdpa_bwd() without the workspace: the caller
 * still provides every input and output, and the chain's scratch memory comes
 * from a 16 MiB device array compiled into the library. It calls no allocator.
 *   - The array occupies 16 MiB on a GPU from the moment the library's code
 *     module holding it is loaded there until the process exits. Under CUDA's
 *     default lazy module loading that is the first call on that GPU, and the
 *     kernels' modules load at their first launch; both take device memory. A
 *     caller whose framework later reserves the whole device pool makes one
 *     small call on each GPU first (or sets CUDA_MODULE_LOADING=EAGER).
 *   - Problems whose sdpa_bwd_workspace_size() exceeds 16 MiB (16777216 bytes)
 *     return SDPA_ERR_WORKSPACE before anything is launched.
 *   - All calls on a device share that array and it keeps what the last call
 *     left; the kernels re-clear what must start at zero on every call, but
 *     calls whose work overlaps on the device race on the array.
 *   - The first call on each device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 */
int sdpa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                     const void* d_o, const float* lse, void* dq, void* dk, void* dv, int B,
                     int H_q, int H_kv, int S_q, int S_kv, int D_qk, int D_v, float scale,
                     int causal, int bottom_right, int window_left, int window_right,
                     int deterministic, const int32_t* seq_q_lens, const int32_t* seq_kv_lens,
                     void* stream);

/* Library ABI version (major * 100 + minor). */
int sdpa_bwd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_BWD_H_ */
