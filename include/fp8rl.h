/*
 * fp8rl.h -- C ABI of the 8-bit rollout linear layer for GB300 (sm_103a).
 *
 * In RL with 8-bit rollouts the trainer updates the bf16 policy weights every
 * step, so the rollout engine must quantize them again after every update and
 * then run its linear layers on 8-bit weights and activations:
 *   - "FP8-RL: A Practical and Stable Low-Precision Stack for LLM Reinforcement
 *     Learning", Abstract: policy weights change every step, requiring repeated
 *     quantization; contribution (i), FP8 W8A8 linear-layer rollout with
 *     blockwise FP8 quantization.
 *   - FlashRL news write-up ("FlashRL: 8Bit Rollouts, Full Power RL"), section
 *     on online quantization (quantizing a model whose parameters are updated)
 *     and Fig. 1 (INT8 and FP8 rollouts).
 * The pages fix neither block sizes nor scale rules.  This library reads
 * "blockwise" as: weight blocks of 128x128 and activation groups of 1x128, one
 * fp32 scale each, scale = fl32(amax / 448) (an all-zero block gets scale 1),
 * code = E4M3FN(round-to-nearest-even, saturate to +-448)(fl32(x / scale)).
 * INT8 uses one symmetric scale per row (weight output channel / token),
 * scale = fl32(amax / 127), code = clamp(rint(fl32(x / scale)), -127, 127),
 * int32 accumulation.  E4M3FN is the OCP OFP8 format.
 *
 * Conventions shared by every call:
 *   - Layout is nn.Linear's: W is [N][K] row-major (out x in), X is [M][K],
 *     Y is [M][N].  bf16 tensors are passed as uint16_t bit patterns.
 *   - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *     never allocates, frees or synchronizes (fp8rl_check_device_error is the
 *     one documented exception: it synchronizes).  All work is enqueued on
 *     `stream` (a cudaStream_t; NULL is the legacy default stream) and is
 *     asynchronous.  The calling thread's current device must own the buffers.
 *   - Validation is synchronous and happens before any launch:
 *       FP8RL_ERR_NULL   a required pointer is NULL (with a non-empty shape),
 *       FP8RL_ERR_SHAPE  N or K not a multiple of 128, a negative size, or a
 *                        leading dimension smaller than the row length,
 *       FP8RL_ERR_ALIGN  a tensor not 16-byte aligned, or a leading
 *                        dimension whose row pitch is not a multiple of 16 B,
 *       FP8RL_ERR_WORKSPACE  workspace smaller than the *_workspace_bytes query
 *                        (where it is required; the GEMMs instead take a
 *                        slower path, as their entries say),
 *       FP8RL_ERR_UNSUPPORTED a size above a documented limit.
 *     A launch failure reported by the runtime returns FP8RL_ERR_CUDA.  Faults
 *     during execution surface, as usual in CUDA, at the caller's next
 *     synchronization.
 *   - M == 0 (an empty batch) is valid and launches nothing.
 *   - Inputs must be finite; NaN/Inf are not checked on this path.
 */
#ifndef FP8RL_H_
#define FP8RL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8RL_OK = 0,
    FP8RL_ERR_NULL = 1,
    FP8RL_ERR_SHAPE = 2,
    FP8RL_ERR_ALIGN = 3,
    FP8RL_ERR_WORKSPACE = 4,
    FP8RL_ERR_CUDA = 5,
    FP8RL_ERR_UNSUPPORTED = 6,
    FP8RL_ERR_TIMEOUT = 7,
    FP8RL_ERR_DEVICE = 8
} fp8rl_status;

#define FP8RL_ABI_VERSION 3

/* Human-readable name of a status code (static storage, never NULL). */
const char* fp8rl_status_string(int status);

/* FP8RL_ABI_VERSION of the loaded library. */
int fp8rl_abi_version(void);

/* ------------------------------------------------------------------------
 * FP8 weight requant (FP8-RL, Abstract: repeated quantization every step;
 * contribution (i): blockwise FP8).  For every 128x128 block (nb, kb) of W:
 *   amax = max |w| (exact, fp32); s = amax == 0 ? 1 : fl32(amax / 448);
 *   Wq[n][k] = E4M3FN_rn_satfinite(fl32(W[n][k] / s)); Ws[nb][kb] = s.
 * W   bf16 [N][ldw], ldw >= K, ldw % 8 == 0, 16-byte aligned.
 * Wq  e4m3 codes [N][K] (contiguous), 16-byte aligned.
 * Ws  fp32 [N/128][K/128] row-major, 4-byte aligned.
 * Output is bit-exact (a pure function of the input bits).
 * ---------------------------------------------------------------------- */
int fp8rl_quant_weight_block(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                             uint8_t* Wq, float* Ws, void* stream);

/* One tensor of a grouped requant: the same operation as
 * fp8rl_quant_weight_block, with the same layout rules per tensor. */
typedef struct {
    const uint16_t* W;
    uint8_t* Wq;
    float* Ws;
    int64_t N, K, ldw;
} fp8rl_wdesc;

/* Requant of n weight tensors (e.g. every linear layer of a model after one
 * policy update) in as few launches as possible.  `descs` is a HOST array of n
 * descriptors (read during the call; the caller may reuse it on return); the
 * pointers inside are device pointers.  Tensors must not overlap.  Any invalid
 * descriptor fails the whole call before anything is launched. */
int fp8rl_quant_weight_block_grouped(const fp8rl_wdesc* descs, int n, void* stream);

/* ------------------------------------------------------------------------
 * FP8 activation quant, 1x128 groups per token (FP8-RL contribution (i), the
 * A8 of W8A8).  For token m and group g (columns 128g .. 128g+127):
 *   s = amax == 0 ? 1 : fl32(amax / 448); Xq[m][k] = E4M3FN_rn_satfinite(fl32(X[m][k] / s)).
 * X   bf16 [M][ldx], ldx >= K, ldx % 8 == 0, 16-byte aligned.
 * Xq  e4m3 [M][K] contiguous, 16-byte aligned.
 * Xs  fp32 [K/128][M]: group-major, so that a GEMM reads the scales of
 *     consecutive tokens contiguously.  4-byte aligned.
 * Bit-exact.
 * ---------------------------------------------------------------------- */
int fp8rl_quant_act_group(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                          uint8_t* Xq, float* Xs, void* stream);

/* ------------------------------------------------------------------------
 * FP8 block-scaled W8A8 GEMM with bf16 output (FP8-RL contribution (i)):
 *   Y[m][n] = bf16_rn( sum_kb Xs[kb][m] * Ws[n/128][kb] * sum_{k in kb} e4m3(Xq[m][k]) * e4m3(Wq[n][k]) )
 * computed with fp32 tensor-core partial sums per 128-wide K block and fp32
 * promotion of each block's scale product.  Accumulation order is not fixed:
 * the result matches the exact value within |y - y_ref| <= 2^-7 |y_ref| +
 * 1e-3 rms(y_ref).  The same call serves decode (small M, weight streaming,
 * HBM-bound) and prefill (large M, tensor-bound); the library picks the kernel.
 * Xq [M][K] e4m3, Xs [K/128][M] fp32, Wq [N][K] e4m3, Ws [N/128][K/128] fp32,
 * Y bf16 [M][ldy], ldy >= N, ldy % 8 == 0.  All 16-byte aligned (scales: 4).
 * workspace: device scratch, 16-byte aligned, of fp8rl_gemm_workspace_bytes(M,
 * N, K) bytes.  It is nonzero for shapes whose K the library splits through
 * memory: most batches of 17..256 tokens on layers with few 128-row weight
 * slabs, small batches on long-K layers (the 27648-wide down projection of a
 * 5120-wide model), and a few hundred tokens against a long K.  The fp32
 * partial tiles are then added in a second launch, in a fixed order
 * (deterministic), so the call launches two kernels instead of one.  With less
 * workspace (or NULL) the call still succeeds, on a split that keeps its
 * partial sums on chip (slower for those shapes).  It does not need to be zeroed and holds
 * nothing between calls, but two calls in flight at once need two workspaces.
 * ---------------------------------------------------------------------- */
size_t fp8rl_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
/* Number of kernels fp8rl_gemm_w8a8_block launches for this shape when given
 * workspace_bytes of workspace (0: none): 1, or 2 when the K split is added by
 * a second launch.  0 for M == 0; -FP8RL_ERR_SHAPE for an invalid shape.  For
 * sizing CUDA graphs and counting launches; host-only, no device access. */
int fp8rl_gemm_kernel_count(int64_t M, int64_t N, int64_t K, size_t workspace_bytes);
int fp8rl_gemm_w8a8_block(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                          const float* Ws, int64_t M, int64_t N, int64_t K,
                          uint16_t* Y, int64_t ldy, void* workspace,
                          size_t workspace_bytes, void* stream);

/* fp8rl_gemm_w8a8_block with flags (same arithmetic, arguments and errors;
 * fp8rl_gemm_w8a8_block is this call with flags = 0).
 * FP8RL_GEMM_WEIGHTS_STABLE: the caller guarantees that the kernel issued
 *     immediately before this call on the same stream did not write Wq (the
 *     usual case in a decode loop: the weights were requantized earlier in the
 *     step, and the call before this one produced the activations).  Every
 *     kernel of this library is launched only after the one before it has
 *     passed its own wait for its predecessor, so anything issued earlier than
 *     the immediately preceding kernel has completed by then.  Small weight
 *     matrices (at most 48 MB) then start streaming into the GEMM before its
 *     wait for that preceding kernel, overlapping its tail.  With a Wq written
 *     by the immediately preceding kernel the result is undefined.
 * Unknown flag bits: FP8RL_ERR_UNSUPPORTED.
 * fp8rl_linear_w8a8_block applies this internally (its GEMM always follows its
 * own activation quantizer). */
#define FP8RL_GEMM_WEIGHTS_STABLE 1u
int fp8rl_gemm_w8a8_block_ex(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                             const float* Ws, int64_t M, int64_t N, int64_t K,
                             uint16_t* Y, int64_t ldy, void* workspace,
                             size_t workspace_bytes, unsigned flags, void* stream);

/* ------------------------------------------------------------------------
 * Grouped block-scaled FP8 GEMM for mixture-of-experts layers (FP8-RL,
 * Abstract: the FP8 rollout stack serves dense and MoE models).  The T token
 * rows are grouped by expert: rows expert_offsets[e] .. expert_offsets[e+1]-1
 * of Xq go through expert e's weights, and for those rows
 *   Y = fp8rl_gemm_w8a8_block(Xq[rows], Xs[:, rows], Wq[e], Ws[e])
 * (same arithmetic and tolerance).  Experts without tokens read none of their
 * weights.  Built on the decode kernel: meant for decode-sized groups.
 * Xq [T][K] e4m3, Xs [K/128][T] fp32, Y bf16 [T][ldy] (ldy >= N, ldy % 8 == 0).
 * Wq  e4m3 [E][N][K] (experts stacked), Ws fp32 [E][N/128][K/128].
 * expert_offsets: DEVICE int32 [E+1], non-decreasing, [0] = 0, [E] = T (the
 *     kernel clamps every range into [0, T], so bad offsets cannot make it
 *     read or write outside the tensors).  It may be written by the previous
 *     kernel in the stream (e.g. a router).
 * max_tokens_per_expert: a host-side bound, 1 <= bound <= T, on every expert's
 *     token count; the grid covers that many rows per expert.  Rows of an
 *     expert beyond it are not computed and the device records it
 *     (fp8rl_check_device_error returns FP8RL_ERR_DEVICE).
 * Limits: K <= 32768 and E * N / 128 <= 65535 (FP8RL_ERR_UNSUPPORTED).
 * ---------------------------------------------------------------------- */
int fp8rl_gemm_w8a8_block_grouped(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                  const float* Ws, const int32_t* expert_offsets, int64_t E,
                                  int64_t T, int64_t N, int64_t K, int64_t max_tokens_per_expert,
                                  uint16_t* Y, int64_t ldy, void* stream);

/* ------------------------------------------------------------------------
 * The whole 8-bit linear layer from bf16 activations: the activation quant
 * above followed by the block-scaled GEMM above, in one call (FP8-RL
 * contribution (i): W8A8 rollout linear layers; the activation side is
 * quantized on the fly, token by token).  The result is
 *   Y = fp8rl_gemm_w8a8_block(Xq, Xs, Wq, Ws)  with  (Xq, Xs) = fp8rl_quant_act_group(X):
 * the same codes and scales (bit-exact) and Y within the GEMM's tolerance.
 * Two kernels run back to back on `stream`: the quantizer, then the GEMM,
 * which is scheduled while the quantizer runs and starts streaming its weights
 * meanwhile (the quantizer writes no weights, so the GEMM loads the weight
 * tiles of its first pipeline stages before its dependency wait, as with
 * FP8RL_GEMM_WEIGHTS_STABLE).  fp8rl_linear_kernel_count gives the count.
 * X   bf16 [M][ldx], ldx >= K, ldx % 8 == 0, 16-byte aligned.
 * Wq, Ws, Y, ldy as for fp8rl_gemm_w8a8_block.
 * Xq_or_null, Xs_or_null: both NULL, or both given ([M][K] e4m3 contiguous,
 *     16-byte aligned; [K/128][M] fp32, 4-byte aligned) to receive the
 *     activation codes and scales.
 * workspace: at least fp8rl_linear_workspace_bytes(M, N, K) bytes, 16-byte
 *     aligned: room for the codes and scales (unused when Xq/Xs are given)
 *     followed by the GEMM's own workspace (see fp8rl_gemm_w8a8_block); no
 *     zeroing needed; calls in flight at once need their own.
 * Limit: M <= 1048560 (FP8RL_ERR_UNSUPPORTED above).
 * ---------------------------------------------------------------------- */
size_t fp8rl_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);
/* Kernels fp8rl_linear_w8a8_block launches for this shape with workspace_bytes
 * of workspace (want_codes != 0 when Xq/Xs are to be returned): the quantizer
 * plus the GEMM's kernel count.  0 for M == 0; -FP8RL_ERR_SHAPE for an invalid
 * shape.  Host-only, no device access. */
int fp8rl_linear_kernel_count(int64_t M, int64_t N, int64_t K, size_t workspace_bytes, int want_codes);
int fp8rl_linear_w8a8_block(const uint16_t* X, int64_t ldx, const uint8_t* Wq, const float* Ws,
                            int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy,
                            uint8_t* Xq_or_null, float* Xs_or_null, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * INT8 per-row quant (FlashRL write-up, Fig. 1: INT8 rollout).  Per row r:
 *   s = amax == 0 ? 1 : fl32(amax / 127); Q[r][k] = clamp(rint(fl32(A[r][k] / s)), -127, 127).
 * The weight variant has one scale per output channel (row of W, Ws [N]); the
 * activation variant one per token (row of X, Xs [M]).
 * A bf16 [R][lda], lda >= K, lda % 8 == 0; Q int8 [R][K] contiguous; S fp32 [R].
 * K <= 32768 (FP8RL_ERR_UNSUPPORTED above).  Bit-exact.
 * ---------------------------------------------------------------------- */
int int8rl_quant_weight_channel(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                int8_t* Wq, float* Ws, void* stream);
int int8rl_quant_act_token(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                           int8_t* Xq, float* Xs, void* stream);

/* ------------------------------------------------------------------------
 * INT8 W8A8 GEMM (FlashRL INT8 rollout):
 *   acc[m][n] = sum_k Xq[m][k] * Wq[n][k]  (int32, exact);
 *   Y[m][n]   = bf16_rn( fl32( fl32(float_rn(acc)) * Xs[m] ) * Ws[n] )  (no FMA).
 * Bit-exact in both acc and Y.  Requires K * 127^2 < 2^31 (K <= 133143) so
 * that no accumulator can overflow; larger K returns FP8RL_ERR_UNSUPPORTED.
 * Xq [M][K] int8, Xs [M] fp32, Wq [N][K] int8, Ws [N] fp32, Y bf16 [M][ldy].
 * acc_or_null: optional int32 [M][N] copy of the accumulators (8-byte aligned).
 * workspace: device scratch, 16-byte aligned, of int8rl_gemm_workspace_bytes(M,
 * N, K) bytes; zero where the small-batch kernel runs (always for up to 64
 * tokens), which needs none.
 *   - 65 to 256 tokens, and up to 512 on layers of at least 2^27 weights: an
 *     fp16 copy of Xq (M * K * 2 bytes, rounded up to 16, exact), loaded in
 *     256-token tiles, and, when those tiles are too few for the GPU, the int32
 *     partial tiles of the K ranges (added exactly by a second launch).
 *   - Larger batches with enough 128 x 256 output tiles (or tiles x K ranges)
 *     for half of the GPU: fp16 copies of Xq and Wq ((M + N) * K * 2 bytes),
 *     and the int32 partial tiles of a K split.
 * With less workspace (or NULL) the call still succeeds on the small-batch
 * kernel (slower for those shapes).  Not zeroed, nothing kept between calls;
 * two calls in flight at once need two workspaces.
 * ---------------------------------------------------------------------- */
size_t int8rl_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
/* Kernels int8rl_gemm_w8a8 launches for this shape and workspace size: 1 on the
 * small-batch kernel; 2 or 3 on the other two paths (conversion, GEMM, and the
 * reduction of a K split).  0 for M == 0; -FP8RL_ERR_SHAPE for an invalid shape. */
int int8rl_gemm_kernel_count(int64_t M, int64_t N, int64_t K, size_t workspace_bytes);
int int8rl_gemm_w8a8(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                     int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy,
                     int32_t* acc_or_null, void* workspace, size_t workspace_bytes,
                     void* stream);

/* ------------------------------------------------------------------------
 * FP8 KV-cache quantization with per-step scale recalibration (FP8-RL,
 * Abstract, contribution (ii): FP8 KV-cache, QKV scales recalibrated every
 * step).  One fp32 scale per K (or V) tensor, recomputed from the tensor:
 *   s = amax == 0 ? 1 : fl32(amax / 448) over all R x C values;
 *   KVq[r][c] = E4M3FN_rn_satfinite(fl32(KV[r][c] / s)); *scale = s.
 * KV    bf16 [R][ld] (e.g. tokens x kv_heads*head_dim), C % 8 == 0, ld >= C,
 *       ld % 8 == 0, 16-byte aligned.
 * KVq   e4m3 [R][C] contiguous, 16-byte aligned.
 * scale one fp32 in device memory (written by the call).
 * workspace: device scratch of at least fp8rl_kv_workspace_bytes(R, C) bytes
 *       (8 bytes per 16384 values, plus 8), 8-byte aligned; it needs no zeroing
 *       (any content is accepted).  Its first 8 bytes carry a call counter from
 *       one call to the next, which the device advances, so the call may be
 *       captured in a CUDA graph and replayed.  Calls in flight at the same time
 *       need their own workspace.  Tensors of up to about 10 M values are done
 *       in one pass (one cooperative launch; a bounded wait that runs out is
 *       reported by fp8rl_check_device_error as FP8RL_ERR_TIMEOUT).  Larger
 *       ones with contiguous rows (ld == C) take one cooperative launch of one
 *       CTA per SM that keeps up to 448 KB of each SM's range on chip between
 *       the amax and the encode (read once up to ~34 M values on GB300, the
 *       rest read again above that; time-outs reported the same way); larger
 *       ones with a row pitch take three launches.
 * Bit-exact.  An empty tensor (R == 0) writes scale 1.
 * ---------------------------------------------------------------------- */
size_t fp8rl_kv_workspace_bytes(int64_t R, int64_t C);
int fp8rl_quant_kv_tensor(const uint16_t* KV, int64_t R, int64_t C, int64_t ld, uint8_t* KVq,
                          float* scale, void* workspace, size_t workspace_bytes, void* stream);

/* The same codes under a scale already fixed for this step (appending new
 * tokens to a KV cache): KVq = E4M3FN_rn_satfinite(fl32(KV / *scale)).
 * scale: one fp32 > 0 in device memory (read by the kernel). */
int fp8rl_quant_kv_with_scale(const uint16_t* KV, int64_t R, int64_t C, int64_t ld,
                              const float* scale, uint8_t* KVq, void* stream);

/* ------------------------------------------------------------------------
 * Token-level importance-sampling rollout correction (FP8-RL, Abstract,
 * contribution (iii): token-level TIS/MIS; FlashRL write-up, section on
 * truncated importance sampling).  For n sampled tokens with log-probabilities
 * under the trainer's policy (logp_train) and under the 8-bit rollout policy
 * (logp_rollout), d = fl32(logp_train - logp_rollout) and, with the threshold
 * C given as log_clip = ln C:
 *   mode FP8RL_IS_TRUNCATE (TIS): w = exp(min(d, log_clip))
 *   mode FP8RL_IS_MASK     (MIS): w = d > log_clip ? 0 : exp(d)
 * Tokens whose mask byte is 0 (padding) get w = 0 and are not counted; mask may
 * be NULL (every token valid).  The clip decision is an fp32 comparison (exact
 * count); w is within a few ulp of exp (CUDA expf).
 * logp_train, logp_rollout, weights: fp32 [n], 4-byte aligned; mask: u8 [n].
 * stats: 4 doubles in device memory: [0] valid tokens, [1] tokens truncated
 * (TIS) or masked (MIS), [2] sum of w, [3] sum of d over valid tokens (its
 * mean is the sample estimate of KL(rollout || train) when the tokens are drawn
 * from the rollout policy).  The sums are reduced in a fixed order
 * (deterministic run to run).
 * workspace: at least fp8rl_rollout_is_workspace_bytes(n) bytes, 8-byte
 * aligned (8 bytes plus 32 bytes per 4096 tokens).  It needs no zeroing; the
 * call leaves a tag in its first word that the next call on the same
 * workspace builds on, so two calls sharing one workspace must not run
 * concurrently (on different streams).
 * ---------------------------------------------------------------------- */
#define FP8RL_IS_TRUNCATE 0
#define FP8RL_IS_MASK 1
size_t fp8rl_rollout_is_workspace_bytes(int64_t n);
int fp8rl_rollout_is_weights(const float* logp_train, const float* logp_rollout,
                             const uint8_t* mask, int64_t n, float log_clip, int mode,
                             float* weights, double* stats, void* workspace,
                             size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Train-inference mismatch of a quantized rollout (FlashRL write-up, Fig. 2,
 * right: the KL divergence between the trainer's policy and the rollout
 * engine's, larger for INT8 rollouts than for FP8 ones).  For every token row
 * m of two logit matrices -- P from the higher-precision policy, Q from the
 * quantized one (e.g. the output of an LM-head GEMM) --
 *   kl[m] = sum_v softmax(P[m])_v * (log softmax(P[m])_v - log softmax(Q[m])_v).
 * P [M][ldp], Q [M][ldq] bf16, V >= 1 logits per row, ld >= V, ld % 8 == 0,
 * 16-byte aligned; kl fp32 [M], 4-byte aligned.  Logits must be finite and
 * |P - Q| < 32 elementwise (keeps every fp32 term finite).  Accuracy: |kl - kl_exact| <= 1e-4 kl_exact + 1e-7
 * (fp32 elementwise terms, fp64 combination; see mismatch_kl.cu).
 * Deterministic.  workspace: at least fp8rl_logits_kl_workspace_bytes(M, V)
 * bytes, 16-byte aligned, no zeroing needed (32 bytes per 4096 logits).
 * Limit: M <= 65535 (FP8RL_ERR_UNSUPPORTED).
 * ---------------------------------------------------------------------- */
size_t fp8rl_logits_kl_workspace_bytes(int64_t M, int64_t V);
int fp8rl_logits_kl(const uint16_t* P, int64_t ldp, const uint16_t* Q, int64_t ldq, int64_t M,
                    int64_t V, float* kl, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * fp8rl_quant_kv_tensor without a workspace.  The paper has no counterpart:
 * this is a calling convention, not part of the method.  It computes exactly
 * what fp8rl_quant_kv_tensor computes, for callers that cannot allocate the
 * workspace -- e.g. an inference engine that reserves nearly all GPU memory
 * for its KV-cache pool at start-up and allows no allocation outside it, or a
 * serving loop that must not call cudaMalloc / cudaFree because they
 * synchronize the device and stall queued work.  It allocates nothing and
 * calls no allocating routine.
 * Scratch: a 64 KB (+ 8 bytes) array in device memory owned by the library (a
 * file-scope __device__ array), held by every GPU that loads the library until
 * the process exits.  Limit: R * C <= 268435456 (16384 x 16384) values; larger
 * tensors return FP8RL_ERR_UNSUPPORTED (use fp8rl_quant_kv_tensor instead).
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  Every call shares the one array: nothing in it needs to start at
 * zero (the three-launch path writes every slot before reading it; the
 * cooperative paths accept a slot only once it carries the call's tag, which
 * the device derives from the previous call's), and two calls
 * whose kernels overlap on the GPU (different streams) race on it -- issue
 * them in one stream, or use fp8rl_quant_kv_tensor with separate workspaces.
 * Other arguments, layouts and errors as for fp8rl_quant_kv_tensor.
 * ---------------------------------------------------------------------- */
int fp8rl_quant_kv_tensor_noalloc(const uint16_t* KV, int64_t R, int64_t C, int64_t ld,
                                  uint8_t* KVq, float* scale, void* stream);

/* ------------------------------------------------------------------------
 * Every wait inside the library's kernels (on an mbarrier filled by TMA or by
 * the tensor core) is bounded.  A wait that runs out records a code in a
 * device-side word, abandons the tile and lets the kernel exit, so the CUDA
 * context stays usable.  This call SYNCHRONIZES the current device, reads and
 * clears that word, and returns FP8RL_OK, FP8RL_ERR_TIMEOUT (a wait ran out)
 * or FP8RL_ERR_DEVICE (a device-side check of the data failed: an expert of
 * the grouped GEMM with more tokens than max_tokens_per_expert).  *detail
 * (may be NULL) receives the raw word (0 if none: kernel id in bits 24..31,
 * the site in bits 16..23, 1 = timeout / 2 = data check in bits 0..15).
 * ---------------------------------------------------------------------- */
int fp8rl_check_device_error(uint32_t* detail);

#ifdef __cplusplus
}
#endif

#endif /* FP8RL_H_ */
