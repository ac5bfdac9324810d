/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the 8-bit rollout
 * linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that the tests, the smoke check and the CPU
 * baseline leg of the benchmark can compare the CUDA library against an
 * independent statement of the method.  It shares no code, header, table or
 * constant generator with the CUDA library.
 *
 * What the method computes, and where it comes from:
 *   - "FP8-RL: A Practical and Stable Low-Precision Stack for LLM Reinforcement
 *     Learning", Abstract, contribution (i): FP8 W8A8 linear-layer rollout with
 *     blockwise FP8 quantization; the policy weights change every step, so they
 *     are quantized again after every update.
 *   - FlashRL news write-up ("FlashRL: 8Bit Rollouts, Full Power RL"), section
 *     on online quantization (weights re-quantized when the trainer updates
 *     them) and the INT8 / FP8 rollout policies of Fig. 1 and Fig. 2.
 * The pages fix neither block sizes nor the scale rule.  This oracle takes the
 * reading the library documents: weight blocks of 128x128 and activation groups
 * of 1x128, scale = fl32(amax / 448) (amax = 0 -> scale 1), codes =
 * E4M3FN(RNE, saturate-to-finite)(fl32(x / scale)); INT8 uses one scale per
 * row, fl32(amax / 127), codes = clamp(rint(fl32(x / scale)), -127, 127).
 * The E4M3FN format itself is the one of the OCP 8-bit Floating Point
 * Specification (OFP8): bias 7, no infinities, S.1111.111 is NaN, largest
 * finite value 448, subnormal step 2^-9.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -shared -fPIC.
 * The flags matter: every fp32 operation below must be one IEEE-754 operation
 * rounded to nearest-even, with no fused multiply-add contraction.
 *
 * Parity pins (see tests/test_oracle_pins.py): the E4M3 encoder against brute
 * force over all 256 codes; the activation quantizer against a hand-worked
 * example (two worked rows plus an all-zero row); round-trip and saturation
 * invariants; the INT8 GEMM against an
 * int64 library matmul; the FP8 GEMM against an exact integer special case and
 * against an unquantized fp64 matmul within the derived quantization bound.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define QBLK 128 /* weight block edge and activation group length */

/* ------------------------------------------------------------------ */
/* number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 -> fp32 is exact: a bf16 is the upper half of an fp32. */
static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float oracle_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }

/* fp32 -> bf16, round to nearest, ties to even (finite inputs). */
uint16_t oracle_f32_to_bf16_rn(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u) {          /* inf / nan: keep, quiet nan */
        uint16_t hi = (uint16_t)(u >> 16);
        if (u & 0x007FFFFFu) hi |= 0x0040u;
        return hi;
    }
    uint32_t keep_lsb = (u >> 16) & 1u;                /* tie goes to the even result */
    u += 0x7FFFu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* E4M3FN decode (OCP OFP8): s.eeee.mmm, bias 7; e == 0 is subnormal
 * (m/8)*2^-6; s.1111.111 is NaN; there is no infinity. */
double oracle_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);             /* (m/8) * 2^(1-7) */
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* E4M3FN encode: round the fp32 value v to the nearest finite E4M3FN value,
 * ties to the even 3-bit mantissa, saturating to +-448 (satfinite).  The sign
 * bit follows v, so -0 and negative values that round to zero give 0x80.
 * Precondition: v is finite. */
uint8_t oracle_e4m3_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    float a = fabsf(v);
    if (a >= 448.0f) return sign | 0x7E;               /* largest finite: 1.75 * 2^8 */
    if (a < 0.015625f) {                               /* below 2^-6: grid step 2^-9 */
        float q = nearbyintf(a * 512.0f);               /* exact scaling, then RNE */
        return sign | (uint8_t)q;                       /* q == 8 is 2^-6, code 0x08 */
    }
    int e2;
    float fr = frexpf(a, &e2);                          /* a = fr * 2^e2, fr in [0.5,1) */
    int E = e2 - 1;                                     /* a = (2 fr) * 2^E, 2fr in [1,2) */
    float t = nearbyintf((2.0f * fr - 1.0f) * 8.0f);    /* every step exact; RNE */
    int mant = (int)t;
    if (mant == 8) { mant = 0; E += 1; }
    int code = ((E + 7) << 3) | mant;
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

void oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------------ */
/* scales                                                              */
/* ------------------------------------------------------------------ */

/* fl32(amax / 448); an all-zero block gets scale 1 (its codes are all zero). */
static float fp8_scale(float amax) { return amax == 0.0f ? 1.0f : amax / 448.0f; }
/* fl32(amax / 127); an all-zero row gets scale 1. */
static float int8_scale(float amax) { return amax == 0.0f ? 1.0f : amax / 127.0f; }

/* ------------------------------------------------------------------ */
/* FP8 weight requant: 128x128 blocks (FP8-RL, Abstract (i): blockwise FP8,
 * re-quantized every step because the policy weights change every step)   */
/* ------------------------------------------------------------------ */

/* W: bf16 bits [N][ldw] (row n, column k).  Wq: e4m3 codes [N][K].
 * Ws: fp32 [N/128][K/128], block (nb, kb) at Ws[nb*(K/128) + kb].
 * Returns 0, or -1 for a shape that is not a whole number of blocks. */
int oracle_fp8_quant_weight_block(const uint16_t* W, int64_t N, int64_t K, int64_t ldw,
                                  uint8_t* Wq, float* Ws) {
    if (N % QBLK || K % QBLK || ldw < K) return -1;
    int64_t KB = K / QBLK;
    for (int64_t nb = 0; nb < N / QBLK; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t i = 0; i < QBLK; ++i)
                for (int64_t j = 0; j < QBLK; ++j) {
                    float x = fabsf(bf16_to_f32(W[(nb * QBLK + i) * ldw + kb * QBLK + j]));
                    if (x > amax) amax = x;
                }
            float s = fp8_scale(amax);
            Ws[nb * KB + kb] = s;
            for (int64_t i = 0; i < QBLK; ++i)
                for (int64_t j = 0; j < QBLK; ++j) {
                    int64_t n = nb * QBLK + i, k = kb * QBLK + j;
                    float x = bf16_to_f32(W[n * ldw + k]);
                    Wq[n * K + k] = oracle_e4m3_encode(x / s);
                }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* FP8 activation quant: 1x128 groups per token (W8A8, FP8-RL Abstract (i)) */
/* ------------------------------------------------------------------ */

/* X: bf16 bits [M][ldx].  Xq: e4m3 codes [M][K].
 * Xs: fp32 [K/128][M] (group-major), group g of token m at Xs[g*M + m]. */
int oracle_fp8_quant_act_group(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                               uint8_t* Xq, float* Xs) {
    if (K % QBLK || ldx < K || M < 0) return -1;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < K / QBLK; ++g) {
            float amax = 0.0f;
            for (int64_t j = 0; j < QBLK; ++j) {
                float x = fabsf(bf16_to_f32(X[m * ldx + g * QBLK + j]));
                if (x > amax) amax = x;
            }
            float s = fp8_scale(amax);
            Xs[g * M + m] = s;
            for (int64_t j = 0; j < QBLK; ++j) {
                float x = bf16_to_f32(X[m * ldx + g * QBLK + j]);
                Xq[m * K + g * QBLK + j] = oracle_e4m3_encode(x / s);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* FP8 KV-cache quant with a per-tensor scale recalibrated from the tensor
 * itself (FP8-RL, Abstract, contribution (ii): FP8 KV-cache with per-step QKV
 * scale recalibration; the reading taken is one scale per K or V tensor,
 * fl32(amax/448) over the whole tensor, recomputed at every call).         */
/* ------------------------------------------------------------------ */

/* X: bf16 bits [R][ldx] with row length C.  Xq: e4m3 codes [R][C].
 * *scale: the tensor's fp32 scale (amax = 0 gives 1). */
int oracle_fp8_quant_tensor(const uint16_t* X, int64_t R, int64_t C, int64_t ldx,
                            uint8_t* Xq, float* scale) {
    if (ldx < C || R < 0 || C < 0) return -1;
    float amax = 0.0f;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            float x = fabsf(bf16_to_f32(X[r * ldx + c]));
            if (x > amax) amax = x;
        }
    float s = fp8_scale(amax);
    *scale = s;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            Xq[r * C + c] = oracle_e4m3_encode(bf16_to_f32(X[r * ldx + c]) / s);
    return 0;
}

/* Codes of X under a given scale s (appending to a KV cache whose scale was
 * fixed for this step): Xq = E4M3FN_rn_satfinite(fl32(X / s)). */
int oracle_fp8_quant_with_scale(const uint16_t* X, int64_t R, int64_t C, int64_t ldx, float s,
                                uint8_t* Xq) {
    if (ldx < C || R < 0 || C < 0 || !(s > 0.0f)) return -1;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            Xq[r * C + c] = oracle_e4m3_encode(bf16_to_f32(X[r * ldx + c]) / s);
    return 0;
}

/* ------------------------------------------------------------------ */
/* INT8 row quant (FlashRL INT8 rollout, Fig. 1 / Fig. 2): one symmetric
 * scale per row over all K.  Used for the weight (per output channel) and
 * for the activation (per token); the two differ only in which rows they
 * are applied to.                                                       */
/* ------------------------------------------------------------------ */

/* A: bf16 bits [R][lda].  Q: int8 [R][K].  S: fp32 [R]. */
int oracle_int8_quant_rows(const uint16_t* A, int64_t R, int64_t K, int64_t lda,
                           int8_t* Q, float* S) {
    if (lda < K || R < 0 || K < 0) return -1;
    for (int64_t r = 0; r < R; ++r) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float x = fabsf(bf16_to_f32(A[r * lda + k]));
            if (x > amax) amax = x;
        }
        float s = int8_scale(amax);
        S[r] = s;
        for (int64_t k = 0; k < K; ++k) {
            float v = bf16_to_f32(A[r * lda + k]) / s;
            float t = nearbyintf(v);                     /* RNE */
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            Q[r * K + k] = (int8_t)t;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* FP8 block-scaled GEMM, fp64 reference                               */
/* ------------------------------------------------------------------ */

/* y[m][n] = sum_kb Xs[kb][m] * Ws[n/128][kb] * sum_{k in kb} dq(Xq[m][k]) dq(Wq[n][k])
 * in fp64.  The inner sum over one 128-wide K block is exact in fp64 (every
 * product of two E4M3 values is a multiple of 2^-18 below 2^18), so this is the
 * dequantize-then-matmul of the codes up to the final fp64 roundings.
 * Xq [M][K], Xs [K/128][M], Wq [N][K], Ws [N/128][K/128], Y [M][N]. */
int oracle_fp8_gemm(const uint8_t* Xq, const float* Xs, const uint8_t* Wq, const float* Ws,
                    int64_t M, int64_t N, int64_t K, double* Y) {
    if (N % QBLK || K % QBLK || M < 0) return -1;
    double dq[256];
    for (int c = 0; c < 256; ++c) dq[c] = oracle_e4m3_decode((uint8_t)c);
    int64_t KB = K / QBLK;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double y = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                double inner = 0.0;
                for (int64_t j = 0; j < QBLK; ++j) {
                    int64_t k = kb * QBLK + j;
                    inner += dq[Xq[m * K + k]] * dq[Wq[n * K + k]];
                }
                double sx = (double)Xs[kb * M + m];
                double sw = (double)Ws[(n / QBLK) * KB + kb];
                y += (sx * sw) * inner;
            }
            Y[m * N + n] = y;
        }
    }
    return 0;
}

/* Unquantized fp64 matmul of the bf16 operands (for reporting the error of the
 * 8-bit path against the full-precision layer; not a parity target).
 * X [M][ldx] bf16, W [N][ldw] bf16, Y [M][N]. */
int oracle_bf16_matmul_f64(const uint16_t* X, int64_t ldx, const uint16_t* W, int64_t ldw,
                           int64_t M, int64_t N, int64_t K, double* Y) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double y = 0.0;
            for (int64_t k = 0; k < K; ++k)
                y += (double)bf16_to_f32(X[m * ldx + k]) * (double)bf16_to_f32(W[n * ldw + k]);
            Y[m * N + n] = y;
        }
    return 0;
}

/* ------------------------------------------------------------------ */
/* INT8 W8A8 GEMM: exact integer accumulation, fp32 epilogue            */
/* ------------------------------------------------------------------ */

/* acc[m][n] = sum_k Xq[m][k] * Wq[n][k], summed in int64 and required to fit
 * int32; y[m][n] = bf16_rn( fl32( fl32(float(acc)) * Xs[m] ) * Ws[n] ), two
 * separately rounded fp32 multiplies (no fused multiply-add).
 * int32 -> fp32 conversion rounds to nearest even (the default rounding mode).
 * Xq [M][K], Wq [N][K], Xs [M], Ws [N]; acc [M][N] may be NULL; Y [M][N] bf16.
 * Returns 0, or -2 if an accumulator leaves the int32 range. */
int oracle_int8_gemm(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                     int64_t M, int64_t N, int64_t K, int32_t* acc, uint16_t* Y) {
    int rc = 0;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            int64_t a = 0;
            for (int64_t k = 0; k < K; ++k) a += (int64_t)Xq[m * K + k] * (int64_t)Wq[n * K + k];
            if (a > INT32_MAX || a < INT32_MIN) rc = -2;
            int32_t a32 = (int32_t)a;
            if (acc) acc[m * N + n] = a32;
            float t = (float)a32;
            float u = t * Xs[m];
            float v = u * Ws[n];
            Y[m * N + n] = oracle_f32_to_bf16_rn(v);
        }
    return rc;
}

/* ------------------------------------------------------------------ */
/* Token-level importance-sampling rollout correction (FP8-RL, Abstract,
 * contribution (iii): token-level TIS/MIS; FlashRL write-up, section on TIS,
 * whose formula is missing from the extracted page).  Reading taken: for a
 * sampled token with log-probabilities lt under the trainer's policy and lr
 * under the 8-bit rollout policy, d = fl32(lt - lr) is the log importance
 * ratio; with a threshold C given as log_clip = ln C,
 *   truncated (TIS): w = exp(min(d, log_clip)),
 *   masked    (MIS): w = d > log_clip ? 0 : exp(d);
 * tokens with mask 0 (padding) get w = 0 and are not counted.  The decision
 * d > log_clip is taken in fp32 (the precision the library uses for it).
 * stats: [0] valid tokens, [1] tokens clipped (TIS) or masked (MIS),
 *        [2] sum of w, [3] sum of d over valid tokens (fp64).             */
/* ------------------------------------------------------------------ */
int oracle_rollout_is(const float* lt, const float* lr, const uint8_t* mask, int64_t n,
                      float log_clip, int mode, double* w, double* stats) {
    if (n < 0 || (mode != 0 && mode != 1)) return -1;
    double nv = 0, nc = 0, sw = 0, sd = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (!mask[i]) { w[i] = 0.0; continue; }
        float d = lt[i] - lr[i];
        int clipped = d > log_clip;
        double wi;
        if (mode == 0) wi = exp((double)(clipped ? log_clip : d));
        else wi = clipped ? 0.0 : exp((double)d);
        w[i] = wi;
        nv += 1; nc += clipped; sw += wi; sd += (double)d;
    }
    stats[0] = nv; stats[1] = nc; stats[2] = sw; stats[3] = sd;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Train-inference mismatch of a quantized rollout (FlashRL write-up,
 * Fig. 2, right: the KL divergence between the trainer's policy and the
 * rollout engine's policy, larger for INT8 rollouts than for FP8 ones).
 * The pages do not give the estimator; this oracle takes the full-vocabulary
 * KL of the two next-token distributions, per token row m:
 *   p = softmax(P[m][:]), q = softmax(Q[m][:]),
 *   kl[m] = sum_v p_v (log p_v - log q_v),
 * P being the higher-precision policy's logits and Q the quantized one's,
 * both bf16 [M][ld].  Plain fp64 log-softmax (max-shifted log-sum-exp).   */
/* ------------------------------------------------------------------ */
static double log_sum_exp_row(const uint16_t* r, int64_t V, double* mx_out) {
    double mx = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double x = (double)oracle_bf16_to_f32(r[v]);
        if (x > mx) mx = x;
    }
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) s += exp((double)oracle_bf16_to_f32(r[v]) - mx);
    *mx_out = mx;
    return mx + log(s);
}

int oracle_logits_kl(const uint16_t* P, int64_t ldp, const uint16_t* Q, int64_t ldq, int64_t M, int64_t V,
                     double* kl) {
    if (M < 0 || V < 1 || ldp < V || ldq < V) return -1;
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* a = P + m * ldp;
        const uint16_t* b = Q + m * ldq;
        double ma, mb;
        double za = log_sum_exp_row(a, V, &ma);
        double zb = log_sum_exp_row(b, V, &mb);
        double acc = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            double lp = (double)oracle_bf16_to_f32(a[v]) - za;
            double lq = (double)oracle_bf16_to_f32(b[v]) - zb;
            acc += exp(lp) * (lp - lq);
        }
        kl[m] = acc;
    }
    return 0;
}
