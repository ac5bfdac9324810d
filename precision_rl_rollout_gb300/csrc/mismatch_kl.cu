// mismatch_kl.cu -- train-inference mismatch of a quantized rollout: the KL
// divergence between the next-token distributions of the higher-precision
// policy and the 8-bit rollout policy (FlashRL write-up, Fig. 2, right: the KL
// between the trainer's and the rollout engine's policies, larger for INT8
// rollouts than for FP8 ones).  Per token row m, with P the higher-precision
// logits and Q the quantized ones (bf16 [M][V]):
//   p = softmax(P[m]), q = softmax(Q[m]),  kl[m] = sum_v p_v (log p_v - log q_v).
//
// Evaluation.  With d_v = P - Q and any constant c (the softmax ignores
// constant shifts), kl = E_p[d - c] + log E_p[exp(-(d - c))]; for nearby
// policies both terms are large next to their sum.  Each row is cut into
// chunks of 4096 logits, staged in shared memory and read twice: first for the
// chunk's largest logit m_j and its position (the centre c_j = d there, so
// every weight w_v = exp(P_v - m_j) <= 1 and the chunk's own distribution puts
// weight >= 1/S_j on x = 0), then for five fp32 sums over x = d - c_j:
//   S = sum w, X = sum w x, F = sum w f(x), U = sum w expm1(-x), G = sum w exp(-x),
// with f(x) = x + expm1(-x) >= 0 (its Taylor series for |x| < 1/16, so no
// cancellation).  Per chunk, r_j = log E[exp(-x)] + E[x] >= 0 is taken as
// F/S + (log1p(U/S) - U/S) when |U/S| < 1/2 -- the bracket from its Taylor
// series, which has no cancellation -- and as X/S + log(G/S) otherwise, and
// z_j = X/S + c_j - r_j is kept in fp64 (only differences of z_j are used
// later).  A second launch (one warp per row) combines the chunks of a row with
// pi_j = S_j exp(m_j - m) / S, m the row's largest logit, in a fixed reduction
// order (deterministic):
//   kl = sum_j pi_j r_j + log1p( sum_j pi_j expm1(-(z_j - zbar)) ),  zbar = sum_j pi_j z_j.
// Every cancellation is in these forms; the terms left (exp of a non-positive
// argument, expm1 of a small one, log1p of a non-negative sum) are evaluated in
// fp32 to ~1e-7 relative error and accumulated in fp64.  (fp64 transcendental
// functions run at a small fraction of the fp32 rate on this GPU; evaluated
// per chunk they took a third of the call.)
//
// The first launch works on pairs of logits with packed fp32 instructions
// (add/mul/fma.rn.f32x2: each lane rounds as the scalar instruction would) and
// 16-byte shared-memory loads; the exponentials are ex2.approx of the argument
// times log2(e) (a few 1e-7 relative error, far inside the result's 1e-4
// bound; x = 0 still gives exact zeros).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace fp8rl {

namespace {

constexpr int kKlThreads = 128;
constexpr int64_t kKlChunk = 4096;                               // logits per CTA (16 KB of P and Q in smem)
constexpr int kKlGroups = (int)(kKlChunk / 8 / kKlThreads);      // groups of 8 logits per thread
constexpr uint16_t kKlPad = 0xFF7Fu;   // the most negative finite bf16: weight 0, every term finite

struct KlPartial {
    double r, z;       // the chunk's Jensen gap and centred mean (see above)
    float m, S;        // its largest logit and sum of weights
    float pad[2];
};

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// packed fp32 pairs (low lane first)
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 up2(uint64_t v) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ uint64_t ex2_2(uint64_t v) {
    const float2 f = up2(v);
    return pk2(ex2_approx(f.x), ex2_approx(f.y));
}
// a word's two bf16 -> two fp32 (exact)
__device__ __forceinline__ uint64_t bf16x2_f32x2(uint32_t w) {
    return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// log(1 + u) - u for |u| < 1/2 from its Taylor series sum_{k>=2} (-1)^(k+1) u^k / k,
// 24 terms in Horner form: the remainder is below 1e-8 of the result at
// |u| = 1/2 (and far smaller for smaller |u|), and nothing cancels.
__device__ __forceinline__ float log1p_minus_u(float u) {
    float t = 1.f / 25.f;
#pragma unroll
    for (int k = 24; k >= 2; --k) t = fmaf(u, t, (k & 1) ? 1.f / (float)k : -1.f / (float)k);
    return u * u * t;
}

__global__ void __launch_bounds__(kKlThreads)
kl_partial_kernel(const uint16_t* __restrict__ P, int64_t ldp, const uint16_t* __restrict__ Q, int64_t ldq,
                  int64_t V, int chunks, KlPartial* __restrict__ part) {
    __shared__ __align__(16) uint16_t sp[kKlChunk];
    __shared__ __align__(16) uint16_t sq[kKlChunk];
    __shared__ float wm[kKlThreads / 32];
    __shared__ int wi[kKlThreads / 32];
    __shared__ float wsum[5][kKlThreads / 32];
    pdl_wait_then_release();
    const int64_t row = blockIdx.y;
    const int64_t v0 = (int64_t)blockIdx.x * kKlChunk;
    const int n = (int)(V - v0 < kKlChunk ? V - v0 : kKlChunk);   // logits in this chunk (>= 1)
    const int ng = (n + 7) / 8;                                     // groups of 8 holding logits
    const uint16_t* __restrict__ a = P + row * ldp + v0;
    const uint16_t* __restrict__ b = Q + row * ldq + v0;
    // stage the chunk (16-byte loads, all in flight together); a group the
    // chunk ends inside is padded
#pragma unroll
    for (int k = 0; k < kKlGroups; ++k) {
        const int g = k * kKlThreads + threadIdx.x;
        if (g * 8 + 8 <= n) {
            *reinterpret_cast<uint4*>(sp + g * 8) = ld_stream_v4(a + g * 8);
            *reinterpret_cast<uint4*>(sq + g * 8) = ld_stream_v4(b + g * 8);
        } else if (g < ng) {
            for (int e = g * 8; e < g * 8 + 8; ++e) {
                sp[e] = e < n ? a[e] : kKlPad;
                sq[e] = e < n ? b[e] : kKlPad;
            }
        }
    }
    __syncthreads();
    // pass 1: the chunk's largest logit (packed bf16 maxima), then the first
    // position holding it (only threads that hold it look)
    uint32_t mw = 0xFF80FF80u;                                      // -inf, -inf
#pragma unroll
    for (int k = 0; k < kKlGroups; ++k) {
        const int g = k * kKlThreads + threadIdx.x;
        if (g < ng) {
            const uint4 v = *reinterpret_cast<const uint4*>(sp + g * 8);
            mw = bf16x2_max(mw, bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w)));
        }
    }
    float mx = fmaxf(__uint_as_float(mw << 16), __uint_as_float(mw & 0xFFFF0000u));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (l == 0) wm[w] = mx;
    __syncthreads();
    mx = wm[0];
#pragma unroll
    for (int k = 1; k < kKlThreads / 32; ++k) mx = fmaxf(mx, wm[k]);
    int ix = 0x7fffffff;
    for (int k = 0; k < kKlGroups && ix == 0x7fffffff; ++k) {
        const int g = k * kKlThreads + threadIdx.x;
        if (g < ng)
            for (int e = g * 8; e < g * 8 + 8; ++e)
                if (bf16f(sp[e]) == mx) {
                    ix = e;
                    break;
                }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ix = min(ix, __shfl_xor_sync(0xffffffffu, ix, off));
    if (l == 0) wi[w] = ix;
    __syncthreads();
    ix = wi[0];
#pragma unroll
    for (int k = 1; k < kKlThreads / 32; ++k) ix = min(ix, wi[k]);
    const float c = bf16f(sp[ix]) - bf16f(sq[ix]);
    // pass 2: the five weighted sums, two logits per instruction
    constexpr float kLog2e = 1.4426950408889634f;
    const uint64_t kL = pk2(kLog2e, kLog2e), kNegL = pk2(-kLog2e, -kLog2e);
    const uint64_t kMxL = pk2(-mx * kLog2e, -mx * kLog2e), kNegC = pk2(-c, -c), kNeg1 = pk2(-1.f, -1.f);
    const uint64_t k720 = pk2(1.f / 720.f, 1.f / 720.f), k120 = pk2(1.f / 120.f, 1.f / 120.f);
    const uint64_t k24 = pk2(1.f / 24.f, 1.f / 24.f), k6 = pk2(1.f / 6.f, 1.f / 6.f), kHalf = pk2(0.5f, 0.5f);
    uint64_t S = 0, X = 0, F = 0, U = 0, G = 0;                     // (+0, +0) pairs
#pragma unroll
    for (int k = 0; k < kKlGroups; ++k) {
        const int g = k * kKlThreads + threadIdx.x;
        if (g < ng) {
            const uint4 pv4 = *reinterpret_cast<const uint4*>(sp + g * 8);
            const uint4 qv4 = *reinterpret_cast<const uint4*>(sq + g * 8);
            const uint32_t pw[4] = {pv4.x, pv4.y, pv4.z, pv4.w}, qw[4] = {qv4.x, qv4.y, qv4.z, qv4.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint64_t pv = bf16x2_f32x2(pw[j]);
                const uint64_t x = add2(fma2(bf16x2_f32x2(qw[j]), kNeg1, pv), kNegC);   // (P - Q) - c
                const uint64_t wv = ex2_2(fma2(pv, kL, kMxL));                          // exp(P - mx)
                const uint64_t ex = ex2_2(mul2(x, kNegL));                              // exp(-x)
                // expm1(-x) and x + expm1(-x): their Taylor series where |x| < 1/16
                // (terms past x^6 are below 1e-9 of the result), else directly
                const uint64_t nx = mul2(x, kNeg1);
                uint64_t t = fma2(nx, k720, k120);
                t = fma2(nx, t, k24);
                t = fma2(nx, t, k6);
                t = fma2(nx, t, kHalf);
                const uint64_t xx = mul2(x, x);
                const float2 fT = up2(mul2(xx, t)), uT = up2(fma2(xx, t, nx));
                const uint64_t uDp = add2(ex, kNeg1);
                const float2 uD = up2(uDp), fD = up2(add2(x, uDp)), xf = up2(x);
                const bool s0 = fabsf(xf.x) < 0.0625f, s1 = fabsf(xf.y) < 0.0625f;
                const uint64_t f = pk2(s0 ? fT.x : fD.x, s1 ? fT.y : fD.y);
                const uint64_t u = pk2(s0 ? uT.x : uD.x, s1 ? uT.y : uD.y);
                S = add2(S, wv);
                X = fma2(wv, x, X);
                F = fma2(wv, f, F);
                U = fma2(wv, u, U);
                G = fma2(wv, ex, G);
            }
        }
    }
    float t5[5];
    const uint64_t acc[5] = {S, X, F, U, G};
#pragma unroll
    for (int q = 0; q < 5; ++q) {
        const float2 v = up2(acc[q]);
        t5[q] = v.x + v.y;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t5[q] += __shfl_xor_sync(0xffffffffu, t5[q], off);
        if (l == 0) wsum[q][w] = t5[q];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float r[5];
        for (int q = 0; q < 5; ++q) {
            r[q] = 0.f;
            for (int k = 0; k < kKlThreads / 32; ++k) r[q] += wsum[q][k];   // fixed order
        }
        const float Sj = r[0], xb = r[1] / Sj, u = r[3] / Sj;
        const float rj = fabsf(u) < 0.5f ? r[2] / Sj + log1p_minus_u(u) : xb + logf(r[4] / Sj);
        part[row * chunks + blockIdx.x] =
            KlPartial{(double)rj, (double)xb + (double)c - (double)rj, mx, r[0], {0.f, 0.f}};
    }
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// One warp per row (one row per CTA, so that the rows spread over the SMs):
// lane l takes chunks l, l+32, ...; fixed shuffle trees.  Each chunk's weight
// S_j exp(m_j - m) is computed once for up to kKlCached chunks per lane (again
// in each sum beyond that).
constexpr int kKlCached = 4;

__global__ void __launch_bounds__(32)
kl_combine_kernel(const KlPartial* __restrict__ part, int chunks, float* __restrict__ kl) {
    pdl_wait_then_release();
    const int64_t row = blockIdx.x;
    const int lane = threadIdx.x;
    const KlPartial* r = part + row * chunks;
    float m = -INFINITY;
    for (int j = lane; j < chunks; j += 32) m = fmaxf(m, r[j].m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    // exp of a non-positive argument (m_j <= m): no overflow, ~1e-7 relative error
    auto weight = [&](int j) { return (double)(r[j].S * expf(r[j].m - m)); };
    double wj[kKlCached];
    double S = 0.0;
#pragma unroll
    for (int i = 0; i < kKlCached; ++i) {
        const int j = lane + 32 * i;
        wj[i] = j < chunks ? weight(j) : 0.0;
        S += wj[i];
    }
    for (int j = lane + 32 * kKlCached; j < chunks; j += 32) S += weight(j);
    S = warp_sum_d(S);
    const double inv_s = 1.0 / S;                      // one fp64 division per lane
    double sr = 0.0, zb = 0.0;
#pragma unroll
    for (int i = 0; i < kKlCached; ++i) {
        const int j = lane + 32 * i;
        if (j < chunks) {
            const double pi = wj[i] * inv_s;
            sr += pi * r[j].r;
            zb += pi * r[j].z;
        }
    }
    for (int j = lane + 32 * kKlCached; j < chunks; j += 32) {
        const double pi = weight(j) * inv_s;
        sr += pi * r[j].r;
        zb += pi * r[j].z;
    }
    sr = warp_sum_d(sr);
    zb = warp_sum_d(zb);
    // the centred differences in fp64, then expm1 of each in fp32
    double g = 0.0;
#pragma unroll
    for (int i = 0; i < kKlCached; ++i) {
        const int j = lane + 32 * i;
        if (j < chunks) g += wj[i] * inv_s * (double)expm1f((float)(zb - r[j].z));
    }
    for (int j = lane + 32 * kKlCached; j < chunks; j += 32)
        g += weight(j) * inv_s * (double)expm1f((float)(zb - r[j].z));
    g = warp_sum_d(g);
    if (lane == 0) kl[row] = (float)(sr + (double)log1pf((float)g));
}

}  // namespace

int kl_chunks(int64_t V) { return (int)((V + kKlChunk - 1) / kKlChunk); }
size_t kl_partial_bytes() { return sizeof(KlPartial); }

cudaError_t launch_logits_kl(const uint16_t* P, int64_t ldp, const uint16_t* Q, int64_t ldq, int64_t M,
                             int64_t V, float* kl, void* ws, cudaStream_t st) {
    const int chunks = kl_chunks(V);
    KlPartial* part = static_cast<KlPartial*>(ws);
    cudaError_t e = launch_pdl(kl_partial_kernel, dim3((unsigned)chunks, (unsigned)M), dim3(kKlThreads), 0, st, P,
                               ldp, Q, ldq, V, chunks, part);
    if (e != cudaSuccess) return e;
    return launch_pdl(kl_combine_kernel, dim3((unsigned)M), dim3(32), 0, st, (const KlPartial*)part, chunks, kl);
}

}  // namespace fp8rl
