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
// chunks of 8192 logits, staged in shared memory and read twice: first for the
// chunk's largest logit m_j and its position (the centre c_j = d there, so
// every weight w_v = exp(P_v - m_j) <= 1 and the chunk's own distribution puts
// weight >= 1/S_j on x = 0), then for five fp32 sums over x = d - c_j:
//   S = sum w, X = sum w x, F = sum w f(x), U = sum w expm1(-x), G = sum w exp(-x),
// with f(x) = x + expm1(-x) >= 0 (its Taylor series for |x| < 1/16, so no
// cancellation).  Per chunk, in fp64, r_j = log E[exp(-x)] + E[x] >= 0 is taken
// as F/S + log1p(U/S) - U/S when |U/S| < 1/2 and as X/S + log(G/S) otherwise,
// and z_j = X/S + c_j - r_j.  A second launch (one warp per row) combines the
// chunks of a row in fp64 with pi_j = S_j exp(m_j - m) / S, m the row's
// largest logit, in a fixed reduction order (deterministic):
//   kl = sum_j pi_j r_j + log1p( sum_j pi_j expm1(-(z_j - zbar)) ),  zbar = sum_j pi_j z_j,
// which is the same quantity with every cancellation left to fp64.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace fp8rl {

namespace {

constexpr int kKlThreads = 256;
constexpr int64_t kKlChunk = 8192;                          // logits per CTA (32 KB of P and Q in smem)
constexpr int kKlPer = (int)(kKlChunk / kKlThreads);        // 32 per thread

struct KlPartial {
    double r, z;       // the chunk's Jensen gap and centred mean (see above)
    float m, S;        // its largest logit and sum of weights
    float pad[2];
};

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

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
    const uint16_t* __restrict__ a = P + row * ldp + v0;
    const uint16_t* __restrict__ b = Q + row * ldq + v0;
    // stage the chunk: 16-byte loads where a whole 8-value group is inside it
    for (int g = threadIdx.x; g * 8 < n; g += kKlThreads) {
        if (g * 8 + 8 <= n) {
            *reinterpret_cast<uint4*>(sp + g * 8) = ld_stream_v4(a + g * 8);
            *reinterpret_cast<uint4*>(sq + g * 8) = ld_stream_v4(b + g * 8);
        } else {
            for (int e = g * 8; e < n; ++e) {
                sp[e] = a[e];
                sq[e] = b[e];
            }
        }
    }
    __syncthreads();
    // pass 1: the chunk's largest logit and its first position
    float mx = -INFINITY;
    int ix = 0x7fffffff;
    for (int k = 0; k < kKlPer; ++k) {
        const int e = k * kKlThreads + threadIdx.x;
        if (e < n) {
            const float v = bf16f(sp[e]);
            if (v > mx) { mx = v; ix = e; }          // e increases: the first maximum is kept
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, off);
        const int oi = __shfl_xor_sync(0xffffffffu, ix, off);
        if (om > mx || (om == mx && oi < ix)) { mx = om; ix = oi; }
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { wm[w] = mx; wi[w] = ix; }
    __syncthreads();
    mx = wm[0];
    ix = wi[0];
    for (int k = 1; k < kKlThreads / 32; ++k)
        if (wm[k] > mx || (wm[k] == mx && wi[k] < ix)) { mx = wm[k]; ix = wi[k]; }
    const float c = bf16f(sp[ix]) - bf16f(sq[ix]);
    // pass 2: the five weighted sums
    float S = 0.f, X = 0.f, F = 0.f, U = 0.f, G = 0.f;
    for (int k = 0; k < kKlPer; ++k) {
        const int e = k * kKlThreads + threadIdx.x;
        if (e < n) {
            const float pv = bf16f(sp[e]);
            // the fast exponential (a few 1e-7 relative error, far inside the
            // result's 1e-4 bound; x = 0 still gives exact zeros below)
            const float wv = __expf(pv - mx);
            const float x = (pv - bf16f(sq[e])) - c;
            const float ex = __expf(-x);
            float u, f;
            if (fabsf(x) < 0.0625f) {
                // expm1(-x) and x + expm1(-x) by their Taylor series (terms past x^6
                // are below 1e-9 of the result)
                float t = fmaf(-x, 1.f / 720.f, 1.f / 120.f);
                t = fmaf(-x, t, 1.f / 24.f);
                t = fmaf(-x, t, 1.f / 6.f);
                t = fmaf(-x, t, 0.5f);
                f = x * x * t;
                u = fmaf(x * x, t, -x);
            } else {
                u = ex - 1.f;                              // |u| >= 0.06: no cancellation
                f = x + u;
            }
            S += wv;
            X = fmaf(wv, x, X);
            F = fmaf(wv, f, F);
            U = fmaf(wv, u, U);
            G = fmaf(wv, ex, G);
        }
    }
    float t[5] = {S, X, F, U, G};
#pragma unroll
    for (int q = 0; q < 5; ++q) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t[q] += __shfl_xor_sync(0xffffffffu, t[q], off);
        if (l == 0) wsum[q][w] = t[q];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float r[5];
        for (int q = 0; q < 5; ++q) {
            r[q] = 0.f;
            for (int k = 0; k < kKlThreads / 32; ++k) r[q] += wsum[q][k];   // fixed order
        }
        const double Sj = r[0], xb = r[1] / Sj, u = r[3] / Sj;
        const double rj = fabs(u) < 0.5 ? r[2] / Sj + (log1p(u) - u) : xb + log(r[4] / Sj);
        part[row * chunks + blockIdx.x] = KlPartial{rj, xb + (double)c - rj, mx, r[0], {0.f, 0.f}};
    }
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// One warp per row: lane l takes chunks l, l+32, ...; fixed shuffle trees.
__global__ void __launch_bounds__(128)
kl_combine_kernel(const KlPartial* __restrict__ part, int64_t M, int chunks, float* __restrict__ kl) {
    pdl_wait_then_release();
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= M) return;                                 // whole warps only
    const KlPartial* r = part + row * chunks;
    float mf = -INFINITY;
    for (int j = lane; j < chunks; j += 32) mf = fmaxf(mf, r[j].m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mf = fmaxf(mf, __shfl_xor_sync(0xffffffffu, mf, off));
    const double m = mf;
    double S = 0.0;
    for (int j = lane; j < chunks; j += 32) S += (double)r[j].S * exp((double)r[j].m - m);
    S = warp_sum_d(S);
    double sr = 0.0, zb = 0.0;
    for (int j = lane; j < chunks; j += 32) {
        const double pi = (double)r[j].S * exp((double)r[j].m - m) / S;
        sr += pi * r[j].r;
        zb += pi * r[j].z;
    }
    sr = warp_sum_d(sr);
    zb = warp_sum_d(zb);
    double g = 0.0;
    for (int j = lane; j < chunks; j += 32) {
        const double pi = (double)r[j].S * exp((double)r[j].m - m) / S;
        g += pi * expm1(-(r[j].z - zb));
    }
    g = warp_sum_d(g);
    if (lane == 0) kl[row] = (float)(sr + log1p(g));
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
    return launch_pdl(kl_combine_kernel, dim3((unsigned)((M + 3) / 4)), dim3(128), 0, st,
                      (const KlPartial*)part, M, chunks, kl);
}

}  // namespace fp8rl
