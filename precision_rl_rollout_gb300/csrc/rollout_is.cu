// rollout_is.cu -- token-level importance-sampling correction of 8-bit rollouts
// (FP8-RL, Abstract, contribution (iii): token-level TIS/MIS; FlashRL write-up,
// section on truncated importance sampling).
//
// The rollout samples tokens from the 8-bit policy while the gradient is taken
// under the trainer's higher-precision policy; each sampled token gets the
// importance weight of the two.  With d = fl32(logp_train - logp_rollout) and a
// threshold C passed as log_clip = ln C:
//   truncated (TIS): w = exp(min(d, log_clip));
//   masked    (MIS): w = d > log_clip ? 0 : exp(d);
// padding tokens (mask 0) get w = 0.  The clip decision is an fp32 comparison,
// so the clipped/masked count is exact; the weights use the CUDA expf.
// Two launches: every CTA of a persistent grid writes the weights of its token
// range and one partial record (valid, clipped, sum w, sum d; fp32 sums inside
// the CTA); one CTA then adds the records in fp64 in a fixed order
// (deterministic statistics for a given GPU).
#include "common.cuh"
#include "internal.h"

namespace fp8rl {

namespace {

constexpr int kIsThreads = 256;
constexpr int kIsPerThread = 16;
constexpr int64_t kIsPerCta = kIsThreads * kIsPerThread;   // 4096 tokens

struct IsPartial {
    double valid, clipped, sum_w, sum_d;
};

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float is_weight(float d, float log_clip, int mode, bool& clipped) {
    clipped = d > log_clip;
    return mode == 0 ? expf(clipped ? log_clip : d) : (clipped ? 0.f : expf(d));
}

// A persistent grid (a few CTAs per SM): CTA c owns the contiguous token range
// [c*per, (c+1)*per), per a multiple of 4096, so every CTA streams the same
// amount and there is no tail wave.  Within the range a thread takes 16
// tokens per step: four groups of four consecutive tokens (16-byte loads of
// both log-prob arrays and a 4-byte load of the mask, all issued before any is
// used).  Ranges that are not whole 4096-token steps, or unaligned pointers,
// take the scalar path.
template <bool kVec>
__global__ void __launch_bounds__(kIsThreads)
rollout_is_kernel(const float* __restrict__ lt, const float* __restrict__ lr,
                  const uint8_t* __restrict__ mask, int64_t n, int64_t per, float log_clip, int mode,
                  float* __restrict__ w, IsPartial* __restrict__ part) {
    pdl_wait_then_release();
    const int64_t r0 = (int64_t)blockIdx.x * per;
    const int64_t r1 = r0 + per < n ? r0 + per : n;
    int nv = 0, nc = 0;
    float sw = 0.f, sd = 0.f;
    for (int64_t base = r0; base < r1; base += kIsPerCta) {
        if (kVec && base + kIsPerCta <= r1) {
            float4 a[4], b[4];
            uint32_t mk[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int64_t i = base + (int64_t)(g * kIsThreads + threadIdx.x) * 4;
                a[g] = *reinterpret_cast<const float4*>(lt + i);
                b[g] = *reinterpret_cast<const float4*>(lr + i);
                mk[g] = mask ? *reinterpret_cast<const uint32_t*>(mask + i) : 0x01010101u;
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float x[4] = {a[g].x, a[g].y, a[g].z, a[g].w};
                const float y[4] = {b[g].x, b[g].y, b[g].z, b[g].w};
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    o[e] = 0.f;
                    if ((mk[g] >> (8 * e)) & 0xFFu) {
                        const float d = __fsub_rn(x[e], y[e]);
                        bool clipped;
                        o[e] = is_weight(d, log_clip, mode, clipped);
                        nv += 1;
                        nc += clipped;
                        sw += o[e];
                        sd += d;
                    }
                }
                const int64_t i = base + (int64_t)(g * kIsThreads + threadIdx.x) * 4;
                *reinterpret_cast<float4*>(w + i) = make_float4(o[0], o[1], o[2], o[3]);
            }
        } else {
            for (int j = 0; j < kIsPerThread; ++j) {
                const int64_t i = base + j * kIsThreads + threadIdx.x;
                if (i >= r1) break;
                float wi = 0.f;
                if (mask == nullptr || mask[i] != 0) {
                    const float d = __fsub_rn(lt[i], lr[i]);
                    bool clipped;
                    wi = is_weight(d, log_clip, mode, clipped);
                    nv += 1;
                    nc += clipped;
                    sw += wi;
                    sd += d;
                }
                w[i] = wi;
            }
        }
    }
    // In-CTA reduction in fp32 (counts exactly, as integers): fp64 arithmetic is
    // a small fraction of the fp32 rate on this GPU.  Only the per-CTA record is
    // widened to fp64.
    nv = __reduce_add_sync(0xffffffffu, nv);
    nc = __reduce_add_sync(0xffffffffu, nc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        sw += __shfl_xor_sync(0xffffffffu, sw, off);
        sd += __shfl_xor_sync(0xffffffffu, sd, off);
    }
    __shared__ int ired[kIsThreads / 32][2];
    __shared__ float fred[kIsThreads / 32][2];
    const int wid = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        ired[wid][0] = nv; ired[wid][1] = nc;
        fred[wid][0] = sw; fred[wid][1] = sd;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int a = 0, b = 0;
        float c = 0.f, e = 0.f;
        for (int k = 0; k < kIsThreads / 32; ++k) {
            a += ired[k][0]; b += ired[k][1]; c += fred[k][0]; e += fred[k][1];
        }
        part[blockIdx.x] = IsPartial{(double)a, (double)b, (double)c, (double)e};
    }
}

__global__ void __launch_bounds__(1024)
rollout_is_stats_kernel(const IsPartial* __restrict__ part, int64_t P, double* __restrict__ stats) {
    pdl_wait_then_release();
    double a[4] = {0.0, 0.0, 0.0, 0.0};
    for (int64_t p = threadIdx.x; p < P; p += 1024) {   // fixed assignment and order
        a[0] += part[p].valid;
        a[1] += part[p].clipped;
        a[2] += part[p].sum_w;
        a[3] += part[p].sum_d;
    }
    __shared__ double red[32][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) a[k] = warp_sum(a[k]);
    if ((threadIdx.x & 31) == 0)
        for (int k = 0; k < 4; ++k) red[threadIdx.x >> 5][k] = a[k];
    __syncthreads();
    if (threadIdx.x < 4) {
        double t = 0.0;
        for (int wv = 0; wv < 32; ++wv) t += red[wv][threadIdx.x];
        stats[threadIdx.x] = t;
    }
}

}  // namespace

// Partial records the workspace must hold: one per 4096 tokens at most (the
// grid never has more CTAs than that).
int64_t rollout_is_max_partials(int64_t n) { return (n + kIsPerCta - 1) / kIsPerCta; }

// CTAs of the persistent grid: up to 4 per SM, each with at least one 4096-token step.
int64_t rollout_is_partials(int64_t n) {
    const int64_t steps = (n + kIsPerCta - 1) / kIsPerCta;
    const int64_t cap = 4 * (int64_t)num_sms();
    return steps < cap ? steps : cap;
}
static int64_t rollout_is_per(int64_t n, int64_t ctas) {
    const int64_t steps = (n + kIsPerCta - 1) / kIsPerCta;
    return ((steps + ctas - 1) / ctas) * kIsPerCta;
}
size_t rollout_is_partial_bytes() { return sizeof(IsPartial); }

cudaError_t launch_rollout_is(const float* lt, const float* lr, const uint8_t* mask, int64_t n,
                              float log_clip, int mode, float* w, double* stats, void* ws,
                              cudaStream_t st) {
    const int64_t P = rollout_is_partials(n);
    if (P > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    IsPartial* part = static_cast<IsPartial*>(ws);
    cudaError_t e;
    if (P > 0) {
        const bool vec = ((reinterpret_cast<uintptr_t>(lt) | reinterpret_cast<uintptr_t>(lr) |
                           reinterpret_cast<uintptr_t>(w)) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(mask) & 3u) == 0;
        const int64_t per = rollout_is_per(n, P);
        e = vec ? launch_pdl(rollout_is_kernel<true>, dim3((unsigned)P), dim3(kIsThreads), 0, st, lt, lr,
                             mask, n, per, log_clip, mode, w, part)
                : launch_pdl(rollout_is_kernel<false>, dim3((unsigned)P), dim3(kIsThreads), 0, st, lt, lr,
                             mask, n, per, log_clip, mode, w, part);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(rollout_is_stats_kernel, dim3(1), dim3(1024), 0, st, (const IsPartial*)part, P,
                      stats);
}

}  // namespace fp8rl
