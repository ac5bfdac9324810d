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
// Two launches: every CTA writes the weights of its 4096 tokens and one
// partial record (valid, clipped, sum w, sum d); one CTA then adds the records
// in a fixed order (deterministic statistics).
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

__global__ void __launch_bounds__(kIsThreads)
rollout_is_kernel(const float* __restrict__ lt, const float* __restrict__ lr,
                  const uint8_t* __restrict__ mask, int64_t n, float log_clip, int mode,
                  float* __restrict__ w, IsPartial* __restrict__ part) {
    pdl_wait_then_release();
    const int64_t base = (int64_t)blockIdx.x * kIsPerCta;
    int nv = 0, nc = 0;
    float sw = 0.f, sd = 0.f;
#pragma unroll 4
    for (int j = 0; j < kIsPerThread; ++j) {
        const int64_t i = base + j * kIsThreads + threadIdx.x;
        if (i >= n) break;
        const bool valid = mask == nullptr || mask[i] != 0;
        float wi = 0.f;
        if (valid) {
            const float d = __fsub_rn(lt[i], lr[i]);
            const bool clipped = d > log_clip;
            wi = mode == 0 ? expf(clipped ? log_clip : d) : (clipped ? 0.f : expf(d));
            nv += 1;
            nc += clipped;
            sw += wi;
            sd += d;
        }
        w[i] = wi;
    }
    double v0 = warp_sum((double)nv), v1 = warp_sum((double)nc), v2 = warp_sum((double)sw),
           v3 = warp_sum((double)sd);
    __shared__ double red[kIsThreads / 32][4];
    const int wid = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[wid][0] = v0; red[wid][1] = v1; red[wid][2] = v2; red[wid][3] = v3;
    }
    __syncthreads();
    if (threadIdx.x < 4) {
        double t = 0.0;
        for (int k = 0; k < kIsThreads / 32; ++k) t += red[k][threadIdx.x];
        reinterpret_cast<double*>(&part[blockIdx.x])[threadIdx.x] = t;
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

int64_t rollout_is_partials(int64_t n) { return (n + kIsPerCta - 1) / kIsPerCta; }
size_t rollout_is_partial_bytes() { return sizeof(IsPartial); }

cudaError_t launch_rollout_is(const float* lt, const float* lr, const uint8_t* mask, int64_t n,
                              float log_clip, int mode, float* w, double* stats, void* ws,
                              cudaStream_t st) {
    const int64_t P = rollout_is_partials(n);
    if (P > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    IsPartial* part = static_cast<IsPartial*>(ws);
    cudaError_t e;
    if (P > 0) {
        e = launch_pdl(rollout_is_kernel, dim3((unsigned)P), dim3(kIsThreads), 0, st, lt, lr, mask, n,
                       log_clip, mode, w, part);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(rollout_is_stats_kernel, dim3(1), dim3(1024), 0, st, (const IsPartial*)part, P,
                      stats);
}

}  // namespace fp8rl
