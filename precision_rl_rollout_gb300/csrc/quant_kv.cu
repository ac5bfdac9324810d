// quant_kv.cu -- FP8 KV-cache quantization with a per-tensor scale recalibrated
// from the tensor itself (FP8-RL, Abstract, contribution (ii): FP8 KV-cache
// with per-step QKV scale recalibration).  One fp32 scale per K or V tensor,
// s = fl32(amax / 448) over the whole tensor (amax = 0 gives 1), recomputed at
// every call; codes as for the weights.
//
// The scale needs the whole tensor's amax before any code can be written, so
// the work is three launches (chained with programmatic dependent launch):
//   1. kv_amax_partial_kernel: every CTA reduces one slice of 2048 chunks
//      (16 K values) to its amax and writes it to partial[cta] (scratch);
//   2. kv_scale_kernel: one CTA reduces the partials and writes the scale;
//   3. kv_quant_kernel: every CTA reads the scale and encodes its slice.
// Deterministic (no atomics, nothing to zero).  Above L2 size the tensor is
// read twice (6.6 B of DRAM traffic per 3 algorithmic bytes); below it the
// second read comes from L2.
#include "common.cuh"
#include "internal.h"

namespace fp8rl {

namespace {

constexpr int kKvThreads = 256;
constexpr int kKvChunksPerThread = 8;
constexpr int64_t kKvChunksPerCta = kKvThreads * kKvChunksPerThread;   // 2048 chunks = 16384 values

// chunk c of a [R][C] tensor with row pitch ld: 8 values at row c / (C/8)
__device__ __forceinline__ int64_t chunk_offset(int64_t c, int64_t cpr, int64_t ld) {
    const int64_t r = c / cpr;
    return r * ld + (c - r * cpr) * 8;
}

__global__ void __launch_bounds__(kKvThreads)
kv_amax_partial_kernel(const uint16_t* __restrict__ X, int64_t total, int64_t cpr, int64_t ld,
                       uint32_t* __restrict__ partial) {
    pdl_wait_then_release();
    const int64_t base = (int64_t)blockIdx.x * kKvChunksPerCta;
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kKvChunksPerThread; ++i) {
        const int64_t c = base + i * kKvThreads + threadIdx.x;
        if (c < total) m = absmax_v4(m, ld_stream_v4(X + chunk_offset(c, cpr, ld)));
    }
    m = __reduce_max_sync(0xffffffffu, max(m & 0xFFFFu, m >> 16));
    __shared__ uint32_t red[kKvThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = red[0];
        for (int w = 1; w < kKvThreads / 32; ++w) r = max(r, red[w]);
        partial[blockIdx.x] = r;                          // bf16 magnitude bits of the slice's amax
    }
}

__global__ void __launch_bounds__(1024)
kv_scale_kernel(const uint32_t* __restrict__ partial, int64_t P, float* __restrict__ scale) {
    pdl_wait_then_release();
    uint32_t m = 0;
    for (int64_t i = threadIdx.x; i < P; i += 1024) m = max(m, partial[i]);
    m = __reduce_max_sync(0xffffffffu, m);
    __shared__ uint32_t red[32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = red[0];
        for (int w = 1; w < 32; ++w) r = max(r, red[w]);
        *scale = fp8_scale_from_amax(__uint_as_float(r << 16));
    }
}

__global__ void __launch_bounds__(kKvThreads)
kv_quant_kernel(const uint16_t* __restrict__ X, int64_t total, int64_t cpr, int64_t ld,
                const float* __restrict__ scale, uint8_t* __restrict__ Xq) {
    pdl_wait_then_release();
    const BlockDivisor d = make_divisor(*scale);
    const int64_t base = (int64_t)blockIdx.x * kKvChunksPerCta;
    uint4 v[kKvChunksPerThread];
#pragma unroll
    for (int i = 0; i < kKvChunksPerThread; ++i) {
        const int64_t c = base + i * kKvThreads + threadIdx.x;
        v[i] = c < total ? ld_stream_v4(X + chunk_offset(c, cpr, ld)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kKvChunksPerThread; ++i) {
        const int64_t c = base + i * kKvThreads + threadIdx.x;
        if (c < total)
            *reinterpret_cast<uint2*>(Xq + c * 8) = d.fast ? quant8_e4m3_t<true>(v[i], d)
                                                           : quant8_e4m3_t<false>(v[i], d);
    }
}

}  // namespace

int64_t kv_partials(int64_t R, int64_t C) {
    const int64_t total = R * (C / 8);
    return (total + kKvChunksPerCta - 1) / kKvChunksPerCta;
}

cudaError_t launch_quant_kv_with_scale(const uint16_t* X, int64_t R, int64_t C, int64_t ld,
                                       const float* scale, uint8_t* Xq, cudaStream_t st) {
    const int64_t total = R * (C / 8), P = kv_partials(R, C);
    if (total == 0) return cudaSuccess;
    if (P > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    return launch_pdl(kv_quant_kernel, dim3((unsigned)P), dim3(kKvThreads), 0, st, X, total, C / 8, ld,
                      scale, Xq);
}

cudaError_t launch_quant_kv_tensor(const uint16_t* X, int64_t R, int64_t C, int64_t ld, uint8_t* Xq,
                                   float* scale, uint32_t* partial, cudaStream_t st) {
    const int64_t total = R * (C / 8), P = kv_partials(R, C);
    if (P > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaError_t e;
    if (P > 0) {
        e = launch_pdl(kv_amax_partial_kernel, dim3((unsigned)P), dim3(kKvThreads), 0, st, X, total, C / 8,
                       ld, partial);
        if (e != cudaSuccess) return e;
    }
    e = launch_pdl(kv_scale_kernel, dim3(1), dim3(1024), 0, st, (const uint32_t*)partial, P, scale);
    if (e != cudaSuccess) return e;
    return launch_quant_kv_with_scale(X, R, C, ld, scale, Xq, st);
}

}  // namespace fp8rl
