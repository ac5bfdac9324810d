// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "internal.h"

namespace fp8rl {

// 16-byte streaming load that bypasses L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// bf16 pair packed in a 32-bit word -> the two fp32 values (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Running per-lane maximum of |bf16| as 16-bit integers: for finite values the
// magnitude bits order like the magnitudes, so integer max == |x| max.
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) {
    return __vmaxu2(acc, w & 0x7FFF7FFFu);
}
__device__ __forceinline__ uint32_t absmax_v4(uint32_t acc, uint4 v) {
    acc = absmax2(acc, v.x);
    acc = absmax2(acc, v.y);
    acc = absmax2(acc, v.z);
    return absmax2(acc, v.w);
}
// Fold the two 16-bit lanes and widen to an fp32 value.
__device__ __forceinline__ float absmax_fold(uint32_t acc) {
    uint32_t m = max(acc & 0xFFFFu, acc >> 16);
    return __uint_as_float(m << 16);
}

// Two fp32 values -> two E4M3FN codes (round to nearest even, saturate to
// +-448), first argument in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// Division of a block's values by its scale s.
//
// The quantizers need the IEEE round-to-nearest quotient fl32(x / s) only up to
// the code it rounds to.  With one scale per block, the reciprocal y = RN(1/s)
// is computed once and each quotient is refined from it with Markstein's
// correction (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
//     q0 = RN(|x| * y),  r = RN(|x| - q0 * s)  (fused, exact),  q = RN(q0 + r * y),
// then the sign of x is put back (so -0 and negative values that round to zero
// keep their sign, as the IEEE quotient does).  For every bf16 x with
// |x| <= amax and every bf16 amax whose scale s is at least 2^-90 (both
// families, s = amax/448 and s = amax/127), this gives the same E4M3 code and
// the same INT8 code as the IEEE quotient; the exhaustive-domain parity tests
// check exactly that against the CPU reference.  A block with a smaller scale
// (all |x| < ~2^-81) uses the IEEE division directly.
struct BlockDivisor {
    float s, y;
    bool fast;
};

__device__ __forceinline__ BlockDivisor make_divisor(float s) {
    return BlockDivisor{s, __frcp_rn(s), s >= 0x1p-90f};
}

template <bool kFast>
__device__ __forceinline__ float div_by_scale(float x, const BlockDivisor& d) {
    if constexpr (!kFast) {
        return __fdiv_rn(x, d.s);
    } else {
        const float a = fabsf(x);
        const float q0 = __fmul_rn(a, d.y);
        const float r = __fmaf_rn(-q0, d.s, a);
        const float q = __fmaf_rn(r, d.y, q0);
        return __uint_as_float(__float_as_uint(q) | (__float_as_uint(x) & 0x80000000u));
    }
}

// The two bf16 values of one 32-bit word (low half first) divided by the block
// scale exactly as div_by_scale<true> divides each, both at once: mul.rn.f32x2
// and fma.rn.f32x2 round each lane as the scalar instructions do, so the
// quotients are the same bits (the residual is formed as RN(|x| + q0 * (-s)),
// which equals RN(|x| - q0 * s)).  Three packed instructions instead of six.
__device__ __forceinline__ float2 div2_by_scale_fast(uint32_t w, const BlockDivisor& d) {
    const uint32_t lo = w << 16, hi = w & 0xFFFF0000u;      // the two values as fp32 bits
    uint64_t a, y2, ns2, q0, r, q;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "r"(lo & 0x7FFFFFFFu), "r"(hi & 0x7FFFFFFFu));
    asm("mov.b64 %0, {%1, %1};" : "=l"(y2) : "f"(d.y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(ns2) : "f"(-d.s));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(a), "l"(y2));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q0), "l"(ns2), "l"(a));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(r), "l"(y2), "l"(q0));
    uint32_t qlo, qhi;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(qlo), "=r"(qhi) : "l"(q));
    return make_float2(__uint_as_float(qlo | (lo & 0x80000000u)), __uint_as_float(qhi | (hi & 0x80000000u)));
}

// Eight bf16 (one 16-byte chunk) divided by the block scale and encoded to
// eight E4M3FN codes, packed little-endian into 8 bytes.
template <bool kFast>
__device__ __forceinline__ uint2 quant8_e4m3_t(uint4 v, const BlockDivisor& d) {
    uint2 o;
    if constexpr (kFast) {
        const float2 a = div2_by_scale_fast(v.x, d), b = div2_by_scale_fast(v.y, d);
        const float2 c = div2_by_scale_fast(v.z, d), e = div2_by_scale_fast(v.w, d);
        o.x = e4m3x2(a.x, a.y) | (e4m3x2(b.x, b.y) << 16);
        o.y = e4m3x2(c.x, c.y) | (e4m3x2(e.x, e.y) << 16);
    } else {
        o.x = e4m3x2(div_by_scale<false>(bf16_lo(v.x), d), div_by_scale<false>(bf16_hi(v.x), d)) |
              (e4m3x2(div_by_scale<false>(bf16_lo(v.y), d), div_by_scale<false>(bf16_hi(v.y), d)) << 16);
        o.y = e4m3x2(div_by_scale<false>(bf16_lo(v.z), d), div_by_scale<false>(bf16_hi(v.z), d)) |
              (e4m3x2(div_by_scale<false>(bf16_lo(v.w), d), div_by_scale<false>(bf16_hi(v.w), d)) << 16);
    }
    return o;
}

__device__ __forceinline__ float fp8_scale_from_amax(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}
__device__ __forceinline__ float int8_scale_from_amax(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 127.0f);
}

// One quotient -> int8 code: clamp(rint(q), -127, 127).
__device__ __forceinline__ uint32_t int8_code(float q) {
    int c = __float2int_rn(q);
    c = min(127, max(-127, c));
    return (uint32_t)(c & 0xFF);
}
// One bf16 -> int8 code: clamp(rint(x / s), -127, 127).
template <bool kFast>
__device__ __forceinline__ uint32_t q_int8(float x, const BlockDivisor& d) {
    return int8_code(div_by_scale<kFast>(x, d));
}
// A word's two bf16 -> two int8 codes (low value in the low byte).
template <bool kFast>
__device__ __forceinline__ uint32_t q_int8x2(uint32_t w, const BlockDivisor& d) {
    if constexpr (kFast) {
        const float2 q = div2_by_scale_fast(w, d);
        return int8_code(q.x) | (int8_code(q.y) << 8);
    } else {
        return q_int8<false>(bf16_lo(w), d) | (q_int8<false>(bf16_hi(w), d) << 8);
    }
}
template <bool kFast>
__device__ __forceinline__ uint2 quant8_int8_t(uint4 v, const BlockDivisor& d) {
    uint2 o;
    o.x = q_int8x2<kFast>(v.x, d) | (q_int8x2<kFast>(v.y, d) << 16);
    o.y = q_int8x2<kFast>(v.z, d) | (q_int8x2<kFast>(v.w, d) << 16);
    return o;
}

// fp32 -> bf16 bits, round to nearest even (the CUDA intrinsic).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return (uint32_t)(*reinterpret_cast<unsigned short*>(&h));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
}

// ---------------------------------------------------------------- launches

// Kernel launch with programmatic stream serialization: the kernel may be
// scheduled while the previous kernel in the stream is still running, and must
// call pdl_wait() before it reads or writes memory that kernel may touch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Wait for the previous kernel of the stream (see launch_pdl), then let the
// next one be scheduled.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// For short kernels whose successor reads inputs of its own first (the GEMM
// after the activation quantizer streams its weights): let the next kernel be
// scheduled at once, then wait for the previous one.  The successor still
// waits for this kernel's completion before it reads what this kernel writes,
// and this kernel completes only after its own wait, so the ordering of the
// stream is kept.
__device__ __forceinline__ void pdl_release_then_wait() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace fp8rl
