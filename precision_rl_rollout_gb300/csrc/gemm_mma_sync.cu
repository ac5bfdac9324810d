// gemm_mma_sync.cu -- warp-level mma.sync FP8 GEMM for the one case the tcgen05
// kernels do not take: fewer than 64 tokens with K beyond the decode kernel's
// split range (K > 32768).
//
// FP8 (FP8-RL, Abstract (i)): Y = sum over 128-wide K blocks of
//   Xs[kb][m] * Ws[nb][kb] * (Xq . Wq over the block),
// partial sums per block from m16n8k32 e4m3 MMAs in fp32, promoted into an
// fp32 accumulator with the block's scale product.
//
// CTA tile: 32 tokens x 128 output channels (one weight block row), 4 warps of
// 16 x 64.  Fragments are read straight from global memory (L1/L2 serve the
// reuse).
#include "common.cuh"
#include "internal.h"

namespace fp8rl {

__device__ __forceinline__ uint32_t ld32(const uint8_t* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}

__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment of m16n8k32 (8-bit): lane (g = lane/4, t = lane%4) holds rows g and
// g+8, columns 4t..4t+3 and 16+4t..16+4t+3 of the 16x32 tile.
__device__ __forceinline__ void load_a_frag(uint32_t (&a)[4], const uint8_t* r0, const uint8_t* r1,
                                            bool v0, bool v1, int64_t k) {
    a[0] = v0 ? ld32(r0 + k) : 0u;
    a[1] = v1 ? ld32(r1 + k) : 0u;
    a[2] = v0 ? ld32(r0 + k + 16) : 0u;
    a[3] = v1 ? ld32(r1 + k + 16) : 0u;
}

__global__ void __launch_bounds__(128)
gemm_fp8_mma_sync_kernel(const uint8_t* __restrict__ Xq, const float* __restrict__ Xs,
                         const uint8_t* __restrict__ Wq, const float* __restrict__ Ws,
                         int64_t M, int64_t N, int64_t K, uint16_t* __restrict__ Y, int64_t ldy) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int64_t nb = blockIdx.x;
    const int64_t n_base = nb * kBlk + (warp >> 1) * 64;
    const int64_t m0 = (int64_t)blockIdx.y * 32 + (warp & 1) * 16 + g, m1 = m0 + 8;
    const bool v0 = m0 < M, v1 = m1 < M;
    const uint8_t* x0 = Xq + (v0 ? m0 : 0) * K;
    const uint8_t* x1 = Xq + (v1 ? m1 : 0) * K;
    const int64_t KB = K / kBlk;

    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    for (int64_t kb = 0; kb < KB; ++kb) {
        float part[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) part[j][0] = part[j][1] = part[j][2] = part[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const int64_t k = kb * kBlk + ks * 32 + t4 * 4;
            uint32_t a[4];
            load_a_frag(a, x0, x1, v0, v1, k);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint8_t* w = Wq + (n_base + j * 8 + g) * K + k;
                mma_e4m3(part[j], a, ld32(w), ld32(w + 16));
            }
        }
        const float sw = Ws[nb * KB + kb];
        const float s0 = v0 ? Xs[kb * M + m0] * sw : 0.f;
        const float s1 = v1 ? Xs[kb * M + m1] * sw : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            acc[j][0] = fmaf(part[j][0], s0, acc[j][0]);
            acc[j][1] = fmaf(part[j][1], s0, acc[j][1]);
            acc[j][2] = fmaf(part[j][2], s1, acc[j][2]);
            acc[j][3] = fmaf(part[j][3], s1, acc[j][3]);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t n = n_base + j * 8 + t4 * 2;
        if (v0) *reinterpret_cast<uint32_t*>(Y + m0 * ldy + n) = pack_bf16x2(acc[j][0], acc[j][1]);
        if (v1) *reinterpret_cast<uint32_t*>(Y + m1 * ldy + n) = pack_bf16x2(acc[j][2], acc[j][3]);
    }
}

cudaError_t launch_gemm_fp8_mma_sync(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                     const float* Ws, int64_t M, int64_t N, int64_t K,
                                     uint16_t* Y, int64_t ldy, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    dim3 grid((unsigned)(N / kBlk), (unsigned)((M + 31) / 32));
    gemm_fp8_mma_sync_kernel<<<grid, 128, 0, st>>>(Xq, Xs, Wq, Ws, M, N, K, Y, ldy);
    return cudaGetLastError();
}

}  // namespace fp8rl
