// quant.cu -- the HBM-bound quantizers of the 8-bit rollout path.
//
//  * FP8 weight requant, 128x128 blocks (FP8-RL, Abstract: weights change every
//    step and are quantized again; contribution (i): blockwise FP8).
//  * FP8 activation quant, 1x128 groups per token (the A8 of W8A8).
//  * INT8 per-row quant for weights (per output channel) and activations (per
//    token) (FlashRL write-up, Fig. 1: INT8 rollout).
//
// Every byte of input is read once with 16-byte streaming loads and every code
// written once; amax is an integer max over the bf16 magnitude bits followed by
// warp reductions; the quotient x / s yields the code of the IEEE round-to-
// nearest fp32 divide (see BlockDivisor in common.cuh) and the conversion is the
// hardware E4M3 convert with round-to-nearest-even and saturation, so every
// output bit is fixed by the input bits.
#include "common.cuh"
#include "internal.h"

namespace fp8rl {

// ---------------------------------------------------------------- FP8 weights

// One launch quantizes the 128x128 blocks of up to kMaxGroup tensors.  Block
// ids are numbered tensor by tensor; block_start[i] is the first block of
// tensor i and block_start[n] the total.
struct WeightGroupParams {
    int n;
    int64_t block_start[kMaxGroup + 1];
    const uint16_t* W[kMaxGroup];
    uint8_t* Wq[kMaxGroup];
    float* Ws[kMaxGroup];
    int64_t ldw[kMaxGroup];
    int64_t K[kMaxGroup];
};

// 256 threads per 128x128 block.  A block row is 256 B of bf16 = 16 chunks of
// 16 B; chunk c = i*256 + t (i = 0..7) lies in row c/16 at column 8*(c%16), so
// a warp reads two full 256-byte row segments per load.  Five CTAs per SM (48
// registers, no spills): the extra resident warps hide the block reduction and
// the encode of the other CTAs (108 -> 102 us on the Qwen2.5-7B layer set,
// against 50 registers and four CTAs per SM).
__global__ void __launch_bounds__(256, 5)
quant_weight_block_kernel(const __grid_constant__ WeightGroupParams p) {
    pdl_wait_then_release();
    const int64_t b = blockIdx.x;
    int lo = 0, hi = p.n - 1;                     // tensor that owns block b
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (p.block_start[mid] <= b) lo = mid; else hi = mid - 1;
    }
    const int ti = lo;
    const int64_t K = p.K[ti], ldw = p.ldw[ti];
    const int64_t KB = K / kBlk;
    const int64_t local = b - p.block_start[ti];
    const int64_t nb = local / KB, kb = local - nb * KB;

    const int t = threadIdx.x;
    const int r0 = t >> 4;                        // row within the block for i = 0
    const int col = (t & 15) * 8;                 // element column within the block
    const uint16_t* src = p.W[ti] + (nb * kBlk + r0) * ldw + kb * kBlk + col;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ld_stream_v4(src + (int64_t)i * 16 * ldw);

    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = absmax_v4(m, v[i]);
    m = __reduce_max_sync(0xffffffffu, max(m & 0xFFFFu, m >> 16));
    __shared__ uint32_t red[8];
    if ((t & 31) == 0) red[t >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = max(m, red[w]);
    const float s = fp8_scale_from_amax(__uint_as_float(m << 16));
    const BlockDivisor d = make_divisor(s);

    uint8_t* dst = p.Wq[ti] + (nb * kBlk + r0) * K + kb * kBlk + col;
    if (d.fast) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint2*>(dst + (int64_t)i * 16 * K) = quant8_e4m3_t<true>(v[i], d);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint2*>(dst + (int64_t)i * 16 * K) = quant8_e4m3_t<false>(v[i], d);
    }
    if (t == 0) p.Ws[ti][nb * KB + kb] = s;
}

cudaError_t launch_quant_weight_block(const WeightDesc* d, int n, cudaStream_t st) {
    for (int base = 0; base < n; base += kMaxGroup) {
        WeightGroupParams p;
        p.n = 0;
        int64_t total = 0;
        for (int i = base; i < n && p.n < kMaxGroup; ++i) {
            const int j = p.n++;
            p.block_start[j] = total;
            p.W[j] = d[i].W;
            p.Wq[j] = d[i].Wq;
            p.Ws[j] = d[i].Ws;
            p.ldw[j] = d[i].ldw;
            p.K[j] = d[i].K;
            total += (d[i].N / kBlk) * (d[i].K / kBlk);
        }
        p.block_start[p.n] = total;
        if (total == 0) continue;
        if (total > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
        cudaError_t e = launch_pdl(quant_weight_block_kernel, dim3((unsigned)total), dim3(256), 0, st, p);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// ---------------------------------------------------------------- FP8 activations

// 256 threads = 16 half-warps; half-warp h quantizes groups G*blockIdx.x ..
// G*blockIdx.x + G-1 of token m = 16*blockIdx.y + h: each of its 16 lanes
// holds one 16-byte chunk (8 values) of each 128-value group.  All G loads of
// a thread are issued before the first group is reduced, so a large tensor
// keeps enough bytes in flight to stream at HBM speed (G = 4: 40 registers,
// six CTAs per SM; measured faster than G = 2, 5 and 8 at every prefill size);
// a small one (decode) takes G = 1 for the most CTAs and the shortest chain.
template <int G>
__global__ void __launch_bounds__(256)
quant_act_group_kernel(const uint16_t* __restrict__ X, int64_t M, int64_t K, int64_t ldx,
                       uint8_t* __restrict__ Xq, float* __restrict__ Xs) {
    pdl_release_then_wait();
    const int t = threadIdx.x;
    const int lane16 = t & 15;
    const int64_t m = (int64_t)blockIdx.y * 16 + (t >> 4);
    const int64_t KG = K / kBlk;
    const int64_t g0 = (int64_t)blockIdx.x * G;
    const bool valid = m < M;
    uint4 v[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        v[j] = make_uint4(0, 0, 0, 0);
        if (valid && g0 + j < KG) v[j] = ld_stream_v4(X + m * ldx + (g0 + j) * kBlk + lane16 * 8);
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
        uint32_t a = absmax_v4(0u, v[j]);
        a = max(a & 0xFFFFu, a >> 16);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) a = max(a, __shfl_xor_sync(0xffffffffu, a, off));
        const float s = fp8_scale_from_amax(__uint_as_float(a << 16));
        const BlockDivisor d = make_divisor(s);
        if (valid && g0 + j < KG) {   // g0 + j < KG is the same for the whole CTA
            uint2 q = d.fast ? quant8_e4m3_t<true>(v[j], d) : quant8_e4m3_t<false>(v[j], d);
            *reinterpret_cast<uint2*>(Xq + m * K + (g0 + j) * kBlk + lane16 * 8) = q;
            if (lane16 == 0) Xs[(g0 + j) * M + m] = s;
        }
    }
}

cudaError_t launch_quant_act_group(const uint16_t* X, int64_t M, int64_t K, int64_t ldx,
                                   uint8_t* Xq, float* Xs, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    const int64_t KG = K / kBlk, MB = (M + 15) / 16;
    // four groups per thread once one group per thread would need more than
    // about eight full waves of CTAs (8 resident per SM)
    if (KG * MB >= 64LL * num_sms())
        return launch_pdl(quant_act_group_kernel<4>, dim3((unsigned)((KG + 3) / 4), (unsigned)MB), dim3(256), 0,
                          st, X, M, K, ldx, Xq, Xs);
    return launch_pdl(quant_act_group_kernel<1>, dim3((unsigned)KG, (unsigned)MB), dim3(256), 0, st, X, M, K,
                      ldx, Xq, Xs);
}

// ---------------------------------------------------------------- INT8 rows

// One CTA of NT threads per row; the row is held in registers between the
// amax pass and the quantization pass: chunk c = i*NT + t for i < CPT.  CPT
// (chunks of 8 values per thread) is the smallest instantiation that covers
// the row, so short rows keep few registers and many CTAs in flight.  Rows of
// up to 8192 values take 128-thread CTAs: twice the CTAs per SM, so twice the
// bytes in flight, and no half-empty last iteration on 5120-wide rows.
template <int CPT, int NT>
__global__ void __launch_bounds__(NT)
quant_int8_rows_kernel(const uint16_t* __restrict__ A, int64_t K, int64_t lda,
                       int8_t* __restrict__ Q, float* __restrict__ S) {
    pdl_wait_then_release();
    const int64_t r = blockIdx.x;
    const int t = threadIdx.x;
    const int chunks = (int)(K / 8);
    const uint16_t* src = A + r * lda;
    uint4 v[CPT];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = i * NT + t;
        v[i] = make_uint4(0, 0, 0, 0);
        if (c < chunks) v[i] = ld_stream_v4(src + (int64_t)c * 8);
        m = absmax_v4(m, v[i]);
    }
    m = __reduce_max_sync(0xffffffffu, max(m & 0xFFFFu, m >> 16));
    __shared__ uint32_t red[NT / 32];
    if ((t & 31) == 0) red[t >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w) m = max(m, red[w]);
    const float s = int8_scale_from_amax(__uint_as_float(m << 16));
    const BlockDivisor d = make_divisor(s);
    int8_t* dst = Q + r * K;
    if (d.fast) {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = i * NT + t;
            if (c < chunks) *reinterpret_cast<uint2*>(dst + (int64_t)c * 8) = quant8_int8_t<true>(v[i], d);
        }
    } else {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = i * NT + t;
            if (c < chunks) *reinterpret_cast<uint2*>(dst + (int64_t)c * 8) = quant8_int8_t<false>(v[i], d);
        }
    }
    if (t == 0) S[r] = s;
}

template <int CPT, int NT>
static cudaError_t launch_int8_rows_cpt(const uint16_t* A, int64_t R, int64_t K, int64_t lda, int8_t* Q,
                                        float* S, cudaStream_t st) {
    return launch_pdl(quant_int8_rows_kernel<CPT, NT>, dim3((unsigned)R), dim3(NT), 0, st, A, K, lda, Q, S);
}

cudaError_t launch_quant_int8_rows(const uint16_t* A, int64_t R, int64_t K, int64_t lda,
                                   int8_t* Q, float* S, cudaStream_t st) {
    if (R == 0) return cudaSuccess;
    if (R > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    const int64_t chunks = K / 8;
    if (chunks <= 128 * 8) {                            // rows of up to 8192 values: 128 threads
        const int64_t need = (chunks + 127) / 128;
        if (need <= 1) return launch_int8_rows_cpt<1, 128>(A, R, K, lda, Q, S, st);
        if (need <= 2) return launch_int8_rows_cpt<2, 128>(A, R, K, lda, Q, S, st);
        if (need <= 3) return launch_int8_rows_cpt<3, 128>(A, R, K, lda, Q, S, st);
        if (need <= 4) return launch_int8_rows_cpt<4, 128>(A, R, K, lda, Q, S, st);
        if (need <= 5) return launch_int8_rows_cpt<5, 128>(A, R, K, lda, Q, S, st);
        if (need <= 6) return launch_int8_rows_cpt<6, 128>(A, R, K, lda, Q, S, st);
        return launch_int8_rows_cpt<8, 128>(A, R, K, lda, Q, S, st);
    }
    const int64_t need = (chunks + 255) / 256;          // chunks per thread
    static_assert(kInt8MaxK / (256 * 8) == 16, "largest instantiation covers kInt8MaxK");
    if (need <= 6) return launch_int8_rows_cpt<6, 256>(A, R, K, lda, Q, S, st);
    if (need <= 8) return launch_int8_rows_cpt<8, 256>(A, R, K, lda, Q, S, st);
    if (need <= 12) return launch_int8_rows_cpt<12, 256>(A, R, K, lda, Q, S, st);
    return launch_int8_rows_cpt<16, 256>(A, R, K, lda, Q, S, st);
}

}  // namespace fp8rl
