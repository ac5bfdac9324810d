// gemm_int8_prefill.cu -- exact INT8 W8A8 GEMM for large token counts, on the
// fp16 tcgen05 path after one conversion pass.
//
// Math (FlashRL write-up, Fig. 1, INT8 rollout): acc[m][n] = sum_k Xq[m][k] Wq[n][k]
// exactly (int32), y = bf16_rn((float(acc) * Xs[m]) * Ws[n]), no FMA.
//
// With many tokens every weight tile meets every token tile, so converting the
// int8 codes to fp16 inside the GEMM (as the small-batch kernel does) would
// repeat the conversion once per tile pair and load shared memory with it.
// Here one launch first writes fp16 copies of X and W into the workspace (every
// int8 code is an exact fp16), and the GEMM runs a plain fp16 pipeline:
//  - persistent, one CTA per SM, 128 tokens x 256 weight rows per tile
//    (tcgen05.mma kind::f16, M=128 N=256 K=16), tiles M-fastest so the CTAs
//    in flight share weight slabs and the L2-resident activations;
//  - a stage holds one 64-wide K atom of both operands (16 + 32 KB, TMA with
//    the 128-byte swizzle); four stages;
//  - TMEM accumulates a group of 8 stages, 512 products per output:
//    |sum| <= 512 * 127^2 < 2^23, so every partial sum is an integer held
//    exactly in fp32 whatever the addition order; two 256-column buffers
//    alternate between groups;
//  - the epilogue converts each group's sums to int32 (exact) and adds them in
//    int32 registers; at the end of a tile it writes Y (bf16, TMA store) and,
//    if asked, the int32 accumulators;
//  - with fewer tiles than SMs (a few hundred tokens), a work unit is a tile's
//    K range; each unit writes its int32 partial tile to the workspace and a
//    second launch adds them (integers: exact in any order) and writes Y.
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {

using namespace sm100;

namespace {

constexpr int kBM = 128, kBN = 256;
constexpr int kStages = 4;
constexpr int kABytes = kBM * 128;                  // 128 tokens x 64 fp16
constexpr int kBBytes = kBN * 128;                  // 256 weight rows x 64 fp16
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kGroup = 8;                           // stages per exact TMEM group (8 x 64 = 512 K)
constexpr int kThreads = 384;
constexpr int kOutBytesPerWarp = 32 * 128;          // 32 rows x 64 bf16 output staging
constexpr int kOutOffset = kStages * kStageBytes;
constexpr int kBarOffset = kOutOffset + 8 * kOutBytesPerWarp;
constexpr int kSmemBytes = kBarOffset + 256 + 1024;
constexpr int kTmemCols = 2 * kBN;
constexpr int kLaunchRegs = 168, kProdRegs = 40, kEpiRegs = 232;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(128 * kProdRegs + 256 * kEpiRegs <= kThreads * kLaunchRegs,
              "register split must fit the CTA's launch allocation");
static_assert(kGroup * 64 * 127 * 127 < (1 << 23), "group sums must stay exact in fp32");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kKernelInt8Prefill = 4;

// kind::f16 instruction descriptor: A = B = fp16, D = fp32, both K-major.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

struct I8pParams {
    uint32_t* err;
    const float* Xs;   // [M]
    const float* Ws;   // [N]
    int32_t* acc;      // [M][N] or null
    int64_t M, N;
    int KS;            // K / 64
    int mtiles, ntiles;
    int split, ks_per;  // K ranges per tile and stages per range (split 1: whole tiles)
    int32_t* part;      // split > 1: int32 partial tiles [tiles * split][128][256]
};

// Work unit u: tile u / split, stages [ks_beg, ks_end) of K.
__device__ __forceinline__ void i8p_unit(int u, const I8pParams& p, int& tile, int& ks_beg, int& ks_end) {
    tile = u / p.split;
    ks_beg = (u - tile * p.split) * p.ks_per;
    ks_end = min(p.KS, ks_beg + p.ks_per);
}

__device__ __forceinline__ void record_timeout(uint32_t* err, uint32_t site, volatile int* abort) {
    atomicCAS(err, 0u, (kKernelInt8Prefill << 24) | (site << 16) | 1u);
    *abort = 1;
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_int8_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ CUtensorMap tmY, const __grid_constant__ I8pParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    const uint32_t tfull0 = smem_u32(bars + 2 * kStages), tempty0 = smem_u32(bars + 2 * kStages + 2);
    const uint32_t warp = warp_id(), lane = lane_id();
    const int units = p.mtiles * p.ntiles * p.split;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 8);          // one arrival per epilogue warp
        }
        *abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmY);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp < 4) {
        regs_dec<kProdRegs>();
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer
            const uint64_t pol_x = policy_evict_last(), pol_w = policy_evict_first();
            uint32_t it = 0;
            for (int u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
                int tile, ks_beg, ks_end;
                i8p_unit(u, p, tile, ks_beg, ks_end);
                const int mt = tile % p.mtiles, nt = tile / p.mtiles;
                for (int ks = ks_beg; ks < ks_end; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, kWaitLimitNs)) {
                        record_timeout(p.err, 1, abort);
                        break;
                    }
                    uint8_t* st = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(full0 + 8 * s, kStageBytes);
                    tma_load_2d(smem_u32(st), &tmX, full0 + 8 * s, ks * 64, mt * kBM, pol_x);
                    tma_load_2d(smem_u32(st + kABytes), &tmW, full0 + 8 * s, ks * 64, nt * kBN, pol_w);
                }
            }
            if (*abort)   // let copies already in flight land before the CTA can exit
                for (uint32_t j = it > (uint32_t)kStages ? it - kStages : 0; j < it; ++j)
                    mbar_drain(full0 + 8 * (j % kStages), (j / kStages) & 1, kWaitLimitNs);
        } else if (warp == 1 && lane == 0) {
            // ---------------- MMA issuer: one group of 8 stages per TMEM buffer
            uint32_t it = 0, gi = 0;
            for (int u = blockIdx.x; u < units && !*abort; u += gridDim.x) {
                int tile, ks_beg, ks_end;
                i8p_unit(u, p, tile, ks_beg, ks_end);
                for (int g0 = ks_beg; g0 < ks_end && !*abort; g0 += kGroup, ++gi) {
                    const uint32_t buf = gi & 1, bph = (gi >> 1) & 1;
                    if (!mbar_wait_bounded(tempty0 + 8 * buf, bph ^ 1, abort, kWaitLimitNs)) {
                        record_timeout(p.err, 3, abort);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + buf * kBN;
                    const int g_end = min(ks_end, g0 + kGroup);
                    for (int ks = g0; ks < g_end; ++ks, ++it) {
                        const int s = it % kStages;
                        const uint32_t ph = (it / kStages) & 1;
                        if (!mbar_wait_bounded(full0 + 8 * s, ph, abort, kWaitLimitNs)) {
                            record_timeout(p.err, 2, abort);
                            break;
                        }
                        tc_fence_after();
                        const uint8_t* st = smem + s * kStageBytes;
                        const uint64_t a = umma_desc_k128_sw128(smem_u32(st));
                        const uint64_t b = umma_desc_k128_sw128(smem_u32(st + kABytes));
#pragma unroll
                        for (int k = 0; k < 4; ++k)      // 4 x K=16 per 64-wide atom; +32 B = +2 in the address field
                            mma_f16(d, a + 2 * k, b + 2 * k, kIdesc, (ks > g0 || k > 0) ? 1u : 0u);
                        tc_commit(empty0 + 8 * s);
                    }
                    tc_commit(tfull0 + 8 * buf);
                }
            }
        }
    } else {
        regs_inc<kEpiRegs>();
        // ---------------- epilogue: exact int32 accumulation of the groups
        const int e = warp - 4;                   // 0..7
        const int q = warp & 3;                   // TMEM lane quadrant
        const int h = e >> 2;                     // column half of the tile
        const int row = 32 * q + lane;
        const int NB = (int)(p.N / 128);
        uint32_t gi = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            int tile, ks_beg, ks_end;
            i8p_unit(u, p, tile, ks_beg, ks_end);
            const int mt = tile % p.mtiles, nt = tile / p.mtiles;
            const int64_t m = (int64_t)mt * kBM + row;
            const int nb = 2 * nt + h;
            int32_t acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0;
            for (int g0 = ks_beg; g0 < ks_end; g0 += kGroup, ++gi) {
                const uint32_t buf = gi & 1, bph = (gi >> 1) & 1;
                // the verdict is made warp-uniform: the TMEM loads below are warp-collective
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(tfull0 + 8 * buf, bph, abort, kWaitLimitNs))) {
                    if (lane == 0) record_timeout(p.err, 4, abort);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + buf * kBN + h * 128;
                uint32_t r[64];
                tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r));
                tmem_ld_32x32b_x32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 64; ++j) acc[j] += __float2int_rn(__uint_as_float(r[j]));
                tmem_ld_32x32b_x32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(r));
                tmem_ld_32x32b_x32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8 * buf);   // buffer free once in registers
#pragma unroll
                for (int j = 0; j < 64; ++j) acc[64 + j] += __float2int_rn(__uint_as_float(r[j]));
            }
            if (!ok) break;
            if (p.split > 1) {
                // this K range's int32 partial: the thread's row, its half's 128 columns
                int4* dst = reinterpret_cast<int4*>(p.part + ((int64_t)u * kBM + row) * kBN + h * 128);
#pragma unroll
                for (int j = 0; j < 32; ++j) dst[j] = make_int4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
                continue;
            }
            if (nb >= NB) continue;                         // N % 256 == 128: no second half
            const bool live = m < p.M;
            if (p.acc != nullptr && live) {             // 8-byte stores: acc is 8-byte aligned
                int2* dst = reinterpret_cast<int2*>(p.acc + m * p.N + (int64_t)nb * 128);
#pragma unroll
                for (int j = 0; j < 64; ++j) dst[j] = make_int2(acc[2 * j], acc[2 * j + 1]);
            }
            // Y = bf16((float(acc) * Xs[m]) * Ws[n]): the warp's 32 rows x 128
            // columns as two 32 x 64 boxes, staged with the 128-byte swizzle and
            // written by TMA stores (rows beyond M are clipped by the store)
            const float xs = live ? __ldg(p.Xs + m) : 0.f;
            const float* wsn = p.Ws + (int64_t)nb * 128;       // 4-byte aligned: scalar loads
            uint8_t* stage = smem + kOutOffset + e * kOutBytesPerWarp;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c0 = c * 64 + 8 * j;
                    float y[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        y[i] = __fmul_rn(__fmul_rn(__int2float_rn(acc[c0 + i]), xs), __ldg(wsn + c0 + i));
                    uint4 o;
                    o.x = pack_bf16x2(y[0], y[1]);
                    o.y = pack_bf16x2(y[2], y[3]);
                    o.z = pack_bf16x2(y[4], y[5]);
                    o.w = pack_bf16x2(y[6], y[7]);
                    *reinterpret_cast<uint4*>(stage + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmY, smem_u32(stage), nt * kBN + h * 128 + c * 64, mt * kBM + 32 * q);
                    bulk_commit();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    __syncwarp();   // warps whose lane 0 alone ran the producer / MMA loop reconverge first
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// int8 -> fp16: v ^ 0x80 = v + 128 in the low byte of the fp16 0x6400 | b =
// 1024 + b, so (1152 + v) - 1152 = v exactly.
__device__ __forceinline__ void i8x16_to_f16(const uint4 v, uint4* dst) {
    const __half2 off = __floats2half2_rn(1152.f, 1152.f);
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t lo = __byte_perm(w[k], 0x64646464u, 0x4140), hi = __byte_perm(w[k], 0x64646464u, 0x4342);
        __half2 hl = __hsub2(*reinterpret_cast<__half2*>(&lo), off);
        __half2 hh = __hsub2(*reinterpret_cast<__half2*>(&hi), off);
        o[2 * k] = *reinterpret_cast<uint32_t*>(&hl);
        o[2 * k + 1] = *reinterpret_cast<uint32_t*>(&hh);
    }
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// X codes then W codes, 16 per chunk, into one fp16 array; each thread has
// four 16-byte loads in flight per step.
__global__ void __launch_bounds__(256)
int8_to_f16_kernel(const int8_t* __restrict__ a, int64_t na16, const int8_t* __restrict__ b, int64_t nb16,
                   uint16_t* __restrict__ out) {
    pdl_wait_then_release();
    const int64_t total = na16 + nb16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < total) v[u] = ld_stream_v4(i < na16 ? a + i * 16 : b + (i - na16) * 16);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < total) i8x16_to_f16(v[u], reinterpret_cast<uint4*>(out + i * 16));
        }
    }
}

// Split-K reduction: one thread per (tile row, 8 columns); the ranges' int32
// partials are added (exact in any order), then Y = bf16((float(acc) * Xs[m]) *
// Ws[n]) as in the GEMM's own epilogue, and acc if asked.
__global__ void __launch_bounds__(256)
i8p_reduce_kernel(const int32_t* __restrict__ part, const float* __restrict__ Xs, const float* __restrict__ Ws,
                  int64_t M, int64_t N, int mtiles, int split, int64_t units8, uint16_t* __restrict__ Y, int64_t ldy,
                  int32_t* __restrict__ acc) {
    pdl_wait_then_release();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= units8) return;
    const int64_t tile = t >> 12;                     // 128 rows x 32 eight-column chunks per tile
    const int r = (int)((t >> 5) & 127), c8 = (int)(t & 31);
    const int mt = (int)(tile % mtiles), nt = (int)(tile / mtiles);
    const int64_t m = (int64_t)mt * kBM + r, n = (int64_t)nt * kBN + c8 * 8;
    if (m >= M || n >= N) return;
    const int32_t* base = part + ((tile * split) * kBM + r) * kBN + c8 * 8;
    const int64_t stride = (int64_t)kBM * kBN;         // one range's partial tile
    int32_t sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int sp0 = 0; sp0 < split; sp0 += 4) {
        int4 v[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (sp0 + j < split) {
                const int4* src = reinterpret_cast<const int4*>(base + (sp0 + j) * stride);
                v[j][0] = src[0];
                v[j][1] = src[1];
            }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (sp0 + j < split) {
                sum[0] += v[j][0].x; sum[1] += v[j][0].y; sum[2] += v[j][0].z; sum[3] += v[j][0].w;
                sum[4] += v[j][1].x; sum[5] += v[j][1].y; sum[6] += v[j][1].z; sum[7] += v[j][1].w;
            }
    }
    if (acc != nullptr) {                              // 8-byte aligned
        int2* d = reinterpret_cast<int2*>(acc + m * N + n);
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] = make_int2(sum[2 * i], sum[2 * i + 1]);
    }
    const float xs = __ldg(Xs + m);
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(__fmul_rn(__int2float_rn(sum[i]), xs), __ldg(Ws + n + i));
    uint4 o;
    o.x = pack_bf16x2(y[0], y[1]);
    o.y = pack_bf16x2(y[2], y[3]);
    o.z = pack_bf16x2(y[4], y[5]);
    o.w = pack_bf16x2(y[6], y[7]);
    *reinterpret_cast<uint4*>(Y + m * ldy + n) = o;
}

// The register split (setmaxnreg) assumes exactly kLaunchRegs registers per
// thread at launch; any other build is refused.  Checked (and the shared memory
// attribute set) once per device.
int i8p_ready(int dev) {
    static int checked[64] = {};   // 0 unknown, 1 ok, -1 refused
    if (dev < 0 || dev >= 64) return -1;
    if (checked[dev] == 0) {
        cudaFuncAttributes fa;
        checked[dev] = (cudaFuncGetAttributes(&fa, gemm_int8_prefill_kernel) == cudaSuccess &&
                        fa.numRegs == kLaunchRegs &&
                        cudaFuncSetAttribute(gemm_int8_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes) == cudaSuccess)
                           ? 1
                           : -1;
        cudaGetLastError();
    }
    return checked[dev];
}

}  // namespace

// K ranges per tile: with fewer tiles than SMs, enough ranges that about one
// wave of units runs, each at least two exact groups (16 stages) long and
// aligned to a group; at most 8.
struct I8pPlan {
    int split, ks_per;
};

static I8pPlan i8p_plan(int64_t M, int64_t N, int64_t K) {
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    const int KS = (int)(K / 64);
    const int64_t sms = num_sms();
    int64_t s = tiles >= sms ? 1 : sms / tiles;
    if (s > KS / 16) s = KS / 16;
    if (s > 8) s = 8;
    if (s < 2) return I8pPlan{1, KS};
    int per = (int)((KS + s - 1) / s);
    per = (per + kGroup - 1) / kGroup * kGroup;
    return I8pPlan{(KS + per - 1) / per, per};
}

// The large-batch path: 256 tokens or more, with enough work units (tiles, or
// tiles x K ranges) for at least half of the SMs.
bool int8_prefill_applies(int64_t M, int64_t N, int64_t K) {
    if (M < 256) return false;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    return tiles * i8p_plan(M, N, K).split * 2 >= num_sms();
}

// fp16 copies of X [M][K] and W [N][K], back to back, then (split K) the int32
// partial tiles.
size_t int8_prefill_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (!int8_prefill_applies(M, N, K)) return 0;
    const I8pPlan pl = i8p_plan(M, N, K);
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    const size_t parts = pl.split > 1 ? (size_t)tiles * pl.split * kBM * kBN * sizeof(int32_t) : 0;
    return (size_t)(M + N) * (size_t)K * 2 + parts;
}

// Kernels of the large-batch path: the conversion, the GEMM and, with split K,
// the reduction.
int int8_prefill_kernel_count(int64_t M, int64_t N, int64_t K) { return i8p_plan(M, N, K).split > 1 ? 3 : 2; }

// fp16 copy of n int8 codes (n % 16 == 0; both pointers 16-byte aligned).
cudaError_t launch_int8_to_f16(const int8_t* src, int64_t n, uint16_t* dst, cudaStream_t st) {
    const int64_t n16 = n / 16;
    if (n16 == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((n16 + 255) / 256, (int64_t)num_sms() * 8);
    return launch_pdl(int8_to_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, src, n16,
                      static_cast<const int8_t*>(nullptr), (int64_t)0, dst);
}

cudaError_t launch_gemm_int8_prefill(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                                     int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy, int32_t* acc,
                                     void* ws, cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (i8p_ready(dev) != 1) return cudaErrorInvalidDeviceFunction;
    const I8pPlan pl = i8p_plan(M, N, K);
    uint16_t* X16 = static_cast<uint16_t*>(ws);
    uint16_t* W16 = X16 + M * K;
    int32_t* part = pl.split > 1 ? reinterpret_cast<int32_t*>(W16 + N * K) : nullptr;   // 16-byte aligned
    CUtensorMap tmX, tmW, tmY;
    if (!make_tmap_f16_load(&tmX, X16, (uint64_t)M, (uint64_t)K, kBM)) return cudaErrorInvalidValue;
    if (!make_tmap_f16_load(&tmW, W16, (uint64_t)N, (uint64_t)K, kBN)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_store(&tmY, Y, (uint64_t)M, (uint64_t)N, (uint64_t)ldy, 64, 32)) return cudaErrorInvalidValue;
    uint32_t* err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    const int64_t na16 = M * K / 16, nb16 = N * K / 16;
    const int64_t cvt_blocks = std::min<int64_t>((na16 + nb16 + 255) / 256, (int64_t)num_sms() * 8);
    cudaError_t e = launch_pdl(int8_to_f16_kernel, dim3((unsigned)cvt_blocks), dim3(256), 0, st, Xq, na16, Wq, nb16,
                               X16);
    if (e != cudaSuccess) return e;
    I8pParams prm{err, Xs, Ws, acc, M, N, (int)(K / 64), (int)((M + kBM - 1) / kBM), (int)((N + kBN - 1) / kBN),
                  pl.split, pl.ks_per, part};
    const int64_t tiles = (int64_t)prm.mtiles * prm.ntiles, units = tiles * pl.split;
    const int grid = units < num_sms() ? (int)units : num_sms();
    e = launch_pdl(gemm_int8_prefill_kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, tmX, tmW, tmY, prm);
    if (e != cudaSuccess || pl.split == 1) return e;
    const int64_t units8 = tiles * kBM * 32;
    return launch_pdl(i8p_reduce_kernel, dim3((unsigned)((units8 + 255) / 256)), dim3(256), 0, st,
                      (const int32_t*)part, Xs, Ws, M, N, prm.mtiles, pl.split, units8, Y, ldy, acc);
}

}  // namespace fp8rl
