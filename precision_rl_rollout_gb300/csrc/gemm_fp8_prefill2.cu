// gemm_fp8_prefill2.cu -- block-scaled FP8 GEMM for large token counts on CTA
// pairs (tcgen05 cta_group::2).
//
// Same math as the one-CTA prefill kernel (FP8-RL, Abstract, contribution (i)):
// per 128-wide K block an fp32 tensor-core partial product, promoted in fp32
// registers with the block's scale product, then one bf16 rounding.
//
// Why pairs: with one CTA per 128x256 tile every K block brings 48 KB into
// shared memory by TMA and the tensor core reads 48 KB back, which saturates
// the SM's shared-memory bandwidth well before the tensor pipe.  A pair of
// CTAs (a cluster of two, on two SMs) computes a 256x256 tile with one
// M=256 MMA issued by the even CTA: each CTA holds its own 128 token rows of
// X and half (128 rows) of the weight tile, so a stage is 32 KB per SM and
// six stages fit.  The MMA reads the other half of the weight tile from the
// peer's shared memory.  Each CTA's TMEM holds its own 128 output rows.
//
// Barriers: the even CTA's full[s] counts both CTAs' TMA bytes; the MMA
// commits to empty[s] and tfull[b] of both CTAs (multicast); both CTAs'
// epilogue warps release a TMEM buffer on the even CTA's tempty[b].
#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {

using namespace sm100;

namespace {

constexpr int kRows = 128;                          // token rows per CTA (256 per pair)
constexpr int kBN = 256;                            // weight rows per pair tile (128 per CTA)
constexpr int kStages = 6;
constexpr int kABytes = kRows * 128;                // X tile: 128 tokens x 128 K
constexpr int kBBytes = 128 * 128;                  // W half tile: 128 rows x 128 K
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 384;
constexpr int kOutBytesPerWarp = 32 * 128;
constexpr int kOutOffset = kStages * kStageBytes;
constexpr int kBarOffset = kOutOffset + 8 * kOutBytesPerWarp;
constexpr int kSmemBytes = kBarOffset + 256 + 1024;
constexpr int kTmemCols = 2 * kBN;
constexpr int kLaunchRegs = 168, kProdRegs = 40, kEpiRegs = 232;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(128 * kProdRegs + 256 * kEpiRegs <= kThreads * kLaunchRegs,
              "register split must fit the CTA's launch allocation");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kKernelPrefillPair = 4;

struct PairParams {
    uint32_t* err;
    const float* Xs;   // [KB][M]
    const float* Ws;   // [N/128][KB]
    int64_t M;
    int KB, NB;
    int mtiles, ntiles;  // ceil(M/256), ceil(N/256)
};

__device__ __forceinline__ void record_timeout(uint32_t* err, uint32_t site, volatile int* abort) {
    atomicCAS(err, 0u, (kKernelPrefillPair << 24) | (site << 16) | 1u);
    *abort = 1;
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_fp8_prefill_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                             const __grid_constant__ CUtensorMap tmY, const __grid_constant__ PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    const uint32_t tfull0 = smem_u32(bars + 2 * kStages), tempty0 = smem_u32(bars + 2 * kStages + 2);
    const uint32_t warp = warp_id(), lane = lane_id();
    const uint32_t rank = cluster_ctarank();        // 0: issues the MMAs; 1: its peer
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int total_tiles = p.mtiles * p.ntiles;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);             // even CTA: its own expect_tx arrival
            mbar_init(empty0 + 8 * s, 1);            // the pair MMA's commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 16);          // 8 epilogue warps in each CTA
        }
        *abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmY);
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    cluster_sync_all();                              // both CTAs' barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();
    const uint32_t full0_leader = map_to_rank(full0, 0);
    const uint32_t tempty0_leader = map_to_rank(tempty0, 0);

    if (warp < 4) {
        regs_dec<kProdRegs>();
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer (both CTAs): own X rows and own weight half
            const uint64_t pol_x = policy_evict_last(), pol_w = policy_evict_first();
            uint32_t it = 0;
            for (int tile = pair; tile < total_tiles && !*abort; tile += npairs) {
                const int mt = tile % p.mtiles, nt = tile / p.mtiles;
                for (int kb = 0; kb < p.KB; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, kWaitLimitNs)) {
                        record_timeout(p.err, 1, abort);
                        break;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(full0 + 8 * s, 2 * kStageBytes);
                    uint8_t* st = smem + s * kStageBytes;
                    tma_load_2d_pair(smem_u32(st), &tmX, full0_leader + 8 * s, kb * 128,
                                     mt * 2 * kRows + (int)rank * kRows, pol_x);
                    tma_load_2d_pair(smem_u32(st + kABytes), &tmW, full0_leader + 8 * s, kb * 128,
                                     nt * kBN + (int)rank * 128, pol_w);
                }
            }
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ---------------- pair MMA issuer (even CTA)
            constexpr uint32_t idesc = idesc_e4m3_f32(2 * kRows, kBN);
            uint32_t it = 0;
            for (int tile = pair; tile < total_tiles && !*abort; tile += npairs) {
                for (int kb = 0; kb < p.KB; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    const uint32_t buf = it & 1, bph = (it >> 1) & 1;
                    if (!mbar_wait_bounded(full0 + 8 * s, ph, abort, kWaitLimitNs)) {
                        record_timeout(p.err, 2, abort);
                        break;
                    }
                    if (!mbar_wait_bounded(tempty0 + 8 * buf, bph ^ 1, abort, kWaitLimitNs)) {
                        record_timeout(p.err, 3, abort);
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* st = smem + s * kStageBytes;
                    const uint64_t a = umma_desc_k128_sw128(smem_u32(st));
                    const uint64_t b = umma_desc_k128_sw128(smem_u32(st + kABytes));
                    const uint32_t d = tmem_base + buf * kBN;
#pragma unroll
                    for (int k = 0; k < 4; ++k) mma_f8f6f4_pair(d, a + 2 * k, b + 2 * k, idesc, k > 0 ? 1u : 0u);
                    tc_commit_pair(empty0 + 8 * s, 0x3);
                    tc_commit_pair(tfull0 + 8 * buf, 0x3);
                }
            }
        }
    } else {
        regs_inc<kEpiRegs>();
        // ---------------- epilogue (both CTAs): own 128 token rows x 256 columns
        const int e = warp - 4;
        const int q = warp & 3;
        const int h = e >> 2;
        const int row = 32 * q + lane;
        uint32_t it = 0;
        for (int tile = pair; tile < total_tiles; tile += npairs) {
            const int mt = tile % p.mtiles, nt = tile / p.mtiles;
            const int64_t m = (int64_t)mt * 2 * kRows + (int64_t)rank * kRows + row;
            const int nb = 2 * nt + h;
            const bool live = m < p.M && nb < p.NB;
            const float* __restrict__ xs = p.Xs + (live ? m : 0);
            const float* __restrict__ ws = p.Ws + (int64_t)(live ? nb : 0) * p.KB;
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.f;
            float sx = live ? __ldg(xs) : 0.f, sw = live ? __ldg(ws) : 0.f;
            bool ok = true;
            for (int kb = 0; kb < p.KB; ++kb, ++it) {
                const float scale = sx * sw;
                if (kb + 1 < p.KB && live) {
                    sx = __ldg(xs + (int64_t)(kb + 1) * p.M);
                    sw = __ldg(ws + kb + 1);
                }
                const uint32_t buf = it & 1, bph = (it >> 1) & 1;
                if (!mbar_wait_bounded(tfull0 + 8 * buf, bph, abort, kWaitLimitNs)) {
                    record_timeout(p.err, 4, abort);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + buf * kBN + h * 128;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + g * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[g * 32 + j] = fmaf(__uint_as_float(r[j]), scale, acc[g * 32 + j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty0_leader + 8 * buf);
            }
            if (!ok) break;
            if (nb < p.NB) {
                uint8_t* stage = smem + kOutOffset + e * kOutBytesPerWarp;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 o;
                        const float* a = acc + c * 64 + 8 * j;
                        o.x = pack_bf16x2(a[0], a[1]);
                        o.y = pack_bf16x2(a[2], a[3]);
                        o.z = pack_bf16x2(a[4], a[5]);
                        o.w = pack_bf16x2(a[6], a[7]);
                        *reinterpret_cast<uint4*>(stage + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmY, smem_u32(stage), nt * kBN + h * 128 + c * 64,
                                     mt * 2 * kRows + (int)rank * kRows + 32 * q);
                        bulk_commit();
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    // the peer's MMAs read this CTA's shared memory and write its TMEM: neither
    // CTA leaves before both are done
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace

// The register split assumes the kernel was built with exactly kLaunchRegs
// registers per thread; anything else could make the epilogue's increase wait
// forever, so the launch is refused (the caller then uses the one-CTA kernel).
bool prefill_pair_available() {
    static int checked = 0;
    if (checked == 0) {
        cudaFuncAttributes fa;
        checked = (cudaFuncGetAttributes(&fa, gemm_fp8_prefill_pair_kernel) == cudaSuccess &&
                   fa.numRegs == kLaunchRegs &&
                   cudaFuncSetAttribute(gemm_fp8_prefill_pair_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) == cudaSuccess)
                      ? 1
                      : -1;
    }
    return checked == 1;
}

cudaError_t launch_gemm_fp8_prefill_pair(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                         const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                                         int64_t ldy, cudaStream_t st) {
    if (!prefill_pair_available()) return cudaErrorInvalidDeviceFunction;
    CUtensorMap tmX, tmW, tmY;
    if (!make_tmap_u8(&tmX, Xq, (uint64_t)M, (uint64_t)K, (uint64_t)K, kRows)) return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tmW, Wq, (uint64_t)N, (uint64_t)K, (uint64_t)K, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_store(&tmY, Y, (uint64_t)M, (uint64_t)N, (uint64_t)ldy, 64, 32)) return cudaErrorInvalidValue;
    uint32_t* err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    PairParams prm{err, Xs, Ws, M, (int)(K / 128), (int)(N / 128), (int)((M + 2 * kRows - 1) / (2 * kRows)),
                   (int)((N + kBN - 1) / kBN)};
    const int tiles = prm.mtiles * prm.ntiles;
    const int pairs = tiles < num_sms() / 2 ? tiles : num_sms() / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_fp8_prefill_pair_kernel, tmX, tmW, tmY, prm);
}

}  // namespace fp8rl
