// gemm_fp8_prefill.cu -- block-scaled FP8 GEMM for large token counts (prefill),
// tensor-core bound, on tcgen05 + TMA.
//
// Same math as the decode kernel (FP8-RL, Abstract, contribution (i)):
//   Y[m][n] = bf16( sum_kb Xs[kb][m] * Ws[n/128][kb] * P_kb[m][n] ),
// with P_kb the fp32 tensor-core product of one 128-wide K block.
//
// Persistent kernel, one CTA per SM.  Output tile 128 tokens x 256 channels:
// one tcgen05.mma M=128 N=256 K=32 group of four per K block into one of two
// 256-column TMEM buffers (double buffered, all 512 columns).  The two column
// halves of the tile are exactly two weight blocks, so the scale that promotes
// a K block's partial product is one fp32 scalar per thread (its token's
// activation scale times its half's weight scale).
// Warpgroup 0: warp 0 issues TMA, warps 1 and 2 issue the MMAs of alternate K
// blocks (warp 1 owns TMEM).
// Warpgroups 1 and 2: epilogue, one per column half; each thread owns one
// token row and keeps 128 fp32 accumulators in registers, which setmaxnreg
// moves over from warpgroup 0 (40 -> 232 registers per thread).
// Tiles go M-fastest, so the CTAs in flight share a few 256-row weight slabs
// and the (L2-resident) activations.
// Split-K: a work unit is (tile, K range); each range writes its fp32 partial
// tile to the caller's workspace by TMA, and a second launch adds the ranges
// of a tile in a fixed order (deterministic) and rounds to bf16.  It serves
// two cases: shapes with fewer tiles than SMs and a long K (a few hundred
// tokens: every tile is split), and the last, partial wave of tiles (only the
// tiles after the last full wave are split, so that wave finishes in a
// fraction of a tile's time; e.g. 1280 tiles on 152 SMs leave 64).
#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {

using namespace sm100;

namespace {

constexpr int kBM = 128, kBN = 256;
constexpr int kStages = 4;
constexpr int kABytes = kBM * 128;                  // X tile: 128 tokens x 128 K
constexpr int kBBytes = kBN * 128;                  // W tile: 256 channels x 128 K
constexpr int kStageBytes = kABytes + kBBytes;
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
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kKernelPrefill = 2;

struct PrefillParams {
    uint32_t* err;
    const float* Xs;   // [KB][M]
    const float* Ws;   // [N/128][KB]
    uint16_t* Y;       // [M][ldy]
    int64_t M, ldy;
    int KB, NB;        // K/128, N/128
    int mtiles, ntiles;
    int group_m;        // token tiles per group of the tile order (see tile_coords)
    int split, kb_per;  // K ranges per split tile and K blocks per range (split 1: no workspace)
    int full_tiles;     // tiles [0, full_tiles) are not split (all of them when split == 1)
};

// Tile order: groups of group_m token tiles; within a group the weight-column
// tile advances slowest and the token tile fastest.  With group_m = mtiles this
// is the token-tile-fastest order over the whole output (every weight tile is
// read by all token tiles while it is in L2); a smaller group keeps the
// activations of the group in L2 while the weight columns stream past, for
// activations larger than L2.
__host__ __device__ __forceinline__ void tile_coords(int64_t tile, int mtiles, int ntiles, int group_m, int& mt,
                                                     int& nt) {
    const int64_t per_group = (int64_t)group_m * ntiles;
    const int64_t g = tile / per_group, r = tile - g * per_group;
    const int rows = min(group_m, mtiles - (int)g * group_m);      // token tiles in this group
    nt = (int)(r / rows);
    mt = (int)(g * group_m + r % rows);
}

// Work unit u: tile, K range [kb_beg, kb_end), and the range's index (-1: the
// whole tile, written as bf16).  Units [0, full_tiles) are whole tiles; each
// later tile is `split` consecutive units.
struct PrefillUnit {
    int tile, sp, kb_beg, kb_end;
};

template <bool kSplit>
__device__ __forceinline__ PrefillUnit prefill_unit(int u, const PrefillParams& p) {
    if (!kSplit || u < p.full_tiles) return PrefillUnit{u, -1, 0, p.KB};
    const int v = u - p.full_tiles, t = v / p.split, sp = v - t * p.split;
    const int kb_beg = sp * p.kb_per;
    return PrefillUnit{p.full_tiles + t, sp, kb_beg, min(p.KB, kb_beg + p.kb_per)};
}

__device__ __forceinline__ void record_timeout(uint32_t* err, uint32_t site, volatile int* abort) {
    atomicCAS(err, 0u, (kKernelPrefill << 24) | (site << 16) | 1u);
    *abort = 1;
}

template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
gemm_fp8_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmP,
                        const __grid_constant__ PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
    const uint32_t tfull0 = smem_u32(bars + 2 * kStages), tempty0 = smem_u32(bars + 2 * kStages + 2);
    const uint32_t warp = warp_id(), lane = lane_id();
    // (kSplit = false: the split code is compiled out)
    const int total_units = kSplit ? p.full_tiles + (p.mtiles * p.ntiles - p.full_tiles) * p.split
                                   : p.mtiles * p.ntiles;

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
        if (kSplit) prefetch_tmap(&tmP);
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
            for (int u = blockIdx.x; u < total_units && !*abort; u += gridDim.x) {
                const PrefillUnit un = prefill_unit<kSplit>(u, p);
                int mt, nt;
                tile_coords(un.tile, p.mtiles, p.ntiles, p.group_m, mt, nt);
                for (int kb = un.kb_beg; kb < un.kb_end; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, kWaitLimitNs)) {
                        record_timeout(p.err, 1, abort);
                        break;
                    }
                    uint8_t* st = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(full0 + 8 * s, kStageBytes);
                    tma_load_2d(smem_u32(st), &tmX, full0 + 8 * s, kb * 128, mt * kBM, pol_x);
                    tma_load_2d(smem_u32(st + kABytes), &tmW, full0 + 8 * s, kb * 128, nt * kBN, pol_w);
                }
            }
            if (*abort)   // let copies already in flight land before the CTA can exit
                for (uint32_t j = it > (uint32_t)kStages ? it - kStages : 0; j < it; ++j)
                    mbar_drain(full0 + 8 * (j % kStages), (j / kStages) & 1, kWaitLimitNs);
        } else if ((warp == 1 || warp == 2) && lane == 0) {
            // ---------------- MMA issuers: warp 1 issues the K blocks that go to
            // TMEM buffer 0, warp 2 those of buffer 1, so one thread's barrier
            // waits and commits overlap the other's MMAs
            constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kBN);
            const uint32_t mine = warp - 1;
            uint32_t it = 0;
            for (int u = blockIdx.x; u < total_units && !*abort; u += gridDim.x) {
                const PrefillUnit un = prefill_unit<kSplit>(u, p);
                const int nkb = un.kb_end - un.kb_beg;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    if ((it & 1) != mine) continue;
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
                    for (int k = 0; k < 4; ++k) mma_f8f6f4(d, a + 2 * k, b + 2 * k, idesc, k > 0 ? 1u : 0u);
                    tc_commit(empty0 + 8 * s);
                    tc_commit(tfull0 + 8 * buf);
                }
            }
        }
    } else {
        regs_inc<kEpiRegs>();
        // ---------------- epilogue: promotion of each K block into fp32 registers
        const int e = warp - 4;                   // 0..7
        const int q = warp & 3;                   // TMEM lane quadrant
        const int h = e >> 2;                     // column half = weight block within the tile
        const int row = 32 * q + lane;
        uint32_t it = 0;
        for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
            const PrefillUnit un = prefill_unit<kSplit>(u, p);
            const int tile = un.tile, sp = un.sp;
            int mt, nt;
            tile_coords(tile, p.mtiles, p.ntiles, p.group_m, mt, nt);
            const int kb_beg = un.kb_beg, kb_end = un.kb_end;
            const int64_t m = (int64_t)mt * kBM + row;
            const int nb = 2 * nt + h;
            const bool live = m < p.M && nb < p.NB;
            const float* __restrict__ xs = p.Xs + (live ? m : 0);
            const float* __restrict__ ws = p.Ws + (int64_t)(live ? nb : 0) * p.KB;
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.f;
            float sx = live ? __ldg(xs + (int64_t)kb_beg * p.M) : 0.f, sw = live ? __ldg(ws + kb_beg) : 0.f;
            bool ok = true;
            for (int kb = kb_beg; kb < kb_end; ++kb, ++it) {
                const float scale = sx * sw;
                if (kb + 1 < kb_end && live) {                // next block's scales, early
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
                // The buffer is released as soon as its last columns are in
                // registers; the second half's promotion runs after the release.
                uint32_t r[64];
                tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r));
                tmem_ld_32x32b_x32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 64; ++j) acc[j] = fmaf(__uint_as_float(r[j]), scale, acc[j]);
                tmem_ld_32x32b_x32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(r));
                tmem_ld_32x32b_x32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
#pragma unroll
                for (int j = 0; j < 64; ++j) acc[64 + j] = fmaf(__uint_as_float(r[j]), scale, acc[64 + j]);
            }
            if (!ok) break;
            if (kSplit && sp >= 0) {
                // fp32 partial of this K range: the warp's 32 rows x 128 columns as
                // four 32 x 32 boxes (128-byte rows, 128-byte swizzle) into the
                // workspace's slot (tile, sp), rows slot*128 .. +127
                uint8_t* stage = smem + kOutOffset + e * kOutBytesPerWarp;
                const int slot_row = ((tile - p.full_tiles) * p.split + sp) * kBM + 32 * q;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float* a = acc + c * 32 + 4 * j;
                        *reinterpret_cast<float4*>(stage + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                            make_float4(a[0], a[1], a[2], a[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmP, smem_u32(stage), h * 128 + c * 32, slot_row);
                        bulk_commit();
                    }
                }
                continue;
            }
            // Output: the warp's 32 rows x 128 columns go out as two 32 x 64 boxes,
            // each staged in this warp's 4 KB buffer with the 128-byte swizzle
            // and written by one asynchronous TMA store (rows beyond M and
            // columns beyond N are clipped by the store).
            if (nb < p.NB) {
                uint8_t* stage = smem + kOutOffset + e * kOutBytesPerWarp;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (lane == 0) bulk_wait_read_all();   // the previous box has left the buffer
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
                        tma_store_2d(&tmY, smem_u32(stage), nt * kBN + h * 128 + c * 64, mt * kBM + 32 * q);
                        bulk_commit();
                    }
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

// Split-K reduction: one thread per (tile row, 8 output columns); the splits
// are added in order in fp32, then rounded to bf16 once.
__global__ void __launch_bounds__(256)
prefill_splitk_reduce_kernel(const float* __restrict__ part, int64_t M, int64_t N, int mtiles, int ntiles,
                             int group_m, int split, int tile0, int64_t units8, uint16_t* __restrict__ Y,
                             int64_t ldy) {
    pdl_wait_then_release();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= units8) return;
    const int64_t slot = t >> 12;                     // 128 rows x 32 eight-column chunks per tile
    const int64_t tile = tile0 + slot;                // split tiles start at tile0
    const int r = (int)((t >> 5) & 127), c8 = (int)(t & 31);
    int mt, nt;
    tile_coords(tile, mtiles, ntiles, group_m, mt, nt);
    const int64_t m = (int64_t)mt * kBM + r, n = (int64_t)nt * kBN + c8 * 8;
    if (m >= M || n >= N) return;
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const float* base = part + ((slot * split) * kBM + r) * kBN + c8 * 8;
    const int64_t stride = (int64_t)kBM * kBN;         // one range's partial tile
    for (int sp0 = 0; sp0 < split; sp0 += 4) {
        // four ranges' loads in flight, then added in range order (deterministic)
        float4 v[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (sp0 + j < split) {
                const float4* src = reinterpret_cast<const float4*>(base + (sp0 + j) * stride);
                v[j][0] = src[0];
                v[j][1] = src[1];
            }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (sp0 + j < split) {
                s[0] += v[j][0].x; s[1] += v[j][0].y; s[2] += v[j][0].z; s[3] += v[j][0].w;
                s[4] += v[j][1].x; s[5] += v[j][1].y; s[6] += v[j][1].z; s[7] += v[j][1].w;
            }
    }
    uint4 o;
    o.x = pack_bf16x2(s[0], s[1]);
    o.y = pack_bf16x2(s[2], s[3]);
    o.z = pack_bf16x2(s[4], s[5]);
    o.w = pack_bf16x2(s[6], s[7]);
    *reinterpret_cast<uint4*>(Y + m * ldy + n) = o;
}

}  // namespace

// Token tiles per group of the tile order: all of them (token-tile fastest over
// the whole output) while the activations fit comfortably in L2, else 16, so
// that 16 token tiles' activations stay in L2 while the weight tiles stream
// past (the 27648-wide down projection at M = 8192: 226 MB of activations).
static int prefill_group_m(int64_t M, int64_t K, int mtiles) {
    constexpr int64_t kActInL2 = 48ll << 20;
    return M * K <= kActInL2 ? mtiles : (mtiles < 16 ? mtiles : 16);
}

// Which tiles are split into K ranges, and into how many (split 1: none).
//  - Fewer tiles than about one wave: every tile, so that about one wave of
//    CTAs runs, keeping at least 8 K blocks per range.
//  - Otherwise the tiles after the last full wave, when they fill at most half
//    a wave: into as many ranges as fill it (at least 8 K blocks each), if the
//    part of a tile's time saved (at about 0.45 us per K block) exceeds what
//    the partial tiles' round trip and the reduction launch cost (3 us plus
//    the partials at 1.4 GB/ms, measured on the 32B shapes at M = 2048 and
//    8192: the 27648-wide down projection gains 3.5% and 27%, the 5120-wide
//    o_proj 6% at M = 2048 and would lose 3% at M = 8192).
struct PrefillPlan {
    int split;        // K ranges per split tile
    int full_tiles;   // tiles [0, full_tiles) run whole
};

static PrefillPlan prefill_plan(int64_t M, int64_t N, int64_t K) {
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    const int64_t sms = num_sms();
    const int kb = (int)(K / 128);
    const PrefillPlan none{1, (int)tiles};
    if (tiles * 4 < sms * 3) {
        int64_t s = sms / tiles;
        if (s > kb / 8) s = kb / 8;
        if (s > 8) s = 8;
        return s < 2 ? none : PrefillPlan{(int)s, 0};
    }
    const int64_t full = tiles / sms * sms, tail = tiles - full;
    if (tail == 0 || tail * 2 > sms) return none;
    int64_t s = sms / tail;
    if (s > kb / 8) s = kb / 8;
    if (s > 8) s = 8;
    if (s < 2) return none;
    const double saved = (1.0 - 1.0 / (double)s) * kb * 0.45;
    const double cost = 3.0 + (double)(tail * s) * kBM * kBN * sizeof(float) / 1.4e6;
    return saved > cost ? PrefillPlan{(int)s, (int)full} : none;
}

static size_t prefill_ws_bytes(int64_t M, int64_t N, const PrefillPlan& pl) {
    if (pl.split <= 1) return 0;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    return (size_t)(tiles - pl.full_tiles) * (size_t)pl.split * kBM * kBN * sizeof(float);
}

// The register split (setmaxnreg) assumes the kernel was built with exactly
// kLaunchRegs registers per thread; anything else could make the epilogue's
// increase wait forever, so such a build is refused.  Checked (and the shared
// memory attribute set) once per device.
template <bool kSplit>
static int prefill_ready(int dev) {
    static int checked[64] = {};   // 0 unknown, 1 ok, -1 refused
    if (checked[dev] == 0) {
        cudaFuncAttributes fa;
        checked[dev] = (cudaFuncGetAttributes(&fa, gemm_fp8_prefill_kernel<kSplit>) == cudaSuccess &&
                        fa.numRegs == kLaunchRegs &&
                        cudaFuncSetAttribute(gemm_fp8_prefill_kernel<kSplit>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) == cudaSuccess)
                           ? 1
                           : -1;
    }
    return checked[dev];
}

cudaError_t launch_gemm_fp8_prefill(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                    const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                                    int64_t ldy, void* ws, size_t ws_bytes, cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (prefill_ready<false>(dev) != 1 || prefill_ready<true>(dev) != 1) return cudaErrorInvalidDeviceFunction;
    PrefillPlan pl = prefill_plan(M, N, K);
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    // with less workspace than the split needs, run without split-K
    if (pl.split > 1 && (ws == nullptr || ws_bytes < prefill_ws_bytes(M, N, pl))) pl = PrefillPlan{1, (int)tiles};
    const int split = pl.split;
    CUtensorMap tmX, tmW, tmY, tmP;
    if (!make_tmap_u8(&tmX, Xq, (uint64_t)M, (uint64_t)K, (uint64_t)K, kBM)) return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tmW, Wq, (uint64_t)N, (uint64_t)K, (uint64_t)K, kBN)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16_store(&tmY, Y, (uint64_t)M, (uint64_t)N, (uint64_t)ldy, 64, 32)) return cudaErrorInvalidValue;
    uint32_t* err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    const int KB = (int)(K / 128);
    const int mtiles = (int)((M + kBM - 1) / kBM);
    PrefillParams prm{err, Xs, Ws, Y, M, ldy, KB, (int)(N / 128),
                      mtiles, (int)((N + kBN - 1) / kBN), prefill_group_m(M, K, mtiles), split,
                      (KB + split - 1) / split, pl.full_tiles};
    const int64_t split_tiles = tiles - pl.full_tiles;
    if (split > 1) {
        if (!make_tmap_f32_store(&tmP, ws, (uint64_t)(split_tiles * split * kBM), (uint64_t)kBN, (uint64_t)kBN, 32,
                                 32))
            return cudaErrorInvalidValue;
    } else {
        tmP = tmY;                                   // not used
    }
    const int64_t units = pl.full_tiles + split_tiles * split;
    const int grid = units < num_sms() ? (int)units : num_sms();
    cudaError_t e = split > 1 ? launch_pdl(gemm_fp8_prefill_kernel<true>, dim3(grid), dim3(kThreads), kSmemBytes,
                                           st, tmX, tmW, tmY, tmP, prm)
                              : launch_pdl(gemm_fp8_prefill_kernel<false>, dim3(grid), dim3(kThreads), kSmemBytes,
                                           st, tmX, tmW, tmY, tmP, prm);
    if (e != cudaSuccess || split == 1) return e;
    const int64_t units8 = split_tiles * kBM * 32;
    return launch_pdl(prefill_splitk_reduce_kernel, dim3((unsigned)((units8 + 255) / 256)), dim3(256), 0, st,
                      (const float*)ws, M, N, prm.mtiles, prm.ntiles, prm.group_m, split, pl.full_tiles, units8, Y,
                      ldy);
}

// The dispatch below takes the prefill kernel for this shape (same rule).
static bool takes_prefill(int64_t M, int64_t N, int64_t K);

size_t gemm_fp8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0) return 0;
    if (!takes_prefill(M, N, K)) return decode_workspace_bytes(M, N, K);
    return prefill_ws_bytes(M, N, prefill_plan(M, N, K));
}

// Estimated prefill-kernel time in microseconds: a fixed 3 us plus the larger of
// the tensor-core time (waves of 128x256 work units, about 0.5 us per 128-wide K
// block) and the HBM time at 5.5 TB/s, plus, with split-K, the partial tiles'
// round trip through L2 and the reduction launch.
static double prefill_cost_us(int64_t M, int64_t N, int64_t K) {
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    const PrefillPlan pl = prefill_plan(M, N, K);
    const int64_t kb_all = K / 128, kb = (kb_all + pl.split - 1) / pl.split, sms = num_sms();
    // whole tiles in waves, then the split tiles' ranges (all of them when full_tiles = 0)
    const int64_t split_units = (tiles - pl.full_tiles) * pl.split;
    const double compute = (double)((pl.full_tiles + sms - 1) / sms) * (double)kb_all * 0.5 +
                           (double)((split_units + sms - 1) / sms) * (double)kb * 0.5;
    const double memory = (double)(N * K + M * K + 2 * M * N) / 5.5e6;
    const double reduce = pl.split > 1 ? 3.0 + (double)prefill_ws_bytes(M, N, pl) / 3e6 : 0.0;
    return 3.0 + (compute > memory ? compute : memory) + reduce;
}

// Up to 256 tokens both tcgen05 kernels apply: the split-K weight-streaming
// decode kernel wins for few, deep weight slabs, the 128x256-tile kernel once
// there are enough tiles (or enough K to split) to fill the GPU; the cheaper
// estimate is taken.  A K beyond the decode kernel's split limit (32768) goes to
// the 128x256-tile kernel at any M.
static bool takes_prefill(int64_t M, int64_t N, int64_t K) {
    if (M > 256 || !decode_supported(K)) return true;
    return prefill_cost_us(M, N, K) < decode_cost_us(M, N, K);
}

// The decode kernel runs a shape when the dispatch picks it and its split fits
// the workspace given (see decode_fits); otherwise the 128x256-tile kernel does.
static bool runs_decode(int64_t M, int64_t N, int64_t K, size_t ws_bytes) {
    return !takes_prefill(M, N, K) && decode_fits(M, N, K, ws_bytes);
}

int gemm_fp8_kernel_count(int64_t M, int64_t N, int64_t K, size_t ws_bytes) {
    if (M <= 0) return 0;
    if (runs_decode(M, N, K, ws_bytes)) return decode_kernel_count(M, N, K, ws_bytes);
    const PrefillPlan pl = prefill_plan(M, N, K);
    return pl.split > 1 && ws_bytes >= prefill_ws_bytes(M, N, pl) ? 2 : 1;
}

cudaError_t launch_gemm_fp8(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                            const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                            int64_t ldy, void* ws, size_t ws_bytes, bool weights_stable, cudaStream_t st) {
    if (runs_decode(M, N, K, ws_bytes))
        return launch_gemm_fp8_decode(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, ws, ws_bytes, weights_stable, st);
    return launch_gemm_fp8_prefill(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, ws, ws_bytes, st);
}

}  // namespace fp8rl
