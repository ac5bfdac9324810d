// gemm_int8_t256.cu -- exact INT8 W8A8 GEMM for mid-size batches (a few
// hundred tokens): weight blocks in tensor memory, 256-token tiles.
//
// Math (FlashRL write-up, Fig. 1, INT8 rollout): acc[m][n] = sum_k Xq[m][k] Wq[n][k]
// exactly (int32), y = bf16_rn((float(acc) * Xs[m]) * Ws[n]), no FMA.
//
// As in the small-batch kernel, the product runs on the fp16 tensor path
// (kind::f16) with the weights as the MMA's A operand in tensor memory: the
// converter warps turn each raw int8 weight block (128 rows x 128 K, TMA) into
// fp16 (exact: fp16(0x6400 | (v ^ 0x80)) - 1152 = v) and store it to TMEM, one
// weight row per lane.  What differs is the token side.  A kind::f16 MMA of
// 128 x N x 16 costs ~140 cycles for any N up to 128, so 64-token tiles spend
// four times the MMAs of one 256-token tile on the same weights.  Here the B
// operand is a 256-token tile of X, converted to fp16 once per call by a small
// launch and loaded by TMA (128-byte swizzle, two 64-wide K atoms per block):
// each weight block costs 8 MMAs of N = 256, for all 256 tokens.
//
// TMEM: two 128-column fp32 half accumulators, tokens 0..127 (half 0) and
// 128..255 (half 1) (token = column, weight row = lane), and four 64-column
// fp16 weight blocks.  A half collects one exact group of at most 2 K blocks
// (256 products, |sum| <= 256 * 127^2 < 2^22: every partial sum is an integer
// held exactly in fp32); its epilogue warps then move it into integer
// registers and release it.  The halves' groups are staggered by one block
// (half 0: blocks {0,1}, {2,3}, ...; half 1: {0}, {1,2}, {3,4}, ...), and each
// half has its own MMA issuer, so while one half is being moved the MMAs of
// the other keep the tensor pipe busy (an issuer's barrier waits drain only
// its own MMAs in flight).  The move is kept short: for an integer v with
// |v| < 2^22, v + 1.5 * 2^23 is exact and its bits are 0x4B400000 + v, so one
// add and one integer add per value replace the quarter-rate float -> int
// conversion; the offsets are taken off once at the end (32-bit wrap-around
// arithmetic).  With at most 128 tokens (one-half form) the token tiles are
// 128 rows, and the two issuers take alternate K blocks into the two
// accumulators, both for tokens 0..127; their int32 tiles are added at the end.
//
// Warps (512 threads): 0 = TMA of the weight blocks, 2 = TMA of the token
// tiles, 1 and 3 = MMA issuers of halves 0 and 1, 4..7 = converters, 8..15 =
// epilogue (warps 8..11 half 0, 12..15 half 1, one per TMEM lane quadrant).
// The int32 tile is transposed through shared memory for coalesced stores of
// Y (or of an int32 partial tile when the K range is split; a second launch
// adds the partials, exact in any order).
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {

using namespace sm100;

namespace {

constexpr int kTok = 256;                          // tokens per tile (the MMA's N)
constexpr int kRawW = 128 * 128;                   // raw int8 weight block
constexpr int kXAtom = kTok * 128;                 // 256 tokens x 64 fp16 K values
constexpr int kXStage = 2 * kXAtom;                // one 128-wide K block
constexpr int kWStages = 4, kXStages = 2, kSlots = 4;
constexpr int kGroupKb = 2;                        // K blocks per exact TMEM group
constexpr int kThreads = 512;
constexpr int kXOffset = kWStages * kRawW;
constexpr int kBarOffset = kXOffset + kXStages * kXStage;
constexpr int kSmemBytes = kBarOffset + 256 + 1024;
constexpr int kTmemCols = 512;                     // half accumulators 0..127, 128..255; weight slots from 256
constexpr int kLaunchRegs = 128, kLowRegs = 72, kEpiRegs = 184;
static_assert(kXOffset % 1024 == 0 && kXAtom % 1024 == 0, "swizzled tiles start on 1024-byte atoms");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kTok * 128 * 4 <= kBarOffset, "the int32 tile is transposed through the stage buffers");
static_assert(256 * kLowRegs + 256 * kEpiRegs <= kThreads * kLaunchRegs,
              "register split must fit the CTA's launch allocation");
static_assert(kGroupKb * 128 * 127 * 127 < (1 << 22), "group sums must stay exact, and within the magic-add range");
constexpr float kMagic = 12582912.0f;              // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;
static_assert((2 * kWStages + 2 * kSlots + 2 * kXStages + 4) * 8 + 8 <= 256, "barrier area");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kKernelInt8T256 = 6;

// kind::f16: A = B = fp16, D = fp32, K-major, M = 128 (weight rows), N = 128 (one half's tokens).
constexpr uint32_t kIdesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr int kHalfRows = 128 * 128;               // bytes of 128 token rows in one swizzled K atom

// Exact groups of half h: half 0 ends a group after every odd block, half 1
// after block 0 and every even block; both also end a group at the last block.
__device__ __forceinline__ bool group_first(int h, int it) { return h == 0 ? (it & 1) == 0 : (it == 0 || (it & 1)); }
__device__ __forceinline__ bool group_last(int h, int it, int nkb) {
    return it == nkb - 1 || (h == 0 ? (it & 1) == 1 : (it & 1) == 0);
}
__device__ __forceinline__ int group_index(int h, int it) { return h == 0 ? it >> 1 : (it + 1) >> 1; }
__device__ __forceinline__ int group_count(int h, int nkb) { return h == 0 ? (nkb + 1) >> 1 : (nkb >> 1) + 1; }

// One-half form (at most 128 tokens): issuer h takes the blocks it = h, h + 2,
// ... into its own accumulator (columns 128 h ..), all for tokens 0..127; its
// own blocks pair up into exact groups, so the two accumulators' drains
// alternate with the other issuer's MMAs.  The two int32 tiles are added at
// the end.
__device__ __forceinline__ bool oh_first(int it) { return ((it >> 1) & 1) == 0; }
__device__ __forceinline__ bool oh_last(int it, int nkb) { return ((it >> 1) & 1) == 1 || it + 2 >= nkb; }
__device__ __forceinline__ int oh_group(int it) { return it >> 2; }
__device__ __forceinline__ int oh_count(int h, int nkb) { return (((nkb - h + 1) >> 1) + 1) >> 1; }

struct T256Params {
    uint32_t* err;
    const float* Xs;    // [M]
    const float* Ws;    // [N]
    uint16_t* Y;        // [M][ldy]
    int32_t* acc;       // [M][N] or null
    int32_t* part;      // split > 1: [split][mtiles][N/128][256][128] int32
    int64_t M, N, ldy;
    int KB;             // K / 128
    int kb_per, split;  // K blocks per range, ranges
    int one_half;       // at most 128 tokens: 128-row token tiles, the issuers take alternate blocks
};

__device__ __forceinline__ void record_timeout(uint32_t* err, uint32_t site, volatile int* abort) {
    atomicCAS(err, 0u, (kKernelInt8T256 << 24) | (site << 16) | 1u);
    *abort = 1;
}

// 4 int8 codes (one 32-bit word) -> 4 fp16 values in two words (exact).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
    const uint32_t y = x ^ 0x80808080u;
    lo = __byte_perm(y, 0x64646464u, 0x4140);   // [y0, 0x64, y1, 0x64]
    hi = __byte_perm(y, 0x64646464u, 0x4342);   // [y2, 0x64, y3, 0x64]
    const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 a = __hsub2(*reinterpret_cast<__half2*>(&lo), off);
    __half2 b = __hsub2(*reinterpret_cast<__half2*>(&hi), off);
    lo = *reinterpret_cast<uint32_t*>(&a);
    hi = *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_int8_t256_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ T256Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
    // wfull[4] wempty[4] sfull[4] sempty[4] xfull[2] xempty[2] afull[2] aempty[2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kWStages + 2 * kSlots + 2 * kXStages + 4);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t wfull0 = smem_u32(bars), wempty0 = wfull0 + 8 * kWStages;
    const uint32_t sfull0 = wempty0 + 8 * kWStages, sempty0 = sfull0 + 8 * kSlots;
    const uint32_t xfull0 = sempty0 + 8 * kSlots, xempty0 = xfull0 + 8 * kXStages;
    const uint32_t afull0 = xempty0 + 8 * kXStages, aempty0 = afull0 + 16;   // per half
    const uint32_t warp = warp_id(), lane = lane_id();
    const int sp = blockIdx.x, mt = blockIdx.y, nt = blockIdx.z;     // K range, token tile, weight slab
    const int kb0 = sp * p.kb_per;
    const int nkb = min(p.KB, kb0 + p.kb_per) - kb0;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(wfull0 + 8 * s, 1);
            mbar_init(wempty0 + 8 * s, 4);           // the four converter warps
        }
        // a block is read by both issuers' MMAs, or in the one-half form by one
        const uint32_t halves = p.one_half ? 1 : 2;
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(sfull0 + 8 * s, 4);
            mbar_init(sempty0 + 8 * s, halves);
        }
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(xfull0 + 8 * s, 1);
            mbar_init(xempty0 + 8 * s, halves);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(afull0 + 8 * h, 1);
            mbar_init(aempty0 + 8 * h, 4);           // the half's four epilogue warps
        }
        *abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp < 8) {
        regs_dec<kLowRegs>();
        if (warp == 0 && lane == 0) {
            // ---------------- TMA: raw int8 weight blocks of this slab
            const uint64_t pol = policy_evict_first();
            int it = 0;
            for (; it < nkb; ++it) {
                const int s = it % kWStages;
                if (!mbar_wait_bounded(wempty0 + 8 * s, ((it / kWStages) & 1) ^ 1, abort, kWaitLimitNs)) {
                    record_timeout(p.err, 1, abort);
                    break;
                }
                mbar_arrive_expect_tx(wfull0 + 8 * s, kRawW);
                tma_load_2d(smem_u32(smem + s * kRawW), &tmW, wfull0 + 8 * s, (kb0 + it) * 128, nt * 128, pol);
            }
            if (*abort)   // let copies already in flight land before the CTA can exit
                for (int j = max(0, it - kWStages); j < it; ++j)
                    mbar_drain(wfull0 + 8 * (j % kWStages), (j / kWStages) & 1, kWaitLimitNs);
        } else if (warp == 2 && lane == 0) {
            // ---------------- TMA: fp16 token tiles (two 64-wide K atoms per block;
            // 128 rows of each atom in the one-half form)
            const uint64_t pol = policy_evict_last();
            const uint32_t bytes = p.one_half ? kXStage / 2 : kXStage;
            int it = 0;
            for (; it < nkb; ++it) {
                const int s = it % kXStages;
                if (!mbar_wait_bounded(xempty0 + 8 * s, ((it / kXStages) & 1) ^ 1, abort, kWaitLimitNs)) {
                    record_timeout(p.err, 2, abort);
                    break;
                }
                uint8_t* st = smem + kXOffset + s * kXStage;
                mbar_arrive_expect_tx(xfull0 + 8 * s, bytes);
                tma_load_2d(smem_u32(st), &tmX, xfull0 + 8 * s, (kb0 + it) * 128, mt * kTok, pol);
                tma_load_2d(smem_u32(st + kXAtom), &tmX, xfull0 + 8 * s, (kb0 + it) * 128 + 64, mt * kTok, pol);
            }
            if (*abort)
                for (int j = max(0, it - kXStages); j < it; ++j)
                    mbar_drain(xfull0 + 8 * (j % kXStages), (j / kXStages) & 1, kWaitLimitNs);
        } else if ((warp == 1 || warp == 3) && lane == 0) {
            // ---------------- MMA issuers, one per half: 8 x (M=128, N=128, K=16)
            // per K block into columns 128 h .. 128 h + 127 (one-half form: the
            // issuers' alternate blocks, both for tokens 0..127)
            const int h = warp == 1 ? 0 : 1;
            const bool oh = p.one_half != 0;
            const uint32_t d = tmem_base + 128 * h;
            for (int it = oh ? h : 0; it < nkb; it += oh ? 2 : 1) {
                const int s = it % kSlots, xs = it % kXStages;
                const bool first = oh ? oh_first(it) : group_first(h, it);
                const int gi = oh ? oh_group(it) : group_index(h, it);
                if (first && !mbar_wait_bounded(aempty0 + 8 * h, (gi & 1) ^ 1, abort, kWaitLimitNs)) {
                    record_timeout(p.err, 3, abort);
                    break;
                }
                if (!mbar_wait_bounded(sfull0 + 8 * s, (it / kSlots) & 1, abort, kWaitLimitNs) ||
                    !mbar_wait_bounded(xfull0 + 8 * xs, (it / kXStages) & 1, abort, kWaitLimitNs)) {
                    record_timeout(p.err, 4, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t a = tmem_base + 256 + s * 64;       // weight block: 64 columns
                const uint32_t xst = smem_u32(smem + kXOffset + xs * kXStage) + (oh ? 0 : h * kHalfRows);
#pragma unroll
                for (int k = 0; k < 8; ++k) {    // K = 16 fp16 = 8 TMEM columns / 32 bytes per step
                    const uint64_t b = umma_desc_k128_sw128(xst + (k >> 2) * kXAtom) + 2 * (k & 3);
                    mma_f16_tmem_a(d, a + 8 * k, b, kIdesc, (first && k == 0) ? 0u : 1u);
                }
                tc_commit(sempty0 + 8 * s);
                tc_commit(xempty0 + 8 * xs);
                if (oh ? oh_last(it, nkb) : group_last(h, it, nkb)) tc_commit(afull0 + 8 * h);
            }
        } else if (warp >= 4) {
            // ---------------- converters: weight row 32 * (warp % 4) + lane of each
            // raw block -> 64 TMEM columns of fp16 pairs (a warp may write only
            // its own quarter of the lanes)
            const int t = (int)(warp & 3) * 32 + (int)lane;
            const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + 256;
            for (int it = 0; it < nkb; ++it) {
                const int ws = it % kWStages, s = it % kSlots;
                const bool got = mbar_wait_bounded(wfull0 + 8 * ws, (it / kWStages) & 1, abort, kWaitLimitNs) &&
                                 mbar_wait_bounded(sempty0 + 8 * s, ((it / kSlots) & 1) ^ 1, abort, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) record_timeout(p.err, 5, abort);
                    break;
                }
                tc_fence_after();
                const uint32_t raw = smem_u32(smem + ws * kRawW) + t * 128;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int c = 4 * h + c4;        // 16-byte chunk: K codes 16c .. 16c + 15
                        const uint4 v = lds128(raw + ((c ^ (t & 7)) << 4));
                        i8x4_to_f16x4(v.x, r[8 * c4 + 0], r[8 * c4 + 1]);
                        i8x4_to_f16x4(v.y, r[8 * c4 + 2], r[8 * c4 + 3]);
                        i8x4_to_f16x4(v.z, r[8 * c4 + 4], r[8 * c4 + 5]);
                        i8x4_to_f16x4(v.w, r[8 * c4 + 6], r[8 * c4 + 7]);
                    }
                    tmem_st_32x32b_x32(lane_addr + s * 64 + 32 * h, r);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(sfull0 + 8 * s);
                    mbar_arrive(wempty0 + 8 * ws);
                }
            }
        }
    } else {
        regs_inc<kEpiRegs>();
        // ---------------- epilogue: exact int32 accumulation; weight row = lane,
        // tokens 128 h .. 128 h + 127 (half h)
        const int q = (int)(warp & 3), h = ((int)warp - 8) >> 2;
        const int n_local = 32 * q + (int)lane;
        const int ngroups = p.one_half ? oh_count(h, nkb) : group_count(h, nkb);
        uint32_t acc[128];                            // sum of (0x4B400000 + group sum) over the groups
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = 0;
        bool ok = true;
        for (int g = 0; g < ngroups; ++g) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(afull0 + 8 * h, g & 1, abort, kWaitLimitNs))) {
                if (lane == 0) record_timeout(p.err, 6, abort);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + h * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + 32 * c, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[32 * c + j] += __float_as_uint(__fadd_rn(__uint_as_float(r[j]), kMagic));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(aempty0 + 8 * h);
        }
        // Once both halves' last groups have been read, every MMA of this CTA
        // has completed (and with them every TMA copy and converter read): the
        // stage buffers are free, and the tile goes there as red[token][weight row].
        named_bar_sync(1, 256);                      // the eight epilogue warps
        int32_t* red = reinterpret_cast<int32_t*>(smem);
        const uint32_t bias = (uint32_t)ngroups * kMagicBits;
        if (!p.one_half) {
            if (ok) {
#pragma unroll
                for (int j = 0; j < 128; ++j) red[(h * 128 + j) * 128 + n_local] = (int32_t)(acc[j] - bias);
            }
        } else {
            // both accumulators hold tokens 0..127: half 1's tile, then half 0 adds its own
            if (ok && h == 1) {
#pragma unroll
                for (int j = 0; j < 128; ++j) red[j * 128 + n_local] = (int32_t)(acc[j] - bias);
            }
            named_bar_sync(1, 256);
            if (ok && h == 0) {
#pragma unroll
                for (int j = 0; j < 128; ++j) red[j * 128 + n_local] += (int32_t)(acc[j] - bias);
            }
        }
        named_bar_sync(1, 256);
        if (!*abort) {
            // thread -> (token, 8 weight rows), 16-byte accesses
            const int et = (int)threadIdx.x - 256;
            const int64_t m0 = (int64_t)mt * kTok;
            const int valid = (int)(p.M - m0 < kTok ? p.M - m0 : kTok);
            for (int c = et; c < valid * 16; c += 256) {
                const int m = c >> 4, n8 = c & 15;
                const int4 a = *reinterpret_cast<const int4*>(red + m * 128 + n8 * 8);
                const int4 b = *reinterpret_cast<const int4*>(red + m * 128 + n8 * 8 + 4);
                if (p.split > 1) {
                    int4* dst = reinterpret_cast<int4*>(
                        p.part + ((((int64_t)sp * gridDim.y + mt) * gridDim.z + nt) * kTok + m) * 128 + n8 * 8);
                    dst[0] = a;
                    dst[1] = b;
                    continue;
                }
                const int32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                const int64_t mg = m0 + m, n0 = (int64_t)nt * 128 + n8 * 8;
                const float xs = __ldg(p.Xs + mg);
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(__int2float_rn(v[e]), xs), __ldg(p.Ws + n0 + e));
                *reinterpret_cast<uint4*>(p.Y + mg * p.ldy + n0) =
                    make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                               pack_bf16x2(y[6], y[7]));
                if (p.acc) {                         // 8-byte stores: the ABI guarantees 8-byte alignment
                    int2* a2 = reinterpret_cast<int2*>(p.acc + mg * p.N + n0);
#pragma unroll
                    for (int e = 0; e < 4; ++e) a2[e] = make_int2(v[2 * e], v[2 * e + 1]);
                }
            }
        }
    }

    __syncwarp();   // warps whose lane 0 alone ran a loop reconverge first
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Split K: one thread per (token, 8 weight rows) adds the ranges' int32
// partials (exact in any order) and writes Y and acc.
__global__ void __launch_bounds__(256)
t256_reduce_kernel(const int32_t* __restrict__ part, const float* __restrict__ Xs, const float* __restrict__ Ws,
                   int64_t M, int64_t N, int mtiles, int split, uint16_t* __restrict__ Y, int64_t ldy,
                   int32_t* __restrict__ acc) {
    pdl_wait_then_release();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t slabs = N / 128;
    const int64_t per_tile = (int64_t)kTok * 16;
    if (t >= (int64_t)mtiles * slabs * per_tile) return;
    const int64_t tile = t / per_tile;                  // mt * slabs + nt
    const int r = (int)(t - tile * per_tile);
    const int m = r >> 4, n8 = r & 15;
    const int mt = (int)(tile / slabs);
    const int64_t nt = tile - (int64_t)mt * slabs;
    const int64_t mg = (int64_t)mt * kTok + m;
    if (mg >= M) return;
    const int64_t stride = (int64_t)mtiles * slabs * kTok * 128;     // one range's partials
    const int32_t* src = part + (tile * kTok + m) * 128 + n8 * 8;
    int32_t s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int k = 0; k < split; ++k) {
        const int4 a = *reinterpret_cast<const int4*>(src + k * stride);
        const int4 b = *reinterpret_cast<const int4*>(src + k * stride + 4);
        s[0] += a.x; s[1] += a.y; s[2] += a.z; s[3] += a.w;
        s[4] += b.x; s[5] += b.y; s[6] += b.z; s[7] += b.w;
    }
    const int64_t n0 = nt * 128 + n8 * 8;
    const float xs = __ldg(Xs + mg);
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(__int2float_rn(s[e]), xs), __ldg(Ws + n0 + e));
    *reinterpret_cast<uint4*>(Y + mg * ldy + n0) =
        make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
    if (acc) {
        int2* a2 = reinterpret_cast<int2*>(acc + mg * N + n0);
#pragma unroll
        for (int e = 0; e < 4; ++e) a2[e] = make_int2(s[2 * e], s[2 * e + 1]);
    }
}

// The register split (setmaxnreg) assumes exactly kLaunchRegs registers per
// thread at launch; any other build is refused.  Checked (and the shared memory
// attribute set) once per device.
int t256_ready(int dev) {
    static int checked[64] = {};   // 0 unknown, 1 ok, -1 refused
    if (dev < 0 || dev >= 64) return -1;
    if (checked[dev] == 0) {
        cudaFuncAttributes fa;
        checked[dev] = (cudaFuncGetAttributes(&fa, gemm_int8_t256_kernel) == cudaSuccess &&
                        fa.numRegs == kLaunchRegs &&
                        cudaFuncSetAttribute(gemm_int8_t256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes) == cudaSuccess)
                           ? 1
                           : -1;
        cudaGetLastError();
    }
    return checked[dev];
}

// K ranges: one CTA per (range, token tile, weight slab), at most one CTA per
// SM.  Estimated time in microseconds, fitted to sweeps of splits 1..8 over
// the Qwen2.5-32B shapes at M = 96, 128 and 256 on GB300 (within 11% of all 96
// points; it picks the fastest split for each of the twelve shape and size
// pairs):
//   5.2 + rounds * (3.9 + t_block * K blocks per range)
//       + (split: 1.9 + 0.055 * partial tiles * tokens per tile / 256)
// with t_block = 0.9 for two token halves and 0.54 for the one-half form
// (rounds of CTAs over the SMs; each split CTA writes an int32 partial of its
// tile's live tokens, which the reduction launch reads back).
struct T256Plan {
    int split, kb_per;
};

T256Plan t256_plan(int64_t M, int64_t N, int64_t K) {
    const int KB = (int)(K / 128);
    const int64_t mtiles = (M + kTok - 1) / kTok;
    const int64_t ctas1 = mtiles * (N / 128);
    const double rows = (double)M / (double)mtiles;     // live tokens per tile, on average
    const int64_t sms = num_sms();
    T256Plan best{1, KB};
    double best_cost = 1e30;
    for (int s = 1; s <= 8 && s <= KB; ++s) {
        const int per = (KB + s - 1) / s;
        if ((int64_t)(s - 1) * per >= KB) continue;
        const int64_t rounds = (ctas1 * s + sms - 1) / sms;
        double cost = 5.2 + (double)rounds * (3.9 + (M <= 128 ? 0.54 : 0.9) * per);
        if (s > 1) cost += 1.9 + 0.055 * (double)(ctas1 * s) * rows / kTok;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = T256Plan{s, per};
        }
    }
    return best;
}

}  // namespace

// fp16 copy of X (M x K x 2 bytes, 16-byte aligned), then the split's partials.
size_t int8_t256_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    const T256Plan pl = t256_plan(M, N, K);
    const size_t x16 = ((size_t)M * K * 2 + 15) / 16 * 16;
    const size_t parts = pl.split > 1 ? (size_t)pl.split * ((M + kTok - 1) / kTok) * N * kTok * sizeof(int32_t) : 0;
    return x16 + parts;
}

int int8_t256_kernel_count(int64_t M, int64_t N, int64_t K) { return t256_plan(M, N, K).split > 1 ? 3 : 2; }

cudaError_t launch_gemm_int8_t256(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                                  int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy, int32_t* acc,
                                  void* ws, cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (t256_ready(dev) != 1) return cudaErrorInvalidDeviceFunction;
    const T256Plan pl = t256_plan(M, N, K);
    uint16_t* X16 = static_cast<uint16_t*>(ws);
    int32_t* part = pl.split > 1 ? reinterpret_cast<int32_t*>(
                                       static_cast<uint8_t*>(ws) + ((size_t)M * K * 2 + 15) / 16 * 16)
                                 : nullptr;
    CUtensorMap tmW, tmX;
    if (!make_tmap_u8(&tmW, Wq, (uint64_t)N, (uint64_t)K, (uint64_t)K, 128)) return cudaErrorInvalidValue;
    const int one_half = M <= 128 ? 1 : 0;             // one token tile with at most 128 live rows
    if (!make_tmap_f16_load(&tmX, X16, (uint64_t)M, (uint64_t)K, one_half ? kTok / 2 : kTok))
        return cudaErrorInvalidValue;
    uint32_t* err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    cudaError_t e = launch_int8_to_f16(Xq, M * K, X16, st);
    if (e != cudaSuccess) return e;
    const int mtiles = (int)((M + kTok - 1) / kTok);
    T256Params prm{err, Xs, Ws, Y, acc, part, M, N, ldy, (int)(K / 128), pl.kb_per, pl.split, one_half};
    e = launch_pdl(gemm_int8_t256_kernel, dim3((unsigned)pl.split, (unsigned)mtiles, (unsigned)(N / 128)),
                   dim3(kThreads), kSmemBytes, st, tmW, tmX, prm);
    if (e != cudaSuccess || pl.split == 1) return e;
    const int64_t threads = (int64_t)mtiles * (N / 128) * kTok * 16;
    return launch_pdl(t256_reduce_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st,
                      (const int32_t*)part, Xs, Ws, M, N, mtiles, pl.split, Y, ldy, acc);
}

}  // namespace fp8rl
