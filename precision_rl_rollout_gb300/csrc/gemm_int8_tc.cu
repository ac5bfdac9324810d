// gemm_int8_tc.cu -- exact INT8 W8A8 GEMM on the 5th-generation tensor cores.
//
// FlashRL write-up (Fig. 1, INT8 rollout): acc[m][n] = sum_k Xq[m][k] Wq[n][k]
// exactly (int32), y = bf16_rn((float(acc) * Xs[m]) * Ws[n]).
//
// sm_103a has no tcgen05 INT8 MMA kind and its legacy INT8 warp MMA is slow, so
// the integer product runs on the fp16 tensor path with exact arithmetic:
//   * every int8 code v (|v| <= 127) is an exact fp16; the conversion is the
//     offset-binary identity fp16(0x6400 | (v ^ 0x80)) = 1152 + v followed by
//     one packed fp16 subtraction of 1152 (exact: the result needs <= 8 bits);
//   * each product is an integer below 2^14, exact in the fp32 accumulator;
//   * a TMEM accumulator collects at most 2 K blocks (256 products per output,
//     |sum| <= 256 * 127^2 < 2^22) so every partial sum is an integer well
//     inside fp32's 24-bit significand and no rounding can occur; it is then
//     moved to 32-bit integer registers exactly (see the epilogue).
// The bit-exact parity tests against the int64 CPU reference include the
// extreme case of every code at +-127.
//
// Layout (swap-AB, as the FP8 decode kernel): the MMA's M side is 128 weight
// rows, its N side a tile of MT tokens; each CTA streams one 128-row weight
// slab.  Warp 0 issues TMA (raw int8 tiles, 128-byte swizzle), warps 1 and 14
// the MMAs of alternate K blocks (each into its own accumulators), warps 2-9
// (two groups, alternate K blocks) convert raw tiles to fp16, warps 10-13
// promote and hold the integer accumulators.  The converted weight
// block goes to tensor memory, where the MMA reads its A operand (one weight
// row per TMEM lane, K packed along the columns); only the small token tile
// is written back to shared memory (UMMA K-major 128-byte-swizzle layout, two
// 64-wide atoms per K block).  Shared memory then carries about 56 KB per
// 16 KB weight block instead of 120 KB: with the fp16 weights in shared memory
// its bandwidth, not HBM, set the pace.  Split-K CTAs of one slab form a
// cluster and add their int32 partials through distributed shared memory.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {

using namespace sm100;

namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kKernelInt8 = 3;
constexpr int kGroupKb = 4;   // K blocks per promotion group, two per MMA issuer (exactness bound)

struct Int8Params {
    uint32_t* err;
    const float* Xs;   // [M]
    const float* Ws;   // [N]
    uint16_t* Y;       // [M][ldy]
    int32_t* acc;      // [M][N] or null
    int64_t M, N, ldy;
    int KB;
    int kb_per_split;
    int split;
    int mtiles;        // token tiles
    int items;         // split == 1: (token tile, slab) work items, taken by CTAs in turn
};

template <int MT>
struct I8Cfg {
    static_assert(MT == 16 || MT == 32 || MT == 64, "token tile");
    static constexpr int kThreads = 480;                       // 15 warps
    static constexpr int kRawW = 128 * 128, kRawX = MT * 128;  // int8 tiles
    static constexpr int kRawStage = kRawW + kRawX;
    // TMEM: four accumulator buffers of MT columns at 0 (two MMA issuers x two
    // alternating groups), then as many fp16 weight blocks (128 lanes x 64
    // columns each) as the rest holds, from column kTmemA
    static constexpr int kTmemA = 4 * MT < 64 ? 64 : 4 * MT;
    static constexpr int kTmemCols = 512;
    static constexpr int kCvtStages = (kTmemCols - kTmemA) / 64;   // fp16 weight blocks = token stages
    static constexpr int kCvtStage = 2 * MT * 128;                 // fp16 token tile: two 64-wide atoms
    // raw int8 stages fill the rest of ~220 KB: the weight bytes in flight per
    // SM keep the HBM stream going
    static constexpr int kRawStages = MT == 16 ? 10 : MT == 32 ? 8 : 5;
    static constexpr int kCvtOffset = kRawStages * kRawStage;
    static constexpr int kRedOffset = kCvtOffset + kCvtStages * kCvtStage;   // int32 tile red[MT][128]
    static constexpr int kBarOffset = kRedOffset + MT * 128 * 4;
    static constexpr int kSmemBytes = kBarOffset + 512 + 1024;
    static_assert(4 * MT <= kTmemA && kTmemA + 64 * kCvtStages <= kTmemCols, "TMEM layout");
    static_assert(kCvtStages >= kGroupKb, "a group's blocks must fit in TMEM at once");
    static_assert((2 * kRawStages + 2 * kCvtStages + 6) * 8 + 8 <= 512, "barrier area");
    static constexpr int kChunk = MT >= 32 ? 32 : 16;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ void record_timeout(uint32_t* err, uint32_t site, volatile int* abort) {
    atomicCAS(err, 0u, (kKernelInt8 << 24) | (site << 16) | 1u);
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

// Chunk c (16 codes) of row r of a raw int8 tile (128 B rows, 128-byte
// swizzle) -> its two 16-byte pieces of the fp16 operand tile (two atoms of 64
// K, each 128 B per row, 128-byte swizzle).
__device__ __forceinline__ void convert_chunk(const uint8_t* raw, uint8_t* cvt, int r, int c, int atom_bytes) {
    const int sw = r & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(raw + r * 128 + ((c ^ sw) << 4));
    uint4 o0, o1;
    i8x4_to_f16x4(v.x, o0.x, o0.y);
    i8x4_to_f16x4(v.y, o0.z, o0.w);
    i8x4_to_f16x4(v.z, o1.x, o1.y);
    i8x4_to_f16x4(v.w, o1.z, o1.w);
    uint8_t* dst = cvt + (c >> 2) * atom_bytes + r * 128;
    const int j = 2 * (c & 3);
    *reinterpret_cast<uint4*>(dst + ((j ^ sw) << 4)) = o0;
    *reinterpret_cast<uint4*>(dst + (((j + 1) ^ sw) << 4)) = o1;
}

// Y[m][n0 .. n0+7] = bf16((float(acc) * Xs[m]) * Ws[n]) and the accumulators if asked.
__device__ __forceinline__ void store_out8(const Int8Params& p, int64_t mg, int64_t n0, const int32_t (&s)[8]) {
    const float xs = p.Xs[mg];
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(__int2float_rn(s[e]), xs), p.Ws[n0 + e]);
    uint4 o;
    o.x = pack_bf16x2(y[0], y[1]);
    o.y = pack_bf16x2(y[2], y[3]);
    o.z = pack_bf16x2(y[4], y[5]);
    o.w = pack_bf16x2(y[6], y[7]);
    *reinterpret_cast<uint4*>(p.Y + mg * p.ldy + n0) = o;
    if (p.acc) {                                 // 8-byte stores: the ABI guarantees 8-byte alignment
        int2* a2 = reinterpret_cast<int2*>(p.acc + mg * p.N + n0);
        a2[0] = make_int2(s[0], s[1]);
        a2[1] = make_int2(s[2], s[3]);
        a2[2] = make_int2(s[4], s[5]);
        a2[3] = make_int2(s[6], s[7]);
    }
}

// Two modes.  Split K (p.split > 1): CTA (split rank, token tile, slab) in a
// cluster of the split CTAs, which add their int32 tiles through distributed
// shared memory.  No split: a persistent grid; CTA c takes the work items
// (token tile, slab) c, c + gridDim.x, ... with every pipeline counter running
// on across items, so the next item's loads and MMAs overlap this item's
// promotion and stores (done by the epilogue warps alone).
template <int MT>
__global__ void __launch_bounds__(I8Cfg<MT>::kThreads, 1)
gemm_int8_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ Int8Params p) {
    using C = I8Cfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    // raw_full[R], raw_empty[R], cvt_full[V], cvt_empty[V], tfull[4] (issuer x buffer), tempty[2]
    constexpr int R = C::kRawStages, V = C::kCvtStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * R + 2 * V + 6);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t rfull0 = smem_u32(bars), rempty0 = smem_u32(bars + R);
    const uint32_t cfull0 = smem_u32(bars + 2 * R), cempty0 = smem_u32(bars + 2 * R + V);
    const uint32_t tfull0 = smem_u32(bars + 2 * R + 2 * V), tempty0 = smem_u32(bars + 2 * R + 2 * V + 4);
    int32_t* red = reinterpret_cast<int32_t*>(smem + C::kRedOffset);

    const uint32_t warp = warp_id(), lane = lane_id();
    const bool persist = p.split == 1;
    const int split_idx = persist ? 0 : (int)blockIdx.x;
    const int w_begin = persist ? (int)blockIdx.x : 0, w_end = persist ? p.items : 1;
    const int w_step = persist ? (int)gridDim.x : 1;
    const int kb0 = split_idx * p.kb_per_split;
    const int nkb = min(p.KB, kb0 + p.kb_per_split) - kb0;
    const int ngroups = (nkb + kGroupKb - 1) / kGroupKb;
#define ITEM_MT(w) (persist ? (w) % p.mtiles : (int)blockIdx.y)
#define ITEM_NT(w) (persist ? (w) / p.mtiles : (int)blockIdx.z)

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(rfull0 + 8 * s, 1);
            mbar_init(rempty0 + 8 * s, 4);           // the four converter warps
        }
        for (int s = 0; s < V; ++s) {
            mbar_init(cfull0 + 8 * s, 4);
            mbar_init(cempty0 + 8 * s, 1);
        }
        for (int b = 0; b < 4; ++b) mbar_init(tfull0 + 8 * b, 1);
        for (int b = 0; b < 2; ++b) mbar_init(tempty0 + 8 * b, 4);   // the four epilogue warps
        *abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ---------------- TMA producer: raw int8 tiles
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            int b = 0;                                   // blocks issued, over all items
            bool ok = true;
            for (int w = w_begin; ok && w < w_end; w += w_step) {
                const int mt = ITEM_MT(w), nt = ITEM_NT(w);
                for (int it = 0; it < nkb; ++it, ++b) {
                    const int s = b % R;
                    const uint32_t ph = (b / R) & 1;
                    if (!mbar_wait_bounded(rempty0 + 8 * s, ph ^ 1, abort, kWaitLimitNs)) {
                        record_timeout(p.err, 1, abort);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * C::kRawStage;
                    mbar_arrive_expect_tx(rfull0 + 8 * s, C::kRawStage);
                    tma_load_2d(smem_u32(st), &tmW, rfull0 + 8 * s, (kb0 + it) * 128, nt * 128, pol_w);
                    tma_load_2d(smem_u32(st + C::kRawW), &tmX, rfull0 + 8 * s, (kb0 + it) * 128, mt * MT, pol_x);
                }
            }
            if (*abort)   // let copies already in flight land before the CTA can exit
                for (int j = max(0, b - R); j < b; ++j)
                    mbar_drain(rfull0 + 8 * (j % R), (j / R) & 1, kWaitLimitNs);
        }
    } else if (warp == 1 || warp == 14) {
        // ---------------- MMA issuers: 8 x (M=128, N=MT, K=16) fp16 MMAs per K
        // block.  Two threads take alternate blocks, each into its own pair of
        // accumulator buffers: a thread's barrier wait returns only after its
        // own MMAs in flight have completed, so with one issuer every block
        // drained the tensor pipe, while the other thread's MMAs keep it busy.
        // Group g (blocks 4g .. 4g+3 of an item) gives each issuer two blocks.
        if (lane == 0) {
            constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(MT >> 3) << 17) | ((128u >> 4) << 24);  // f16 x f16 -> f32
            const int me = warp == 1 ? 0 : 1;
            int b0 = 0, G0 = 0;                          // blocks and groups of earlier items
            bool ok = true;
            for (int w = w_begin; ok && w < w_end; w += w_step) {
                for (int g = 0; ok && g < ngroups; ++g) {
                    const int G = G0 + g;
                    const uint32_t buf = G & 1, bph = (G >> 1) & 1;
                    const int g_beg = g * kGroupKb, g_end = min(nkb, g_beg + kGroupKb);
                    if (g_beg + me >= g_end) {
                        // issuer 1 in a one-block group: no MMAs, but its barrier
                        // phases stay in step with the epilogue's
                        if (!mbar_wait_bounded(tempty0 + 8 * buf, bph ^ 1, abort, kWaitLimitNs)) {
                            record_timeout(p.err, 3, abort);
                            ok = false;
                            break;
                        }
                        mbar_arrive(tfull0 + 8 * (2 * me + buf));
                        continue;
                    }
                    for (int it = g_beg + me; it < g_end; it += 2) {
                        const bool first = it == g_beg + me, last = it + 2 >= g_end;
                        const int bb = b0 + it, s = bb % V;
                        const uint32_t ph = (bb / V) & 1;
                        if (!mbar_wait_bounded(cfull0 + 8 * s, ph, abort, kWaitLimitNs)) {
                            record_timeout(p.err, 2, abort);
                            ok = false;
                            break;
                        }
                        if (first && !mbar_wait_bounded(tempty0 + 8 * buf, bph ^ 1, abort, kWaitLimitNs)) {
                            record_timeout(p.err, 3, abort);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint8_t* st = smem + C::kCvtOffset + s * C::kCvtStage;
                        const uint32_t d = tmem_base + (2 * me + buf) * MT;
                        const uint32_t a = tmem_base + C::kTmemA + s * 64;     // weight block s: 64 columns
#pragma unroll
                        for (int k = 0; k < 8; ++k) {    // K = 16 fp16 = 8 TMEM columns / 32 bytes per step
                            const uint64_t bd = umma_desc_k128_sw128(smem_u32(st + (k >> 2) * (MT * 128))) + 2 * (k & 3);
                            mma_f16_tmem_a(d, a + 8 * k, bd, idesc, (first && k == 0) ? 0u : 1u);
                        }
                        tc_commit(cempty0 + 8 * s);
                        if (last) tc_commit(tfull0 + 8 * (2 * me + buf));
                    }
                }
                b0 += nkb;
                G0 += ngroups;
            }
        }
    } else if (warp < 10) {
        // ---------------- converters: raw int8 -> fp16.  Two groups of four
        // warps take alternate blocks (block b goes to TMEM weight block and
        // token stage b % V), so two blocks are converted concurrently.  A warp
        // may write only its own quarter of the TMEM lanes, so its thread
        // converts weight row 32 * (warp % 4) + lane.
        const int grp = (warp - 2) >> 2;
        const int t = (int)(warp & 3) * 32 + lane;  // 0..127
        const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + C::kTmemA;
        const int nblocks = nkb * ((w_end - w_begin + w_step - 1) / w_step);
        for (int b = grp; b < nblocks; b += 2) {
            const int rs = b % R, cs = b % V;
            const uint32_t rph = (b / R) & 1, cph = (b / V) & 1;
            const bool got = mbar_wait_bounded(rfull0 + 8 * rs, rph, abort, kWaitLimitNs) &&
                             mbar_wait_bounded(cempty0 + 8 * cs, cph ^ 1, abort, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) record_timeout(p.err, 4, abort);
                break;
            }
            const uint8_t* raw = smem + rs * C::kRawStage;
            uint8_t* cvt = smem + C::kCvtOffset + cs * C::kCvtStage;
            // weight row t: 128 codes -> 64 columns of fp16 pairs in TMEM
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int c = 4 * h + c4;        // 16-byte chunk: K codes 16c .. 16c + 15
                    const uint4 v = *reinterpret_cast<const uint4*>(raw + t * 128 + ((c ^ (t & 7)) << 4));
                    i8x4_to_f16x4(v.x, r[8 * c4 + 0], r[8 * c4 + 1]);
                    i8x4_to_f16x4(v.y, r[8 * c4 + 2], r[8 * c4 + 3]);
                    i8x4_to_f16x4(v.z, r[8 * c4 + 4], r[8 * c4 + 5]);
                    i8x4_to_f16x4(v.w, r[8 * c4 + 6], r[8 * c4 + 7]);
                }
                tmem_st_32x32b_x32(lane_addr + cs * 64 + 32 * h, r);
            }
            // the token tile (MT rows x 8 chunks of 16 codes), spread over all 128
            // threads of the group so that no warp does twice the work
#pragma unroll
            for (int i = t; i < MT * 8; i += 128) convert_chunk(raw + C::kRawW, cvt, i >> 3, i & 7, MT * 128);
            tmem_wait_st();
            fence_proxy_async_smem();                // generic writes -> tensor-core reads
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(cfull0 + 8 * cs);
                mbar_arrive(rempty0 + 8 * rs);
            }
        }
    } else {
        // ---------------- epilogue: exact promotion into integer registers.  Per
        // group, each issuer's accumulator holds at most two blocks' products
        // (256 per output, |sum| <= 256 * 127^2 < 2^22), so v + 1.5 * 2^23 is
        // exact and its bits are 0x4B400000 + v: one add and one integer add per
        // value; the offsets come off at the end of the item (32-bit wrap-around).
        const int q = warp & 3;
        const int n_local = 32 * q + lane;
        const int et = (int)threadIdx.x - 320;      // 0..127 over the four epilogue warps
        int G0 = 0;
        for (int w = w_begin; w < w_end; w += w_step) {
            const int mt = ITEM_MT(w), nt = ITEM_NT(w);
            uint32_t acc[MT];
#pragma unroll
            for (int j = 0; j < MT; ++j) acc[j] = 0;
            uint32_t reads = 0;
            bool ok = true;
            for (int g = 0; g < ngroups; ++g) {
                const int G = G0 + g;
                const uint32_t buf = G & 1, bph = (G >> 1) & 1;
                const int nblk = min(nkb - g * kGroupKb, kGroupKb);
                // both issuers arrive once per group (issuer 1 without MMAs in a one-block group)
                const bool got = mbar_wait_bounded(tfull0 + 8 * buf, bph, abort, kWaitLimitNs) &&
                                 mbar_wait_bounded(tfull0 + 8 * (2 + buf), bph, abort, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0) record_timeout(p.err, 5, abort);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int nacc = nblk >= 2 ? 2 : 1;
                for (int i = 0; i < nacc; ++i) {
                    const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (2 * i + buf) * MT;
#pragma unroll
                    for (int ch = 0; ch < MT / C::kChunk; ++ch) {
                        uint32_t r[C::kChunk];
                        if constexpr (C::kChunk == 32) tmem_ld_32x32b_x32(taddr + ch * 32, r);
                        else tmem_ld_32x32b_x16(taddr + ch * 16, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < C::kChunk; ++j)
                            acc[ch * C::kChunk + j] += __float_as_uint(__fadd_rn(__uint_as_float(r[j]), 12582912.0f));
                    }
                    ++reads;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
            }
            G0 += ngroups;
            if (ok) {
                const uint32_t bias = reads * 0x4B400000u;
#pragma unroll
                for (int j = 0; j < MT; ++j) red[j * 128 + n_local] = (int32_t)(acc[j] - bias);
            }
            if (!persist) break;                         // split K: the whole CTA adds and stores below
            // persistent: the four epilogue warps store this item's tile while
            // the other warps go on with the next item
            named_bar_sync(1, 128);
            if (ok && !*abort) {
                const int64_t m_tile0 = (int64_t)mt * MT;
                const int valid_m = (int)(p.M - m_tile0 < MT ? p.M - m_tile0 : MT);
                for (int c = et; c < valid_m * 16; c += 128) {
                    const int m = c >> 4, n8 = c & 15;
                    const int4 u0 = *reinterpret_cast<const int4*>(red + m * 128 + n8 * 8);
                    const int4 u1 = *reinterpret_cast<const int4*>(red + m * 128 + n8 * 8 + 4);
                    const int32_t v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                    store_out8(p, m_tile0 + m, (int64_t)nt * 128 + n8 * 8, v);
                }
            }
            // red is free again, and every epilogue thread takes the same decision
            if (bar_red_or(1, 128, !ok || *abort)) break;
        }
    }
#undef ITEM_MT
#undef ITEM_NT

    // ---------------- split K: reduction over the cluster (int32: exact) and stores
    // (warps 0, 1 and 14 ran their loops on lane 0 alone: reconverged before the
    // .aligned barriers, which every lane of a warp must execute together)
    __syncwarp();
    tc_fence_before();
    if (!persist) {
        cluster_sync_all();
        const int mt = blockIdx.y, nt = blockIdx.z;
        const int64_t m_tile0 = (int64_t)mt * MT;
        const int valid_m = (int)(p.M - m_tile0 < MT ? p.M - m_tile0 : MT);
        const int total = valid_m * 16;
        const int per = (total + p.split - 1) / p.split;
        const int begin = split_idx * per, end = min(total, begin + per);
        const uint32_t red_addr = smem_u32(red);
        for (int c = begin + (int)threadIdx.x; c < end && !*abort; c += C::kThreads) {
            const int m = c >> 4, n8 = c & 15;
            const uint32_t off = (uint32_t)(m * 128 + n8 * 8) * 4u;
            int32_t sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int rk = 0; rk < p.split; ++rk) {
                const uint32_t a = map_to_rank(red_addr + off, (uint32_t)rk);
                const float4 v0 = ld_cluster_v4(a), v1 = ld_cluster_v4(a + 16);
                sum[0] += __float_as_int(v0.x); sum[1] += __float_as_int(v0.y);
                sum[2] += __float_as_int(v0.z); sum[3] += __float_as_int(v0.w);
                sum[4] += __float_as_int(v1.x); sum[5] += __float_as_int(v1.y);
                sum[6] += __float_as_int(v1.z); sum[7] += __float_as_int(v1.w);
            }
            store_out8(p, m_tile0 + m, (int64_t)nt * 128 + n8 * 8, sum);
        }
        __syncwarp();
        cluster_sync_all();
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// Split-K factor: fill the GPU (one CTA per SM) without starving each CTA.
int choose_split_i8(int64_t tiles, int KB) {
    const int sms = num_sms();
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= 8 && s <= KB; ++s) {
        const int per = (KB + s - 1) / s;
        if ((int64_t)(s - 1) * per >= KB) continue;
        const int64_t ctas = tiles * s;
        const int64_t busiest = (ctas + sms - 1) / sms;
        const double cost = 3.0 * busiest + 0.55 * busiest * per + 1.0 * s;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

template <int MT>
cudaError_t launch_i8_mt(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws, int64_t M,
                         int64_t N, int64_t K, uint16_t* Y, int64_t ldy, int32_t* acc, cudaStream_t st) {
    using C = I8Cfg<MT>;
    CUtensorMap tmW, tmX;
    if (!make_tmap_u8(&tmW, Wq, (uint64_t)N, (uint64_t)K, (uint64_t)K, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tmX, Xq, (uint64_t)M, (uint64_t)K, (uint64_t)K, MT)) return cudaErrorInvalidValue;
    const int KB = (int)(K / 128);
    const int64_t mtiles = (M + MT - 1) / MT;
    const int split = choose_split_i8((N / 128) * mtiles, KB);
    const int per = (KB + split - 1) / split;
    uint32_t* err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    const int64_t items = mtiles * (N / 128);
    if (items > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    Int8Params prm{err, Xs, Ws, Y, acc, M, N, ldy, KB, per, split, (int)mtiles, (int)items};
    auto kern = gemm_int8_tc_kernel<MT>;
    static bool attr_set[64] = {};     // the attribute belongs to the device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    // no split: a persistent grid of at most one CTA per SM over the work items
    cfg.gridDim = split > 1 ? dim3((unsigned)split, (unsigned)mtiles, (unsigned)(N / 128))
                            : dim3((unsigned)(items < num_sms() ? items : num_sms()));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmX, prm);
}

}  // namespace

cudaError_t launch_gemm_int8_tc(const int8_t* Xq, const float* Xs, const int8_t* Wq, const float* Ws,
                                int64_t M, int64_t N, int64_t K, uint16_t* Y, int64_t ldy, int32_t* acc,
                                cudaStream_t st) {
    if (M <= 16) return launch_i8_mt<16>(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, acc, st);
    if (M <= 32) return launch_i8_mt<32>(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, acc, st);
    return launch_i8_mt<64>(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, acc, st);
}

// Dispatch (32B shapes measured at M = 64 .. 4096, graphs over weight copies):
//  - up to 64 tokens: this kernel (64-token tiles at most, weights in TMEM);
//  - 65 .. 256 tokens, and up to 512 on layers of at least 2^27 weights: the
//    256-token kernel (an fp16 copy of X and, for a K split, int32 partials in
//    the workspace);
//  - larger batches with enough tiles: fp16 copies of X and W and the
//    128 x 256 tile kernel;
//  - anything else, or too little workspace for the chosen path: this kernel.
static bool int8_t256_applies(int64_t M, int64_t N, int64_t K) {
    return M > 64 && (M <= 256 || (M <= 512 && N * K >= (int64_t(1) << 27)));
}
size_t gemm_int8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (int8_t256_applies(M, N, K)) return int8_t256_workspace_bytes(M, N, K);
    return int8_prefill_workspace_bytes(M, N, K);
}
int gemm_int8_kernel_count(int64_t M, int64_t N, int64_t K, size_t ws_bytes) {
    if (M <= 0) return 0;
    const size_t need = gemm_int8_workspace_bytes(M, N, K);
    if (need == 0 || ws_bytes < need) return 1;
    return int8_t256_applies(M, N, K) ? int8_t256_kernel_count(M, N, K) : int8_prefill_kernel_count(M, N, K);
}
cudaError_t launch_gemm_int8(const int8_t* Xq, const float* Xs, const int8_t* Wq,
                             const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                             int64_t ldy, int32_t* acc, void* ws, size_t ws_bytes, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    const size_t need = gemm_int8_workspace_bytes(M, N, K);
    if (need > 0 && ws != nullptr && ws_bytes >= need) {
        if (int8_t256_applies(M, N, K)) return launch_gemm_int8_t256(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, acc, ws, st);
        return launch_gemm_int8_prefill(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, acc, ws, st);
    }
    return launch_gemm_int8_tc(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, acc, st);
}

}  // namespace fp8rl
