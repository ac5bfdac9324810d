// gemm_fp8_tc.cu -- block-scaled FP8 W8A8 GEMMs on the 5th-generation tensor
// cores (tcgen05) of sm_103a, fed by TMA.
//
// Math (FP8-RL, Abstract, contribution (i): FP8 W8A8 linear layers with
// blockwise scales; block 128x128 for W and 1x128 for X in this library):
//   Y[m][n] = bf16( sum_kb Xs[kb][m] * Ws[n/128][kb] * P_kb[m][n] ),
//   P_kb[m][n] = sum_{k in block kb} e4m3(Xq[m][k]) * e4m3(Wq[n][k])   (fp32)
// The block scales are arbitrary fp32 values (amax/448), which the tensor
// core's own block-scaled MMA kinds (power-of-two / E4M3 scales on 16- or
// 32-element blocks) cannot express, so each 128-wide K block is one MMA
// group into its own TMEM buffer and the epilogue warps promote it into fp32
// registers with that block's scale product.  Several TMEM buffers (two in
// the prefill kernel, four to eight here) let the MMAs of later blocks run
// while the epilogue promotes earlier ones.
//
// Decode kernel (small M, HBM-bound; the long-tail rollout batches of "Taming
// the Long Tail" (ASPLOS'26 blog), section 3.2 roofline and section 4.3.1):
// swap-AB -- the MMA's M side is 128 weight rows, its N side the (padded)
// tokens -- so each CTA streams a disjoint 128-row weight slab exactly once.
// The split-K CTAs of one slab add their fp32 partials in a fixed order
// (deterministic) in one of three ways: in a cluster, through distributed
// shared memory or through the caller's workspace in L2; or, without a
// cluster, through the workspace and a second launch (see the plan below).
//
// Grouped form (mixture-of-experts layers; FP8-RL, Abstract: dense and MoE
// models): the weights of E experts are stacked as [E*N][K] and the token rows
// are grouped by expert, expert e owning rows offsets[e] .. offsets[e+1]-1.
// Grid z runs over (expert, 128-row slab); each CTA reads its expert's token
// range after the dependency wait (the router may have just written it), and
// a CTA whose token tile is empty streams nothing.  With more such items than
// CTAs fit at once, the persistent kernel below takes them in turn instead.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace fp8rl {

using namespace sm100;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
enum : uint32_t { kKernelDecode = 1 };

__device__ __forceinline__ void record_timeout(uint32_t* err, uint32_t kernel, uint32_t site,
                                               volatile int* abort) {
    atomicCAS(err, 0u, (kernel << 24) | (site << 16) | 1u);
    *abort = 1;
}

// ------------------------------------------------------------------ decode kernel

struct DecodeParams {
    uint32_t* err;     // device error word (bounded waits)
    const float* Xs;   // [KB][M]
    const float* Ws;   // [N/128][KB]
    uint16_t* Y;       // [M][ldy]
    int64_t M, ldy;
    int KB;            // K / 128
    int kb_per_split;  // K blocks per split-K CTA
    int split;         // CTAs per cluster (split-K factor)
    // grouped form only (offs == nullptr: one dense GEMM; M is then the token count)
    const int32_t* offs;   // [E+1] first token row of each expert, device memory
    int ntiles;            // 128-row weight slabs per expert (N / 128)
    int64_t tok_bound;     // token rows per expert the grid covers (M tiles * MT)
    // split-K exchange (kXchg*): through distributed shared memory (part ==
    // nullptr), or through fp32 partial tiles [slabs * M tiles * split][MT][128]
    // in the workspace, added by a second launch or, in a cluster, by the CTAs
    // themselves after one cluster barrier
    float* part;
    int xmode;
    // weight tiles of the first pipeline stages are loaded before the
    // dependency wait (the caller guarantees that the kernel immediately
    // preceding this one in the stream did not write Wq)
    int early_w;
};

enum : int { kXchgSmem = 0, kXchgReduceLaunch = 1, kXchgClusterMem = 2 };

template <int MT>
struct DecodeCfg {
    static_assert(MT == 16 || MT == 32 || MT == 64 || MT == 128, "token tile");
    static constexpr int kEpiWarps = MT >= 128 ? 8 : 4;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kCols = MT / (kEpiWarps / 4);         // TMEM columns per epilogue thread
    static constexpr int kStageBytes = 16384 + MT * 128;       // W tile + X tile
    // MT <= 64: two CTAs per SM (2 x (smem + 1 KB reserved) <= 228 KB); larger: one.
    static constexpr int kStages = MT == 16 ? 6 : MT == 32 ? 5 : MT == 64 ? 4 : 5;
    static constexpr int kMaxKbPerSplit = 32;                     // K blocks per split-K CTA
    static constexpr int kMaxSplit = 8;                           // portable cluster size
    static constexpr int kPrefetchKb = 8;                         // weight blocks sent to L2 early
    static constexpr int kScaleBytes = kMaxKbPerSplit * MT * 4;   // per-block scale products
    // TMEM accumulator buffers: enough that the MMAs of several K blocks are in
    // flight while the epilogue drains earlier ones (a block's four dependent
    // MMAs take far longer to complete than to issue); the columns of two
    // co-resident CTAs (MT <= 64) or of one (MT = 128) fill at most 512
    static constexpr int kTmemBufs = MT <= 32 ? 8 : 4;
    static constexpr int kTmemCols = kTmemBufs * MT;
    static constexpr int kMinBlocks = MT <= 64 ? 2 : 1;             // CTAs per SM the registers allow
    static constexpr int kChunk = kCols >= 32 ? 32 : 16;               // TMEM load width
    static constexpr int kGroup = kCols < 64 ? kCols : 64;             // columns per tcgen05.wait::ld
    static constexpr int kBarOffset = kStages * kStageBytes + kScaleBytes;
    static constexpr int kSmemBytes = kBarOffset + 256 + 1024;   // barriers + alignment slack
    static_assert((2 * kStages + 2 * kTmemBufs) * 8 + 8 <= 256, "barrier area");
    static_assert(kTmemCols >= 32 && (kTmemCols & (kTmemCols - 1)) == 0 &&
                      kTmemCols * (MT <= 64 ? 2 : 1) <= 512, "TMEM allocation");
    static_assert(MT * 128 * 4 <= kStages * kStageBytes, "reduction buffer must fit the stage area");
};

// ---- pieces shared by the decode kernels (the per-slab kernel and the
// persistent kernel below run the same roles on the same shared-memory layout)

// One thread: the stage barriers full/empty, the TMEM buffer barriers
// tfull/tempty (one arrival per epilogue warp) and the abort flag.
template <int MT>
__device__ __forceinline__ void decode_init_barriers(uint32_t full0, uint32_t empty0, uint32_t tfull0,
                                                     uint32_t tempty0, volatile int* abort) {
    using C = DecodeCfg<MT>;
    for (int s = 0; s < C::kStages; ++s) {
        mbar_init(full0 + 8 * s, 1);
        mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < C::kTmemBufs; ++b) {
        mbar_init(tfull0 + 8 * b, 1);
        mbar_init(tempty0 + 8 * b, C::kEpiWarps);
    }
    *abort = 0;
    fence_mbar_init();
}

// MMA thread: one 128-wide K block of the stage at `st` (weight tile, then the
// token tile 16 KB on) into TMEM columns d .. d + MT - 1, as 4 MMAs of K = 32;
// the stage and the buffer are then handed on (released / filled) when the
// MMAs complete.
template <int MT>
__device__ __forceinline__ void decode_mma_block(const uint8_t* st, uint32_t d, uint32_t empty_bar,
                                                 uint32_t tfull_bar) {
    constexpr uint32_t idesc = idesc_e4m3_f32(128, MT);
    tc_fence_after();
    const uint64_t a = umma_desc_k128_sw128(smem_u32(st));
    const uint64_t b = umma_desc_k128_sw128(smem_u32(st + 16384));
#pragma unroll
    for (int k = 0; k < 4; ++k)     // +32 B along K = +2 in the descriptors' address field
        mma_f8f6f4(d, a + 2 * k, b + 2 * k, idesc, k > 0 ? 1u : 0u);
    tc_commit(empty_bar);
    tc_commit(tfull_bar);
}

// Epilogue threads (thread et of kThreadsFill): the per-block scale products
// c[b][j] = ws[b] * xs[b * M + j] for b < nblk, j < MT (0 for j >= rows).  The
// loads are issued in batches of 8 so that their latencies overlap.
template <int MT, int kThreadsFill>
__device__ __forceinline__ void decode_fill_scales(float* cscale, const float* __restrict__ ws,
                                                   const float* __restrict__ xs, int64_t M, int nblk,
                                                   int64_t rows, int et) {
    const int total = nblk * MT;
    for (int base = et; base < total; base += 8 * kThreadsFill) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = base + u * kThreadsFill;
            const int b = idx / MT, j = idx - b * MT;
            v[u] = (idx < total && j < rows) ? __ldg(ws + b) * __ldg(xs + (int64_t)b * M + j) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (base + u * kThreadsFill < total) cscale[base + u * kThreadsFill] = v[u];
    }
}

// Epilogue warp, after the buffer's tfull wait: this thread's kCols columns of
// one K block (TMEM address taddr) into registers, all in flight under one
// wait; the buffer is released as soon as they are there, before the
// promotion, so the next MMAs into it need not wait for the FMAs.  Then
// acc += block * c (c: this thread's scale products of the block).
template <int MT>
__device__ __forceinline__ void decode_promote_block(uint64_t (&acc)[DecodeCfg<MT>::kCols / 2], uint32_t taddr,
                                                     const float* cs, uint32_t tempty_bar, uint32_t lane) {
    using C = DecodeCfg<MT>;
    static_assert(C::kCols == C::kGroup, "one load group per block");
    tc_fence_after();
    uint32_t r[C::kGroup];
#pragma unroll
    for (int ch = 0; ch < C::kGroup / C::kChunk; ++ch) {
        uint32_t(&rc)[C::kChunk] = *reinterpret_cast<uint32_t(*)[C::kChunk]>(r + ch * C::kChunk);
        const uint32_t a = taddr + ch * C::kChunk;
        if constexpr (C::kChunk == 32) tmem_ld_32x32b_x32(a, rc);
        else tmem_ld_32x32b_x16(a, rc);
    }
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tempty_bar);
    const uint64_t* cs2 = reinterpret_cast<const uint64_t*>(cs);
#pragma unroll
    for (int j = 0; j < C::kGroup / 2; ++j)
        fma_f32x2(acc[j], f32x2_pack(r[2 * j], r[2 * j + 1]), cs2[j]);
}

template <int MT>
__global__ void __launch_bounds__(DecodeCfg<MT>::kThreads, DecodeCfg<MT>::kMinBlocks)
gemm_fp8_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ DecodeParams p) {
    using C = DecodeCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* cscale = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    // bars: full[S], empty[S], tfull[B], tempty[B] (B TMEM buffers)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 2 * C::kTmemBufs);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + C::kStages);
    const uint32_t tfull0 = smem_u32(bars + 2 * C::kStages);
    const uint32_t tempty0 = smem_u32(bars + 2 * C::kStages + C::kTmemBufs);

    const uint32_t warp = warp_id(), lane = lane_id();
    const int split_idx = blockIdx.x;                  // rank within the cluster
    const int mt = blockIdx.y;                        // M tiles of one slab are adjacent
    const int z = blockIdx.z;                         // weight slab: rows 128 z .. of [E*N][K]
    const int nt = p.offs ? z % p.ntiles : z;         // output column block
    const int kb0 = split_idx * p.kb_per_split;
    const int nkb = min(p.KB, kb0 + p.kb_per_split) - kb0;   // >= 1 by construction

    if (warp == 0 && lane == 0) {
        decode_init_barriers<MT>(full0, empty0, tfull0, tempty0, abort);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
        // The first weight blocks of this slab start moving into L2 while the
        // previous kernel of the stream finishes (the weights are read-only
        // here; an L2 prefetch cannot return stale data).
        // (grouped form: not before the expert is known to have tokens here)
        const int pre0 = (p.early_w && (p.M - (int64_t)mt * MT) > 0) ? min(nkb, C::kStages) : 0;
        const int npf = p.offs ? 0 : min(nkb - pre0, C::kPrefetchKb);
        for (int it = 0; it < npf; ++it) tma_prefetch_l2_2d(&tmW, (kb0 + pre0 + it) * 128, z * 128);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // With early_w (dense form only), the weight tiles of the first stages
    // start moving into shared memory now.  A kernel is launched only after
    // the one before it has passed its own dependency wait, so everything
    // earlier in the stream than the immediately preceding kernel has
    // completed; that kernel not writing Wq is the caller's guarantee.
    const int pre = (p.early_w && (p.M - (int64_t)mt * MT) > 0) ? min(nkb, C::kStages) : 0;
    if (pre > 0 && warp == 0 && lane == 0) {
        const uint64_t pol_w = policy_evict_first();
        for (int it = 0; it < pre; ++it) {
            mbar_arrive_expect_tx(full0 + 8 * it, C::kStageBytes);   // the token tile joins after the wait
            tma_load_2d(smem_u32(smem + it * C::kStageBytes), &tmW, full0 + 8 * it, (kb0 + it) * 128, z * 128,
                        pol_w);
        }
    }
    // Programmatic dependent launch: the set-up above overlapped the tail of the
    // previous kernel in the stream; nothing else in global memory is touched
    // before it has completed.  The next kernel may then be scheduled (it
    // waits the same way).
    grid_dependency_wait();
    grid_launch_dependents();

    // this CTA's token rows: row0 .. row0 + rows - 1 (rows <= 0: nothing to do;
    // the decision is the same for every CTA of a cluster)
    int64_t row0 = (int64_t)mt * MT, rows = p.M - row0;
    if (p.offs) {
        const int e = z / p.ntiles;
        int64_t b = p.offs[e], en = p.offs[e + 1];
        b = b < 0 ? 0 : (b > p.M ? p.M : b);
        en = en < b ? b : (en > p.M ? p.M : en);
        row0 = b + (int64_t)mt * MT;
        rows = en - row0;
        if (mt == 0 && split_idx == 0 && nt == 0 && threadIdx.x == 0 && en - b > p.tok_bound)
            atomicCAS(p.err, 0u, (kKernelDecode << 24) | (7u << 16) | 2u);   // tokens beyond the bound
    }
    const int nrun = rows > 0 ? nkb : 0;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            int it = 0;
            // stages whose weight tile is already on its way: only the token tile
            for (const int pre_run = nrun > 0 ? pre : 0; it < pre_run; ++it)
                tma_load_2d(smem_u32(smem + it * C::kStageBytes + 16384), &tmX, full0 + 8 * it, (kb0 + it) * 128,
                            (int32_t)row0, pol_x);
            for (; it < nrun; ++it) {
                const int s = it % C::kStages;
                const uint32_t ph = (it / C::kStages) & 1;
                if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, kWaitLimitNs)) {
                    record_timeout(p.err, kKernelDecode, 1, abort);
                    break;
                }
                uint8_t* st = smem + s * C::kStageBytes;
                mbar_arrive_expect_tx(full0 + 8 * s, C::kStageBytes);
                tma_load_2d(smem_u32(st), &tmW, full0 + 8 * s, (kb0 + it) * 128, z * 128, pol_w);
                tma_load_2d(smem_u32(st + 16384), &tmX, full0 + 8 * s, (kb0 + it) * 128, (int32_t)row0, pol_x);
            }
            if (*abort) {   // let copies already in flight land before the CTA can exit
                for (int j = max(0, it - C::kStages); j < it; ++j)
                    mbar_drain(full0 + 8 * (j % C::kStages), (j / C::kStages) & 1, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (one thread)
        if (lane == 0) {
            for (int it = 0; it < nrun; ++it) {
                const int s = it % C::kStages;
                const uint32_t ph = (it / C::kStages) & 1;
                const int buf = it % C::kTmemBufs;
                const uint32_t bph = (it / C::kTmemBufs) & 1;
                if (!mbar_wait_bounded(full0 + 8 * s, ph, abort, kWaitLimitNs)) {
                    record_timeout(p.err, kKernelDecode, 2, abort);
                    break;
                }
                if (!mbar_wait_bounded(tempty0 + 8 * buf, bph ^ 1, abort, kWaitLimitNs)) {
                    record_timeout(p.err, kKernelDecode, 3, abort);
                    break;
                }
                decode_mma_block<MT>(smem + s * C::kStageBytes, tmem_base + buf * MT, empty0 + 8 * s,
                                     tfull0 + 8 * buf);
            }
        }
    } else {
        // ---------------- epilogue: per-block promotion in fp32 registers
        const int e = warp - 2;
        const int q = warp & 3;                          // TMEM lane quadrant of this warp
        const int colbase = (e >> 2) * C::kCols;         // token columns of this thread
        const int n_local = 32 * q + lane;               // weight row within the slab
        const int et = e * 32 + lane;
        // c[it][j] = Ws[z][kb0+it] * Xs[kb0+it][row0 + j]
        decode_fill_scales<MT, C::kEpiWarps * 32>(cscale, p.Ws + (int64_t)z * p.KB + kb0,
                                                  p.Xs + (int64_t)kb0 * p.M + row0, p.M, nrun, rows, et);
        named_bar_sync(1, C::kEpiWarps * 32);

        uint64_t acc[C::kCols / 2];              // fp32 accumulators as packed pairs
#pragma unroll
        for (int j = 0; j < C::kCols / 2; ++j) acc[j] = 0ull;
        for (int it = 0; it < nrun; ++it) {
            const int buf = it % C::kTmemBufs;
            const uint32_t bph = (it / C::kTmemBufs) & 1;
            // the verdict is made warp-uniform: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(tfull0 + 8 * buf, bph, abort, kWaitLimitNs))) {
                if (lane == 0) record_timeout(p.err, kKernelDecode, 4, abort);
                break;
            }
            decode_promote_block<MT>(acc, tmem_base + ((uint32_t)(32 * q) << 16) + buf * MT + colbase,
                                     cscale + it * MT + colbase, tempty0 + 8 * buf, lane);
        }
        // every MMA of this CTA has completed: the stage area is free for the
        // transposed partial tile red[m][n_local]
        float* red = reinterpret_cast<float*>(smem);
#pragma unroll
        for (int j = 0; j < C::kCols / 2; ++j) {
            const float2 v = f32x2_unpack(acc[j]);
            red[(colbase + 2 * j) * 128 + n_local] = v.x;
            red[(colbase + 2 * j + 1) * 128 + n_local] = v.y;
        }
    }

    // ---------------- split-K: the split CTAs' partials are added in rank order,
    // then rounded to bf16 once.  Warps 0 and 1 ran their producer / MMA loop on
    // lane 0 alone: the warp is reconverged before the .aligned barriers below,
    // which every lane of a warp must execute together.
    __syncwarp();
    tc_fence_before();
    const bool clustered = p.split > 1 && p.xmode != kXchgReduceLaunch;
    // self-check: the launch shape the exchange relies on (`split` CTAs per slab
    // along x; in a cluster, ranked by blockIdx.x); a mismatch is recorded and
    // the exchange skipped
    const bool shape_ok = gridDim.x == (unsigned)p.split &&
                          (!clustered || (cluster_nctarank() == (uint32_t)p.split &&
                                          cluster_ctarank() == (uint32_t)split_idx));
    if (!shape_ok && threadIdx.x == 0) atomicCAS(p.err, 0u, (kKernelDecode << 24) | (8u << 16) | 2u);
    const int64_t ncols = (int64_t)(p.offs ? p.ntiles : (int)gridDim.z) * 128;   // output columns
    const int valid_m = rows <= 0 ? 0 : (int)(rows < MT ? rows : MT);
    // this slab's first partial slot in the workspace (memory exchanges)
    float* const slot0 = p.part != nullptr ? p.part + ((int64_t)z * gridDim.y + mt) * p.split * (MT * 128) : nullptr;
    if (slot0 != nullptr) {
        // this CTA's partial rows to its slot: coalesced 16-byte stores of red[m][0..127]
        __syncthreads();
        if (shape_ok) {
            float4* dst = reinterpret_cast<float4*>(slot0 + (int64_t)split_idx * (MT * 128));
            const float4* src = reinterpret_cast<const float4*>(smem);
            for (int i = threadIdx.x; i < valid_m * 32; i += C::kThreads) dst[i] = src[i];
        }
    }
    if (p.xmode != kXchgReduceLaunch) {
        // every rank's partial is complete (and, through memory, visible to the
        // cluster) after this barrier; each CTA then adds 1/split of the chunks
        if (clustered) cluster_sync_all(); else __syncthreads();
        if (shape_ok) {
            const int total = valid_m * 16;                   // chunks of 8 output channels
            const int per = (total + p.split - 1) / p.split;
            const int begin = split_idx * per, end = min(total, begin + per);
            const uint32_t red_addr = smem_u32(smem);
            for (int c = begin + (int)threadIdx.x; c < end; c += C::kThreads) {
                const int m = c >> 4, n8 = c & 15;
                const uint32_t off = (uint32_t)(m * 128 + n8 * 8) * 4u;
                float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (clustered) {
                    // every rank's loads are in flight before the first add: one
                    // round trip per chunk, not one per rank
                    float4 v[C::kMaxSplit][2];
                    if (p.xmode == kXchgClusterMem) {
                        const float* src = slot0 + m * 128 + n8 * 8;
#pragma unroll
                        for (int r = 0; r < C::kMaxSplit; ++r)
                            if (r < p.split) {
                                const float4* q4 = reinterpret_cast<const float4*>(src + (int64_t)r * (MT * 128));
                                v[r][0] = __ldcg(q4);
                                v[r][1] = __ldcg(q4 + 1);
                            }
                    } else {
#pragma unroll
                        for (int r = 0; r < C::kMaxSplit; ++r)
                            if (r < p.split) {
                                const uint32_t a = map_to_rank(red_addr + off, (uint32_t)r);
                                v[r][0] = ld_cluster_v4(a);
                                v[r][1] = ld_cluster_v4(a + 16);
                            }
                    }
#pragma unroll
                    for (int r = 0; r < C::kMaxSplit; ++r)   // fixed order: deterministic
                        if (r < p.split) {
                            s[0] += v[r][0].x; s[1] += v[r][0].y; s[2] += v[r][0].z; s[3] += v[r][0].w;
                            s[4] += v[r][1].x; s[5] += v[r][1].y; s[6] += v[r][1].z; s[7] += v[r][1].w;
                        }
                } else {
                    const float4* l = reinterpret_cast<const float4*>(smem + off);
                    const float4 v0 = l[0], v1 = l[1];
                    s[0] += v0.x; s[1] += v0.y; s[2] += v0.z; s[3] += v0.w;
                    s[4] += v1.x; s[5] += v1.y; s[6] += v1.z; s[7] += v1.w;
                }
                uint4 o;
                o.x = pack_bf16x2(s[0], s[1]);
                o.y = pack_bf16x2(s[2], s[3]);
                o.z = pack_bf16x2(s[4], s[5]);
                o.w = pack_bf16x2(s[6], s[7]);
                const int64_t col = (int64_t)nt * 128 + n8 * 8;
                if (row0 + m < p.M && col + 8 <= ncols)        // self-check of the output index
                    *reinterpret_cast<uint4*>(p.Y + (row0 + m) * p.ldy + col) = o;
                else
                    atomicCAS(p.err, 0u, (kKernelDecode << 24) | (9u << 16) | 2u);
            }
        }
    }
    // a CTA whose shared memory its peers read stays until they are done
    __syncwarp();
    if (clustered && p.xmode == kXchgSmem) cluster_sync_all(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// Split-K without a cluster: one thread per (slab, token row, 8 channels) adds
// the split partials in order and rounds to bf16 once.
template <int MT>
__global__ void __launch_bounds__(256)
decode_splitk_reduce_kernel(const float* __restrict__ part, int64_t M, int mtiles, int split, int64_t units,
                            uint16_t* __restrict__ Y, int64_t ldy) {
    pdl_wait_then_release();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= units) return;
    const int64_t tile = t / (MT * 16);
    const int rem = (int)(t - tile * (MT * 16));
    const int m = rem >> 4, c8 = rem & 15;
    const int64_t z = tile / mtiles, mt = tile - z * mtiles;
    const int64_t row = mt * MT + m;
    if (row >= M) return;
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const float* base = part + ((tile * split) * MT + m) * 128 + c8 * 8;
    const int64_t stride = (int64_t)MT * 128;          // one split's partial tile
    for (int sp0 = 0; sp0 < split; sp0 += 4) {
        // four splits' loads in flight, then added in split order (deterministic)
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
    *reinterpret_cast<uint4*>(Y + row * ldy + z * 128 + c8 * 8) = o;
}

// ------------------------------------------------------------------ persistent decode kernel
//
// For shapes with several waves of (weight slab, token tile) items and K not
// split (the grouped form's experts: thousands of short items).  One CTA per
// SM slot takes items w = blockIdx.x, w + gridDim.x, ...; item w is token tile
// w % mtiles of weight slab w / mtiles.  The TMA ring and the TMEM buffers run
// on from one item to the next, so each CTA pays its set-up once and the
// weight blocks of the next item stream while the epilogue finishes the
// current one; the epilogue writes Y straight from its registers.  The roles
// and the per-block promotion are the shared pieces above.
struct PersistParams {
    uint32_t* err;
    const float* Xs;       // [KB][M]
    const float* Ws;       // [slabs][KB]
    uint16_t* Y;           // [M][ldy]
    int64_t M, ldy;
    int KB;                // K / 128 (at most kMaxKbPerSplit)
    int items, mtiles;     // items = mtiles x weight slabs
    const int32_t* offs;   // grouped form: [E+1] first token row of each expert (nullptr: dense)
    int ntiles;            // 128-row slabs per expert (grouped) or per matrix (dense)
    int64_t tok_bound;     // grouped form: token rows per expert the items cover
};

// Token rows of item (mt, z): row0 .. row0 + rows - 1 (rows <= 0: none).  The
// same for every thread that asks (offs is not written while the kernel runs).
template <int MT>
__device__ __forceinline__ void persist_item_rows(const PersistParams& p, int mt, int z, int64_t& row0,
                                                  int64_t& rows) {
    row0 = (int64_t)mt * MT;
    rows = p.M - row0;
    if (p.offs) {
        const int e = z / p.ntiles;
        int64_t b = p.offs[e], en = p.offs[e + 1];
        b = b < 0 ? 0 : (b > p.M ? p.M : b);
        en = en < b ? b : (en > p.M ? p.M : en);
        row0 = b + (int64_t)mt * MT;
        rows = en - row0;
    }
}

template <int MT>
__global__ void __launch_bounds__(DecodeCfg<MT>::kThreads, DecodeCfg<MT>::kMinBlocks)
gemm_fp8_decode_persistent_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                                  const __grid_constant__ PersistParams p) {
    using C = DecodeCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* cscale = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 2 * C::kTmemBufs);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + C::kStages);
    const uint32_t tfull0 = smem_u32(bars + 2 * C::kStages);
    const uint32_t tempty0 = smem_u32(bars + 2 * C::kStages + C::kTmemBufs);
    const uint32_t warp = warp_id(), lane = lane_id();
    const int KB = p.KB;

    if (warp == 0 && lane == 0) {
        decode_init_barriers<MT>(full0, empty0, tfull0, tempty0, abort);
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // nothing in global memory is read before the previous kernel has completed
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ---------------- TMA producer: one pipeline counter over all items
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            uint32_t it = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < p.items; w += gridDim.x) {
                const int mt = w % p.mtiles, z = w / p.mtiles;
                int64_t row0, rows;
                persist_item_rows<MT>(p, mt, z, row0, rows);
                if (rows <= 0) continue;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % C::kStages;
                    const uint32_t ph = (it / C::kStages) & 1;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1, abort, kWaitLimitNs)) {
                        record_timeout(p.err, kKernelDecode, 11, abort);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + s * C::kStageBytes;
                    mbar_arrive_expect_tx(full0 + 8 * s, C::kStageBytes);
                    tma_load_2d(smem_u32(st), &tmW, full0 + 8 * s, kb * 128, z * 128, pol_w);
                    tma_load_2d(smem_u32(st + 16384), &tmX, full0 + 8 * s, kb * 128, (int32_t)row0, pol_x);
                }
            }
            if (*abort) {   // let copies already in flight land before the CTA can exit
                for (uint32_t j = it > (uint32_t)C::kStages ? it - C::kStages : 0; j < it; ++j)
                    mbar_drain(full0 + 8 * (j % C::kStages), (j / C::kStages) & 1, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (one thread), the same counter
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < p.items; w += gridDim.x) {
                const int mt = w % p.mtiles, z = w / p.mtiles;
                int64_t row0, rows;
                persist_item_rows<MT>(p, mt, z, row0, rows);
                if (rows <= 0) continue;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % C::kStages;
                    const uint32_t ph = (it / C::kStages) & 1;
                    const int buf = it % C::kTmemBufs;
                    const uint32_t bph = (it / C::kTmemBufs) & 1;
                    if (!mbar_wait_bounded(full0 + 8 * s, ph, abort, kWaitLimitNs)) {
                        record_timeout(p.err, kKernelDecode, 12, abort);
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_bounded(tempty0 + 8 * buf, bph ^ 1, abort, kWaitLimitNs)) {
                        record_timeout(p.err, kKernelDecode, 13, abort);
                        ok = false;
                        break;
                    }
                    decode_mma_block<MT>(smem + s * C::kStageBytes, tmem_base + buf * MT, empty0 + 8 * s,
                                         tfull0 + 8 * buf);
                }
            }
        }
    } else {
        // ---------------- epilogue: per-block promotion, then Y from registers
        constexpr int kEpiThreads = C::kEpiWarps * 32;
        const int e = warp - 2;
        const int q = warp & 3;                          // TMEM lane quadrant of this warp
        const int colbase = (e >> 2) * C::kCols;         // token columns of this thread
        const int n_local = 32 * q + lane;               // weight row within the slab
        const int et = e * 32 + lane;
        uint32_t it = 0;
        for (int w = blockIdx.x; w < p.items; w += gridDim.x) {
            const int mt = w % p.mtiles, z = w / p.mtiles;
            const int nt = p.offs ? z % p.ntiles : z;
            int64_t row0, rows;
            persist_item_rows<MT>(p, mt, z, row0, rows);
            if (rows <= 0) continue;
            if (p.offs && et == 0 && mt == 0 && nt == 0) {
                const int ex = z / p.ntiles;
                if ((int64_t)p.offs[ex + 1] - p.offs[ex] > p.tok_bound)
                    atomicCAS(p.err, 0u, (kKernelDecode << 24) | (7u << 16) | 2u);   // tokens beyond the bound
            }
            // every epilogue thread is done with the previous item's scales, and
            // all of them take the same decision on going on
            if (bar_red_or(1, kEpiThreads, *abort != 0)) break;
            // c[kb][j] = Ws[z][kb] * Xs[kb][row0 + j]
            decode_fill_scales<MT, kEpiThreads>(cscale, p.Ws + (int64_t)z * KB, p.Xs + row0, p.M, KB, rows, et);
            named_bar_sync(1, kEpiThreads);
            uint64_t acc[C::kCols / 2];
#pragma unroll
            for (int j = 0; j < C::kCols / 2; ++j) acc[j] = 0ull;
            bool ok = true;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int buf = it % C::kTmemBufs;
                const uint32_t bph = (it / C::kTmemBufs) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(tfull0 + 8 * buf, bph, abort, kWaitLimitNs))) {
                    if (lane == 0) record_timeout(p.err, kKernelDecode, 14, abort);
                    ok = false;
                    break;
                }
                decode_promote_block<MT>(acc, tmem_base + ((uint32_t)(32 * q) << 16) + buf * MT + colbase,
                                         cscale + kb * MT + colbase, tempty0 + 8 * buf, lane);
            }
            if (!ok) continue;   // the abort flag is set: the next item's barrier ends the loop
            // Y[row0 + colbase + j][nt * 128 + n_local]: per token column, a warp
            // writes 32 consecutive channels (64 bytes)
            const int valid = rows < MT ? (int)rows : MT;
            uint16_t* yp = p.Y + (row0 + colbase) * p.ldy + (int64_t)nt * 128 + n_local;
#pragma unroll
            for (int j = 0; j < C::kCols / 2; ++j) {
                const float2 v = f32x2_unpack(acc[j]);
                const uint32_t pk = pack_bf16x2(v.x, v.y);
                if (colbase + 2 * j < valid) yp[(int64_t)(2 * j) * p.ldy] = (uint16_t)(pk & 0xffffu);
                if (colbase + 2 * j + 1 < valid) yp[(int64_t)(2 * j + 1) * p.ldy] = (uint16_t)(pk >> 16);
            }
        }
    }
    __syncwarp();   // warps 0 and 1 ran their loops on lane 0 alone
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// Split-K factor for `tiles` weight slabs of KB blocks and a token tile of MT.
// Cost model fitted to a sweep of cluster splits 1..8 over the Qwen2.5-7B/32B
// decode shapes at M = 1..256 on GB300.  It underrates larger splits on short
// weight streams (up to 20% slower than the best split at M = 1), so the dense
// GEMM's plan below uses it only as a fallback; it also prices the decode
// kernel for the decode/prefill dispatch and sets the grouped form's split:
//   cost = 3 * waves + busiest-SM CTAs * blocks per CTA * (0.4 + 0.3 MT/128) + 2 * split * MT/128
// (microseconds, roughly): a fixed cost per wave of CTAs, the weight stream of
// the busiest SM (heavier per block for wide token tiles), and the cluster
// reduction, which grows with the split and the tile.
static int choose_split(int64_t tiles, int KB, int MT, int max_kb_per_split, double* cost_out = nullptr) {
    const int sms = num_sms();
    const int per_sm = MT <= 64 ? 2 : 1;              // CTAs of this tile co-resident on one SM
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= DecodeCfg<16>::kMaxSplit && s <= KB; ++s) {
        const int per = (KB + s - 1) / s;
        if (per > max_kb_per_split) continue;
        if ((int64_t)(s - 1) * per >= KB) continue;  // no empty split
        const int64_t ctas = tiles * s;
        const int64_t busiest = (ctas + sms - 1) / sms;
        const int64_t waves = (busiest + per_sm - 1) / per_sm;
        const double cost = 3.0 * waves + (double)busiest * per * (0.4 + 0.3 * MT / 128.0) +
                            2.0 * s * MT / 128.0;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = s;
        }
    }
    if (cost_out) *cost_out = best_cost;
    return best;
}

// Split for the exchange through distributed shared memory, which is used
// only for token tiles of up to 32 (partial tiles of at most 16 KB per CTA);
// wider tiles without a workspace run unsplit.
template <int MT>
static int smem_exchange_split(int64_t tiles, int KB) {
    if (MT > 32) return 1;
    return choose_split(tiles, KB, MT, DecodeCfg<MT>::kMaxKbPerSplit);
}

static int token_tile(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

// Estimated decode-kernel time in microseconds (the split model above scaled
// by 0.8, its median ratio of measured to modelled time on GB300).
double decode_cost_us(int64_t M, int64_t N, int64_t K) {
    const int MT = token_tile(M);
    const int64_t tiles = (N / 128) * ((M + MT - 1) / MT);
    double c = 1e30;
    choose_split(tiles, (int)(K / 128), MT, DecodeCfg<16>::kMaxKbPerSplit, &c);
    return 0.8 * c;
}

template <int MT>
static cudaError_t set_decode_smem(int dev) {
    static bool attr_set[64] = {};     // the attribute belongs to the device
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_fp8_decode_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             DecodeCfg<MT>::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return cudaSuccess;
}

template <int MT>
static cudaError_t set_persist_smem(int dev) {
    static bool attr_set[64] = {};     // the attribute belongs to the device
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_fp8_decode_persistent_kernel<MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, DecodeCfg<MT>::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return cudaSuccess;
}

// Clusters of `split` CTAs of this kernel that can run at once on the device
// (the occupancy API counts one CTA of a cluster per SM; this kernel fits
// kMinBlocks per SM, so that many times more run).  0 if unknown.
template <int MT>
static int64_t clusters_per_wave(int split) {
    static int cache[64][9] = {};      // device x split; -1: unknown
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || split < 1 || split > 8) return 0;
    if (cache[dev][split] == 0) {
        int n = -1;
        if (set_decode_smem<MT>(dev) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)split, 1, 1024);
            cfg.blockDim = dim3(DecodeCfg<MT>::kThreads);
            cfg.dynamicSmemBytes = DecodeCfg<MT>::kSmemBytes;
            cudaLaunchAttribute a[1];
            a[0].id = cudaLaunchAttributeClusterDimension;
            a[0].val.clusterDim.x = (unsigned)split;
            a[0].val.clusterDim.y = 1;
            a[0].val.clusterDim.z = 1;
            cfg.attrs = a;
            cfg.numAttrs = 1;
            int c = 0;
            if (cudaOccupancyMaxActiveClusters(&c, gemm_fp8_decode_kernel<MT>, &cfg) == cudaSuccess && c > 0) n = c;
        }
        cudaGetLastError();            // a failed query leaves no sticky error
        cache[dev][split] = n;
    }
    return cache[dev][split] > 0 ? (int64_t)cache[dev][split] * DecodeCfg<MT>::kMinBlocks : 0;
}

// Split-K plan of the dense decode GEMM, from a sweep of the three exchanges
// and splits 1..16 over the Qwen2.5-7B/32B decode shapes at M = 1..128 on
// GB300 (in the order tried):
//  - token tiles of 64, with a workspace: the largest split whose clusters all
//    run at once, exchanging through L2 (below);
//  - token tiles of 128 (or 64 without such a split), with a workspace: the
//    split CTAs run without a cluster, about one per SM, and a second launch
//    adds their partials;
//  - token tiles of up to 32: a cluster split whose clusters all run at once
//    (per the occupancy API).  Without a workspace the largest such split, i.e.
//    more, shorter weight streams per slab as long as no second wave of
//    clusters is needed, exchanging through distributed shared memory.  With
//    a workspace the partials go through L2 and the CTAs add them after one
//    cluster barrier (at 16-32 tokens 7-9% faster than through distributed
//    shared memory, which needs a second barrier before any CTA may exit), and
//    the split is l2_exchange_split's;
//  - when no such split exists (long K on few slabs: the 27648-wide down
//    projection), through the workspace and a second launch, as many CTAs per
//    slab as one wave holds;
//  - else the cost model above (without a workspace, tiles of 64 and more: it
//    picks the best cluster split there).
struct DecodePlan {
    int split;
    int xmode;   // kXchg*: how the split CTAs exchange their partials
    bool uses_memory() const { return xmode != kXchgSmem; }
};

static bool split_fits(int KB, int s, int max_per) {
    const int per = (KB + s - 1) / s;
    return per <= max_per && (s - 1) * per < KB;   // no empty split
}

// Split of a token tile of up to 32 whose exchange goes through L2, among the
// splits whose clusters all run at once (one_wave: the largest of them).  In a
// sweep of every such split over 12 shapes (N, K from 1536 to 10240) at M = 1,
// 8 and 32 on GB300, the fastest was, in this order:
//  - the largest split that leaves at most one CTA per SM, if it keeps at least
//    90% of the SMs busy with weight streams of at most 8 K blocks (128 KB) per
//    CTA: a CTA alone on its SM streams faster than two sharing one;
//  - else the smallest split whose CTAs cover every SM with streams of at most
//    8 blocks: a larger split adds ranks to the exchange, not bandwidth;
//  - else the largest one-wave split.
// Against the largest one-wave split alone this took, e.g., Qwen2.5-7B qkv at
// M = 8 from 6.5 to 5.8 us and Qwen2.5-32B o_proj at M = 1 from 8.2 to 7.7 us.
template <int MT>
static int l2_exchange_split(int64_t tiles, int KB, int one_wave) {
    constexpr int kMaxKbPerCta = 8;
    const int64_t sms = num_sms();
    auto usable = [&](int s) {
        return split_fits(KB, s, DecodeCfg<MT>::kMaxKbPerSplit) && clusters_per_wave<MT>(s) >= tiles;
    };
    int alone = 0;   // largest split with at most one CTA per SM
    for (int s = 1; s <= one_wave; ++s)
        if (tiles * s <= sms && usable(s)) alone = s;
    if (alone > 0 && tiles * alone * 10 >= sms * 9 && (KB + alone - 1) / alone <= kMaxKbPerCta) return alone;
    for (int s = 1; s <= one_wave; ++s)
        if (tiles * s >= sms && (KB + s - 1) / s <= kMaxKbPerCta && usable(s)) return s;
    return one_wave;
}

template <int MT>
static DecodePlan decode_plan(int64_t tiles, int KB, bool may_use_memory) {
    using C = DecodeCfg<MT>;
    constexpr int kMaxMemSplit = 16;
    const int64_t sms = num_sms();
    // the largest split whose clusters all run at once (0: none)
    int one_wave = 0;
    for (int s = C::kMaxSplit; s >= 1 && one_wave == 0; --s)
        if (split_fits(KB, s, C::kMaxKbPerSplit) && clusters_per_wave<MT>(s) >= tiles) one_wave = s;
    // 64-token tiles: the largest one-wave cluster split, exchanging through
    // L2.  Against the second launch at one CTA per SM, over 12 shapes (N, K
    // from 1536 to 10240) at M = 64: 127.1 -> 120.0 us in all, e.g. an 8192 x
    // 8192 GEMM 20.6 -> 16.4 us, Qwen2.5-32B qkv 13.7 -> 13.0 us, 7B down
    // 18.1 -> 16.9 us; the worst case, 7B qkv, 8.4 -> 8.8 us
    if (may_use_memory && MT == 64 && one_wave >= 2) return DecodePlan{one_wave, kXchgClusterMem};
    if (may_use_memory && MT >= 64) {
        int64_t t = sms / tiles;
        int s = (int)(t < kMaxMemSplit ? t : kMaxMemSplit);
        while (s >= 2 && !split_fits(KB, s, C::kMaxKbPerSplit)) --s;
        if (s >= 2) return DecodePlan{s, kXchgReduceLaunch};
    }
    if (MT <= 32 && one_wave > 0) {
        if (!may_use_memory || one_wave == 1) return DecodePlan{one_wave, kXchgSmem};
        const int s = l2_exchange_split<MT>(tiles, KB, one_wave);
        return DecodePlan{s, s > 1 ? kXchgClusterMem : kXchgSmem};
    }
    if (may_use_memory && clusters_per_wave<MT>(1) > 0) {   // occupancy known: clusters did not fit
        int64_t t = sms * C::kMinBlocks / tiles;
        int s = (int)(t < kMaxMemSplit ? t : kMaxMemSplit);
        while (s >= 2 && !split_fits(KB, s, C::kMaxKbPerSplit)) --s;
        if (s >= 2) return DecodePlan{s, kXchgReduceLaunch};
    }
    return DecodePlan{smem_exchange_split<MT>(tiles, KB), kXchgSmem};
}

template <int MT>
static size_t decode_ws_bytes_mt(int64_t M, int64_t N, int64_t K) {
    const int64_t mtiles = (M + MT - 1) / MT, tiles = (N / 128) * mtiles;
    const DecodePlan pl = decode_plan<MT>(tiles, (int)(K / 128), true);
    return pl.uses_memory() ? (size_t)tiles * pl.split * MT * 128 * sizeof(float) : 0;
}

template <int MT>
static int decode_kernels_mt(int64_t M, int64_t N, int64_t K, size_t ws_bytes) {
    const int64_t mtiles = (M + MT - 1) / MT, tiles = (N / 128) * mtiles;
    const int KB = (int)(K / 128);
    DecodePlan pl = decode_plan<MT>(tiles, KB, true);
    if (pl.uses_memory() && ws_bytes < (size_t)tiles * pl.split * MT * 128 * sizeof(float))
        pl = decode_plan<MT>(tiles, KB, false);
    return pl.xmode == kXchgReduceLaunch ? 2 : 1;
}

template <int MT>
static bool decode_fits_mt(int64_t M, int64_t N, int64_t K, size_t ws_bytes) {
    const int64_t mtiles = (M + MT - 1) / MT, tiles = (N / 128) * mtiles;
    const int KB = (int)(K / 128);
    DecodePlan pl = decode_plan<MT>(tiles, KB, true);
    if (pl.uses_memory() && ws_bytes < (size_t)tiles * pl.split * MT * 128 * sizeof(float))
        pl = decode_plan<MT>(tiles, KB, false);
    return (KB + pl.split - 1) / pl.split <= DecodeCfg<MT>::kMaxKbPerSplit;
}

// Whether the dense decode kernel can run this shape with `ws_bytes` of
// workspace: without a workspace, token tiles of 64 and more run unsplit (the
// exchange through distributed shared memory is kept to tiles of up to 32), so
// a K beyond one CTA's 32 blocks then goes to the 128 x 256 tile kernel.
bool decode_fits(int64_t M, int64_t N, int64_t K, size_t ws_bytes) {
    if (M <= 0 || !decode_supported(K)) return false;
    if (M <= 16) return decode_fits_mt<16>(M, N, K, ws_bytes);
    if (M <= 32) return decode_fits_mt<32>(M, N, K, ws_bytes);
    if (M <= 64) return decode_fits_mt<64>(M, N, K, ws_bytes);
    return decode_fits_mt<128>(M, N, K, ws_bytes);
}

// Kernels the dense decode GEMM launches for this shape and workspace size.
int decode_kernel_count(int64_t M, int64_t N, int64_t K, size_t ws_bytes) {
    if (M <= 16) return decode_kernels_mt<16>(M, N, K, ws_bytes);
    if (M <= 32) return decode_kernels_mt<32>(M, N, K, ws_bytes);
    if (M <= 64) return decode_kernels_mt<64>(M, N, K, ws_bytes);
    return decode_kernels_mt<128>(M, N, K, ws_bytes);
}

size_t decode_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || !decode_supported(K)) return 0;
    if (M <= 16) return decode_ws_bytes_mt<16>(M, N, K);
    if (M <= 32) return decode_ws_bytes_mt<32>(M, N, K);
    if (M <= 64) return decode_ws_bytes_mt<64>(M, N, K);
    return decode_ws_bytes_mt<128>(M, N, K);
}

// M: token rows (all experts together in the grouped form); rows_per_group:
// the token rows one weight matrix may have (M, or the per-expert bound);
// groups: experts (1 for the dense GEMM, offs == nullptr).  ws: workspace for
// split-K without a cluster (dense form only; may be too small or NULL).
// Weights of at most this many bytes are streamed before the dependency wait
// when the caller allows it: on the Qwen2.5-7B/32B qkv and o_proj layers
// (13-37 MB) this saves 0.3-1.2 us per call; on the larger layers the early
// traffic delayed the preceding kernel's tail by more than it saved.
constexpr int64_t kEarlyWeightMaxBytes = 48ll << 20;

template <int MT>
static cudaError_t launch_decode_mt(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                    const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                                    int64_t ldy, const int32_t* offs, int64_t groups, int64_t rows_per_group,
                                    void* ws, size_t ws_bytes, bool weights_stable, cudaStream_t st) {
    using C = DecodeCfg<MT>;
    CUtensorMap tmW, tmX;
    if (!make_tmap_u8(&tmW, Wq, (uint64_t)(groups * N), (uint64_t)K, (uint64_t)K, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tmX, Xq, (uint64_t)M, (uint64_t)K, (uint64_t)K, MT)) return cudaErrorInvalidValue;
    const int KB = (int)(K / 128);
    const int64_t mtiles = (rows_per_group + MT - 1) / MT;
    const int64_t tiles = groups * (N / 128) * mtiles;
    DecodePlan pl = offs ? DecodePlan{smem_exchange_split<MT>(tiles, KB), kXchgSmem}
                         : decode_plan<MT>(tiles, KB, true);
    if (pl.uses_memory() && (ws == nullptr || ws_bytes < (size_t)tiles * pl.split * MT * 128 * sizeof(float)))
        pl = decode_plan<MT>(tiles, KB, false);
    const int split = pl.split;
    const int per = (KB + split - 1) / split;
    if (per > C::kMaxKbPerSplit) return cudaErrorInvalidValue;
    uint32_t* err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // grouped form, K not split, more items than CTAs fit at once: persistent CTAs
    const int64_t slots = (int64_t)num_sms() * C::kMinBlocks;
    if (offs != nullptr && split == 1 && tiles > slots && tiles < (1ll << 31)) {
        e = set_persist_smem<MT>(dev);
        if (e != cudaSuccess) return e;
        PersistParams pp{err, Xs, Ws, Y, M, ldy, KB, (int)tiles, (int)mtiles, offs, (int)(N / 128), mtiles * MT};
        return launch_pdl(gemm_fp8_decode_persistent_kernel<MT>, dim3((unsigned)slots), dim3(C::kThreads),
                          C::kSmemBytes, st, tmW, tmX, pp);
    }
    const int early_w = (weights_stable && offs == nullptr && N * K <= kEarlyWeightMaxBytes) ? 1 : 0;
    DecodeParams prm{err, Xs, Ws, Y, M, ldy, KB, per, split, offs, (int)(N / 128), mtiles * MT,
                     pl.uses_memory() ? static_cast<float*>(ws) : nullptr, pl.xmode, early_w};
    e = set_decode_smem<MT>(dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)split, (unsigned)mtiles, (unsigned)(groups * (N / 128)));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)split;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pl.xmode == kXchgReduceLaunch ? 1 : 2;    // no cluster for the reduction launch
    e = cudaLaunchKernelEx(&cfg, gemm_fp8_decode_kernel<MT>, tmW, tmX, prm);
    if (e != cudaSuccess || pl.xmode != kXchgReduceLaunch) return e;
    const int64_t units = tiles * MT * 16;
    return launch_pdl(decode_splitk_reduce_kernel<MT>, dim3((unsigned)((units + 255) / 256)), dim3(256), 0, st,
                      (const float*)ws, M, (int)mtiles, split, units, Y, ldy);
}

bool decode_supported(int64_t K) { return K / 128 <= 8 * DecodeCfg<16>::kMaxKbPerSplit; }

cudaError_t launch_gemm_fp8_decode(const uint8_t* Xq, const float* Xs, const uint8_t* Wq,
                                   const float* Ws, int64_t M, int64_t N, int64_t K, uint16_t* Y,
                                   int64_t ldy, void* ws, size_t ws_bytes, bool weights_stable,
                                   cudaStream_t st) {
    const bool w = weights_stable;
    if (M <= 16) return launch_decode_mt<16>(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, nullptr, 1, M, ws, ws_bytes, w, st);
    if (M <= 32) return launch_decode_mt<32>(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, nullptr, 1, M, ws, ws_bytes, w, st);
    if (M <= 64) return launch_decode_mt<64>(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, nullptr, 1, M, ws, ws_bytes, w, st);
    return launch_decode_mt<128>(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, nullptr, 1, M, ws, ws_bytes, w, st);
}

cudaError_t launch_gemm_fp8_grouped(const uint8_t* Xq, const float* Xs, const uint8_t* Wq, const float* Ws,
                                    const int32_t* offs, int64_t E, int64_t T, int64_t N, int64_t K,
                                    int64_t max_rows, uint16_t* Y, int64_t ldy, cudaStream_t st) {
    if (max_rows <= 16)
        return launch_decode_mt<16>(Xq, Xs, Wq, Ws, T, N, K, Y, ldy, offs, E, max_rows, nullptr, 0, false, st);
    if (max_rows <= 32)
        return launch_decode_mt<32>(Xq, Xs, Wq, Ws, T, N, K, Y, ldy, offs, E, max_rows, nullptr, 0, false, st);
    if (max_rows <= 64)
        return launch_decode_mt<64>(Xq, Xs, Wq, Ws, T, N, K, Y, ldy, offs, E, max_rows, nullptr, 0, false, st);
    return launch_decode_mt<128>(Xq, Xs, Wq, Ws, T, N, K, Y, ldy, offs, E, max_rows, nullptr, 0, false, st);
}

// ------------------------------------------------------------------ linear layer

size_t linear_codes_bytes(int64_t M, int64_t K) { return ((size_t)M * (size_t)K + 255) & ~(size_t)255; }

static size_t linear_codes_and_scales_bytes(int64_t M, int64_t K) {
    return linear_codes_bytes(M, K) + (((size_t)M * (size_t)(K / 128) * 4 + 255) & ~(size_t)255);
}

// [codes | scales | the GEMM's workspace], each part 256-byte aligned
size_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0) return 0;
    return linear_codes_and_scales_bytes(M, K) + gemm_fp8_workspace_bytes(M, N, K);
}

// The activation quantizer releases its dependent at launch, so the GEMM's
// CTAs are resident and have started pulling their first weight blocks while
// the activations are quantized; the GEMM then reads the codes from L2.  The
// kernel right before the GEMM is the quantizer, which writes only Xq and Xs,
// so the GEMM may load weight tiles before its dependency wait.
cudaError_t launch_linear_fp8(const uint16_t* X, int64_t ldx, const uint8_t* Wq, const float* Ws, int64_t M,
                              int64_t N, int64_t K, uint16_t* Y, int64_t ldy, uint8_t* Xq_out,
                              float* Xs_out, void* ws, cudaStream_t st) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint8_t* Xq = Xq_out ? Xq_out : base;
    float* Xs = Xs_out ? Xs_out : reinterpret_cast<float*>(base + linear_codes_bytes(M, K));
    cudaError_t e = launch_quant_act_group(X, M, K, ldx, Xq, Xs, st);
    if (e != cudaSuccess) return e;
    const size_t g = gemm_fp8_workspace_bytes(M, N, K);
    void* gws = (base && g) ? base + linear_codes_and_scales_bytes(M, K) : nullptr;
    return launch_gemm_fp8(Xq, Xs, Wq, Ws, M, N, K, Y, ldy, gws, gws ? g : 0, true, st);
}

}  // namespace fp8rl
