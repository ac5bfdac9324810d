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
//
// When every slice's CTA can be resident at once (tensors up to ~10 M values,
// e.g. one step's keys or values), one cooperative launch does all three: each
// CTA keeps its slice in registers and publishes its partial amax in an 8-byte
// slot tagged with the call's tag; CTA 0 waits (bounded) until every slot
// carries that tag and publishes the tensor amax in the header word, which
// the other CTAs wait for (bounded); every CTA then encodes its slice from
// registers.  One read of the tensor and no launch gaps; the scale and codes
// are the same bits as the three-launch path's.  Larger tensors with
// contiguous rows take a cooperative launch of one CTA per SM that keeps the
// first part of each SM's range on chip (kv_resident_kernel below), so only
// the rest is read twice.
//
// The call's tag is derived on the device from the tag the previous call left
// in the header word (next tag = previous + 1, top bit set), so a CUDA graph
// that replays one launch still gives every replay a new tag, and a slot left
// by an earlier call never carries the current one.  The workspace needs no
// zeroing: the three-launch path's partials (bf16 magnitude bits, below
// 0x8000) never have the top bit of a tag, and anything else a reused
// workspace holds matches a tag only by chance.
//
// Workspace layout (64-bit words): word 0 is the one-pass header, words
// 1 .. P the one-pass slots; the three-launch path keeps its 32-bit partials
// from byte 8 on, so it never overwrites the header.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"
#include "tagged_slots.cuh"

namespace fp8rl {

namespace {

constexpr int kKvThreads = 256;
constexpr int kKvChunksPerThread = 8;
constexpr int64_t kKvChunksPerCta = kKvThreads * kKvChunksPerThread;   // 2048 chunks = 16384 values

// chunk c of a [R][C] tensor with row pitch ld: 8 values at row c / (C/8).
// Contiguous rows (the usual cache layout) skip the 64-bit division.
__device__ __forceinline__ int64_t chunk_offset(int64_t c, int64_t cpr, int64_t ld) {
    if (ld == cpr * 8) return c * 8;
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

constexpr uint64_t kKvWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait
constexpr uint32_t kKernelKv = 5;
constexpr int kKvMaxSlots = 768;                      // slices one gathering CTA polls at most
constexpr uint32_t kKvAborted = 0xFFFFFFFFu;          // header amax of a call whose gather ran out

// Maximum of v over the CTA, returned to every thread.  red: kThreads / 32
// words of shared memory, free again when this returns.
template <int kThreads>
__device__ __forceinline__ uint32_t cta_max_u32(uint32_t v, uint32_t* red) {
    v = __reduce_max_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t r = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) r = max(r, red[w]);
    __syncthreads();
    return r;
}

// Grid-wide maximum of a cooperative launch (every CTA resident) over the
// header word and P slots: slot[1 + i] = tag << 32 | the maximum of CTA i; the
// header, slot[0], ends as tag << 32 | the grid maximum.  Every CTA reads the
// header before it publishes its slot, and CTA 0 overwrites the header only
// after it has seen every slot of this call, so all CTAs derive the same tag
// (release stores and relaxed polling: each slot word carries its own tag and
// value, and relaxed loads stay in flight together where acquire loads would
// complete one after another).  Polling
// traffic stays O(P) per round (CTA 0 reads the P slots, the rest read one
// word), backing off between rounds so it does not crowd the loads of CTAs
// still reading their part.  v_cta: this CTA's maximum (the same in every
// thread).  Returns false in every thread of a CTA whose wait ran out (the
// time-out is recorded in the error word); if CTA 0's gather runs out it still
// advances the header (with an abort marker), so the next call's tag differs
// from this one's.
template <int kThreads>
__device__ bool kv_grid_max(uint64_t* __restrict__ slot, int64_t P, uint32_t tag, uint32_t v_cta,
                            uint32_t* red, uint32_t* err, uint32_t* out) {
    constexpr int kSlotsPerThread = (kKvMaxSlots + kThreads - 1) / kThreads;
    __shared__ uint32_t bcast[2];                          // grid maximum, wait ok
    if (threadIdx.x == 0) st_release_u64(slot + 1 + blockIdx.x, ((uint64_t)tag << 32) | v_cta);
    bool ok = true;
    if (blockIdx.x == 0) {
        // each thread polls up to kSlotsPerThread slots, all loads of a round in flight together
        uint32_t a = 0;
        uint64_t sv[kSlotsPerThread];
        uint32_t pending = 0;
#pragma unroll
        for (int j = 0; j < kSlotsPerThread; ++j) {
            const int64_t i = threadIdx.x + (int64_t)j * kThreads;
            sv[j] = 0;
            if (i < P) {
                sv[j] = ld_relaxed_u64(slot + 1 + i);
                pending |= 1u << j;
            }
        }
        const uint64_t t0 = sm100::globaltimer_ns();
        for (;;) {
#pragma unroll
            for (int j = 0; j < kSlotsPerThread; ++j)
                if (((pending >> j) & 1u) && (uint32_t)(sv[j] >> 32) == tag) {
                    a = max(a, (uint32_t)sv[j]);
                    pending &= ~(1u << j);
                }
            if (!pending) break;
            if (sm100::globaltimer_ns() - t0 > kKvWaitLimitNs) {
                ok = false;
                break;
            }
            __nanosleep(16);
#pragma unroll
            for (int j = 0; j < kSlotsPerThread; ++j)
                if ((pending >> j) & 1u) sv[j] = ld_relaxed_u64(slot + 1 + threadIdx.x + (int64_t)j * kThreads);
        }
        ok = __syncthreads_and(ok);
        a = cta_max_u32<kThreads>(a, red);
        if (threadIdx.x == 0) {
            // a release store: the slots this CTA saw (through the barriers
            // above) are ordered before it; readers take only this word
            st_release_u64(slot, ((uint64_t)tag << 32) | (ok ? a : kKvAborted));
            bcast[0] = a;
            bcast[1] = ok;
        }
    } else if (threadIdx.x == 0) {
        const uint64_t t0 = sm100::globaltimer_ns();
        uint64_t sv = ld_relaxed_u64(slot);
        while ((uint32_t)(sv >> 32) != tag) {
            if (sm100::globaltimer_ns() - t0 > kKvWaitLimitNs) {
                ok = false;
                break;
            }
            __nanosleep(16);
            sv = ld_relaxed_u64(slot);
        }
        if ((uint32_t)sv == kKvAborted) ok = false;      // CTA 0's gather ran out (it recorded that)
        bcast[0] = (uint32_t)sv;
        bcast[1] = ok;
    }
    __syncthreads();
    ok = bcast[1] != 0;
    if (!ok && threadIdx.x == 0) atomicCAS(err, 0u, (kKernelKv << 24) | (1u << 16) | 1u);
    *out = bcast[0];
    return ok;
}

// One cooperative launch over slices of kKvChunksPerCta chunks (the grid
// maximum above).  Each CTA keeps its slice in registers, so the tensor is
// read once; a CTA whose wait ran out writes no codes.
__global__ void __launch_bounds__(kKvThreads, 4)   // four CTAs per SM: 608 slices resident at once
kv_onepass_kernel(const uint16_t* __restrict__ X, int64_t total, int64_t cpr, int64_t ld,
                  uint64_t* __restrict__ slot, int64_t P, float* __restrict__ scale,
                  uint8_t* __restrict__ Xq, uint32_t* __restrict__ err) {
    const int64_t base = (int64_t)blockIdx.x * kKvChunksPerCta;
    uint4 v[kKvChunksPerThread];
#pragma unroll
    for (int i = 0; i < kKvChunksPerThread; ++i) {
        const int64_t c = base + i * kKvThreads + threadIdx.x;
        v[i] = c < total ? ld_stream_v4(X + chunk_offset(c, cpr, ld)) : make_uint4(0, 0, 0, 0);
    }
    // the header is read after the slice's loads are in flight; a relaxed load
    // suffices, as the release store of this CTA's slot orders it first
    __shared__ uint32_t s_tag;
    __shared__ uint32_t red[kKvThreads / 32];
    if (threadIdx.x == 0) s_tag = next_call_tag((uint32_t)(ld_relaxed_u64(slot) >> 32));
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kKvChunksPerThread; ++i) m = absmax_v4(m, v[i]);
    m = cta_max_u32<kKvThreads>(max(m & 0xFFFFu, m >> 16), red);    // bf16 magnitude bits of the slice's amax
    uint32_t r;
    if (!kv_grid_max<kKvThreads>(slot, P, s_tag, m, red, err, &r)) return;
    const float s = fp8_scale_from_amax(__uint_as_float(r << 16));
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
    const BlockDivisor d = make_divisor(s);
#pragma unroll
    for (int i = 0; i < kKvChunksPerThread; ++i) {
        const int64_t c = base + i * kKvThreads + threadIdx.x;
        if (c < total)
            *reinterpret_cast<uint2*>(Xq + c * 8) = d.fast ? quant8_e4m3_t<true>(v[i], d)
                                                           : quant8_e4m3_t<false>(v[i], d);
    }
}

// Tensors too large for one slice per CTA (contiguous rows, 16-byte aligned):
// one cooperative launch of one 512-thread CTA per SM.  The tensor is cut into
// batches of kResBatch rounds (a round is one 16-byte chunk per thread, so a
// batch is 64 KB), dealt to the CTAs in turn -- CTA b takes batches b, b + G,
// b + 2G, ... -- which spreads every SM's share over the whole tensor.  While
// its batches are read for the amax (the next batch's loads in flight while
// one is reduced and stored), a CTA keeps its first kResResident on chip --
// kResTmemBatches in tensor memory (32 columns of each warp's lane quadrant per
// batch), then kResSmemBatches in shared memory, 448 KB per CTA -- so after
// the grid maximum only the rest is read again.  Tensors up to the on-chip
// total (152 x 448 KB of bf16 on GB300, ~34 M values) are read once; larger
// ones save that much of the second read.
constexpr int kResThreads = 512;
constexpr int kResBatch = 8;                            // rounds per batch: loads in flight per thread
constexpr int kResTmemBatches = 4;                      // 4 x 32 columns per warp: all 512 TMEM columns
constexpr int kResSmemBatches = 3;                      // 3 x 64 KB of shared memory
constexpr int kResResident = kResTmemBatches + kResSmemBatches;
constexpr int64_t kResChunksPerBatch = (int64_t)kResBatch * kResThreads;
constexpr int kResSmemBytes = kResSmemBatches * kResBatch * kResThreads * 16;
constexpr uint32_t kResTmemCols = 512;
static_assert((kResThreads / 32 / 4) * kResTmemBatches * 32 == (int)kResTmemCols, "TMEM columns per warp");

__device__ __forceinline__ void encode_batch(const uint4 (&v)[kResBatch], int64_t c, int64_t total,
                                             const BlockDivisor& d, uint8_t* __restrict__ Xq) {
#pragma unroll
    for (int i = 0; i < kResBatch; ++i, c += kResThreads)
        if (c < total)
            *reinterpret_cast<uint2*>(Xq + c * 8) = d.fast ? quant8_e4m3_t<true>(v[i], d)
                                                           : quant8_e4m3_t<false>(v[i], d);
}

__device__ __forceinline__ void load_batch(uint4 (&v)[kResBatch], const uint16_t* __restrict__ X, int64_t c,
                                           int64_t total) {
#pragma unroll
    for (int i = 0; i < kResBatch; ++i, c += kResThreads)
        v[i] = c < total ? ld_stream_v4(X + c * 8) : make_uint4(0, 0, 0, 0);
}

// Pass 1, batch b (in v): its amax into m, and on chip if it is resident.
__device__ __forceinline__ void keep_batch(int b, const uint4 (&v)[kResBatch], uint32_t& m, uint32_t tw,
                                           uint4* sres) {
#pragma unroll
    for (int i = 0; i < kResBatch; ++i) m = absmax_v4(m, v[i]);
    if (b < kResTmemBatches) {
        sm100::tmem_st_32x32b_x32(tw + b * 32, *reinterpret_cast<const uint32_t(*)[32]>(v));
    } else if (b < kResResident) {
        uint4* dst = sres + (int64_t)(b - kResTmemBatches) * kResBatch * kResThreads + threadIdx.x;
#pragma unroll
        for (int i = 0; i < kResBatch; ++i) dst[i * kResThreads] = v[i];
    }
}

__global__ void __launch_bounds__(kResThreads, 1)
kv_resident_kernel(const uint16_t* __restrict__ X, int64_t total, uint64_t* __restrict__ slot, int64_t P,
                   float* __restrict__ scale, uint8_t* __restrict__ Xq, uint32_t* __restrict__ err) {
    extern __shared__ uint4 sres[];                    // [kResSmemBatches][kResBatch][kResThreads]
    __shared__ uint32_t tmem_slot, s_tag;
    __shared__ uint32_t red[kResThreads / 32];
    const uint32_t warp = threadIdx.x >> 5;
    if (warp == 0) sm100::tmem_alloc(sm100::smem_u32(&tmem_slot), kResTmemCols);
    if (threadIdx.x == 32) s_tag = next_call_tag((uint32_t)(ld_relaxed_u64(slot) >> 32));
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
    // this warp's TMEM: its lane quadrant, 128 columns from (warp / 4) * 128
    const uint32_t tw = tmem_slot + ((32u * (warp & 3)) << 16) + (warp >> 2) * (kResTmemBatches * 32);
    const int64_t G = gridDim.x;
    const int64_t tb = (total + kResChunksPerBatch - 1) / kResChunksPerBatch;   // batches in the tensor
    const int nb = (int)((tb - blockIdx.x + G - 1) / G);                      // this CTA's: b + j G < tb
    const int64_t c0 = (int64_t)blockIdx.x * kResChunksPerBatch + threadIdx.x;   // its first chunk
    const int64_t cstride = G * kResChunksPerBatch;                           // chunks between its batches

    // pass 1: the range's amax, its first batches kept on chip; two batches
    // alternate in registers so that one is always being loaded
    uint32_t m = 0;
    {
        uint4 va[kResBatch], vb[kResBatch];
        if (nb > 0) load_batch(va, X, c0, total);
        for (int b = 0; b < nb; b += 2) {
            if (b + 1 < nb) load_batch(vb, X, c0 + (b + 1) * cstride, total);
            keep_batch(b, va, m, tw, sres);
            if (b + 1 >= nb) break;
            if (b + 2 < nb) load_batch(va, X, c0 + (b + 2) * cstride, total);
            keep_batch(b + 1, vb, m, tw, sres);
        }
    }
    sm100::tmem_wait_st();
    m = cta_max_u32<kResThreads>(max(m & 0xFFFFu, m >> 16), red);   // bf16 magnitude bits of the range's amax
    uint32_t r;
    if (kv_grid_max<kResThreads>(slot, P, s_tag, m, red, err, &r)) {
        const float s = fp8_scale_from_amax(__uint_as_float(r << 16));
        if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
        const BlockDivisor d = make_divisor(s);
        // pass 2: the resident batches are encoded while the first batch read
        // again is in flight
        uint4 nxt[kResBatch];
        if (nb > kResResident) load_batch(nxt, X, c0 + kResResident * cstride, total);
        for (int b = 0; b < kResTmemBatches && b < nb; ++b) {
            uint4 v[kResBatch];
            sm100::tmem_ld_32x32b_x32(tw + b * 32, *reinterpret_cast<uint32_t(*)[32]>(v));
            sm100::tmem_wait_ld();
            encode_batch(v, c0 + b * cstride, total, d, Xq);
        }
        for (int b = kResTmemBatches; b < kResResident && b < nb; ++b) {
            uint4 v[kResBatch];
            const uint4* src = sres + (int64_t)(b - kResTmemBatches) * kResBatch * kResThreads + threadIdx.x;
#pragma unroll
            for (int i = 0; i < kResBatch; ++i) v[i] = src[i * kResThreads];
            encode_batch(v, c0 + b * cstride, total, d, Xq);
        }
        for (int b = kResResident; b < nb; ++b) {
            uint4 v[kResBatch];
#pragma unroll
            for (int i = 0; i < kResBatch; ++i) v[i] = nxt[i];
            if (b + 1 < nb) load_batch(nxt, X, c0 + (b + 1) * cstride, total);
            encode_batch(v, c0 + b * cstride, total, d, Xq);
        }
    }
    sm100::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        sm100::tc_fence_after();
        sm100::tmem_dealloc(tmem_slot, kResTmemCols);
    }
}

// CTAs of the one-pass kernel that can be resident at once on the current
// device (0 if unknown); cached per device.
int64_t kv_onepass_capacity() {
    static int cache[64] = {};                            // 0 unknown, -1 none, else CTAs
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int per_sm = 0, coop = 0;
        const bool ok = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
                        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kv_onepass_kernel, kKvThreads, 0) ==
                            cudaSuccess && per_sm > 0;
        cudaGetLastError();
        cache[dev] = ok ? per_sm * num_sms() : -1;
    }
    return cache[dev] > 0 ? cache[dev] : 0;
}

// CTAs of the resident kernel (one per SM) if it can run on the current
// device: cooperative launch, its shared memory, one CTA per SM; else 0.
int64_t kv_resident_ctas() {
    static int cache[64] = {};                            // 0 unknown, -1 no, else CTAs
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int per_sm = 0, coop = 0;
        const bool ok =
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
            cudaFuncSetAttribute(kv_resident_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kResSmemBytes) ==
                cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kv_resident_kernel, kResThreads, kResSmemBytes) ==
                cudaSuccess &&
            per_sm == 1 && num_sms() <= kKvMaxSlots;
        cudaGetLastError();
        cache[dev] = ok ? num_sms() : -1;
    }
    return cache[dev] > 0 ? cache[dev] : 0;
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
    uint64_t* slots = reinterpret_cast<uint64_t*>(partial);
    if (P > 0 && P <= kv_onepass_capacity() && P <= kKvMaxSlots) {
        int64_t cpr = C / 8;
        uint32_t* err = device_error_word();
        if (!err) return cudaErrorInvalidValue;
        void* args[] = {(void*)&X,     (void*)&total, (void*)&cpr, (void*)&ld, (void*)&slots,
                        (void*)&P,     (void*)&scale, (void*)&Xq,  (void*)&err};
        return cudaLaunchCooperativeKernel((const void*)kv_onepass_kernel, dim3((unsigned)P), dim3(kKvThreads),
                                           args, 0, st);
    }
    // larger, contiguous and 16-byte aligned: one CTA per SM, part of each range
    // kept on chip (the workspace holds P + 1 >= G + 1 slots: P exceeds the
    // one-pass capacity, at least 4 slices per SM)
    const int64_t G = kv_resident_ctas();
    if (P > 0 && G > 0 && G <= P && ld == C && (reinterpret_cast<uintptr_t>(X) & 15) == 0) {
        uint32_t* err = device_error_word();
        if (!err) return cudaErrorInvalidValue;
        int64_t Pr = G;
        void* args[] = {(void*)&X, (void*)&total, (void*)&slots, (void*)&Pr, (void*)&scale, (void*)&Xq, (void*)&err};
        return cudaLaunchCooperativeKernel((const void*)kv_resident_kernel, dim3((unsigned)G), dim3(kResThreads),
                                           args, kResSmemBytes, st);
    }
    uint32_t* part = P > 0 ? partial + 2 : partial;       // past the one-pass header word
    if (P > 0) {
        e = launch_pdl(kv_amax_partial_kernel, dim3((unsigned)P), dim3(kKvThreads), 0, st, X, total, C / 8,
                       ld, part);
        if (e != cudaSuccess) return e;
    }
    e = launch_pdl(kv_scale_kernel, dim3(1), dim3(1024), 0, st, (const uint32_t*)part, P, scale);
    if (e != cudaSuccess) return e;
    return launch_quant_kv_with_scale(X, R, C, ld, scale, Xq, st);
}

// ---------------------------------------------------------------- no-allocation variant
//
// Some callers cannot hand the library a workspace: an inference engine that
// reserves almost all GPU memory for its KV-cache pool when it starts and
// allows no allocation outside that pool afterwards, or a serving loop that
// must not call cudaMalloc / cudaFree because those calls synchronize the
// device and would stall the work already queued.  For them the partial maxima
// live in this file-scope device array instead of a caller workspace.  Every
// GPU that loads the library holds the array (64 KB + 8 B) until the process exits.

constexpr int64_t kKvNoAllocSlots = 16384;   // partial maxima: tensors up to 16384 x 16384 values
// 32-bit words: the 8-byte one-pass header, then one word per partial (the
// three-launch path) or two per slot (the one-pass path)
static __device__ __align__(256) uint32_t g_kv_noalloc_partials[2 + kKvNoAllocSlots];

static_assert((kKvMaxSlots + 1) * 2 <= 2 + kKvNoAllocSlots, "one-pass slots fit the array");

int64_t kv_noalloc_max_values() { return kKvNoAllocSlots * kKvChunksPerCta * 8; }

// Device address of the array on the current device.  The host-side name of a
// __device__ variable is only a stand-in, never a device address, so it is
// resolved once per device with cudaGetSymbolAddress (with that device
// current) and cached.  Returns nullptr if the runtime reports an error.
static uint32_t* kv_noalloc_scratch() {
    constexpr int kMaxDevices = 64;
    static uint32_t* cache[kMaxDevices] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kv_noalloc_partials) != cudaSuccess || !p) return nullptr;
        cache[dev] = static_cast<uint32_t*>(p);
    }
    return cache[dev];
}

cudaError_t launch_quant_kv_tensor_noalloc(const uint16_t* X, int64_t R, int64_t C, int64_t ld,
                                           uint8_t* Xq, float* scale, cudaStream_t st) {
    if (kv_partials(R, C) > kKvNoAllocSlots) return cudaErrorInvalidValue;
    uint32_t* partial = kv_noalloc_scratch();
    if (!partial) return cudaErrorInvalidDevicePointer;
    return launch_quant_kv_tensor(X, R, C, ld, Xq, scale, partial, st);
}

}  // namespace fp8rl
