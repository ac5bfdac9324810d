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
// are the same bits as the three-launch path's.
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
constexpr int kKvSlotsPerThread = 3;                  // one pass polls at most 768 slots
constexpr uint32_t kKvAborted = 0xFFFFFFFFu;          // header amax of a call whose gather ran out

// Cooperative launch (every CTA resident) over the header word and P slots:
// slot[1 + i] = tag << 32 | amax bits of slice i; the header, slot[0], ends as
// tag << 32 | tensor amax bits.  Every CTA reads the header before it
// publishes its slot, and CTA 0 overwrites the header only after it has seen
// every slot of this call, so all CTAs derive the same tag (release stores,
// relaxed polling and a fence before the header write: each slot word carries
// its own tag and value, and relaxed loads stay in flight together where
// acquire loads would complete one after another).  Polling traffic stays
// O(P) per round (CTA 0 reads the P slots, the
// rest read one word), backing off between rounds so it does not crowd the
// loads of CTAs still reading their slice.  A CTA whose wait runs out records
// a time-out in the error word and writes no codes; if CTA 0's gather runs out
// it still advances the header (with an abort marker), so the next call's tag
// differs from this one's.
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
    // suffices, as the release store of this CTA's slot below orders it first
    __shared__ uint32_t s_tag;
    if (threadIdx.x == 0) s_tag = next_call_tag((uint32_t)(ld_relaxed_u64(slot) >> 32));
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kKvChunksPerThread; ++i) m = absmax_v4(m, v[i]);
    __shared__ uint32_t red[kKvThreads / 32];
    m = __reduce_max_sync(0xffffffffu, max(m & 0xFFFFu, m >> 16));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    const uint32_t tag = s_tag;
    if (threadIdx.x == 0) {
        uint32_t r = red[0];
        for (int w = 1; w < kKvThreads / 32; ++w) r = max(r, red[w]);
        st_release_u64(slot + 1 + blockIdx.x, ((uint64_t)tag << 32) | r);   // bf16 magnitude bits of the amax
    }
    // CTA 0 gathers every slice's amax of this call (each thread polls up to
    // kKvSlotsPerThread slots, all loads of a round in flight together) and
    // publishes the tensor amax in the header; the other CTAs wait for that word.
    __shared__ uint32_t bcast[2];                          // tensor amax bits, wait ok
    bool ok = true;
    if (blockIdx.x == 0) {
        uint32_t a = 0;
        uint64_t sv[kKvSlotsPerThread];
        uint32_t pending = 0;
#pragma unroll
        for (int j = 0; j < kKvSlotsPerThread; ++j) {
            const int64_t i = threadIdx.x + (int64_t)j * kKvThreads;
            sv[j] = 0;
            if (i < P) {
                sv[j] = ld_relaxed_u64(slot + 1 + i);
                pending |= 1u << j;
            }
        }
        const uint64_t t0 = sm100::globaltimer_ns();
        for (;;) {
#pragma unroll
            for (int j = 0; j < kKvSlotsPerThread; ++j)
                if (((pending >> j) & 1u) && (uint32_t)(sv[j] >> 32) == tag) {
                    a = max(a, (uint32_t)sv[j]);
                    pending &= ~(1u << j);
                }
            if (!pending) break;
            if (sm100::globaltimer_ns() - t0 > kKvWaitLimitNs) {
                ok = false;
                break;
            }
            __nanosleep(64);
#pragma unroll
            for (int j = 0; j < kKvSlotsPerThread; ++j)
                if ((pending >> j) & 1u) sv[j] = ld_relaxed_u64(slot + 1 + threadIdx.x + (int64_t)j * kKvThreads);
        }
        ok = __syncthreads_and(ok);
        a = __reduce_max_sync(0xffffffffu, a);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;   // red[] free: __syncthreads_and above
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t r = red[0];
            for (int w = 1; w < kKvThreads / 32; ++w) r = max(r, red[w]);
            __threadfence();       // the slots seen above happen before the header write
            st_release_u64(slot, ((uint64_t)tag << 32) | (ok ? r : kKvAborted));
            bcast[0] = r;
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
            __nanosleep(64);
            sv = ld_relaxed_u64(slot);
        }
        if ((uint32_t)sv == kKvAborted) ok = false;      // CTA 0's gather ran out (it recorded that)
        bcast[0] = (uint32_t)sv;
        bcast[1] = ok;
    }
    __syncthreads();
    if (!bcast[1]) {
        if (threadIdx.x == 0) atomicCAS(err, 0u, (kKernelKv << 24) | (1u << 16) | 1u);
        return;
    }
    const uint32_t r = bcast[0];
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
    if (P > 0 && P <= kv_onepass_capacity() && P <= (int64_t)kKvSlotsPerThread * kKvThreads) {
        int64_t cpr = C / 8;
        uint64_t* slots = reinterpret_cast<uint64_t*>(partial);
        uint32_t* err = device_error_word();
        if (!err) return cudaErrorInvalidValue;
        void* args[] = {(void*)&X,     (void*)&total, (void*)&cpr, (void*)&ld, (void*)&slots,
                        (void*)&P,     (void*)&scale, (void*)&Xq,  (void*)&err};
        return cudaLaunchCooperativeKernel((const void*)kv_onepass_kernel, dim3((unsigned)P), dim3(kKvThreads),
                                           args, 0, st);
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

static_assert((kKvSlotsPerThread * kKvThreads + 1) * 2 <= 2 + kKvNoAllocSlots, "one-pass slots fit the array");

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
