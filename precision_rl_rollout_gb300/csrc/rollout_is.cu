// rollout_is.cu -- token-level importance-sampling correction of 8-bit rollouts
// (FP8-RL, Abstract, contribution (iii): token-level TIS/MIS; FlashRL write-up,
// section on truncated importance sampling).
//
// The rollout samples tokens from the 8-bit policy while the gradient is taken
// under the trainer's higher-precision policy; each sampled token gets the
// importance weight of the two.  With d = fl32(logp_train - logp_rollout) and a
// threshold C passed as log_clip = ln C:
//   truncated (TIS): w = exp(min(d, log_clip));
//   masked    (MIS): w = d > log_clip ? 0 : exp(d);
// padding tokens (mask 0) get w = 0.  The clip decision is an fp32 comparison,
// so the clipped/masked count is exact; the weights use the CUDA expf.
// Every CTA of a persistent grid writes the weights of its token range and
// one partial record (valid, clipped, sum w, sum d; fp32 sums inside the CTA);
// the records are added in a fixed order, the counts exactly and the sums in
// compensated fp32 (deterministic statistics for a given GPU).  One
// cooperative launch (the grid, at most four CTAs per SM, is resident at once)
// does both: each CTA publishes its record as four tagged words (see
// tagged_slots.cuh) and CTA 0, after its own range, gathers them (bounded
// wait) and writes the statistics.
#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"
#include "tagged_slots.cuh"

namespace fp8rl {

namespace {

constexpr int kIsThreads = 256;
constexpr int kIsPerThread = 16;
constexpr int64_t kIsPerCta = kIsThreads * kIsPerThread;   // 4096 tokens
constexpr int kIsRecsPerThread = 3;                         // the gather covers up to 768 CTAs
constexpr uint64_t kIsWaitLimitNs = 2000000000ull;          // 2 s: far above any legitimate wait
constexpr uint32_t kKernelIs = 7;
constexpr uint32_t kIsAborted = 0xFFFFFFFFu;                // header payload of a call whose gather ran out

// Compensated fp32 sums: (hi, lo) with hi + lo the exact sum of what was
// added, up to the rounding of lo.  fp64 is a small fraction of the fp32 rate
// on this GPU, and the gather below is on the kernel's critical path.
struct F2 {
    float hi, lo;
};
__device__ __forceinline__ F2 f2_add(F2 a, float b) {   // error-free two-sum of a.hi and b
    const float s = __fadd_rn(a.hi, b);
    const float bp = __fsub_rn(s, a.hi);
    const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bp)), __fsub_rn(b, bp));
    return F2{s, __fadd_rn(a.lo, e)};
}
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    const F2 r = f2_add(a, b.hi);
    return F2{r.hi, __fadd_rn(r.lo, b.lo)};
}
__device__ __forceinline__ F2 f2_warp_sum(F2 v) {       // fixed shuffle order: deterministic
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v = f2_add(v, F2{__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)});
    return v;
}

// The inputs are read once and the weights written once: streaming loads that
// skip L1, and evict-first stores.
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
    const uint4 u = ld_stream_v4(p);
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}
__device__ __forceinline__ uint32_t ld_stream_u32(const uint8_t* p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}
__device__ __forceinline__ void st_stream_f4(float* p, float a, float b, float c, float d) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ float is_weight(float d, float log_clip, int mode, bool& clipped) {
    clipped = d > log_clip;
    return mode == 0 ? expf(clipped ? log_clip : d) : (clipped ? 0.f : expf(d));
}

// Workspace (64-bit words): word 0 is the header, words 1 + 4c .. 4 + 4c CTA
// c's tagged record (valid, clipped, sum w bits, sum d bits).
//
// A persistent grid (a few CTAs per SM): CTA c owns the contiguous token range
// [c*per, (c+1)*per), per a multiple of 4096, so every CTA streams the same
// amount and there is no tail wave.  Within the range a thread takes 16
// tokens per step: four groups of four consecutive tokens (16-byte loads of
// both log-prob arrays and a 4-byte load of the mask, all issued before any is
// used).  Ranges that are not whole 4096-token steps, or unaligned pointers,
// take the scalar path.
template <bool kVec>
__global__ void __launch_bounds__(kIsThreads, 4)
rollout_is_kernel(const float* __restrict__ lt, const float* __restrict__ lr,
                  const uint8_t* __restrict__ mask, int64_t n, int64_t per, float log_clip, int mode,
                  float* __restrict__ w, uint64_t* __restrict__ ws, double* __restrict__ stats,
                  uint32_t* __restrict__ err) {
    pdl_wait_then_release();
    __shared__ uint32_t s_tag;
    if (threadIdx.x == 0) s_tag = next_call_tag((uint32_t)(ld_relaxed_u64(ws) >> 32));
    const int64_t r0 = (int64_t)blockIdx.x * per;
    const int64_t r1 = r0 + per < n ? r0 + per : n;
    int nv = 0, nc = 0;
    float sw = 0.f, sd = 0.f;
    for (int64_t base = r0; base < r1; base += kIsPerCta) {
        if (kVec && base + kIsPerCta <= r1) {
            float4 a[4], b[4];
            uint32_t mk[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int64_t i = base + (int64_t)(g * kIsThreads + threadIdx.x) * 4;
                a[g] = ld_stream_f4(lt + i);
                b[g] = ld_stream_f4(lr + i);
                mk[g] = mask ? ld_stream_u32(mask + i) : 0x01010101u;
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float x[4] = {a[g].x, a[g].y, a[g].z, a[g].w};
                const float y[4] = {b[g].x, b[g].y, b[g].z, b[g].w};
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    o[e] = 0.f;
                    if ((mk[g] >> (8 * e)) & 0xFFu) {
                        const float d = __fsub_rn(x[e], y[e]);
                        bool clipped;
                        o[e] = is_weight(d, log_clip, mode, clipped);
                        nv += 1;
                        nc += clipped;
                        sw += o[e];
                        sd += d;
                    }
                }
                const int64_t i = base + (int64_t)(g * kIsThreads + threadIdx.x) * 4;
                st_stream_f4(w + i, o[0], o[1], o[2], o[3]);
            }
        } else {
            for (int j = 0; j < kIsPerThread; ++j) {
                const int64_t i = base + j * kIsThreads + threadIdx.x;
                if (i >= r1) break;
                float wi = 0.f;
                if (mask == nullptr || mask[i] != 0) {
                    const float d = __fsub_rn(lt[i], lr[i]);
                    bool clipped;
                    wi = is_weight(d, log_clip, mode, clipped);
                    nv += 1;
                    nc += clipped;
                    sw += wi;
                    sd += d;
                }
                w[i] = wi;
            }
        }
    }
    // In-CTA reduction in fp32 (counts exactly, as integers): fp64 arithmetic is
    // a small fraction of the fp32 rate on this GPU.  Only the per-CTA record is
    // widened to fp64.
    nv = __reduce_add_sync(0xffffffffu, nv);
    nc = __reduce_add_sync(0xffffffffu, nc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        sw += __shfl_xor_sync(0xffffffffu, sw, off);
        sd += __shfl_xor_sync(0xffffffffu, sd, off);
    }
    __shared__ int ired[kIsThreads / 32][2];
    __shared__ float fred[kIsThreads / 32][2];
    const int wid = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        ired[wid][0] = nv; ired[wid][1] = nc;
        fred[wid][0] = sw; fred[wid][1] = sd;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int a = 0, b = 0;
        float c = 0.f, e = 0.f;
        for (int k = 0; k < kIsThreads / 32; ++k) {
            a += ired[k][0]; b += ired[k][1]; c += fred[k][0]; e += fred[k][1];
        }
        const uint64_t t = (uint64_t)s_tag << 32;
        uint64_t* rec = ws + 1 + 4 * (int64_t)blockIdx.x;
        st_release_u64(rec + 0, t | (uint32_t)a);
        st_release_u64(rec + 1, t | (uint32_t)b);
        st_release_u64(rec + 2, t | __float_as_uint(c));
        st_release_u64(rec + 3, t | __float_as_uint(e));
    }
    if (blockIdx.x != 0) return;
    // ---------------- CTA 0: gather every CTA's record of this call, in a fixed
    // assignment (thread t: records t, t + 256, t + 512) and order.  Each word
    // carries its own tag and value, so relaxed loads suffice, and they stay in
    // flight together (acquire loads would complete one after another).
    __syncthreads();
    const uint32_t tag = s_tag;
    const int P = (int)gridDim.x;
    uint64_t v[kIsRecsPerThread][4];
    uint32_t pending = 0;                    // bit 4 j + k: word k of record j not yet of this call
#pragma unroll
    for (int j = 0; j < kIsRecsPerThread; ++j) {
        const int r = threadIdx.x + j * kIsThreads;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[j][k] = 0;
            if (r < P) pending |= 1u << (4 * j + k);
        }
    }
    bool ok = true;
    const uint64_t t0 = sm100::globaltimer_ns();
    for (;;) {
#pragma unroll
        for (int j = 0; j < kIsRecsPerThread; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if ((pending >> (4 * j + k)) & 1u) {
                    v[j][k] = ld_relaxed_u64(ws + 1 + 4 * (int64_t)(threadIdx.x + j * kIsThreads) + k);
                    if ((uint32_t)(v[j][k] >> 32) == tag) pending &= ~(1u << (4 * j + k));
                }
        if (!pending) break;
        if (sm100::globaltimer_ns() - t0 > kIsWaitLimitNs) {
            ok = false;
            break;
        }
        __nanosleep(64);
    }
    ok = __syncthreads_and(ok);
    // counts: exact 64-bit integer sums; sums: compensated fp32
    long long cnt0 = 0, cnt1 = 0;
    F2 sum_w{0.f, 0.f}, sum_d{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kIsRecsPerThread; ++j)
        if (threadIdx.x + j * kIsThreads < P) {
            cnt0 += (int)(uint32_t)v[j][0];
            cnt1 += (int)(uint32_t)v[j][1];
            sum_w = f2_add(sum_w, __uint_as_float((uint32_t)v[j][2]));
            sum_d = f2_add(sum_d, __uint_as_float((uint32_t)v[j][3]));
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        cnt0 += __shfl_xor_sync(0xffffffffu, cnt0, off);
        cnt1 += __shfl_xor_sync(0xffffffffu, cnt1, off);
    }
    sum_w = f2_warp_sum(sum_w);
    sum_d = f2_warp_sum(sum_d);
    __shared__ long long cred[kIsThreads / 32][2];
    __shared__ F2 sred[kIsThreads / 32][2];
    if ((threadIdx.x & 31) == 0) {
        cred[threadIdx.x >> 5][0] = cnt0;
        cred[threadIdx.x >> 5][1] = cnt1;
        sred[threadIdx.x >> 5][0] = sum_w;
        sred[threadIdx.x >> 5][1] = sum_d;
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        long long c = 0;
        F2 t{0.f, 0.f};
        for (int wv = 0; wv < kIsThreads / 32; ++wv) {     // fixed order
            c += cred[wv][threadIdx.x];
            t = f2_add(t, sred[wv][threadIdx.x]);
        }
        if (ok) {
            stats[threadIdx.x] = (double)c;
            stats[2 + threadIdx.x] = (double)t.hi + (double)t.lo;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // the next call's tag follows this one's even if the gather ran out.
        // The fence makes the records seen above happen before the header
        // write, so no CTA can have read this call's header after it.
        if (!ok) atomicCAS(err, 0u, (kKernelIs << 24) | (1u << 16) | 1u);
        __threadfence();
        st_release_u64(ws, ((uint64_t)tag << 32) | (ok ? 0u : kIsAborted));
    }
}

}  // namespace

// Partial records the workspace must hold: one per 4096 tokens at most (the
// grid never has more CTAs than that).
int64_t rollout_is_max_partials(int64_t n) { return (n + kIsPerCta - 1) / kIsPerCta; }

// CTAs of the persistent grid: up to 4 per SM, each with at least one 4096-token step.
int64_t rollout_is_partials(int64_t n) {
    const int64_t steps = (n + kIsPerCta - 1) / kIsPerCta;
    const int64_t cap = 4 * (int64_t)num_sms();
    return steps < cap ? steps : cap;
}
static int64_t rollout_is_per(int64_t n, int64_t ctas) {
    const int64_t steps = (n + kIsPerCta - 1) / kIsPerCta;
    return ((steps + ctas - 1) / ctas) * kIsPerCta;
}
size_t rollout_is_partial_bytes() { return 4 * sizeof(uint64_t); }   // one tagged record

// CTAs of the one-launch kernel that can be resident at once on the current
// device (0 if unknown or if cooperative launches are not supported); cached
// per device.
static int64_t rollout_is_capacity() {
    static int cache[64] = {};                            // 0 unknown, -1 none, else CTAs
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int a = 0, b = 0, coop = 0;
        const bool ok =
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, rollout_is_kernel<true>, kIsThreads, 0) ==
                cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, rollout_is_kernel<false>, kIsThreads, 0) ==
                cudaSuccess &&
            a > 0 && b > 0;
        cudaGetLastError();
        cache[dev] = ok ? (a < b ? a : b) * num_sms() : -1;
    }
    return cache[dev] > 0 ? cache[dev] : 0;
}

// One launch: cooperative (every CTA resident, which the gather in CTA 0
// relies on) and, where the runtime accepts both attributes, scheduled early
// behind the previous kernel of the stream (programmatic dependent launch).
template <bool kVec>
static cudaError_t launch_is_one(int64_t P, const float* lt, const float* lr, const uint8_t* mask, int64_t n,
                                 int64_t per, float log_clip, int mode, float* w, uint64_t* words,
                                 double* stats, uint32_t* err, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P);
    cfg.blockDim = dim3(kIsThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, rollout_is_kernel<kVec>, lt, lr, mask, n, per, log_clip, mode,
                                       w, words, stats, err);
    if (e == cudaSuccess) return e;
    cudaGetLastError();                                   // not accepted together: cooperative alone
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rollout_is_kernel<kVec>, lt, lr, mask, n, per, log_clip, mode, w, words,
                              stats, err);
}

cudaError_t launch_rollout_is(const float* lt, const float* lr, const uint8_t* mask, int64_t n,
                              float log_clip, int mode, float* w, double* stats, void* ws,
                              cudaStream_t st) {
    const int64_t P = rollout_is_partials(n);
    if (P > (int64_t)kIsRecsPerThread * kIsThreads) return cudaErrorInvalidValue;
    if (P > rollout_is_capacity()) return cudaErrorNotSupported;   // cannot be resident at once
    uint64_t* words = static_cast<uint64_t*>(ws);
    uint32_t* err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    if (P == 0) return cudaMemsetAsync(stats, 0, 4 * sizeof(double), st);   // no tokens: zero statistics
    const bool vec = ((reinterpret_cast<uintptr_t>(lt) | reinterpret_cast<uintptr_t>(lr) |
                       reinterpret_cast<uintptr_t>(w)) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(mask) & 3u) == 0;
    const int64_t per = rollout_is_per(n, P);
    return vec ? launch_is_one<true>(P, lt, lr, mask, n, per, log_clip, mode, w, words, stats, err, st)
               : launch_is_one<false>(P, lt, lr, mask, n, per, log_clip, mode, w, words, stats, err, st);
}

}  // namespace fp8rl
