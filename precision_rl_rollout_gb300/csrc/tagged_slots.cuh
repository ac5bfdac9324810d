// tagged_slots.cuh -- per-call tags for one-launch grid reductions.
//
// A kernel whose CTAs publish partial results for one CTA to gather keeps a
// header word and the CTAs' slots in the caller's workspace.  Each 64-bit slot
// word is tag << 32 | 32 bits of payload.  At the start every CTA reads the
// header (the tag of the previous call) and derives this call's tag; the
// gathering CTA waits until every slot word it needs carries that tag, then
// writes the header with the new tag.  Each word carries its own tag and
// payload, so the polling uses relaxed loads (which stay in flight together;
// acquire loads complete one after another), and the header is written with a
// release store, which orders the slots seen before it (a kernel that writes
// other results for the readers of the header fences those first).  A CUDA graph that replays one launch
// still gives each replay a new tag, and the workspace needs no zeroing: a
// word left by an earlier call carries an older tag.
#pragma once

#include <cstdint>

namespace fp8rl {

// The tag of the call after the one whose tag is `prev`: top bit always set,
// the low 31 bits counting up.
__device__ __forceinline__ uint32_t next_call_tag(uint32_t prev) {
    return ((prev + 1u) & 0x7FFFFFFFu) | 0x80000000u;
}

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

}  // namespace fp8rl
