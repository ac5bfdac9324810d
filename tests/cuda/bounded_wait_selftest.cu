// Test-only kernel: exercises the library's bounded mbarrier waits on a
// barrier that nothing completes, so every wait must give up after its limit
// and report it, and the CUDA context must stay usable afterwards.
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm100_ptx.cuh"

using namespace fp8rl::sm100;

// out[0]: 1 if the bounded wait reported success (it must not), 0 if it gave up
// out[1]: elapsed ns of the bounded wait;  out[2]: elapsed ns of the drain
__global__ void bounded_wait_kernel(uint64_t limit_ns, unsigned long long* out) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = globaltimer_ns();
        const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, limit_ns);   // nobody arrives
        const uint64_t t1 = globaltimer_ns();
        mbar_drain(smem_u32(&bar), 0, limit_ns);
        const uint64_t t2 = globaltimer_ns();
        out[0] = ok ? 1ull : 0ull;
        out[1] = t1 - t0;
        out[2] = t2 - t1;
    }
}

extern "C" int run_bounded_wait(unsigned long long limit_ns, unsigned long long* out_device) {
    bounded_wait_kernel<<<1, 32>>>(limit_ns, out_device);
    return (int)cudaGetLastError();
}
