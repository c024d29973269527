// wait_probe.cu — test hook for the bounded device waits that every pipelined kernel of the library
// uses (mbar_wait in common.cuh). One CTA waits on an mbarrier that no thread ever arrives at and no
// copy ever completes, so only the wait's own time limit, or the CTA's abort flag raised by a second
// warp, can end it. Either way the kernel must return and leave bit 0 (and bit 4, naming this wait)
// in the device error word, exactly as a pipeline stage that never fills would.
// The pattern follows the error-word convention of the collectives in dsv41-offload worker/tp2.py
// (a wait that gives up sets a bit the host reads, instead of trapping).
#include "common.cuh"
#include "internal.h"

namespace strata {

__global__ void __launch_bounds__(64) wait_probe_kernel(int64_t limit_ns, int64_t abort_after_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int s_abort;
    pdl_wait();
    pdl_launch();
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);  // one arrival would complete phase 0; none ever comes
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0 && !mbar_wait(smem_u32(&bar), 0, &s_abort, uint64_t(limit_ns)))
            atomicOr(&g_strata_device_error, 1 | 16);
    } else if (lane == 0 && abort_after_ns >= 0) {
        // the abort path: raise the flag after a set time (the loop is bounded by that time)
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < uint64_t(abort_after_ns)) __nanosleep(1000);
        s_abort = 1;
    }
}

cudaError_t launch_wait_probe(int64_t limit_ns, int64_t abort_after_ns, cudaStream_t stream)
{
    return launch_pdl(wait_probe_kernel, dim3(1), dim3(64), 0, stream, limit_ns, abort_after_ns);
}

cudaError_t read_device_error_probe(int* out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_strata_device_error, sizeof(int));
    if (e != cudaSuccess || !clear) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_strata_device_error, &zero, sizeof(int));
}

}  // namespace strata
