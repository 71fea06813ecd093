// k_selftest.cu -- a check of the failure path every kernel of the library
// relies on: one warp waits on an mbarrier phase that nothing completes.  The
// bounded wait must give up after its time limit (kWaitTimeoutNs of global
// time), record kErrWaitTimeout in the device error word and return, so the
// kernel ends and the context stays usable.  Nothing faults, traps or spins
// without a limit.
#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

__device__ uint32_t g_gave_up;   // 1 once the wait has given up, 2 if it (wrongly) completed

__global__ void __launch_bounds__(32) wait_selftest(uint32_t *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);   // one arrival expected; none is made
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(smem_u32(&bar), 0, err);
    if (threadIdx.x == 0) g_gave_up = ok ? 2u : 1u;
}

}  // namespace

cudaError_t run_wait_selftest(uint32_t *err, bool *gave_up, cudaStream_t s) {
    const uint32_t zero = 0;
    cudaError_t e = cudaMemcpyToSymbolAsync(g_gave_up, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    wait_selftest<<<1, 32, 0, s>>>(err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    uint32_t v = 0;
    e = cudaMemcpyFromSymbolAsync(&v, g_gave_up, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *gave_up = v == 1u;
    return cudaSuccess;
}

}  // namespace da
