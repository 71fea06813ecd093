// k_selftest.cu -- checks of the failure paths every kernel of the library
// relies on.  Wait: one warp waits on an mbarrier phase that nothing
// completes; the bounded wait must give up after its time limit
// (kWaitTimeoutNs of global time), record kErrWaitTimeout in the error word
// and return, so the kernel ends and the context stays usable.  Bounds: one
// warp tests an index past the end of a buffer through DA_CHECK.  Nothing
// faults, traps, writes out of range or spins without a limit.
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

__device__ uint32_t g_bounds_buf[32];
__device__ uint32_t g_bounds_passed;

// Lane l writes entry l + 1 of the 32-entry buffer: lane 31's index is one
// past the end.  The write happens only where the plain test passes too, so
// the release build (where DA_CHECK is true) writes nothing out of range
// either; the debug build records kErrBounds for lane 31.
__global__ void __launch_bounds__(32) bounds_selftest(uint32_t *err) {
    const int idx = static_cast<int>(threadIdx.x) + 1;
    const bool inside = idx < 32;
    const bool checked = DA_CHECK(inside, err);
    if (inside && checked) g_bounds_buf[idx] = 1u;
    if (!inside && checked && kDebugChecks) atomicOr(&g_bounds_passed, 1u);   // the check let it through
}

}  // namespace

cudaError_t run_bounds_selftest(uint32_t *err, bool *wrote, cudaStream_t s) {
    const uint32_t zero = 0;
    cudaError_t e = cudaMemcpyToSymbolAsync(g_bounds_passed, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    bounds_selftest<<<1, 32, 0, s>>>(err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    uint32_t v = 0;
    e = cudaMemcpyFromSymbolAsync(&v, g_bounds_passed, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *wrote = v != 0;   // an index past the end passed the check
    return cudaSuccess;
}

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
