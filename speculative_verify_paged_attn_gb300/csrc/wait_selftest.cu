// wait_selftest.cu -- a diagnostic of the device-side wait limit.
//
// Every wait in the library's kernels is an mbarrier wait bounded in wall
// time (mbar_wait); when the limit passes, the kernel raises
// SVPA_DEVERR_TIMEOUT, releases what it holds and returns, so that the host
// reads a status instead of finding a hung GPU.  svpa_wait_selftest runs that
// path on purpose: one CTA allocates tensor memory, waits with the same
// mbar_wait, under a caller-chosen limit, on an mbarrier that no thread ever
// arrives on, then frees the tensor memory and returns.  No copy is in flight
// while it waits.
#include "svpa_device.cuh"
#include "svpa_internal.h"

namespace svpa {

namespace {

__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(unsigned long long limit_ns, int32_t *err,
                                                              int32_t *reached) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival completes a phase; none ever comes
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        // the wait runs out after limit_ns, raises SVPA_DEVERR_TIMEOUT and
        // returns false; reaching the line below shows it returned
        const bool done = mbar_wait(&bar, 0, err, limit_ns);
        atomicAdd(reached, done ? 2 : 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 32);
}

}  // namespace

}  // namespace svpa

extern "C" {

svpa_status svpa_wait_selftest(uint64_t limit_ns, int32_t *error_flag, int32_t *reached, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_wait_selftest");
    if (!error_flag || !reached || limit_ns == 0 || limit_ns > 10000000000ull) return SVPA_ERR_INVALID_ARG;
    svpa::wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, error_flag, reached);
    return cudaGetLastError() == cudaSuccess ? SVPA_OK : SVPA_ERR_CUDA;
}

}  // extern "C"
