// selftest.cu -- a check of the library's failure detection that faults nothing: one CTA
// waits, with the same bounded mbarrier wait every kernel here uses, on a barrier no one
// completes. The wait gives up after the limit and the CTA records MLA_ERR_TIMEOUT (detail:
// the microseconds it waited) in the workspace error word, as a real kernel would.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mla {

namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint64_t limit_ns,
                                                                   uint32_t *err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        sm100::mbar_init(b, 1);  // one arrival expected, none ever made
        sm100::fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = sm100::globaltimer_ns();
        const bool done = sm100::mbar_wait(b, 0, &abort_flag, limit_ns);
        const uint64_t waited = sm100::globaltimer_ns() - t0;
        if (!done) flag_error(err, MLA_ERR_TIMEOUT, static_cast<uint32_t>(waited / 1000));
    }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, uint32_t *err, cudaStream_t stream) {
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace mla
