// kda_selftest.cu -- a check that the library's device-side waits give up.
//
// Every wait in the tensor-core prefill is bounded: after a time limit it
// records KDA_DEVICE_TIMEOUT in the workspace status word and the CTA leaves
// instead of hanging.  This entry point exercises that path on purpose with a
// barrier that nothing ever arrives on, so a caller (and the test suite) can
// see the timeout reported without any fault.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = tc::smem_u32(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    // phase 0 never completes: no thread arrives and no copy is in flight
    if (threadIdx.x == 0 && !tc::mbar_wait(b, 0, limit_ns)) flag_status(status, KDA_DEVICE_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t limit_ns, int32_t *status, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
