// Self-test of the device error path: a bounded wait that runs out.
//
// Every wait of the library's kernels on an mbarrier is bounded: after the limit
// it raises MSA_FLAG_TIMEOUT in the caller's error word and the kernel drains and
// returns, so the context stays usable and msa_check reports MSA_ERR_TIMEOUT.
// This kernel exercises exactly that path without any fault: one thread waits
// on an mbarrier that nothing ever arrives on.
#include "msa_device.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

__global__ void __launch_bounds__(32) k_selftest_timeout(int32_t *err) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort = 0;
        fence_mbar_init();
    }
    __syncwarp();
    // phase 0 of `bar` never completes: the wait gives up after its limit
    if (threadIdx.x == 0) mbar_wait(&bar, 0, err, &abort);
}

}  // namespace

cudaError_t launch_selftest_timeout(int32_t *err, cudaStream_t st) {
    k_selftest_timeout<<<1, 32, 0, st>>>(err);
    return cudaGetLastError();
}

}  // namespace msa
