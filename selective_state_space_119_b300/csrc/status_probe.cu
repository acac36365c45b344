// status_probe.cu -- a kernel for tests of the failure path.
//
// It waits, with the same bounded mbarrier wait the scan kernels use on their
// TMA copies, on a barrier that nothing ever arrives on, gives up after
// max_polls probes and sets the workspace status word exactly as a scan kernel
// whose copy never landed would. Nothing faults and nothing hangs: the wait is
// bounded, the CTA returns, and the context stays usable.
#include <cuda_runtime.h>

#include "ssm_internal.h"
#include "ssm_tma.cuh"

namespace ssm {
namespace {

constexpr uint32_t kStatusTimeout = 7;    // -SSM_ERR_TIMEOUT

__global__ void timeout_probe_kernel(unsigned int* status, uint32_t max_polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // phase 0 of a fresh barrier completes only when one arrival lands: none does
    const bool ok = mbar_wait_bounded(&bar, 0u, max_polls);
    if (!ok && threadIdx.x == 0) atomicExch(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_timeout_probe(unsigned int* status, uint32_t max_polls, cudaStream_t s) {
    timeout_probe_kernel<<<1, 32, 0, s>>>(status, max_polls);
    return cudaGetLastError();
}

}  // namespace ssm
