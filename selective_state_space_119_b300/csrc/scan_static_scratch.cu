// scan_static_scratch.cu -- ssm_selective_scan_fwd_static: the selective scan
// for callers that cannot allocate device memory.
//
// Some callers have no way to allocate: plain C hosts and plugins that live
// inside another runtime and are handed only their input and output buffers,
// and latency-critical callers that must not call cudaMalloc on the hot path
// (it can synchronize the device and can fail under memory pressure at an
// arbitrary point). For them the chunked scan's scratch (its chunk carries and
// status header) lives in a fixed-size array inside the library instead of a
// caller-supplied workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads libssm
// holds SSM_STATIC_SCRATCH_BYTES of it until the process exits. Host code may
// not pass the array's name to a kernel (on the host it names a host-side
// stand-in, not device memory), so every call looks up its device address on
// the current device with cudaGetSymbolAddress. The lookup is host work of a
// few microseconds; it is not cached, so an address from a context that was
// torn down (cudaDeviceReset) is never reused.
#include <cuda_runtime.h>

#include "ssm.h"
#include "ssm_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scan_scratch[SSM_STATIC_SCRATCH_BYTES];

// Device address of g_scan_scratch in the current context.
int scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scan_scratch);
    if (e != cudaSuccess || p == nullptr) return SSM_ERR_CUDA;
    *out = p;
    return SSM_OK;
}

}  // namespace

extern "C" int ssm_selective_scan_fwd_static(const void* x, const void* delta, const float* A,
                                             const void* B, const void* C, const float* D,
                                             const void* z, const float* delta_bias,
                                             int delta_softplus, void* out, float* final_state,
                                             const ssm_dims* dims, ssm_stream_t stream) {
    if (!dims) return SSM_ERR_NULL;
    ssm_dims d = *dims;
    d.workspace = nullptr;
    d.workspace_bytes = 0;
    const size_t need = ssm_scan_workspace_bytes(&d);
    if (need > size_t(SSM_STATIC_SCRATCH_BYTES)) return SSM_ERR_WORKSPACE;
    if (need > 0) {
        void* p = nullptr;
        const int rc = scratch_address(&p);
        if (rc != SSM_OK) return rc;
        d.workspace = p;
        d.workspace_bytes = SSM_STATIC_SCRATCH_BYTES;
    }
    // Same validation, plan and kernels as the workspace entry point; only the
    // scratch differs. Nothing in the scratch has to start at zero: every carry
    // is written before it is read within a call, and the status word at its
    // start is only ever set (by a wait that gave up) and cleared by
    // ssm_get_static_status.
    return ssm_selective_scan_fwd(x, delta, A, B, C, D, z, delta_bias, delta_softplus, out,
                                  final_state, &d, stream);
}

// The status word at the start of the library's scratch: the same word a
// caller workspace holds, read and cleared the same way as ssm_get_device_status.
extern "C" int ssm_get_static_status(ssm_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SSM_ERR_CUDA;
    void* p = nullptr;
    int rc = scratch_address(&p);
    if (rc != SSM_OK) return rc;
    uint32_t status = 0;
    if (cudaMemcpy(&status, p, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SSM_ERR_CUDA;
    if (status == 0) return SSM_OK;
    if (cudaMemset(p, 0, sizeof(status)) != cudaSuccess) return SSM_ERR_CUDA;
    return -static_cast<int>(status);
}

// For tests of the failure path on this scratch: the bounded-wait probe of
// ssm_debug_timeout_probe aimed at the library's status word.
extern "C" int ssm_debug_timeout_probe_static(uint32_t max_polls, ssm_stream_t stream) {
    if (max_polls == 0 || max_polls > (1u << 24)) return SSM_ERR_DIMS;
    void* p = nullptr;
    const int rc = scratch_address(&p);
    if (rc != SSM_OK) return rc;
    const cudaError_t e = ssm::launch_timeout_probe(static_cast<unsigned int*>(p), max_polls,
                                                    reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
