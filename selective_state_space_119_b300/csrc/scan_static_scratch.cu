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
// stand-in, not device memory), so its device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "ssm.h"

namespace {

static __device__ __align__(256) unsigned char g_scan_scratch[SSM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scan_scratch on the current device (looked up on the
// first call for that device, then cached).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_scan_scratch);
        if (e != cudaSuccess || p == nullptr) return SSM_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
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
    // is written before it is read within a call.
    return ssm_selective_scan_fwd(x, delta, A, B, C, D, z, delta_bias, delta_softplus, out,
                                  final_state, &d, stream);
}
