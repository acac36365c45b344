// ssm_internal.h -- launch interface between the C ABI layer (libssm.cu) and
// the kernel files. Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

// Host-side plan of one scan call (pure function of the sizes).
struct ScanPlan {
    int64_t chunk_len = 0;     // tokens per L-chunk
    int64_t nchunks = 0;       // L-chunks per channel
    int64_t tiles = 0;         // channel tiles per batch row
    int64_t channels_per_cta = 0;
    int64_t ctas = 0;          // CTAs per phase kernel (tiles * batch * nchunks)
    int kernels = 0;           // launches per call
    size_t ws_bytes = 0;       // workspace bytes (0: single pass)
    size_t ws_off_H = 0;       // byte offsets inside the workspace
    size_t ws_off_S = 0;
};

// Workspace header (first 256 bytes of every non-empty workspace).
struct WsHeader {
    uint32_t status;           // SSM_OK or SSM_ERR_TIMEOUT (as uint32)
    uint32_t reserved[63];
};
constexpr size_t kWsHeaderBytes = 256;

struct ScanArgs {
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    int softplus;
    void* out;
    float* final_state;
    int64_t batch, L, dim;
    int64_t chunk_len, nchunks, tiles;
    float* ws_H;   // [batch][nchunks-1][dim][N]: chunk-local end states, then carries
    float* ws_S;   // [batch][nchunks-1][dim]: sum of dt over each chunk
};

struct StepArgs {
    float* state;
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    int softplus;
    void* out;
    int64_t batch, dim;
};

constexpr int kScanThreads = 128;   // threads per scan CTA
constexpr int kScanCPT = 2;         // channels per thread

// Enqueue one full scan (all phases). io: 0 = fp32, 1 = bf16.
cudaError_t launch_scan(const ScanArgs& a, const ScanPlan& p, int io, int N, cudaStream_t s);
// Enqueue one decode step.
cudaError_t launch_state_update(const StepArgs& a, int io, int N, cudaStream_t s);

}  // namespace ssm
