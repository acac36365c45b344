// ssm_internal.h -- launch interface between the C ABI layer (libssm.cu) and
// the kernel files. Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

// Scan tiling shared by the planner and the kernels. A tile configuration
// fixes the channels per CTA and how many threads share one channel:
//   id 0: 64 channels, 1 thread per channel      id 1: 64 channels, 2 per channel
//   id 2: 32 channels, 4 per channel             id 3: 16 channels, 8 per channel
// (dstate 16; smaller dstate always uses id 1). Tokens stream through shared
// memory in stages of kScanStageTokens; L-chunks are a whole number of stages
// so that only the sequence end is ragged.
constexpr int kScanStageTokens = 16;
constexpr int kScanTileConfigs = 4;
inline int scan_tile_channels(int cfg) {
    static const int ch[kScanTileConfigs] = {64, 64, 32, 16};
    return ch[cfg];
}
inline int scan_threads_per_channel(int cfg) {
    static const int t[kScanTileConfigs] = {1, 2, 4, 8};
    return t[cfg];
}

// Host-side plan of one scan call (pure function of the sizes and hints).
struct ScanPlan {
    int64_t chunk_len = 0;     // tokens per L-chunk
    int64_t nchunks = 0;       // L-chunks per channel
    int64_t tiles = 0;         // channel tiles per batch row
    int64_t channels_per_cta = 0;
    int tile_cfg = 1;          // tile configuration id
    int64_t ctas = 0;          // CTAs per phase kernel (tiles * batch * nchunks)
    int kernels = 0;           // launches per call
    size_t ws_bytes = 0;       // workspace bytes (0: empty problem)
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
    unsigned int* status;  // workspace status word (sticky; 0 = ok)
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

// Enqueue one full scan (all phases). io: 0 = fp32, 1 = bf16.
cudaError_t launch_scan(const ScanArgs& a, const ScanPlan& p, int io, int N, cudaStream_t s);
// Enqueue one decode step.
cudaError_t launch_state_update(const StepArgs& a, int io, int N, cudaStream_t s);

}  // namespace ssm
