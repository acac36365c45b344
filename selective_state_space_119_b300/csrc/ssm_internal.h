// ssm_internal.h -- launch interface between the C ABI layer (libssm.cu) and
// the kernel files. Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

// Scan tiling shared by the planner and the kernels. A CTA has SW "state"
// warps, which run the recurrence, and RW "row" warps, which stage the inputs,
// compute dt and write the gated output. NS lanes of a state warp share one
// channel's N states (each holds N / NS of them), so a state warp covers
// 32 / NS channels and a CTA SW * 32 / NS channels:
//   id 0: NS 4, SW 4, RW 2   id 1: NS 8, SW 4, RW 2
//   id 2: NS 4, SW 2, RW 1   id 3: NS 2, SW 4, RW 2
// For N < NS the lanes per channel drop to N, and a CTA keeps at most 64
// channels. Tokens stream through shared memory in stages of kScanStageTokens;
// L-chunks are a whole number of stages so that only the sequence end is
// ragged.
constexpr int kScanStageTokens = 32;
constexpr int kScanTileConfigs = 4;
inline int scan_lanes_per_channel(int cfg, int64_t N) {
    static const int ns[kScanTileConfigs] = {4, 8, 4, 2};
    return ns[cfg] < N ? ns[cfg] : static_cast<int>(N);
}
inline int scan_tile_channels(int cfg, int64_t N) {
    static const int sw[kScanTileConfigs] = {4, 4, 2, 4};
    const int cpw = 32 / scan_lanes_per_channel(cfg, N);
    const int warps = sw[cfg] * cpw <= 64 ? sw[cfg] : (64 / cpw > 0 ? 64 / cpw : 1);
    return warps * cpw;
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
