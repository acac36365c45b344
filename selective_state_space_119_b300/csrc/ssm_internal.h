// ssm_internal.h -- launch interface between the C ABI layer (libssm.cu) and
// the kernel files. Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

// Scan tiling shared by the planner and the kernels. Every lane of the scan
// owns one channel (and, with its partner lane, the states of a channel
// pair); a CTA has W warps, so it covers 32 * W channels of one batch row and
// one L-chunk:
//   id 0: W 4 (128 channels)   id 1: W 2 (64)   id 2: W 1 (32)   id 3: W 3 (96)
// B_t / C_t rows go through shared memory in stages of kScanStageTokens;
// L-chunks are a whole number of stages so that only the sequence end is
// ragged.
constexpr int kScanStageTokens = 32;
constexpr int kScanTileConfigs = 4;
inline int scan_tile_channels(int cfg) {
    static const int w[kScanTileConfigs] = {4, 2, 1, 3};
    return 32 * w[cfg];
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
    const float* h0;  // [batch][dim][N] state before the first token, or NULL (zero)
    const float* conv_w;  // [dim][conv_k] causal conv taps of the fused input stage, or NULL
    const float* conv_b;  // [dim] conv bias, or NULL
    int conv_k;           // conv width (1 .. 4) when conv_w is given
    float* ckpt;          // [batch][nckpt][dim][N]: state before every kCkptTokens-th token, or NULL
    int64_t nckpt;        // ceil(L / kCkptTokens)
    int zoh;              // exact zero-order-hold Bbar instead of dt * B
    float* ws_H;   // [batch][nchunks-1][dim][N]: chunk-local end states (from h = 0)
    float* ws_S;   // [batch][nchunks-1][dim]: sum of dt over each chunk
    unsigned int* status;  // workspace status word (sticky; 0 = ok; no current kernel sets it)
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
    int zoh;              // exact zero-order-hold Bbar instead of dt * B
    int bc_per_channel;   // B, C of shape [batch, dim, N] instead of [batch, N]
};

// Tokens between two saved states of a checkpointing forward (the backward
// recomputes the states in between). Chunks and stages are multiples of it.
constexpr int kCkptTokens = 8;
static_assert(kScanStageTokens % kCkptTokens == 0, "stages start on a checkpoint");

// Widest causal conv of the Mamba block's input stage (d_conv = 4 on the pages).
constexpr int kMaxConvK = 4;

struct ConvArgs {
    const void* x;          // [batch][L][dim]
    const float* w;         // [dim][k]
    const float* b;         // [dim] or NULL
    void* u;                // [batch][L][dim]
    int64_t batch, L, dim;
    int k;
};

// Gradients of the input stage for dLoss/du = du.
struct ConvBwdArgs {
    const void* x;          // [batch][L][dim]
    const float* w;         // [dim][k]
    const float* b;         // [dim] or NULL
    const void* du;         // [batch][L][dim]
    void* dx;               // [batch][L][dim]
    float* dw;              // [dim][k]
    float* db;              // [dim] or NULL
    float* part;            // workspace: the per-block shares of dw | dbias
    int64_t batch, L, dim;
    int k;
};
// fp32 values of the per-block shares (the workspace after its header).
size_t conv1d_bwd_partial_floats(int64_t batch, int64_t L, int64_t dim, int k);
cudaError_t launch_conv1d_silu_bwd(const ConvBwdArgs& a, int io, cudaStream_t s);

// The gradient pass of the scan (dstate 16). Chunking follows the forward's
// plan with 128-channel tiles.
struct BwdArgs {
    const void* x;
    const void* delta;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* delta_bias;
    int softplus;
    const float* ckpt;    // [batch][nckpt][dim][N] from the checkpointing forward
    int64_t nckpt;
    const void* dout;     // [batch][L][dim]
    const float* dfinal;  // [batch][dim][N] or NULL
    void* dx;             // [batch][L][dim] io
    void* ddelta;
    void* dz;             // NULL without the gate
    float* dh0;           // [batch][dim][N] or NULL
    void* dB;             // [batch][L][N] io ([batch][L][dim][N] with per-channel rows)
    void* dC;
    float* dA;            // [dim][N]
    float* dD;            // [dim] or NULL
    float* dbias;         // [dim] or NULL
    int64_t batch, L, dim;
    int64_t chunk_len, nchunks, tiles;
    int zoh;              // exact zero-order-hold input term
    // workspace
    float* wsQ;    // [batch][nchunks-1][dim][N]: reverse carry of chunks 1.. from zero
    float* wsS;    // [batch][nchunks-1][dim]: sum of dt over those chunks
    float* pBC;    // [batch][tiles][L][2N]: each tile's share of dB | dC
    float* pA;     // [batch][nchunks][dim][N]
    float* pD;     // [batch][nchunks][dim]
    float* pbias;  // [batch][nchunks][dim]
};

// Enqueue one full scan (all phases). io: 0 = fp32, 1 = bf16.
cudaError_t launch_scan(const ScanArgs& a, const ScanPlan& p, int io, int N, cudaStream_t s);
// The same for dstate 16 with 128-channel tiles and no fused input stage,
// checkpoints or variant (one lane per channel, structured-A fast path).
cudaError_t launch_scan16(const ScanArgs& a, const ScanPlan& p, int io, cudaStream_t s);
// Enqueue one decode step.
cudaError_t launch_state_update(const StepArgs& a, int io, int N, cudaStream_t s);
// Enqueue the scan with per-channel B and C ([batch][L][dim][N], dstate 16).
cudaError_t launch_scan_bcd(const ScanArgs& a, const ScanPlan& p, int io, cudaStream_t s);
// Enqueue the gradient passes (reverse carries, gradients, reduction).
cudaError_t launch_scan_bwd(const BwdArgs& a, int io, cudaStream_t s);
// The same for per-channel B and C (dB, dC [batch][L][dim][N]; pBC unused).
cudaError_t launch_scan_bcd_bwd(const BwdArgs& a, int io, cudaStream_t s);
// Mamba-2's SSD layer (bf16 I/O, d_head 64, d_state 128): one launch.
struct SsdLaunch {
    const void* x;            // [batch, L, H, 64] bf16
    const void* dt;           // [batch, L, H] bf16
    const float* A;           // [H]
    const void* B;            // [batch, L, G, 128] bf16
    const void* C;
    const float* D;           // [H] or NULL
    const float* dt_bias;     // [H] or NULL
    int softplus;
    const float* h0;          // [batch, H, 64, 128] or NULL
    void* y;                  // [batch, L, H, 64] bf16
    float* final_state;       // [batch, H, 64, 128] or NULL
    int64_t batch, L, H, G;
    unsigned int* status;     // workspace status word
};
cudaError_t launch_ssd(const SsdLaunch& l, cudaStream_t s);

// Enqueue the failure-path probe: a bounded wait that runs out and sets *status.
cudaError_t launch_timeout_probe(unsigned int* status, uint32_t max_polls, cudaStream_t s);
// Enqueue the standalone causal depthwise conv1d + SiLU.
cudaError_t launch_conv1d_silu(const ConvArgs& a, int io, cudaStream_t s);

}  // namespace ssm
