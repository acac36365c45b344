// conv1d.cu -- the Mamba block's input stage on its own: causal depthwise
// conv1d followed by SiLU.
//
// "State Space Models -- Mamba, S4, and Beyond", "Mamba (S6 -- Selective
// State Space)", MambaBlock: a depthwise Conv1d of width d_conv (4 there) with
// d_conv - 1 zeros of padding on the left, cut back to seq_len, then SiLU.
// Its output u feeds both x_proj (which forms delta, B and C from it) and the
// scan, so u has to exist in memory before the scan starts. Per channel d and
// token t, with x = 0 before the first token:
//   u[b,t,d] = silu(bias[d] + sum_{k<K} w[d,k] * x[b, t-K+1+k, d])
//
// The op is bound by HBM: one read of x and one write of u per element. A
// thread owns one 16-byte vector of channels (8 bf16 or 4 fp32) and a run of
// kRun consecutive tokens. It issues every load of the run, with the 3 rows
// before it, ahead of any arithmetic (kRun + 3 independent 16-byte loads in
// flight per thread) and keeps the window in registers. A CTA is 32 lanes of
// consecutive channel vectors (a warp's load of one row is 512 contiguous
// bytes) by 4 warps of consecutive runs; the halo rows a run re-reads were
// loaded by the warp before it and come from L1/L2. The taps of the CTA's
// channels are one contiguous block of [channel][K] floats: they are staged
// through shared memory with coalesced loads (per-lane loads of them would
// touch 32 cache lines per instruction), at an odd float4 stride per lane so
// that the lanes' 16-byte reads do not conflict. K is a template parameter.
#include <cuda_bf16.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kConvThreads = 128;   // (a launch-shape sweep on b4 L2048 d1536: 128 x 4 per SM best)
constexpr int kRun = 8;                    // tokens per thread
constexpr int kHalo = kMaxConvK - 1;       // rows before the run

// The 16 bytes of one load as VE fp32 values.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& r, float (&v)[16 / sizeof(T)]) {
    if constexpr (sizeof(T) == 2) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
        v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
        v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
    }
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float (&v)[16 / sizeof(T)]) {
    if constexpr (sizeof(T) == 2) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&p);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu on a pair, with packed FP32 arithmetic: z / (1 + 2^(-z log2 e)); below
// z = -88 the exponential is inf, its reciprocal 0 and the result -0.
__device__ __forceinline__ float2 silu2(float2 z) {
    const float2 s = __fmul2_rn(z, make_float2(-kLog2e, -kLog2e));
    const float2 d = __ffma2_rn(make_float2(ex2(s.x), ex2(s.y)), make_float2(1.f, 1.f),
                                make_float2(1.f, 1.f));
    return __fmul2_rn(z, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

template <typename T, int K, int RUN = kRun, int THREADS = kConvThreads, int MINB = 4>
__global__ void __launch_bounds__(THREADS, MINB) conv1d_silu_kernel(const ConvArgs a) {
    constexpr int kRun = RUN;
    constexpr int kConvThreads = THREADS;
    constexpr int VE = 16 / sizeof(T);     // channels per thread
    constexpr int NF = VE * K / 4;         // float4 of taps per lane
    constexpr int NFP = NF + 1;            // padded lane stride in shared memory
    constexpr int RUNS = kConvThreads / 32;
    __shared__ float4 s_w[32 * NFP];
    __shared__ float4 s_b[32 * VE / 4];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t G = a.dim / VE;          // channel vectors per token
    const int64_t GB = (G + 31) / 32;      // channel blocks
    const int64_t RB = (a.L + kRun * RUNS - 1) / (kRun * RUNS);
    const int64_t gb = blockIdx.x % GB, rest = blockIdx.x / GB;
    const int64_t rb = rest % RB, b = rest / RB;
    const int64_t g0 = gb * 32;
    const int nvalid = static_cast<int>(G - g0 < 32 ? G - g0 : 32);
    const int64_t d0 = (g0 + lane) * VE;
    const int64_t t0 = (rb * RUNS + warp) * kRun;
    const bool active = lane < nvalid && t0 < a.L;
    const T* x = static_cast<const T*>(a.x) + b * a.L * a.dim + d0;
    T* u = static_cast<T*>(a.u) + b * a.L * a.dim + d0;

    // rows t0 - kHalo .. t0 + kRun - 1, zero outside [0, L)
    uint4 raw[kHalo + kRun];
#pragma unroll
    for (int i = 0; i < kHalo + kRun; ++i) {
        const int64_t t = t0 - kHalo + i;
        raw[i] = (active && t >= 0 && t < a.L)
                     ? __ldg(reinterpret_cast<const uint4*>(x + t * a.dim))
                     : make_uint4(0u, 0u, 0u, 0u);
    }
    // The block's taps ([channel][K], contiguous for its 32 channel vectors)
    // and bias, staged through shared memory with coalesced 16-byte loads.
    const float4* wsrc = reinterpret_cast<const float4*>(a.w + g0 * VE * K);
    for (int i = threadIdx.x; i < nvalid * NF; i += kConvThreads)
        s_w[(i / NF) * NFP + i % NF] = __ldg(wsrc + i);
    if (a.b) {
        const float4* bsrc = reinterpret_cast<const float4*>(a.b + g0 * VE);
        for (int i = threadIdx.x; i < nvalid * VE / 4; i += kConvThreads) s_b[i] = __ldg(bsrc + i);
    }
    __syncthreads();
    if (!active) return;

    // taps and bias of channel pairs (c, c + 1), for packed FP32 arithmetic
    float tap[VE * K], bias[VE];
#pragma unroll
    for (int j = 0; j < NF; ++j) {
        const float4 v = s_w[lane * NFP + j];
        tap[4 * j] = v.x; tap[4 * j + 1] = v.y; tap[4 * j + 2] = v.z; tap[4 * j + 3] = v.w;
    }
#pragma unroll
    for (int j = 0; j < VE / 4; ++j) {
        const float4 v = a.b ? s_b[lane * (VE / 4) + j] : make_float4(0.f, 0.f, 0.f, 0.f);
        bias[4 * j] = v.x; bias[4 * j + 1] = v.y; bias[4 * j + 2] = v.z; bias[4 * j + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < kRun; ++i) {
        float2 acc[VE / 2];
#pragma unroll
        for (int c = 0; c < VE / 2; ++c) acc[c] = make_float2(bias[2 * c], bias[2 * c + 1]);
        // tap k multiplies the row K - 1 - k tokens before t (row kHalo + i is t)
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float v[VE];
            unpack16<T>(raw[kHalo + i - (K - 1) + k], v);
#pragma unroll
            for (int c = 0; c < VE / 2; ++c)
                acc[c] = __ffma2_rn(make_float2(tap[2 * c * K + k], tap[(2 * c + 1) * K + k]),
                                    make_float2(v[2 * c], v[2 * c + 1]), acc[c]);
        }
        float o[VE];
#pragma unroll
        for (int c = 0; c < VE / 2; ++c) {
            const float2 r = silu2(acc[c]);
            o[2 * c] = r.x;
            o[2 * c + 1] = r.y;
        }
        if (t0 + i < a.L) *reinterpret_cast<uint4*>(u + (t0 + i) * a.dim) = pack16<T>(o);
    }
}

template <typename T, int K>
cudaError_t launch_k(const ConvArgs& a, cudaStream_t s) {
    constexpr int VE = 16 / sizeof(T);
    constexpr int RUNS = kConvThreads / 32;
    const int64_t GB = (a.dim / VE + 31) / 32;
    const int64_t RB = (a.L + kRun * RUNS - 1) / (kRun * RUNS);
    const int64_t blocks = a.batch * RB * GB;
    if (blocks >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
    conv1d_silu_kernel<T, K><<<static_cast<unsigned>(blocks), kConvThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const ConvArgs& a, cudaStream_t s) {
    switch (a.k) {
        case 1: return launch_k<T, 1>(a, s);
        case 2: return launch_k<T, 2>(a, s);
        case 3: return launch_k<T, 3>(a, s);
        case 4: return launch_k<T, 4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_conv1d_silu(const ConvArgs& a, int io, cudaStream_t s) {
    return io == 1 ? launch_typed<__nv_bfloat16>(a, s) : launch_typed<float>(a, s);
}

}  // namespace ssm
