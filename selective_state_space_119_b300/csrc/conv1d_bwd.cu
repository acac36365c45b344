// conv1d_bwd.cu -- gradients of the Mamba block's input stage, the causal
// depthwise conv1d followed by SiLU ("State Space Models -- Mamba, S4, and
// Beyond", "Mamba (S6 -- Selective State Space)", MambaBlock: Conv1d of width
// d_conv, padding d_conv - 1 cut back to seq_len, then F.silu), for a loss
// whose gradient with respect to the stage's output u is du. Per channel d:
//   pre_t  = bias + sum_{k<K} w[k] x_{t-K+1+k},   u_t = silu(pre_t)
//   dpre_t = du_t * silu'(pre_t),  silu'(p) = s (1 + p (1 - s)), s = sigmoid(p)
//   dx_s   = sum_{k<K} w[k] dpre_{s+K-1-k}        (terms past the sequence end are 0)
//   dw[k]  = sum_{b,t} dpre_t x_{t-K+1+k},   dbias = sum_{b,t} dpre_t
// (the chain rule on the forward's loop; the same derivative the training
// section's "gradient flows through" asks of every stage.)
//
// Like the forward, a thread owns a vector of VE consecutive channels and a run
// of kRun tokens; it loads the x rows its run and the K - 1 tokens on either
// side need, and the du rows of its run and the K - 1 after it, forms dpre on
// those kRun + K - 1 tokens, and writes dx of its run. dw and dbias of the
// run's own tokens are summed over the CTA's warps in shared memory and written
// as the CTA's share; a second kernel adds the shares of every (batch row,
// token block) in a fixed order, so the sums do not depend on scheduling.
#include <cuda_bf16.h>


#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kThreads = 128;                // 3 CTAs (12 warps) per SM at <= 170 registers
constexpr int kRun = 8;                      // tokens per thread
constexpr int kRuns = kThreads / 32;         // runs (warps) per CTA
constexpr int kVE = 4;                       // channels per thread

template <typename T>
__device__ __forceinline__ void ld4ch(const T* p, float (&v)[kVE]) {
    if constexpr (sizeof(T) == 2) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
        const float4 u = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
}

template <typename T>
__device__ __forceinline__ void st4ch(T* p, const float (&v)[kVE]) {
    if constexpr (sizeof(T) == 2) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
        *reinterpret_cast<uint2*>(p) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
    } else {
        *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// silu'(p) = sigmoid(p) (1 + p (1 - sigmoid(p)))
__device__ __forceinline__ float dsilu(float p) {
    const float s = __fdividef(1.f, 1.f + __expf(-p));
    return s * fmaf(p, 1.f - s, 1.f);
}

template <typename T, int K, int RUN = kRun, int THREADS = kThreads, int MINB = 3>
__global__ void __launch_bounds__(THREADS, MINB) conv1d_silu_bwd_kernel(const ConvBwdArgs a) {
    constexpr int kRun = RUN;
    constexpr int kRuns = THREADS / 32;
    constexpr int NX = kRun + 2 * (K - 1);   // x rows: t0 - K + 1 .. t0 + kRun + K - 2
    constexpr int ND = kRun + K - 1;         // du / dpre rows: t0 .. t0 + kRun + K - 2
    __shared__ float s_part[kRuns][32][kVE * (K + 1)];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t G = a.dim / kVE;
    const int64_t GB = (G + 31) / 32;
    const int64_t RB = (a.L + kRun * kRuns - 1) / (kRun * kRuns);
    const int64_t gb = blockIdx.x % GB, rest = blockIdx.x / GB;
    const int64_t rb = rest % RB, b = rest / RB;
    const int64_t g = gb * 32 + lane;
    const bool ch_ok = g < G;
    const int64_t d0 = (ch_ok ? g : 0) * kVE;
    const int64_t t0 = (rb * kRuns + warp) * kRun;
    const bool active = ch_ok && t0 < a.L;
    const T* x = static_cast<const T*>(a.x) + b * a.L * a.dim + d0;
    const T* du = static_cast<const T*>(a.du) + b * a.L * a.dim + d0;

    float w[kVE][K], bias[kVE];
#pragma unroll
    for (int c = 0; c < kVE; ++c) {
#pragma unroll
        for (int k = 0; k < K; ++k) w[c][k] = __ldg(a.w + (d0 + c) * K + k);
        bias[c] = a.b ? __ldg(a.b + d0 + c) : 0.f;
    }
    float xr[NX][kVE], dp[ND][kVE];
#pragma unroll
    for (int i = 0; i < NX; ++i) {
        const int64_t t = t0 - (K - 1) + i;
        if (active && t >= 0 && t < a.L) {
            ld4ch<T>(x + t * a.dim, xr[i]);
        } else {
#pragma unroll
            for (int c = 0; c < kVE; ++c) xr[i][c] = 0.f;
        }
    }
#pragma unroll
    for (int i = 0; i < ND; ++i) {
        const int64_t t = t0 + i;
        if (active && t < a.L) {
            ld4ch<T>(du + t * a.dim, dp[i]);
        } else {
#pragma unroll
            for (int c = 0; c < kVE; ++c) dp[i][c] = 0.f;
        }
    }
    // dpre on tokens t0 .. t0 + ND - 1 (du is 0 past the end: dpre 0 there)
#pragma unroll
    for (int i = 0; i < ND; ++i) {
#pragma unroll
        for (int c = 0; c < kVE; ++c) {
            float pre = bias[c];
#pragma unroll
            for (int k = 0; k < K; ++k) pre = fmaf(w[c][k], xr[i + k][c], pre);   // x_{t-K+1+k}
            dp[i][c] *= dsilu(pre);
        }
    }
    // dx of the run's tokens
    if (active) {
        T* dx = static_cast<T*>(a.dx) + b * a.L * a.dim + d0;
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
            if (t0 + j >= a.L) break;
            float v[kVE];
#pragma unroll
            for (int c = 0; c < kVE; ++c) {
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < K; ++k) acc = fmaf(w[c][k], dp[j + K - 1 - k][c], acc);
                v[c] = acc;
            }
            st4ch<T>(dx + (t0 + j) * a.dim, v);
        }
    }
    // this run's share of dw and dbias (its own tokens only)
    float part[kVE * (K + 1)];
#pragma unroll
    for (int c = 0; c < kVE; ++c) {
#pragma unroll
        for (int k = 0; k <= K; ++k) part[c * (K + 1) + k] = 0.f;
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
#pragma unroll
            for (int k = 0; k < K; ++k)
                part[c * (K + 1) + k] = fmaf(dp[j][c], xr[j + k][c], part[c * (K + 1) + k]);
            part[c * (K + 1) + K] += dp[j][c];
        }
    }
#pragma unroll
    for (int i = 0; i < kVE * (K + 1); ++i) s_part[warp][lane][i] = part[i];
    __syncthreads();
    // the CTA's share: warps summed in order, one channel vector per thread of warp 0
    if (warp == 0 && ch_ok) {
        float* dst = a.part + ((b * RB + rb) * a.dim + d0) * (K + 1);
#pragma unroll
        for (int i = 0; i < kVE * (K + 1); ++i) {
            float s = 0.f;
#pragma unroll
            for (int r = 0; r < kRuns; ++r) s += s_part[r][lane][i];
            dst[i] = s;   // [channel][K + 1]: dw[0..K-1], dbias
        }
    }
}

// dw[d][k] and dbias[d]: the shares of every (batch row, token block). A CTA
// owns 32 outputs; its 8 warps sum the rows q = w, w + 8, w + 16, ... of each
// (4 running sums each, added in order), and warp 0 adds the 8 slices in
// order: a fixed order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(256) conv1d_bwd_reduce_kernel(const ConvBwdArgs a,
                                                                 int64_t nblocks, int K) {
    constexpr int kSlices = 8;
    __shared__ float s_slice[kSlices][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t n = a.dim * (K + 1);
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 32 + lane;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (i < n) {
        int64_t q = w;
        for (; q + 3 * kSlices < nblocks; q += 4 * kSlices) {
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] += a.part[(q + j * kSlices) * n + i];
        }
        for (int j = 0; q < nblocks; q += kSlices, ++j) acc[j] += a.part[q * n + i];
    }
    s_slice[w][lane] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    __syncthreads();
    if (w == 0 && i < n) {
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < kSlices; ++r) s += s_slice[r][lane];
        const int64_t d = i / (K + 1), k = i % (K + 1);
        if (k < K)
            a.dw[d * K + k] = s;
        else if (a.db)
            a.db[d] = s;
    }
}

template <typename T, int K>
cudaError_t launch_bwd_k(const ConvBwdArgs& a, cudaStream_t s) {
    const int64_t G = a.dim / kVE;
    const int64_t GB = (G + 31) / 32;
    const int64_t RB = (a.L + kRun * kRuns - 1) / (kRun * kRuns);
    const int64_t blocks = a.batch * RB * GB;
    if (blocks >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
    conv1d_silu_bwd_kernel<T, K><<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(a);
    const int64_t n = a.dim * (K + 1);
    const int64_t rblocks = (n + 31) / 32;
    if (rblocks >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
    conv1d_bwd_reduce_kernel<<<static_cast<unsigned>(rblocks), 256, 0, s>>>(a, a.batch * RB, K);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_typed(const ConvBwdArgs& a, cudaStream_t s) {
    switch (a.k) {
        case 1: return launch_bwd_k<T, 1>(a, s);
        case 2: return launch_bwd_k<T, 2>(a, s);
        case 3: return launch_bwd_k<T, 3>(a, s);
        case 4: return launch_bwd_k<T, 4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t conv1d_bwd_partial_floats(int64_t batch, int64_t L, int64_t dim, int k) {
    const int64_t RB = (L + kRun * kRuns - 1) / (kRun * kRuns);
    return size_t(batch) * size_t(RB) * size_t(dim) * size_t(k + 1);
}

cudaError_t launch_conv1d_silu_bwd(const ConvBwdArgs& a, int io, cudaStream_t s) {
    return io == 1 ? launch_bwd_typed<__nv_bfloat16>(a, s) : launch_bwd_typed<float>(a, s);
}

}  // namespace ssm
