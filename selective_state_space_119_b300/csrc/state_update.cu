// state_update.cu -- one token of recurrent generation on a cached state.
//
// "State-space models (Mamba, S4)", "Training vs Inference Modes": keep h,
// take the new token, h <- Abar h + Bbar x, y = C h, O(1) work per token.
// With the selective parameters of "State Space Models -- Mamba, S4, and
// Beyond", "Mamba (S6 -- Selective State Space)", this is one t-iteration of
// the scan: dt = softplus?(delta + bias), h <- exp(dt A[d,:]) h + dt B x,
// y = C . h + D x, out = y * silu(z); the fp32 state is updated in place.
//
// The step is bound by HBM traffic on the state (N fp32 read + written per
// channel). L = N / kNPL lanes share a channel, each holding kNPL = 4 states
// (one 128-bit load and store), so a warp reads and writes 512 contiguous
// bytes of state per instruction. The partial C . h sums meet through
// butterfly shuffles; lane 0 of each group writes y.
#include <cuda_bf16.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kStepThreads = 256;

template <typename T, int N>
__global__ void __launch_bounds__(kStepThreads) state_update_kernel(const StepArgs a) {
    constexpr int NPL = N >= 4 ? 4 : N;        // states per lane
    constexpr int LANES = N / NPL;             // lanes per channel (1, 2 or 4)
    constexpr int CH_PER_CTA = kStepThreads / LANES;

    const int lane_in_ch = threadIdx.x % LANES;
    const int64_t ch = static_cast<int64_t>(blockIdx.x) * CH_PER_CTA + threadIdx.x / LANES;
    const int64_t nch = a.batch * a.dim;
    // Whole groups of LANES lanes share the same `ch`, so the shuffle below
    // always runs with every participant present.
    const bool active = ch < nch;
    const int64_t b = active ? ch / a.dim : 0;
    const int64_t d = active ? ch % a.dim : 0;
    const int n0 = lane_in_ch * NPL;

    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ delta = static_cast<const T*>(a.delta);
    const T* __restrict__ Bg = static_cast<const T*>(a.B);
    const T* __restrict__ Cg = static_cast<const T*>(a.C);
    const T* __restrict__ z = static_cast<const T*>(a.z);

    float y = 0.f, xv = 0.f;
    if (active) {
        xv = IO<T>::ld(x + ch);
        float dt = IO<T>::ld(delta + ch);
        if (a.delta_bias) dt += __ldg(a.delta_bias + d);
        if (a.softplus) dt = softplus(dt);
        const float dtx = dt * xv;

        float h[NPL], A2[NPL];
        float* st = a.state + ch * N + n0;
        if constexpr (NPL == 4) {
            const float4 hv = *reinterpret_cast<const float4*>(st);
            h[0] = hv.x; h[1] = hv.y; h[2] = hv.z; h[3] = hv.w;
            const float4 av = __ldg(reinterpret_cast<const float4*>(a.A + d * N + n0));
            A2[0] = av.x; A2[1] = av.y; A2[2] = av.z; A2[3] = av.w;
        } else {
#pragma unroll
            for (int j = 0; j < NPL; ++j) { h[j] = st[j]; A2[j] = __ldg(a.A + d * N + n0 + j); }
        }
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            const float Bn = IO<T>::ld(Bg + b * N + n0 + j);
            const float Cn = IO<T>::ld(Cg + b * N + n0 + j);
            h[j] = fmaf(ex2(dt * (A2[j] * kLog2e)), h[j], dtx * Bn);
            y = fmaf(Cn, h[j], y);
        }
        if constexpr (NPL == 4) {
            *reinterpret_cast<float4*>(st) = make_float4(h[0], h[1], h[2], h[3]);
        } else {
#pragma unroll
            for (int j = 0; j < NPL; ++j) st[j] = h[j];
        }
    }
#pragma unroll
    for (int off = 1; off < LANES; off <<= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
    if (active && lane_in_ch == 0) {
        if (a.D) y = fmaf(__ldg(a.D + d), xv, y);
        if (z) y *= silu(IO<T>::ld(z + ch));
        IO<T>::st(static_cast<T*>(a.out) + ch, y);
    }
}

template <typename T, int N>
cudaError_t launch_typed(const StepArgs& a, cudaStream_t s) {
    constexpr int NPL = N >= 4 ? 4 : N;
    constexpr int CH_PER_CTA = kStepThreads / (N / NPL);
    const int64_t nch = a.batch * a.dim;
    const int64_t grid = (nch + CH_PER_CTA - 1) / CH_PER_CTA;
    state_update_kernel<T, N><<<static_cast<unsigned>(grid), kStepThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_n(const StepArgs& a, int N, cudaStream_t s) {
    switch (N) {
        case 1: return launch_typed<T, 1>(a, s);
        case 2: return launch_typed<T, 2>(a, s);
        case 4: return launch_typed<T, 4>(a, s);
        case 8: return launch_typed<T, 8>(a, s);
        case 16: return launch_typed<T, 16>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_state_update(const StepArgs& a, int io, int N, cudaStream_t s) {
    return io == 1 ? launch_n<__nv_bfloat16>(a, N, s) : launch_n<float>(a, N, s);
}

}  // namespace ssm
