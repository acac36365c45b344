// state_update.cu -- one token of recurrent generation on a cached state.
//
// "State-space models (Mamba, S4)", "Training vs Inference Modes": keep h,
// take the new token, h <- Abar h + Bbar x, y = C h, O(1) work per token.
// With the selective parameters of "State Space Models -- Mamba, S4, and
// Beyond", "Mamba (S6 -- Selective State Space)", this is one t-iteration of
// the scan: dt = softplus?(delta + bias), h <- exp(dt A[d,:]) h + dt B x,
// y = C . h + D x, out = y * silu(z); the fp32 state is updated in place.
// With the exact zero-order hold ("State-space models (Mamba, S4)", "From
// Continuous to Discrete: The Key Step") the input term is (e^{dt A} - 1)/A B x.
// With per-channel B, C ("Mamba: State Space Models Challenge Transformers",
// "Selective Scan Algorithm": B, C of shape [B, L, D, N]) the token's rows are
// [batch, dim, N], one per channel, read like the state.
//
// The step is bound by HBM traffic on the state (N fp32 read + written per
// channel). LANES = N / NPL lanes share a channel, each holding NPL = 4 states
// (one 128-bit load and store), so a warp reads and writes 512 contiguous
// bytes of state per instruction; the state is streamed (read once, written
// once) with evict-first cache hints. A CTA covers CH_PER_CTA channels of
// kItems consecutive batch rows (the grid's y index; one row measured fastest,
// below); each lane group handles its channel in all kItems rows, so A, the
// bias and D are loaded once for them, with all loads issued before any
// arithmetic. The partial C . h sums meet through butterfly shuffles; lane 0 of
// each group writes y.
#include <cuda_bf16.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kStepThreads = 256;
// batch rows per lane group (a sweep on b256 d5120 bf16: 1 row 32.8 us, 2 rows
// 34.8, 4 rows 40.1, 8 rows 61.6: more, smaller CTAs keep more loads in flight
// than more rows per thread)
constexpr int kItems = 1;

// NPL consecutive I/O elements widened to fp32 (NPL <= 4; 8-byte aligned for
// bf16 x 4 and 16-byte aligned for fp32 x 4).
template <typename T, int NPL>
__device__ __forceinline__ void ld_vec(const T* p, float (&v)[NPL]) {
    if constexpr (NPL == 4 && sizeof(T) == 2) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xffff0000u);
    } else if constexpr (NPL == 4 && sizeof(T) == 4) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    } else {
#pragma unroll
        for (int j = 0; j < NPL; ++j) v[j] = IO<T>::ld(p + j);
    }
}

// m = dt phi(dt A) = (e^{dt A} - 1) / A of the exact zero-order hold (Taylor
// series for |dt A| < 0.1, where the difference e^z - 1 would cancel).
__device__ __forceinline__ float zoh_m(float dt, float A, float dA) {
    const float zz = dt * A;
    float p = fmaf(zz, 1.f / 120.f, 1.f / 24.f);
    p = fmaf(zz, p, 1.f / 6.f);
    p = fmaf(zz, p, 0.5f);
    p = fmaf(zz, p, 1.f);
    return fabsf(zz) < 0.1f ? dt * p : (dA - 1.f) / A;
}

template <typename T, int N, bool ZOH, bool BCD, int ITEMS = kItems>
__global__ void __launch_bounds__(kStepThreads) state_update_kernel(const StepArgs a) {
    constexpr int kItems = ITEMS;
    constexpr int NPL = N >= 4 ? 4 : N;        // states per lane
    constexpr int LANES = N / NPL;             // lanes per channel (1, 2 or 4)
    constexpr int CH_PER_CTA = kStepThreads / LANES;

    const int lane_in_ch = threadIdx.x % LANES;
    const int n0 = lane_in_ch * NPL;
    // One channel per lane group; the kItems items are kItems batch rows of that
    // channel (2-D grid: the y index picks the rows), so A, the bias and D are
    // loaded once and serve every row.
    const int64_t dd = static_cast<int64_t>(blockIdx.x) * CH_PER_CTA + threadIdx.x / LANES;
    const bool d_ok = dd < a.dim;
    const int64_t d = d_ok ? dd : 0;
    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ delta = static_cast<const T*>(a.delta);
    const T* __restrict__ Bg = static_cast<const T*>(a.B);
    const T* __restrict__ Cg = static_cast<const T*>(a.C);
    const T* __restrict__ z = static_cast<const T*>(a.z);

    float A2[NPL];
    if constexpr (NPL == 4) {
        const float4 av = __ldg(reinterpret_cast<const float4*>(a.A + d * N + n0));
        A2[0] = av.x; A2[1] = av.y; A2[2] = av.z; A2[3] = av.w;
    } else {
#pragma unroll
        for (int j = 0; j < NPL; ++j) A2[j] = __ldg(a.A + d * N + n0 + j);
    }
    const float bias = a.delta_bias ? __ldg(a.delta_bias + d) : 0.f;
    const float Dd = a.D ? __ldg(a.D + d) : 0.f;

    // ---- loads of every item first ----
    int64_t ch[kItems];
    bool active[kItems];
    float xv[kItems], dt[kItems], zv[kItems], h[kItems][NPL], Bv[kItems][NPL], Cv[kItems][NPL];
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        // Whole groups of LANES lanes share the same channel and row, so the
        // shuffles below always run with every participant present.
        const int64_t bb = static_cast<int64_t>(blockIdx.y) * kItems + it;
        active[it] = d_ok && bb < a.batch;
        const int64_t b = bb < a.batch ? bb : 0;
        ch[it] = b * a.dim + d;
        const int64_t c = ch[it];
        xv[it] = IO<T>::ld(x + c);
        dt[it] = IO<T>::ld(delta + c) + bias;
        zv[it] = z ? IO<T>::ld(z + c) : 0.f;
        const float* st = a.state + c * N + n0;
        if constexpr (NPL == 4) {
            const float4 hv = __ldcs(reinterpret_cast<const float4*>(st));
            h[it][0] = hv.x; h[it][1] = hv.y; h[it][2] = hv.z; h[it][3] = hv.w;
        } else {
#pragma unroll
            for (int j = 0; j < NPL; ++j) h[it][j] = __ldcs(st + j);
        }
        // shared rows [batch, N], or the channel's own rows [batch, dim, N]
        const int64_t row = BCD ? c : b;
        ld_vec<T, NPL>(Bg + row * N + n0, Bv[it]);
        ld_vec<T, NPL>(Cg + row * N + n0, Cv[it]);
    }

    // ---- arithmetic and stores ----
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const int64_t c = ch[it];
        float dtv = dt[it];
        if (a.softplus) dtv = softplus(dtv);
        const float dtx = dtv * xv[it];
        float y = 0.f;
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            const float dA = ex2(dtv * (A2[j] * kLog2e));
            // first order: Bbar x = dt x B; exact zero-order hold: x B m
            const float bx = ZOH ? xv[it] * Bv[it][j] * zoh_m(dtv, A2[j], dA) : dtx * Bv[it][j];
            h[it][j] = fmaf(dA, h[it][j], bx);
            y = fmaf(Cv[it][j], h[it][j], y);
        }
        if (active[it]) {
            float* st = a.state + c * N + n0;
            if constexpr (NPL == 4) {
                __stcs(reinterpret_cast<float4*>(st),
                       make_float4(h[it][0], h[it][1], h[it][2], h[it][3]));
            } else {
#pragma unroll
                for (int j = 0; j < NPL; ++j) __stcs(st + j, h[it][j]);
            }
        }
#pragma unroll
        for (int off = 1; off < LANES; off <<= 1) y += __shfl_xor_sync(0xffffffffu, y, off);
        if (active[it] && lane_in_ch == 0) {
            y = fmaf(Dd, xv[it], y);
            if (z) y *= silu(zv[it]);
            IO<T>::st(static_cast<T*>(a.out) + c, y);
        }
    }
}

template <typename T, int N, bool ZOH, bool BCD>
cudaError_t launch_zoh(const StepArgs& a, cudaStream_t s) {
    constexpr int NPL = N >= 4 ? 4 : N;
    constexpr int CH_PER_CTA = kStepThreads / (N / NPL);
    constexpr int64_t kMaxRows = 65535 * kItems;   // rows of one launch (grid y limit)
    // kItems batch rows per CTA row of the grid, in slices of at most kMaxRows rows
    for (int64_t b0 = 0; b0 < a.batch; b0 += kMaxRows) {
        StepArgs p = a;
        p.batch = a.batch - b0 < kMaxRows ? a.batch - b0 : kMaxRows;
        const int64_t e = b0 * a.dim;      // elements before the slice
        p.state = a.state + e * N;
        p.x = static_cast<const T*>(a.x) + e;
        p.delta = static_cast<const T*>(a.delta) + e;
        p.z = a.z ? static_cast<const T*>(a.z) + e : nullptr;
        p.out = static_cast<T*>(a.out) + e;
        p.B = static_cast<const T*>(a.B) + (BCD ? e : b0) * N;
        p.C = static_cast<const T*>(a.C) + (BCD ? e : b0) * N;
        const dim3 grid(static_cast<unsigned>((a.dim + CH_PER_CTA - 1) / CH_PER_CTA),
                        static_cast<unsigned>((p.batch + kItems - 1) / kItems));
        state_update_kernel<T, N, ZOH, BCD><<<grid, kStepThreads, 0, s>>>(p);
    }
    return cudaGetLastError();
}

template <typename T, int N>
cudaError_t launch_typed(const StepArgs& a, cudaStream_t s) {
    if (a.bc_per_channel)
        return a.zoh ? launch_zoh<T, N, true, true>(a, s) : launch_zoh<T, N, false, true>(a, s);
    return a.zoh ? launch_zoh<T, N, true, false>(a, s) : launch_zoh<T, N, false, false>(a, s);
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
