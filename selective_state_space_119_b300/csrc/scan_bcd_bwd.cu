// scan_bcd_bwd.cu -- gradients of the scan with per-channel B and C.
//
// "Mamba: State Space Models Challenge Transformers", "Selective Scan
// Algorithm": B and C of shape [B, L, D, N], one row per channel and token.
// Channel d is then a one-channel scan with rows B[b,t,d,:], C[b,t,d,:], and its
// gradients are the chain rule on that recurrence ("State Space Models --
// Mamba, S4, and Beyond", "Verification Checklist": gradients flow through the
// discretization). Per token, from the end, with Q[n] = a_{t+1}[n] dL/dh_{t+1}[n]:
//   dy = dout silu(z) (dout without the gate),  g[n] = Q[n] + dy C[n]
//   dC[n] = dy h[n],  dB[n] = g[n] dt x,  dA[n] += g[n] dt (h[n] - dt x B[n])
//   dx = dt sum_n g[n] B[n] + dy D,  ddt = x sum_n g[n] B[n] + sum_n g[n] A[n] (h[n] - dt x B[n])
//   ddelta = ddt sigmoid(delta + bias) (softplus) or ddt,  dz = dout y silu'(z),
//   Q[n] <- e^{dt A[n]} g[n]
// (h[n] - dt x B[n] is a[n] h_{t-1}[n], the decayed previous state). Nothing
// sums over channels here: dB and dC are one row per (b, t, d), written as they
// are formed. dA, dD and dbias sum over batch rows and tokens: every CTA writes
// its share, and a last kernel adds the shares in a fixed order.
//
// Layout: one lane per channel (128 channels per CTA), all 16 states in
// registers, as in the per-channel forward. The sequence is split into the
// forward's L-chunks. The carry pass runs the reverse recurrence of every chunk
// but the first from Q = 0 and keeps its Q at the chunk's first token and its
// sum of dt; the gradient pass of chunk k starts from dL/dfinal_state and
// composes the carries of the chunks to its right, Q <- e^{A S_i} Q + Q_i. It
// then walks its chunk in 8-token blocks from the end: the block's checkpoint
// (the state before its first token) is reloaded, the block's 8 states are
// recomputed forward into the lane's own slots of shared memory, and the
// reverse sweep reads them back. The slots are private to the lane, so the
// passes need no barrier.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kThreads = 128;          // channels per CTA
constexpr int kN = 16;                 // states per channel
constexpr int kTB = kCkptTokens;       // tokens per recomputed block (8)
constexpr float kLn2f = 0.6931471805599453f;

// shared memory of the gradient pass: the states after each token of the
// block, float4 [kTB][kN / 4][kThreads] (lane-consecutive, no bank conflict),
// then dt and sigmoid(delta + bias) per token, float [kTB][kThreads] each
constexpr int kHistBytes = kTB * (kN / 4) * kThreads * 16;
constexpr int kGradSmem = kHistBytes + 2 * kTB * kThreads * 4;

// the 16 values of one channel's B or C row as fp32
template <typename T>
__device__ __forceinline__ void ld_row(const T* p, float (&v)[kN]) {
    if constexpr (sizeof(T) == 2) {
        const uint4* q = reinterpret_cast<const uint4*>(p);
        const uint4 u0 = __ldg(q), u1 = __ldg(q + 1);
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
        const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
        for (int i = 0; i < kN / 4; ++i) {
            const float4 f = __ldg(q + i);
            v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
        }
    }
}

template <typename T>
__device__ __forceinline__ void st_row(T* p, const float (&v)[kN]) {
    if constexpr (sizeof(T) == 2) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        uint4* q = reinterpret_cast<uint4*>(p);
        q[0] = make_uint4(w[0], w[1], w[2], w[3]);
        q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
        float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
        for (int i = 0; i < kN / 4; ++i)
            q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
}

__device__ __forceinline__ float sigmoid(float v) { return 1.f / (1.f + __expf(-v)); }

// silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z)))
__device__ __forceinline__ float dsilu(float z) {
    const float s = sigmoid(z);
    return s * fmaf(z, 1.f - s, 1.f);
}

// The reverse carry of chunks 1 .. nchunks-1 from Q = 0: Q at the chunk's
// first token and the chunk's sum of dt.
template <typename T, bool SOFTPLUS, bool GATE>
__global__ void __launch_bounds__(kThreads) bcd_carry_kernel(const BwdArgs a) {
    const int64_t lin = blockIdx.x;   // ((k - 1) * batch + b) * tiles + tile
    const int64_t tile = lin % a.tiles;
    const int64_t b = (lin / a.tiles) % a.batch;
    const int64_t k = 1 + lin / (a.tiles * a.batch);
    const int64_t d = tile * kThreads + threadIdx.x;
    if (d >= a.dim) return;
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(a.L, t_begin + a.chunk_len);

    float A2[kN], Q[kN];
#pragma unroll
    for (int q = 0; q < kN; ++q) {
        A2[q] = __ldg(a.A + d * kN + q) * kLog2e;
        Q[q] = 0.f;
    }
    const float bias = a.delta_bias ? __ldg(a.delta_bias + d) : 0.f;
    const int64_t e0 = b * a.L * a.dim + d;
    const T* dl = static_cast<const T*>(a.delta) + e0;
    const T* go = static_cast<const T*>(a.dout) + e0;
    const T* zg = GATE ? static_cast<const T*>(a.z) + e0 : nullptr;
    const T* Cg = static_cast<const T*>(a.C) + e0 * kN;
    float dt_sum = 0.f;
#pragma unroll 2
    for (int64_t t = t_end - 1; t >= t_begin; --t) {
        const int64_t e = t * a.dim;
        float dt = IO<T>::ld(dl + e) + bias;
        if constexpr (SOFTPLUS) dt = softplus(dt);
        float dy = IO<T>::ld(go + e);
        if constexpr (GATE) dy *= silu(IO<T>::ld(zg + e));
        float c[kN];
        ld_row(Cg + e * kN, c);
#pragma unroll
        for (int q = 0; q < kN; ++q) Q[q] = ex2(A2[q] * dt) * fmaf(dy, c[q], Q[q]);
        dt_sum += dt;
    }
    const int64_t idx = (b * (a.nchunks - 1) + (k - 1)) * a.dim + d;
#pragma unroll
    for (int q = 0; q < kN; ++q) a.wsQ[idx * kN + q] = Q[q];
    a.wsS[idx] = dt_sum;
}

// The gradients of one L-chunk of 128 channels of one batch row.
template <typename T, bool SOFTPLUS, bool GATE>
__global__ void __launch_bounds__(kThreads, 3) bcd_grad_kernel(const BwdArgs a) {
    extern __shared__ float4 smem4[];
    float4* hist = smem4;                                                   // [kTB][kN/4][kThreads]
    float* sdt = reinterpret_cast<float*>(smem4 + kTB * (kN / 4) * kThreads);   // [kTB][kThreads]
    float* ssig = sdt + kTB * kThreads;                                      // [kTB][kThreads]

    const int tid = threadIdx.x;
    const int64_t lin = blockIdx.x;   // (k * batch + b) * tiles + tile
    const int64_t tile = lin % a.tiles;
    const int64_t b = (lin / a.tiles) % a.batch;
    const int64_t k = lin / (a.tiles * a.batch);
    const int64_t d = tile * kThreads + tid;
    if (d >= a.dim) return;   // every lane works on its own slots only
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(a.L, t_begin + a.chunk_len);

    float A2[kN], Q[kN], gA[kN];
#pragma unroll
    for (int q = 0; q < kN; ++q) {
        A2[q] = __ldg(a.A + d * kN + q) * kLog2e;
        Q[q] = a.dfinal ? a.dfinal[(b * a.dim + d) * kN + q] : 0.f;
        gA[q] = 0.f;
    }
    // dL/dh at the chunk's last token: the carries of the chunks to the right
    for (int64_t i = a.nchunks - 1; i > k; --i) {
        const int64_t idx = (b * (a.nchunks - 1) + (i - 1)) * a.dim + d;
        const float S = a.wsS[idx];
#pragma unroll
        for (int q = 0; q < kN; ++q) Q[q] = fmaf(ex2(A2[q] * S), Q[q], a.wsQ[idx * kN + q]);
    }
    const float bias = a.delta_bias ? __ldg(a.delta_bias + d) : 0.f;
    const float Dd = a.D ? __ldg(a.D + d) : 0.f;
    const int64_t e0 = b * a.L * a.dim + d;
    const T* xg = static_cast<const T*>(a.x) + e0;
    const T* dl = static_cast<const T*>(a.delta) + e0;
    const T* go = static_cast<const T*>(a.dout) + e0;
    const T* zg = GATE ? static_cast<const T*>(a.z) + e0 : nullptr;
    const T* Bg = static_cast<const T*>(a.B) + e0 * kN;
    const T* Cg = static_cast<const T*>(a.C) + e0 * kN;
    T* dxg = static_cast<T*>(a.dx) + e0;
    T* ddg = static_cast<T*>(a.ddelta) + e0;
    T* dzg = GATE ? static_cast<T*>(a.dz) + e0 : nullptr;
    T* dBg = static_cast<T*>(a.dB) + e0 * kN;
    T* dCg = static_cast<T*>(a.dC) + e0 * kN;
    float gD = 0.f, gbias = 0.f;

    const int64_t m_first = t_begin / kTB, m_last = (t_end - 1) / kTB;
    for (int64_t m = m_last; m >= m_first; --m) {
        const int64_t u0 = m * kTB;
        const int cnt = t_end - u0 < kTB ? static_cast<int>(t_end - u0) : kTB;
        // the state before token u0, then the states after each of the block's tokens
        float h[kN];
        {
            const float4* ck =
                reinterpret_cast<const float4*>(a.ckpt + ((b * a.nckpt + m) * a.dim + d) * kN);
#pragma unroll
            for (int i = 0; i < kN / 4; ++i) {
                const float4 v = ck[i];
                h[4 * i] = v.x; h[4 * i + 1] = v.y; h[4 * i + 2] = v.z; h[4 * i + 3] = v.w;
            }
        }
#pragma unroll
        for (int j = 0; j < kTB; ++j) {
            if (j < cnt) {
                const int64_t e = (u0 + j) * a.dim;
                const float xv = IO<T>::ld(xg + e);
                const float v = IO<T>::ld(dl + e) + bias;
                const float dt = SOFTPLUS ? softplus(v) : v;
                sdt[j * kThreads + tid] = dt;
                if constexpr (SOFTPLUS) ssig[j * kThreads + tid] = sigmoid(v);
                float bb[kN];
                ld_row(Bg + e * kN, bb);
                const float dtx = dt * xv;
#pragma unroll
                for (int q = 0; q < kN; ++q) h[q] = fmaf(ex2(A2[q] * dt), h[q], dtx * bb[q]);
#pragma unroll
                for (int i = 0; i < kN / 4; ++i)
                    hist[(j * (kN / 4) + i) * kThreads + tid] =
                        make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
            }
        }
        // the reverse sweep over the block
#pragma unroll 2
        for (int j = cnt - 1; j >= 0; --j) {
            const int64_t e = (u0 + j) * a.dim;
            const float xv = IO<T>::ld(xg + e);
            const float dt = sdt[j * kThreads + tid];
            const float dout = IO<T>::ld(go + e);
            float zv = 0.f, dy = dout;
            if constexpr (GATE) {
                zv = IO<T>::ld(zg + e);
                dy = dout * silu(zv);
            }
            float bb[kN], cc[kN], hh[kN];
            ld_row(Bg + e * kN, bb);
            ld_row(Cg + e * kN, cc);
#pragma unroll
            for (int i = 0; i < kN / 4; ++i) {
                const float4 v = hist[(j * (kN / 4) + i) * kThreads + tid];
                hh[4 * i] = v.x; hh[4 * i + 1] = v.y; hh[4 * i + 2] = v.z; hh[4 * i + 3] = v.w;
            }
            const float dtx = dt * xv;
            float dB[kN], dC[kN];
            float sgb = 0.f, sga = 0.f, y = Dd * xv;
#pragma unroll
            for (int q = 0; q < kN; ++q) {
                const float g = fmaf(dy, cc[q], Q[q]);
                const float ahp = fmaf(-dtx, bb[q], hh[q]);   // e^{dt A} h_{t-1}
                const float gahp = g * ahp;
                dC[q] = dy * hh[q];
                dB[q] = g * dtx;
                sgb = fmaf(g, bb[q], sgb);
                sga = fmaf(gahp, A2[q], sga);
                gA[q] = fmaf(gahp, dt, gA[q]);
                Q[q] = ex2(A2[q] * dt) * g;
                if constexpr (GATE) y = fmaf(cc[q], hh[q], y);
            }
            st_row(dBg + e * kN, dB);
            st_row(dCg + e * kN, dC);
            const float ddt = fmaf(xv, sgb, sga * kLn2f);
            const float dd = SOFTPLUS ? ddt * ssig[j * kThreads + tid] : ddt;
            IO<T>::st(dxg + e, fmaf(dt, sgb, dy * Dd));
            IO<T>::st(ddg + e, dd);
            if constexpr (GATE) IO<T>::st(dzg + e, dout * y * dsilu(zv));
            gD = fmaf(dy, xv, gD);
            gbias += dd;
        }
    }
    if (k == 0 && a.dh0) {
#pragma unroll
        for (int q = 0; q < kN; ++q) a.dh0[(b * a.dim + d) * kN + q] = Q[q];
    }
    const int64_t row = b * a.nchunks + k;
#pragma unroll
    for (int q = 0; q < kN; ++q) a.pA[(row * a.dim + d) * kN + q] = gA[q];
    a.pD[row * a.dim + d] = gD;
    a.pbias[row * a.dim + d] = gbias;
}

// dA, dD, dbias: the shares of every (batch row, chunk), added in order.
__global__ void __launch_bounds__(256) bcd_bwd_reduce_kernel(const BwdArgs a) {
    const int64_t nA = a.dim * kN, nd = a.dim;
    const int64_t total = nA + 2 * nd, rows = a.batch * a.nchunks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (i < nA) {
            float s = 0.f;
            for (int64_t r = 0; r < rows; ++r) s += a.pA[r * nA + i];
            a.dA[i] = s;
        } else {
            const int64_t e = i - nA;
            const bool is_bias = e >= nd;
            float* out = is_bias ? a.dbias : a.dD;
            if (!out) continue;
            const int64_t dd = is_bias ? e - nd : e;
            const float* part = is_bias ? a.pbias : a.pD;
            float s = 0.f;
            for (int64_t r = 0; r < rows; ++r) s += part[r * nd + dd];
            out[dd] = s;
        }
    }
}

template <typename T, bool SOFTPLUS, bool GATE>
cudaError_t launch_flags(const BwdArgs& a, cudaStream_t s) {
    static std::mutex mu;
    static bool done[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(bcd_grad_kernel<T, SOFTPLUS, GATE>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kGradSmem);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    const int64_t per_chunk = a.tiles * a.batch;
    if (a.nchunks > 1)
        bcd_carry_kernel<T, SOFTPLUS, GATE>
            <<<static_cast<unsigned>(per_chunk * (a.nchunks - 1)), kThreads, 0, s>>>(a);
    bcd_grad_kernel<T, SOFTPLUS, GATE>
        <<<static_cast<unsigned>(per_chunk * a.nchunks), kThreads, kGradSmem, s>>>(a);
    const int64_t total = a.dim * kN + 2 * a.dim;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, 148 * 16);
    bcd_bwd_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const BwdArgs& a, cudaStream_t s) {
    const bool gate = a.z != nullptr;
    if (a.softplus)
        return gate ? launch_flags<T, true, true>(a, s) : launch_flags<T, true, false>(a, s);
    return gate ? launch_flags<T, false, true>(a, s) : launch_flags<T, false, false>(a, s);
}

}  // namespace

cudaError_t launch_scan_bcd_bwd(const BwdArgs& a, int io, cudaStream_t s) {
    if (a.tiles * kThreads < a.dim) return cudaErrorInvalidValue;
    return io == 1 ? launch_typed<__nv_bfloat16>(a, s) : launch_typed<float>(a, s);
}

}  // namespace ssm
