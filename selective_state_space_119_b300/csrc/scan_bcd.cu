// scan_bcd.cu -- the selective scan with per-channel B and C.
//
// "Mamba: State Space Models Challenge Transformers", "Selective Scan
// Algorithm": the docstring of selective_scan gives B and C the shape
// [B, L, D, N], one input / output projection per channel and token, where the
// method's code shares one [B, L, N] row by all channels. The recurrence is the
// same per channel: h = exp(dt A) h + dt B[b,t,d,:] x, y = C[b,t,d,:] . h + D x,
// out = y silu(z).
//
// With per-channel B and C nothing is shared between lanes: each channel reads
// 2 N values per token (64 bytes in bf16 for N = 16) on top of x, delta, z and
// y, so the scan is bound by HBM (72 bytes per element) rather than by the SFU.
// One lane owns one channel and all N of its states. A warp's 32 consecutive
// channels read one contiguous 1 KB row of B (and of C) per token, so the loads
// are fully coalesced and go straight from global memory into a ring of 4
// (bf16) or 2 (fp32) tokens held in registers (twice that in the chunk-state
// pass, which reads no C); the loads of a later token are issued while a token
// computes.
// The L-chunk plan, the chunk-state pass and the carry composition are those of
// the shared-B scan (same workspace layout).
#include <cuda_bf16.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kBcdThreads = 128;    // = the 128-channel tile of configuration 0
// tokens of loads in flight per lane: the chunk-state pass reads no C (half
// the bytes per token), so it keeps twice as many tokens in flight; fp32 rows
// are twice as wide as bf16 ones
template <typename T, int MODE>
struct RingTokens {
    static constexpr int value = (sizeof(T) == 2 ? 4 : 2) * (MODE == 1 ? 1 : 2);
};

template <typename T, int N>
struct Row;   // N values of one channel and token, as raw 16-byte words

template <int N>
struct Row<__nv_bfloat16, N> {
    static constexpr int W = N * 2 / 16;   // uint4 words
    uint4 w[W];
    __device__ __forceinline__ void load(const __nv_bfloat16* p, bool ok) {
#pragma unroll
        for (int i = 0; i < W; ++i)
            w[i] = ok ? __ldg(reinterpret_cast<const uint4*>(p) + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    // values q, q + 1 as fp32
    __device__ __forceinline__ float2 pair(int q) const {
        const uint4& u = w[q / 8];
        const int k = (q % 8) / 2;
        const uint32_t v = k == 0 ? u.x : k == 1 ? u.y : k == 2 ? u.z : u.w;
        return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    }
};

template <int N>
struct Row<float, N> {
    static constexpr int W = N * 4 / 16;
    uint4 w[W];
    __device__ __forceinline__ void load(const float* p, bool ok) {
#pragma unroll
        for (int i = 0; i < W; ++i)
            w[i] = ok ? __ldg(reinterpret_cast<const uint4*>(p) + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    __device__ __forceinline__ float2 pair(int q) const {
        const uint4& u = w[q / 4];
        const int k = q % 4;   // 0 or 2
        return k == 0 ? make_float2(__uint_as_float(u.x), __uint_as_float(u.y))
                      : make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
};

template <typename T>
__device__ __forceinline__ uint32_t ld_raw(const T* p, bool ok) {
    if constexpr (sizeof(T) == 2)
        return ok ? static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16
                  : 0u;
    else
        return ok ? __float_as_uint(__ldg(p)) : 0u;
}

// The per-token loads of one lane: x, delta (, z) and the channel's B (, C) row.
template <typename T, int N, bool WITH_C, bool WITH_Z>
struct Slot {
    uint32_t x, dl, z;
    Row<T, N> B, C;
};

// MODE 1: the output pass (composes the chunk carries, writes y and the final
// state; with CKPT, the training forward's, it also saves the state before
// every kCkptTokens-th token for the backward); MODE 0: the chunk-state pass
// (end state from 0 and sum of dt of every chunk but the last). One lane = one
// channel. The saving pass walks whole groups of kCkptTokens tokens, the save
// at a fixed position of the unrolled group: a save behind a per-token test of
// the token index split the token body and ran the pass 3x slower, and a
// separate pass that re-read x, delta and B cost 111 us on b4 L2048 d1536
// against the 74 us the in-pass saves add.
template <typename T, int N, int MODE, bool SOFTPLUS, bool GATE, bool CKPT = false>
__global__ void __launch_bounds__(kBcdThreads) scan_bcd_kernel(const ScanArgs a) {
    constexpr bool WITH_C = MODE == 1, WITH_Z = MODE == 1 && GATE;
    using S = Slot<T, N, WITH_C, WITH_Z>;
    constexpr int kRing = RingTokens<T, MODE>::value;
    // the token loop walks whole groups of kCkptTokens (the ring reused), so
    // that a saved state sits at a fixed position of the unrolled group
    constexpr int kGroup = CKPT ? kCkptTokens : kRing;
    static_assert(kGroup % kRing == 0, "whole rings per group");
    const int64_t lin = blockIdx.x;   // chunk-major: ((k * batch) + b) * tiles + tile
    const int64_t tile = lin % a.tiles;
    const int64_t b = (lin / a.tiles) % a.batch;
    const int64_t k = lin / (a.tiles * a.batch);
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(a.L, t_begin + a.chunk_len);
    const int64_t d = tile * kBcdThreads + threadIdx.x;
    const bool ch_ok = d < a.dim;
    const int64_t dsafe = ch_ok ? d : 0;

    float A2[N], h[N];
#pragma unroll
    for (int q = 0; q < N; ++q) {
        A2[q] = ch_ok ? __ldg(a.A + dsafe * N + q) * kLog2e : 0.f;
        h[q] = 0.f;
    }
    if (MODE != 0 && ch_ok) {
        if (a.h0) {
#pragma unroll
            for (int q = 0; q < N; ++q) h[q] = a.h0[(b * a.dim + d) * N + q];
        }
        // the state entering chunk k: h <- exp(A S_i) h + H_i over chunks 0 .. k-1
        for (int64_t i = 0; i < k; ++i) {
            const int64_t idx = (b * (a.nchunks - 1) + i) * a.dim + d;
            const float Si = a.ws_S[idx];
            const float* Hi = a.ws_H + idx * N;
#pragma unroll
            for (int q = 0; q < N; ++q) h[q] = fmaf(ex2(A2[q] * Si), h[q], Hi[q]);
        }
    }
    const float bias = (a.delta_bias && ch_ok) ? __ldg(a.delta_bias + dsafe) : 0.f;
    const float Dd = (MODE == 1 && a.D && ch_ok) ? __ldg(a.D + dsafe) : 0.f;

    const int64_t e0 = b * a.L * a.dim + dsafe;   // element (b, 0, d)
    const T* xg = static_cast<const T*>(a.x) + e0;
    const T* dg = static_cast<const T*>(a.delta) + e0;
    const T* zg = WITH_Z ? static_cast<const T*>(a.z) + e0 : nullptr;
    const T* Bg = static_cast<const T*>(a.B) + e0 * N;
    const T* Cg = WITH_C ? static_cast<const T*>(a.C) + e0 * N : nullptr;
    T* og = MODE == 1 ? static_cast<T*>(a.out) + e0 : nullptr;

    auto load = [&](S& s, int64_t t) {
        const bool ok = ch_ok && t < t_end;
        const int64_t e = ok ? t * a.dim : 0;
        s.x = ld_raw(xg + e, ok);
        s.dl = ld_raw(dg + e, ok);
        if constexpr (WITH_Z) s.z = ld_raw(zg + e, ok);
        s.B.load(Bg + e * N, ok);
        if constexpr (WITH_C) s.C.load(Cg + e * N, ok);
    };
    S ring[kRing];
#pragma unroll
    for (int u = 0; u < kRing; ++u) load(ring[u], t_begin + u);

    float dt_sum = 0.f;
    for (int64_t t0 = t_begin; t0 < t_end; t0 += kGroup) {
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int64_t t = t0 + u;
            const S cur = ring[u % kRing];
            load(ring[u % kRing], t + kRing);   // the loads of a later token, in flight meanwhile
            const bool valid = ch_ok && t < t_end;
            if constexpr (CKPT) {
                // chunks start on a checkpoint: t0 is one, the state before token t0
                if (u == 0 && valid) {
                    float4* ck = reinterpret_cast<float4*>(
                        a.ckpt + ((b * a.nckpt + t / kCkptTokens) * a.dim + d) * N);
#pragma unroll
                    for (int q = 0; q < N / 4; ++q)
                        ck[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                }
            }
            const float xv = __uint_as_float(cur.x);
            float dt = __uint_as_float(cur.dl) + bias;
            if constexpr (SOFTPLUS) dt = softplus(dt);
            dt = valid ? dt : 0.f;      // dt = 0 leaves the state unchanged
            const float2 dt2 = make_float2(dt, dt), dtx2 = make_float2(dt * xv, dt * xv);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < N; q += 2) {
                const float2 arg = __fmul2_rn(dt2, make_float2(A2[q], A2[q + 1]));
                const float2 bx = __fmul2_rn(dtx2, cur.B.pair(q));
                const float2 hn = __ffma2_rn(make_float2(ex2(arg.x), ex2(arg.y)),
                                             make_float2(h[q], h[q + 1]), bx);
                h[q] = hn.x;
                h[q + 1] = hn.y;
                if constexpr (WITH_C) acc = __ffma2_rn(cur.C.pair(q), hn, acc);
            }
            if constexpr (MODE == 1) {
                float y = fmaf(Dd, xv, acc.x + acc.y);
                if constexpr (GATE) y *= silu(__uint_as_float(cur.z));
                if (valid) IO<T>::st(og + t * a.dim, y);
            } else if constexpr (MODE == 0) {
                dt_sum += dt;
            }
        }
    }

    if (!ch_ok) return;
    if constexpr (MODE == 1) {
        if (a.final_state && k == a.nchunks - 1) {
#pragma unroll
            for (int q = 0; q < N; ++q) a.final_state[(b * a.dim + d) * N + q] = h[q];
        }
    } else if constexpr (MODE == 0) {
        const int64_t idx = (b * (a.nchunks - 1) + k) * a.dim + d;
#pragma unroll
        for (int q = 0; q < N; ++q) a.ws_H[idx * N + q] = h[q];
        a.ws_S[idx] = dt_sum;
    }
}

template <typename T, int N, bool SOFTPLUS, bool GATE>
cudaError_t launch_flags(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    if (p.channels_per_cta != kBcdThreads) return cudaErrorInvalidValue;
    const int64_t per_chunk = p.tiles * a.batch;
    if (p.nchunks > 1)
        scan_bcd_kernel<T, N, 0, SOFTPLUS, false>
            <<<static_cast<unsigned>(per_chunk * (p.nchunks - 1)), kBcdThreads, 0, s>>>(a);
    if (a.ckpt)
        scan_bcd_kernel<T, N, 1, SOFTPLUS, GATE, true>
            <<<static_cast<unsigned>(per_chunk * p.nchunks), kBcdThreads, 0, s>>>(a);
    else
        scan_bcd_kernel<T, N, 1, SOFTPLUS, GATE>
            <<<static_cast<unsigned>(per_chunk * p.nchunks), kBcdThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    constexpr int N = 16;
    const bool gate = a.z != nullptr;
    if (a.softplus)
        return gate ? launch_flags<T, N, true, true>(a, p, s) : launch_flags<T, N, true, false>(a, p, s);
    return gate ? launch_flags<T, N, false, true>(a, p, s) : launch_flags<T, N, false, false>(a, p, s);
}

}  // namespace

cudaError_t launch_scan_bcd(const ScanArgs& a, const ScanPlan& p, int io, cudaStream_t s) {
    return io == 1 ? launch_typed<__nv_bfloat16>(a, p, s) : launch_typed<float>(a, p, s);
}

}  // namespace ssm
