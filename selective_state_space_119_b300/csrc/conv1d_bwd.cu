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
// A CTA owns a tile of kTT tokens x kDC channels of one batch row. Its x rows
// (the tile's tokens and the K - 1 on either side) and du rows (its tokens and
// the K - 1 after them) are copied into shared memory with 16-byte cp.async
// (rows outside the sequence, channels past dim: zeros). One thread per pair
// of channels (packed FP32 arithmetic) then walks the rows in order with a
// window of K x values and K dpre values in registers: dpre of each row, dx of
// the row K - 1 back (written over that row's du, already read), and the
// tile's own tokens' shares of dw and dbias; the tile's dx rows then leave
// with 16-byte stores. The shares of every
// (batch row, tile) are added by a second kernel in a fixed order, so the sums
// do not depend on scheduling.
#include <cuda_bf16.h>

#include <mutex>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kTT = 32;                // tokens per tile
constexpr int kDC = 128;               // channels per tile
constexpr int kConvBwdThreads = kDC / 2;   // a pair of channels per thread

template <typename T, int K>
struct ConvBwdSmem {
    static constexpr int NX = kTT + 2 * (K - 1);   // x rows: t0 - K + 1 .. t0 + kTT + K - 2
    static constexpr int ND = kTT + K - 1;         // du rows: t0 .. t0 + kTT + K - 2
    static constexpr int kBytes = (NX + ND) * kDC * int(sizeof(T));
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
};

// 16 bytes global -> shared, asynchronously; valid = false writes zeros.
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

// two consecutive channels of a shared-memory row
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld2(const __nv_bfloat16* p) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ void st2(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void st2(__nv_bfloat16* p, float2 v) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __float22bfloat162_rn(v);
}

// silu'(p) = sigmoid(p) (1 + p (1 - sigmoid(p))), for a pair of channels
// (sigmoid as a fast reciprocal of 1 + e^-p: 0 once e^-p overflows)
__device__ __forceinline__ float2 dsilu2(float2 p) {
    const float2 q = __fmul2_rn(p, make_float2(-kLog2e, -kLog2e));
    const float2 den = __ffma2_rn(make_float2(ex2(q.x), ex2(q.y)), make_float2(1.f, 1.f),
                                  make_float2(1.f, 1.f));
    const float2 s = make_float2(__fdividef(1.f, den.x), __fdividef(1.f, den.y));
    const float2 oms = __ffma2_rn(s, make_float2(-1.f, -1.f), make_float2(1.f, 1.f));
    return __fmul2_rn(s, __ffma2_rn(p, oms, make_float2(1.f, 1.f)));
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvBwdThreads) conv1d_silu_bwd_kernel(const ConvBwdArgs a) {
    using Sm = ConvBwdSmem<T, K>;
    constexpr int VEC = 16 / int(sizeof(T)), ROWC = kDC / VEC, NT = kConvBwdThreads;
    constexpr int NX = Sm::NX, ND = Sm::ND;
    extern __shared__ __align__(16) unsigned char smem[];
    T* sx = reinterpret_cast<T*>(smem);   // [NX][kDC]
    T* sdu = sx + NX * kDC;                // [ND][kDC]; dx of the first kTT rows afterwards

    const int tid = threadIdx.x;
    const int64_t DB = (a.dim + kDC - 1) / kDC, RB = (a.L + kTT - 1) / kTT;
    const int64_t dblk = blockIdx.x % DB, rest = blockIdx.x / DB;
    const int64_t rb = rest % RB, b = rest / RB;
    const int64_t dbase = dblk * kDC, t0 = rb * kTT;
    const int64_t base = b * a.L * a.dim;
    const T* xg = static_cast<const T*>(a.x) + base;
    const T* dug = static_cast<const T*>(a.du) + base;
    // lane tid copies the 16-byte piece cc of rows tid / ROWC, + NT / ROWC, ...
    static_assert(NT % ROWC == 0, "whole rows per pass");
    constexpr int RSTEP = NT / ROWC;
    const int cc = (tid % ROWC) * VEC, r0 = tid / ROWC;
    const bool c_ok = dbase + cc < a.dim;
    {
        int64_t t = t0 - (K - 1) + r0;
        const T* src = xg + t * a.dim + dbase + cc;
        for (int r = r0; r < NX; r += RSTEP, t += RSTEP, src += RSTEP * a.dim) {
            const bool valid = c_ok && t >= 0 && t < a.L;
            cp16(sx + r * kDC + cc, valid ? src : xg, valid);
        }
        t = t0 + r0;
        src = dug + t * a.dim + dbase + cc;
        for (int r = r0; r < ND; r += RSTEP, t += RSTEP, src += RSTEP * a.dim) {
            const bool valid = c_ok && t < a.L;
            cp16(sdu + r * kDC + cc, valid ? src : dug, valid);
        }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");

    // this thread's channels c, c + 1 of the tile (dim is even: both or neither exist)
    const int c = 2 * tid;
    const bool ch_ok = dbase + c < a.dim;
    const int64_t d = ch_ok ? dbase + c : 0;
    float2 w[K];
#pragma unroll
    for (int k = 0; k < K; ++k) w[k] = make_float2(__ldg(a.w + d * K + k), __ldg(a.w + (d + 1) * K + k));
    const float2 bias = a.b ? make_float2(__ldg(a.b + d), __ldg(a.b + d + 1)) : make_float2(0.f, 0.f);
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();

    // row i: du row i (token t0 + i) with the x window xw[k] = x row i + k
    // (token t0 + i - K + 1 + k); dq holds dpre of rows i - K + 1 .. i
    const float2 zero = make_float2(0.f, 0.f), one = make_float2(1.f, 1.f);
    float2 xw[K], dq[K], dwp[K], dbp = zero;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        xw[k] = k < K - 1 ? ld2(sx + k * kDC + c) : zero;
        dq[k] = zero;
        dwp[k] = zero;
    }
    auto row = [&](const int i, const bool own, const bool emit) {
        xw[K - 1] = ld2(sx + (i + K - 1) * kDC + c);
        float2 pre = bias;
#pragma unroll
        for (int k = 0; k < K; ++k) pre = __ffma2_rn(w[k], xw[k], pre);
        const float2 dp = __fmul2_rn(ld2(sdu + i * kDC + c), dsilu2(pre));
#pragma unroll
        for (int k = 0; k < K - 1; ++k) dq[k] = dq[k + 1];
        dq[K - 1] = dp;
        if (own) {   // a token of this tile: its share of dw and dbias
#pragma unroll
            for (int k = 0; k < K; ++k) dwp[k] = __ffma2_rn(dp, xw[k], dwp[k]);
            dbp = __ffma2_rn(dp, one, dbp);
        }
        if (emit) {  // dx of row i - K + 1 = sum_k w[k] dpre of row i - k
            float2 acc = zero;
#pragma unroll
            for (int k = 0; k < K; ++k) acc = __ffma2_rn(w[k], dq[K - 1 - k], acc);
            st2(sdu + (i - (K - 1)) * kDC + c, acc);
        }
#pragma unroll
        for (int k = 0; k < K - 1; ++k) xw[k] = xw[k + 1];
    };
#pragma unroll
    for (int i = 0; i < K - 1; ++i) row(i, true, false);
#pragma unroll
    for (int i = K - 1; i < kTT; ++i) row(i, true, true);
#pragma unroll
    for (int i = kTT; i < ND; ++i) row(i, false, true);
    if (ch_ok) {
        // [channel][K + 1]: dw[0..K-1], dbias
        float* dst = a.part + ((b * RB + rb) * a.dim + d) * (K + 1);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            dst[k] = dwp[k].x;
            dst[K + 1 + k] = dwp[k].y;
        }
        dst[K] = dbp.x;
        dst[2 * K + 1] = dbp.y;
    }
    __syncthreads();
    // the tile's dx rows, 16 bytes at a time
    if (c_ok) {
        T* dst = static_cast<T*>(a.dx) + base + (t0 + r0) * a.dim + dbase + cc;
        for (int r = r0; r < kTT && t0 + r < a.L; r += RSTEP, dst += RSTEP * a.dim)
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(sdu + r * kDC + cc);
    }
}

// dw[d][k] and dbias[d]: the shares of every (batch row, token block). A CTA
// owns 32 outputs; its 8 warps sum the rows q = w, w + 8, w + 16, ... of each
// (4 running sums each, added in order), and warp 0 adds the 8 slices in
// order: a fixed order, so the result does not depend on scheduling. (Eight
// running sums per warp measured slower.)
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
#pragma unroll
        for (int j = 0; j < 3; ++j)
            if (q + j * kSlices < nblocks) acc[j] += a.part[(q + j * kSlices) * n + i];
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
    using Sm = ConvBwdSmem<T, K>;
    static std::mutex mu;
    static bool done[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(conv1d_silu_bwd_kernel<T, K>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kBytes);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    const int64_t DB = (a.dim + kDC - 1) / kDC;
    const int64_t RB = (a.L + kTT - 1) / kTT;
    const int64_t blocks = a.batch * RB * DB;
    if (blocks >= (int64_t(1) << 31)) return cudaErrorInvalidConfiguration;
    conv1d_silu_bwd_kernel<T, K><<<static_cast<unsigned>(blocks), kConvBwdThreads, Sm::kBytes, s>>>(a);
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
    const int64_t RB = (L + kTT - 1) / kTT;
    return size_t(batch) * size_t(RB) * size_t(dim) * size_t(k + 1);
}

cudaError_t launch_conv1d_silu_bwd(const ConvBwdArgs& a, int io, cudaStream_t s) {
    return io == 1 ? launch_bwd_typed<__nv_bfloat16>(a, s) : launch_bwd_typed<float>(a, s);
}

}  // namespace ssm
