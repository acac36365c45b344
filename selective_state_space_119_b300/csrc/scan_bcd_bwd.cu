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
// The sequence is split into the backward's L-chunks. The carry pass runs the
// reverse recurrence of every chunk but the first from Q = 0 and keeps its Q
// at the chunk's first token and its sum of dt; the gradient pass of chunk k
// starts from dL/dfinal_state and composes the carries of the chunks to its
// right, Q <- e^{A S_i} Q + Q_i. It then walks its chunk in 8-token blocks from
// the end: the block's checkpoint (the state before its first token) is
// reloaded, the block's states are recomputed forward into shared memory, and
// the reverse sweep reads them back.
//
// Two layouts. bf16 rows (the fast path): both passes stage each block's rows
// through shared memory with cp.async, a block or two ahead (the staged
// kernels below); the carry has one lane per channel, the gradient pass two (8
// states each). fp32 rows: one lane per channel, all 16 states in registers,
// each lane loading its own rows token by token, as in the per-channel forward
// (bcd_carry_kernel, bcd_grad_kernel); the recomputed states go to the lane's
// own slots of shared memory, so those passes need no barrier.
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

// (a fast quotient: the denominator is at least 1; where it exceeds 2^126 the
// quotient, then 0, is below the smallest normal float anyway)
__device__ __forceinline__ float sigmoid(float v) { return __fdividef(1.f, 1.f + __expf(-v)); }

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
    // (unrolled: their loads do not depend on Q)
#pragma unroll 4
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

// The gradient pass for bf16 rows, staged through shared memory.
//
// The same arithmetic as bcd_grad_kernel, laid out for more warps and with the
// loads taken off the lanes:
// - Each 8-token block's B and C rows (32 bytes per channel and token), its x,
//   delta, z and dout rows and its checkpoint are copied into one of two
//   shared-memory buffers with 16-byte cp.async, the next block's (in reverse
//   order) while this one computes, so a block's 80 KB are in flight at once.
// - Two lanes per channel, 8 states each (256 threads for 128 channels): one
//   CTA per SM (the buffers take 208 KB) still holds 8 warps, and the sums over
//   the states (sum_n g B, sum_n g A a h, sum_n C h) take one exchange of the
//   pair. The per-token scalars (dt, sigmoid(delta + bias), dy, dout silu'(z))
//   are formed once per channel in a pass over the block.
// - Only the states after the block's even tokens are kept; the sweep forms an
//   odd token's state from the even one before it, h_j = e^{dt A} h_{j-1} +
//   dt x B, the step the recompute took.
// Requires dim % 8 == 0 and 16-byte aligned rows, which the bf16 entry points
// check.
constexpr int kGThreads = 2 * kThreads;              // two lanes per channel
constexpr int kNH = kN / 2;                          // states per lane
constexpr int kSRows = kTB * kThreads * kN * 2;      // a block's B (or C) rows, bytes
constexpr int kSScal = kTB * kThreads * 2;           // a block's x (or delta, z, dout) row set
constexpr int kSCkpt = kThreads * kN * 4;            // a block's checkpoint
constexpr int kSOffScal = 2 * kSRows, kSOffCkpt = 2 * kSRows + 4 * kSScal;
constexpr int kSBuf = kSOffCkpt + kSCkpt;            // one buffer (80 KB)
constexpr int kSHist = kTB / 2 * 2 * kGThreads * 16; // states after the even tokens
constexpr int kSTok = kTB * kThreads * 16;           // per token and channel: dt, sig, dy, gz
constexpr int kStagedSmem = 2 * kSBuf + kSHist + kSTok;
static_assert(kStagedSmem <= 227 * 1024, "shared memory per CTA");
static_assert(kThreads == 128 && kTB == 8 && kN == 16, "the copy and lane maps below");

// Byte offset of 16-byte piece `half` (0, 1) of channel ch's row within one
// token's 128 rows (the two lanes of channel ch read one piece each; lanes of a
// quarter-warp read 128 consecutive bytes).
__device__ __forceinline__ int row_piece(int ch, int half) { return ch * 32 + (half << 4); }
// Byte offset of float4 `part` (0..3) of channel ch's checkpoint: parts rotate
// with ch / 2 so that the 8 lanes of a quarter-warp reading part 2 half + i
// of channels ch .. ch + 3 cover all 32 banks.
__device__ __forceinline__ int ckpt_piece(int ch, int part) {
    return ch * 64 + ((part ^ ((ch >> 1) & 3)) << 4);
}

// 16 bytes global -> shared, asynchronously; valid = false writes zeros.
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int K>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(K) : "memory");
}

// 8 floats -> 8 bf16 (16 bytes)
__device__ __forceinline__ void st_half(__nv_bfloat16* p, const float2 (&v)[kNH / 2]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __float22bfloat162_rn(v[i]);
        w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool SOFTPLUS, bool GATE>
__global__ void __launch_bounds__(kGThreads, 1) bcd_grad_staged_kernel(const BwdArgs a) {
    using T = __nv_bfloat16;
    extern __shared__ __align__(16) unsigned char smem[];
    float4* hist = reinterpret_cast<float4*>(smem + 2 * kSBuf);          // [kTB/2][2][kGThreads]
    float4* stok = reinterpret_cast<float4*>(smem + 2 * kSBuf + kSHist); // [kTB][kThreads]

    const int tid = threadIdx.x;
    const int c = tid >> 1, half = tid & 1;   // this lane: channel c of the tile, states 8 half ..
    const int64_t lin = blockIdx.x;           // (k * batch + b) * tiles + tile
    const int64_t tile = lin % a.tiles;
    const int64_t b = (lin / a.tiles) % a.batch;
    const int64_t k = lin / (a.tiles * a.batch);
    const int64_t dbase = tile * kThreads;
    // lanes past dim (a ragged last tile) compute on zeros and store nothing;
    // every lane takes part in the copies and the barriers
    const int nch = a.dim - dbase < kThreads ? static_cast<int>(a.dim - dbase) : kThreads;
    const bool ch_ok = c < nch;
    const int64_t d = ch_ok ? dbase + c : dbase;
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(a.L, t_begin + a.chunk_len);
    const int q0 = kNH * half;

    // states in pairs (packed FP32 arithmetic): pair p holds states q0 + 2p, q0 + 2p + 1
    constexpr int kP2 = kNH / 2;
    float2 A2[kP2], Q[kP2], gA[kP2];
#pragma unroll
    for (int p = 0; p < kP2; ++p) {
        A2[p] = make_float2(__ldg(a.A + d * kN + q0 + 2 * p) * kLog2e,
                            __ldg(a.A + d * kN + q0 + 2 * p + 1) * kLog2e);
        Q[p] = (a.dfinal && ch_ok)
                   ? *reinterpret_cast<const float2*>(a.dfinal + (b * a.dim + d) * kN + q0 + 2 * p)
                   : make_float2(0.f, 0.f);
        gA[p] = make_float2(0.f, 0.f);
    }
    // dL/dh at the chunk's last token: the carries of the chunks to the right
    // (unrolled: their loads do not depend on Q)
#pragma unroll 4
    for (int64_t i = a.nchunks - 1; i > k; --i) {
        const int64_t idx = (b * (a.nchunks - 1) + (i - 1)) * a.dim + d;
        const float S = a.wsS[idx];
#pragma unroll
        for (int p = 0; p < kP2; ++p) {
            const float2 qc = *reinterpret_cast<const float2*>(a.wsQ + idx * kN + q0 + 2 * p);
            const float2 e = make_float2(ex2(A2[p].x * S), ex2(A2[p].y * S));
            Q[p] = __ffma2_rn(e, Q[p], qc);
        }
    }
    const float Dd = a.D ? __ldg(a.D + d) : 0.f;
    // the scalar pass's channel (tid mod 128) and its bias
    const int pc = tid & (kThreads - 1);
    const float pbias = (a.delta_bias && pc < nch) ? __ldg(a.delta_bias + dbase + pc) : 0.f;
    const int64_t e0 = b * a.L * a.dim + d;
    T* dxg = static_cast<T*>(a.dx) + e0;
    T* ddg = static_cast<T*>(a.ddelta) + e0;
    T* dzg = GATE ? static_cast<T*>(a.dz) + e0 : nullptr;
    T* dBg = static_cast<T*>(a.dB) + e0 * kN + q0;
    T* dCg = static_cast<T*>(a.dC) + e0 * kN + q0;
    float gD = 0.f, gbias = 0.f;

    // the copies of block m (tokens 8m ..) into buffer `buf`: consecutive lanes
    // take consecutive 16-byte pieces of global memory; rows past the chunk's
    // end or the last channel read as zeros
    auto stage = [&](int64_t m, int buf) {
        unsigned char* base = smem + buf * kSBuf;
        const int64_t u0 = m * kTB;
        const int cnt = t_end - u0 < kTB ? static_cast<int>(t_end - u0) : kTB;
        const int64_t rstride = a.dim * kN, roff = ((b * a.L + u0) * a.dim + d) * kN + q0;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const T* g = static_cast<const T*>(which ? a.C : a.B);
            const T* src = g + roff;
#pragma unroll
            for (int j = 0; j < kTB; ++j, src += rstride) {
                const bool valid = j < cnt && ch_ok;
                cp16(base + which * kSRows + j * (kThreads * 32) + row_piece(c, half), valid ? src : g, valid);
            }
        }
        // x, delta (lanes 0..127) and z, dout (lanes 128..255): channels
        // 8 (tid mod 16) .. of token (tid mod 128) / 16
        {
            const int j = pc >> 4, c8 = (pc & 15) * 8;
            const bool valid = j < cnt && c8 < nch;
            const int64_t off = valid ? (b * a.L + u0 + j) * a.dim + dbase + c8 : 0;
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const int which = 2 * w + (tid >> 7);   // uniform per warp
                if (!GATE && which == 2) continue;
                const T* g = static_cast<const T*>(which == 0 ? a.x : which == 1 ? a.delta
                                                   : which == 2 ? a.z : a.dout);
                cp16(base + kSOffScal + which * kSScal + (j * kThreads + c8) * 2, g + off, valid);
            }
        }
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int piece = p * kGThreads + tid, ch = piece >> 2, part = piece & 3;
            const bool valid = ch < nch;
            const float* src = a.ckpt + (valid ? ((b * a.nckpt + m) * a.dim + dbase + ch) * kN + part * 4 : 0);
            cp16(base + kSOffCkpt + ckpt_piece(ch, part), src, valid);
        }
        cp_commit();
    };

    const int64_t m_first = t_begin / kTB, m_last = (t_end - 1) / kTB;
    stage(m_last, 0);
    int buf = 0;
    for (int64_t m = m_last; m >= m_first; --m, buf ^= 1) {
        const int64_t u0 = m * kTB;
        const int cnt = t_end - u0 < kTB ? static_cast<int>(t_end - u0) : kTB;
        if (m > m_first) {
            stage(m - 1, buf ^ 1);   // in flight while this block computes
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();   // every lane's copies of this block have landed
        const unsigned char* base = smem + buf * kSBuf;
        const T* xs = reinterpret_cast<const T*>(base + kSOffScal);   // [kTB][kThreads] each
        const T* ds = xs + kTB * kThreads;
        const T* zs = ds + kTB * kThreads;
        const T* gs = zs + kTB * kThreads;
        // the per-token scalars of channel pc, tokens (tid / 128) + 2 i
#pragma unroll
        for (int i = 0; i < kTB / 2; ++i) {
            const int j = 2 * i + (tid >> 7);
            const int o = j * kThreads + pc;
            const float v = __bfloat162float(ds[o]) + pbias;
            const float dout = __bfloat162float(gs[o]);
            float4 s;
            s.x = SOFTPLUS ? softplus(v) : v;
            s.y = SOFTPLUS ? sigmoid(v) : 1.f;
            s.z = dout;
            s.w = 0.f;
            if constexpr (GATE) {
                const float zv = __bfloat162float(zs[o]);
                s.z = dout * silu(zv);
                s.w = dout * dsilu(zv);
            }
            stok[o] = s;
        }
        __syncthreads();
        // this lane's half of channel c's B (which 0) or C (which 1) row of token j
        auto row = [&](int which, int j, float2 (&v)[kP2]) {
            const uint4 u = *reinterpret_cast<const uint4*>(base + which * kSRows + j * (kThreads * 32) +
                                                            row_piece(c, half));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < kP2; ++i)
                v[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
        };
        auto e_pair = [&](const float2 A22, const float2 dt2) {
            const float2 arg = __fmul2_rn(A22, dt2);
            return make_float2(ex2(arg.x), ex2(arg.y));
        };
        // the state before token u0, then forward over the block, the states
        // after the even tokens kept
        float2 h[kP2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float4 v = *reinterpret_cast<const float4*>(base + kSOffCkpt + ckpt_piece(c, 2 * half + i));
            h[2 * i] = make_float2(v.x, v.y);
            h[2 * i + 1] = make_float2(v.z, v.w);
        }
#pragma unroll
        for (int j = 0; j < kTB; ++j) {
            if (j < cnt) {
                const float xv = __bfloat162float(xs[j * kThreads + c]);
                const float dt = stok[j * kThreads + c].x;
                float2 bb[kP2];
                row(0, j, bb);
                const float2 dt2 = make_float2(dt, dt), dtx2 = make_float2(dt * xv, dt * xv);
#pragma unroll
                for (int p = 0; p < kP2; ++p)
                    h[p] = __ffma2_rn(e_pair(A2[p], dt2), h[p], __fmul2_rn(dtx2, bb[p]));
                if ((j & 1) == 0) {
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        hist[((j >> 1) * 2 + i) * kGThreads + tid] =
                            make_float4(h[2 * i].x, h[2 * i].y, h[2 * i + 1].x, h[2 * i + 1].y);
                }
            }
        }
        // one token of the reverse sweep; odd: the kept state is h_{j-1}
        auto sweep = [&](const int j, const bool odd) {
            const float xv = __bfloat162float(xs[j * kThreads + c]);
            const float4 s = stok[j * kThreads + c];
            const float dt = s.x, dy = s.z;
            float2 bb[kP2], cc[kP2], hk[kP2];
            row(0, j, bb);
            row(1, j, cc);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float4 v = hist[((j >> 1) * 2 + i) * kGThreads + tid];
                hk[2 * i] = make_float2(v.x, v.y);
                hk[2 * i + 1] = make_float2(v.z, v.w);
            }
            const float dtx = dt * xv;
            const float2 dt2 = make_float2(dt, dt), dtx2 = make_float2(dtx, dtx),
                         ndtx2 = make_float2(-dtx, -dtx), dy2 = make_float2(dy, dy);
            float2 dB[kP2], dC[kP2];
            float2 sgb2 = make_float2(0.f, 0.f), sga2 = sgb2, y2 = sgb2;
#pragma unroll
            for (int p = 0; p < kP2; ++p) {
                const float2 e = e_pair(A2[p], dt2);
                float2 hh, ahp;   // h_j and e^{dt A} h_{j-1}
                if (odd) {
                    ahp = __fmul2_rn(e, hk[p]);
                    hh = __ffma2_rn(dtx2, bb[p], ahp);
                } else {
                    hh = hk[p];
                    ahp = __ffma2_rn(ndtx2, bb[p], hh);
                }
                const float2 g = __ffma2_rn(dy2, cc[p], Q[p]);
                const float2 gahp = __fmul2_rn(g, ahp);
                dC[p] = __fmul2_rn(dy2, hh);
                dB[p] = __fmul2_rn(g, dtx2);
                sgb2 = __ffma2_rn(g, bb[p], sgb2);
                sga2 = __ffma2_rn(gahp, A2[p], sga2);
                gA[p] = __ffma2_rn(gahp, dt2, gA[p]);
                Q[p] = __fmul2_rn(e, g);
                if constexpr (GATE) y2 = __ffma2_rn(cc[p], hh, y2);
            }
            float sgb = sgb2.x + sgb2.y, sga = sga2.x + sga2.y, y = y2.x + y2.y;
            // the pair's sums over all 16 states
            sgb += __shfl_xor_sync(0xffffffffu, sgb, 1);
            sga += __shfl_xor_sync(0xffffffffu, sga, 1);
            if constexpr (GATE) y += __shfl_xor_sync(0xffffffffu, y, 1);
            if (ch_ok) {
                const int64_t e = (u0 + j) * a.dim;
                st_half(dBg + e * kN, dB);
                st_half(dCg + e * kN, dC);
                if (half == 0) {
                    const float ddt = fmaf(xv, sgb, sga * kLn2f);
                    const float dd = SOFTPLUS ? ddt * s.y : ddt;
                    IO<T>::st(dxg + e, fmaf(dt, sgb, dy * Dd));
                    IO<T>::st(ddg + e, dd);
                    gD = fmaf(dy, xv, gD);
                    gbias += dd;
                } else if constexpr (GATE) {
                    IO<T>::st(dzg + e, s.w * fmaf(Dd, xv, y));
                }
            }
        };
        for (int j = cnt - 1; j >= 0; --j) {
            if (j & 1)
                sweep(j, true);
            else
                sweep(j, false);
        }
        __syncthreads();   // this buffer and the scalars are free for what follows
    }
    if (!ch_ok) return;
    if (k == 0 && a.dh0) {
#pragma unroll
        for (int p = 0; p < kP2; ++p)
            *reinterpret_cast<float2*>(a.dh0 + (b * a.dim + d) * kN + q0 + 2 * p) = Q[p];
    }
    const int64_t prow = b * a.nchunks + k;
#pragma unroll
    for (int p = 0; p < kP2; ++p)
        *reinterpret_cast<float2*>(a.pA + (prow * a.dim + d) * kN + q0 + 2 * p) = gA[p];
    if (half == 0) {
        a.pD[prow * a.dim + d] = gD;
        a.pbias[prow * a.dim + d] = gbias;
    }
}

// The reverse carry for bf16 rows, staged through shared memory: the same
// recurrence as bcd_carry_kernel, one lane per channel with all 16 states.
// Each 4-token block's C rows and delta, dout and z rows of 128 channels are
// copied with cp.async, three blocks in flight per CTA (57 KB of shared
// memory, three CTAs per SM). A lane reads its channel's C row as two 16-byte
// pieces whose order alternates every 4 channels, so that the 8 lanes of a
// quarter-warp cover all 32 banks. (Two lanes per channel, 8 states each,
// executed three times the instructions per channel and token: each lane
// repeated the channel's softplus and SiLU.)
constexpr int kCCh = 128;                              // channels per CTA, one per lane
constexpr int kCTB = 4;                                // tokens per block
constexpr int kCStages = 3;
constexpr int kCRows = kCTB * kCCh * kN * 2;           // a block's C rows, bytes
constexpr int kCScal = kCTB * kCCh * 2;                // a block's delta (dout, z) rows
constexpr int kCBuf = kCRows + 3 * kCScal;
constexpr int kCarrySmem = kCStages * kCBuf;

__device__ __forceinline__ int crow_piece(int ch, int h) { return ch * 32 + ((h ^ ((ch >> 2) & 1)) << 4); }

template <bool SOFTPLUS, bool GATE>
__global__ void __launch_bounds__(kCCh) bcd_carry_staged_kernel(const BwdArgs a, int64_t ctiles) {
    using T = __nv_bfloat16;
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x;
    const int64_t lin = blockIdx.x;   // ((k - 1) * batch + b) * ctiles + tile
    const int64_t tile = lin % ctiles;
    const int64_t b = (lin / ctiles) % a.batch;
    const int64_t k = 1 + lin / (ctiles * a.batch);
    const int64_t dbase = tile * kCCh;
    const int nch = a.dim - dbase < kCCh ? static_cast<int>(a.dim - dbase) : kCCh;
    const bool ch_ok = tid < nch;
    const int64_t d = ch_ok ? dbase + tid : dbase;
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(a.L, t_begin + a.chunk_len);

    float2 A2[kN / 2], Q[kN / 2];
#pragma unroll
    for (int p = 0; p < kN / 2; ++p) {
        A2[p] = make_float2(__ldg(a.A + d * kN + 2 * p) * kLog2e, __ldg(a.A + d * kN + 2 * p + 1) * kLog2e);
        Q[p] = make_float2(0.f, 0.f);
    }
    const float bias = a.delta_bias ? __ldg(a.delta_bias + d) : 0.f;

    auto stage = [&](int64_t m, int buf) {
        unsigned char* base = smem + buf * kCBuf;
        const int64_t u0 = m * kCTB;
        const int cnt = t_end - u0 < kCTB ? static_cast<int>(t_end - u0) : kCTB;
        const T* Cg = static_cast<const T*>(a.C);
        // C rows: lane tid copies piece tid & 1 of channels tid / 2 and 64 + tid / 2
        // of every token (consecutive lanes, consecutive global bytes)
        const int h = tid & 1, chp = tid >> 1;
        const T* rowsrc = Cg + ((b * a.L + u0) * a.dim + dbase) * kN + h * 8;
#pragma unroll
        for (int j = 0; j < kCTB; ++j, rowsrc += a.dim * kN) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int ch = half * (kCCh / 2) + chp;
                const bool valid = j < cnt && ch < nch;
                cp16(base + j * (kCCh * 32) + crow_piece(ch, h), valid ? rowsrc + ch * kN : Cg, valid);
            }
        }
        // delta, dout, z: 3 arrays x 4 tokens x 16 pieces of 8 channels
        for (int piece = tid; piece < 3 * kCTB * (kCCh / 8); piece += kCCh) {
            const int which = piece / (kCTB * (kCCh / 8)), r = piece % (kCTB * (kCCh / 8));
            if (!GATE && which == 2) continue;
            const int j = r / (kCCh / 8), c8 = (r % (kCCh / 8)) * 8;
            const T* g = static_cast<const T*>(which == 0 ? a.delta : which == 1 ? a.dout : a.z);
            const bool valid = j < cnt && c8 < nch;
            const T* src = g + (valid ? (b * a.L + u0 + j) * a.dim + dbase + c8 : 0);
            cp16(base + kCRows + which * kCScal + (j * kCCh + c8) * 2, src, valid);
        }
    };

    const int64_t m_first = t_begin / kCTB, m_last = (t_end - 1) / kCTB;
    const int64_t nblk = m_last - m_first + 1;
#pragma unroll
    for (int s = 0; s < kCStages - 1; ++s) {
        if (s < nblk) stage(m_last - s, s);
        cp_commit();
    }
    float dt_sum = 0.f;
    for (int64_t i = 0; i < nblk; ++i) {
        const int64_t m = m_last - i;
        if (i + kCStages - 1 < nblk)
            stage(m - (kCStages - 1), static_cast<int>((i + kCStages - 1) % kCStages));
        cp_commit();
        cp_wait<kCStages - 1>();
        __syncthreads();   // block m's copies (every lane's) have landed
        const unsigned char* base = smem + (i % kCStages) * kCBuf;
        const T* dls = reinterpret_cast<const T*>(base + kCRows);
        const T* gos = dls + kCTB * kCCh;
        const T* zs = gos + kCTB * kCCh;
        const int cnt = t_end - m * kCTB < kCTB ? static_cast<int>(t_end - m * kCTB) : kCTB;
        for (int j = cnt - 1; j >= 0; --j) {
            float dt = __bfloat162float(dls[j * kCCh + tid]) + bias;
            if constexpr (SOFTPLUS) dt = softplus(dt);
            float dy = __bfloat162float(gos[j * kCCh + tid]);
            if constexpr (GATE) dy *= silu(__bfloat162float(zs[j * kCCh + tid]));
            const unsigned char* rowp = base + j * (kCCh * 32);
            const uint4 u0v = *reinterpret_cast<const uint4*>(rowp + crow_piece(tid, 0));
            const uint4 u1v = *reinterpret_cast<const uint4*>(rowp + crow_piece(tid, 1));
            const uint32_t w[8] = {u0v.x, u0v.y, u0v.z, u0v.w, u1v.x, u1v.y, u1v.z, u1v.w};
            const float2 dt2 = make_float2(dt, dt), dy2 = make_float2(dy, dy);
#pragma unroll
            for (int p = 0; p < kN / 2; ++p) {
                const float2 cc = make_float2(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xffff0000u));
                const float2 arg = __fmul2_rn(A2[p], dt2);
                Q[p] = __fmul2_rn(make_float2(ex2(arg.x), ex2(arg.y)), __ffma2_rn(dy2, cc, Q[p]));
            }
            dt_sum += dt;
        }
        __syncthreads();   // this buffer is refilled two blocks later
    }
    if (!ch_ok) return;
    const int64_t idx = (b * (a.nchunks - 1) + (k - 1)) * a.dim + d;
#pragma unroll
    for (int p = 0; p < kN / 2; ++p) *reinterpret_cast<float2*>(a.wsQ + idx * kN + 2 * p) = Q[p];
    a.wsS[idx] = dt_sum;
}

// dA, dD, dbias: the shares of every (batch row, chunk), added in a fixed
// order. An output is a lane quad's: lane p of the quad adds rows p, p + 4,
// ..., and two xor exchanges add the four partial sums (the same bits in every
// lane: float addition commutes). The quads' range, 4 (16 + 2) dim, is a
// multiple of 32 (dim is a multiple of 4), so a quad is always whole.
__global__ void __launch_bounds__(256) bcd_bwd_reduce_kernel(const BwdArgs a) {
    const int64_t nA = a.dim * kN, nd = a.dim;
    const int64_t total = 4 * (nA + 2 * nd), rows = a.batch * a.nchunks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t o = i >> 2;
        const int part = static_cast<int>(i & 3);
        const float* src;
        int64_t stride;
        if (o < nA) {
            src = a.pA + o;
            stride = nA;
        } else if (o < nA + nd) {
            src = a.pD + (o - nA);
            stride = nd;
        } else {
            src = a.pbias + (o - nA - nd);
            stride = nd;
        }
        float s = 0.f;
        for (int64_t r = part; r < rows; r += 4) s += src[r * stride];
        const unsigned mask = __activemask();
        s += __shfl_xor_sync(mask, s, 1);
        s += __shfl_xor_sync(mask, s, 2);
        if (part == 0) {
            if (o < nA)
                a.dA[o] = s;
            else if (o < nA + nd) {
                if (a.dD) a.dD[o - nA] = s;
            } else if (a.dbias) {
                a.dbias[o - nA - nd] = s;
            }
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
    constexpr bool kStaged = sizeof(T) == 2;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            if constexpr (kStaged) {
                e = cudaFuncSetAttribute(bcd_grad_staged_kernel<SOFTPLUS, GATE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kStagedSmem);
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(bcd_carry_staged_kernel<SOFTPLUS, GATE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kCarrySmem);
            } else
                e = cudaFuncSetAttribute(bcd_grad_kernel<T, SOFTPLUS, GATE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kGradSmem);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    const int64_t per_chunk = a.tiles * a.batch;
    if (a.nchunks > 1) {
        if constexpr (kStaged) {
            const int64_t ctiles = (a.dim + kCCh - 1) / kCCh;
            bcd_carry_staged_kernel<SOFTPLUS, GATE>
                <<<static_cast<unsigned>(ctiles * a.batch * (a.nchunks - 1)), kCCh, kCarrySmem, s>>>(
                    a, ctiles);
        } else {
            bcd_carry_kernel<T, SOFTPLUS, GATE>
                <<<static_cast<unsigned>(per_chunk * (a.nchunks - 1)), kThreads, 0, s>>>(a);
        }
    }
    if constexpr (kStaged)
        bcd_grad_staged_kernel<SOFTPLUS, GATE>
            <<<static_cast<unsigned>(per_chunk * a.nchunks), kGThreads, kStagedSmem, s>>>(a);
    else
        bcd_grad_kernel<T, SOFTPLUS, GATE>
            <<<static_cast<unsigned>(per_chunk * a.nchunks), kThreads, kGradSmem, s>>>(a);
    const int64_t total = 4 * (a.dim * kN + 2 * a.dim);
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
