// scan_fwd.cu -- the selective scan (Mamba S6) over whole sequences, sm_103a.
//
// Per channel (b, d) with an N-wide diagonal fp32 state h, starting at 0:
//   dt = softplus?(delta + bias);  h <- exp(dt A[d,:]) * h + dt B_t x;
//   y = C_t . h + D x;  out = y * silu(z)
// ("State Space Models -- Mamba, S4, and Beyond", "Mamba (S6 -- Selective
// State Space)", _selective_scan; "Mamba: State Space Models Challenge
// Transformers", "Selective Scan Algorithm" and "Mamba's Innovation:
// Selection".)
//
// L-chunks. The recurrence is linear in h, so the sequence can be cut into
// chunks joined by composing affine maps h -> P h + H, (P1, H1) then (P2, H2)
// = (P2 P1, P2 H1 + H2): the associative operator behind the pages' parallel
// scan ("State Space Models -- Mamba, S4, and Beyond", "Hardware-Efficient
// Scan (for Training)"; "State-space models (Mamba, S4)", "Training vs
// Inference Modes"). For a chunk P = prod_t exp(dt_t A) = exp(A sum_t dt_t), so
// only the sum of dt is kept. When a sequence is split, three stream-ordered
// phases run (no CTA ever waits for another CTA):
//   1. chunk state : every chunk but the last runs from h = 0 and stores its
//                    end state H and S = sum(dt)            (MODE 0)
//   2. carry       : per (b, d, n), h_in(k+1) = exp(A S_k) h_in(k) + H_k
//   3. output      : every chunk runs from its entering state, writes y; the
//                    last chunk writes final_state           (MODE 1)
// An unsplit sequence runs phase 3 alone.
//
// Work layout. One CTA = one (chunk, batch row, tile of DT channels) and WARPS
// warps. A warp owns CPW = 32 / NS consecutive channels of the tile; lane
// (c, j) = (lane / NS, lane % NS) holds states [j*SPL, j*SPL + SPL) of channel
// c in fp32 registers (SPL = N / NS). Each warp works on its own channels from
// start to end; the only CTA-wide barrier is one per stage of TS = 32 tokens.
//
// Per stage:
//   * TMA (cp.async.bulk.tensor) has loaded the [TS x DT] tiles of x, delta and
//     z into an NST-deep ring of shared-memory buffers (mbarrier completion);
//     B_t and C_t rows of the stage were converted to fp32 in shared memory
//     during the previous stage by all threads of the CTA, and are read by
//     every warp.
//   * prologue (lane = token of the stage): dt = softplus(delta + bias) and
//     dt * x for the warp's CPW channels, into a warp-private buffer; tokens
//     past the chunk end get dt = dt*x = 0, which leaves h unchanged exactly
//     (exp(0) = 1), so the state loop needs no ragged bounds.
//   * states: for each token, exp2(dt * A log2 e) on the SFU, h = Abar h +
//     (dt x) B_t and the lane's partial C_t . h, in packed f32x2 arithmetic.
//     Each lane stores its partial sums to a warp-private buffer, four tokens
//     per store.
//   * epilogue (lane = token again): y = sum of the NS partials + D x, times
//     silu(z), rounded to the I/O type, into the output tile.
//   * one elected thread TMA-stores the stage's output tile (triple-buffered)
//     and refills the input ring.
// Every mbarrier wait is bounded; a wait that gives up sets the workspace
// status word and the CTA stops.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssm_tma.cuh"

namespace ssm {
namespace {

constexpr uint32_t kMaxPolls = 1u << 24;  // bound on one mbarrier wait (about a second)
constexpr uint32_t kStatusTimeout = 7;    // -SSM_ERR_TIMEOUT

template <int NS_, int SW_, int RW_>
struct TileCfg {
    static constexpr int NS = NS_, SW = SW_, RW = RW_;
};

template <typename T, int N, typename TC>
struct Cfg {
    static constexpr int NS = TC::NS < N ? TC::NS : N;   // lanes per channel
    static constexpr int SPL = N / NS;                    // states per lane
    static constexpr int CPW = 32 / NS;                   // channels per state warp
    // state warps (small dstate: at most 64 channels per CTA)
    static constexpr int SW = TC::SW * CPW <= 64 ? TC::SW : (64 / CPW > 0 ? 64 / CPW : 1);
    static constexpr int RW = TC::RW;                     // row warps
    static constexpr int DT = SW * CPW;                   // channels per CTA
    static constexpr int CPR = DT / RW;                   // channels per row lane
    static constexpr int THREADS = (SW + RW) * 32;
    static constexpr int ROW_THREADS = RW * 32;
    static constexpr int TS = kScanStageTokens;           // tokens per stage (= 32 lanes)
    static constexpr int TILE = TS * DT;                  // elements per [TS x DT] tile
    static constexpr int NST = 3;                         // input ring depth (stages)
    static constexpr int R = 2;                           // dt / B,C / partial-sum ring depth
    static_assert(TS == 32, "a row lane owns one token of the stage");
    static_assert(N % NS == 0 && 32 % NS == 0, "state split");
    static_assert(DT % RW == 0 && CPR >= 4, "row lanes own whole vectors of channels");
    static_assert(DT * sizeof(T) % 16 == 0, "TMA rows must be whole 16-byte units");
};

constexpr int align128(int v) { return (v + 127) & ~127; }

template <typename T, int N, typename TC, int MODE>
struct Smem {
    using C = Cfg<T, N, TC>;
    static constexpr int NT = MODE == 1 ? 3 : 2;  // x, delta (, z) tiles per stage
    // B (and, for the output pass, C) rows travel with the stage's TMA
    // transaction when a row is a whole number of 16-byte units; otherwise the
    // row warps read them from global memory while converting.
    static constexpr bool BC_TMA = (N * sizeof(T)) % 16 == 0;
    static constexpr int NBC = MODE == 1 ? 2 : 1;
    static constexpr int BC_ELEMS = BC_TMA ? NBC * C::TS * N : 0;
    static constexpr int STAGE_ELEMS = NT * C::TILE + BC_ELEMS;
    // padded row strides (floats): row-lane writes and column reads then hit
    // distinct banks
    static constexpr int DTP_ROW = 2 * C::DT + 4;     // one token's (dt, dt*x) pairs
    static constexpr int YS_ROW = C::TS + 4;          // one (channel, lane) row of partials
    static constexpr int BCF = C::TS * 2 * N;         // floats per B/C slot
    static constexpr int kIn = 0;                                                   // [NST][STAGE_ELEMS] T
    static constexpr int kBC = align128(kIn + C::NST * STAGE_ELEMS * int(sizeof(T)));  // [R][TS][NS][2*SPL] f32
    static constexpr int kDtp = align128(kBC + C::R * BCF * 4);                     // [R][TS][DTP_ROW] f32
    static constexpr int kYs = align128(kDtp + C::R * C::TS * DTP_ROW * 4);         // [R][DT*NS][YS_ROW] f32
    static constexpr int kOut = align128(kYs + (MODE == 1 ? C::R * C::DT * C::NS * YS_ROW * 4 : 0));  // [2][TS][DT] T
    static constexpr int kPar = align128(kOut + (MODE == 1 ? 2 * C::TILE * int(sizeof(T)) : 0));  // [2][DT] f32: bias, D
    static constexpr int kBar = align128(kPar + 2 * C::DT * 4);
    // barriers: full[NST], prep_full[R], prep_empty[R], ys_full[R], ys_empty[R]
    static constexpr int kBytes = align128(kBar + (C::NST + 4 * C::R) * 8);
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
    static_assert((STAGE_ELEMS * sizeof(T)) % 128 == 0 && (C::TILE * sizeof(T)) % 128 == 0,
                  "TMA destinations stay 128-byte aligned");
};

// ---- shared-memory element access ----------------------------------------
__device__ __forceinline__ float lds1(const float* p) { return *p; }
__device__ __forceinline__ float lds1(const __nv_bfloat16* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16);
}
__device__ __forceinline__ void sts1(float* p, float v) { *p = v; }
__device__ __forceinline__ void sts1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
}

// K consecutive elements of one shared-memory row (K * sizeof(T) bytes,
// aligned to min(16, K * sizeof(T))) widened to fp32.
template <int K>
__device__ __forceinline__ void lds_row(const __nv_bfloat16* p, float* v) {
    if constexpr (K % 8 == 0) {
#pragma unroll
        for (int i = 0; i < K; i += 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(p + i);
            unpack_bf16x2(u.x, v[i], v[i + 1]);
            unpack_bf16x2(u.y, v[i + 2], v[i + 3]);
            unpack_bf16x2(u.z, v[i + 4], v[i + 5]);
            unpack_bf16x2(u.w, v[i + 6], v[i + 7]);
        }
    } else if constexpr (K == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        unpack_bf16x2(u.x, v[0], v[1]);
        unpack_bf16x2(u.y, v[2], v[3]);
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) v[i] = lds1(p + i);
    }
}
template <int K>
__device__ __forceinline__ void lds_row(const float* p, float* v) {
    if constexpr (K % 4 == 0) {
#pragma unroll
        for (int i = 0; i < K; i += 4) {
            const float4 u = *reinterpret_cast<const float4*>(p + i);
            v[i] = u.x; v[i + 1] = u.y; v[i + 2] = u.z; v[i + 3] = u.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) v[i] = p[i];
    }
}

// K floats from shared memory (16-byte vectors where K allows).
template <int K>
__device__ __forceinline__ void lds_f(const float* p, float* v) { lds_row<K>(p, v); }

template <int K>
__device__ __forceinline__ void sts_f(float* p, const float* v) {
    if constexpr (K % 4 == 0) {
#pragma unroll
        for (int i = 0; i < K; i += 4)
            *reinterpret_cast<float4*>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else if constexpr (K == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) p[i] = v[i];
    }
}

// K consecutive elements of one shared-memory row from fp32, rounded to T.
template <int K>
__device__ __forceinline__ void sts_row(float* p, const float* v) { sts_f<K>(p, v); }
template <int K>
__device__ __forceinline__ void sts_row(__nv_bfloat16* p, const float* v) {
    auto pk = [](float lo, float hi) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
        return *reinterpret_cast<const uint32_t*>(&b);
    };
    if constexpr (K % 8 == 0) {
#pragma unroll
        for (int i = 0; i < K; i += 8)
            *reinterpret_cast<uint4*>(p + i) = make_uint4(pk(v[i], v[i + 1]), pk(v[i + 2], v[i + 3]),
                                                          pk(v[i + 4], v[i + 5]), pk(v[i + 6], v[i + 7]));
    } else if constexpr (K == 4) {
        *reinterpret_cast<uint2*>(p) = make_uint2(pk(v[0], v[1]), pk(v[2], v[3]));
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) sts1(p + i, v[i]);
    }
}

// One state-lane step for one token: h <- exp2(dt * A2) h + dtx * B, and
// (MODE 1) the partial C . h over the lane's states.
template <int SPL, bool READOUT>
__device__ __forceinline__ float state_step(float dt, float dtx, const float* __restrict__ bc,
                                            const float (&A2)[SPL], float (&h)[SPL]) {
    if constexpr (SPL % 2 == 0) {
        float2 acc = make_float2(0.f, 0.f);
        const float2 dt2 = make_float2(dt, dt), dtx2 = make_float2(dtx, dtx);
#pragma unroll
        for (int q = 0; q < SPL; q += 2) {
            const float2 arg = __fmul2_rn(dt2, make_float2(A2[q], A2[q + 1]));
            const float2 dA = make_float2(ex2(arg.x), ex2(arg.y));
            const float2 bx = __fmul2_rn(dtx2, make_float2(bc[q], bc[q + 1]));
            const float2 hn = __ffma2_rn(dA, make_float2(h[q], h[q + 1]), bx);
            h[q] = hn.x;
            h[q + 1] = hn.y;
            if constexpr (READOUT)
                acc = __ffma2_rn(make_float2(bc[SPL + q], bc[SPL + q + 1]), hn, acc);
        }
        return acc.x + acc.y;
    } else {
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < SPL; ++q) {
            h[q] = fmaf(ex2(dt * A2[q]), h[q], dtx * bc[q]);
            if constexpr (READOUT) acc = fmaf(bc[SPL + q], h[q], acc);
        }
        return acc;
    }
}

// The token's discretized parameters for the lane's states:
// Abar = exp2(dt * A log2 e) and (dt x) B.
template <int SPL>
__device__ __forceinline__ void discretize(float dt, float dtx, const float* __restrict__ bv,
                                           const float (&A2)[SPL], float (&ea)[SPL],
                                           float (&bx)[SPL]) {
    if constexpr (SPL % 2 == 0) {
        const float2 dt2 = make_float2(dt, dt), dtx2 = make_float2(dtx, dtx);
#pragma unroll
        for (int q = 0; q < SPL; q += 2) {
            const float2 arg = __fmul2_rn(dt2, make_float2(A2[q], A2[q + 1]));
            ea[q] = ex2(arg.x);
            ea[q + 1] = ex2(arg.y);
            const float2 u = __fmul2_rn(dtx2, make_float2(bv[q], bv[q + 1]));
            bx[q] = u.x;
            bx[q + 1] = u.y;
        }
    } else {
#pragma unroll
        for (int q = 0; q < SPL; ++q) {
            ea[q] = ex2(dt * A2[q]);
            bx[q] = dtx * bv[q];
        }
    }
}

// h <- Abar h + (dt x) B and the lane's partial C . h.
template <int SPL>
__device__ __forceinline__ float recur_readout(const float (&ea)[SPL], const float (&bx)[SPL],
                                               const float* __restrict__ cv, float (&h)[SPL]) {
    if constexpr (SPL % 2 == 0) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < SPL; q += 2) {
            const float2 hn = __ffma2_rn(make_float2(ea[q], ea[q + 1]), make_float2(h[q], h[q + 1]),
                                         make_float2(bx[q], bx[q + 1]));
            h[q] = hn.x;
            h[q + 1] = hn.y;
            acc = __ffma2_rn(make_float2(cv[q], cv[q + 1]), hn, acc);
        }
        return acc.x + acc.y;
    } else {
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < SPL; ++q) {
            h[q] = fmaf(ea[q], h[q], bx[q]);
            acc = fmaf(cv[q], h[q], acc);
        }
        return acc;
    }
}

template <typename T, int N, typename TC, int MODE>
__global__ void __launch_bounds__(Cfg<T, N, TC>::THREADS, 1)
scan_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
            const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_out,
            const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
            const ScanArgs a) {
    using Cf = Cfg<T, N, TC>;
    using Sm = Smem<T, N, TC, MODE>;
    constexpr int NS = Cf::NS, SPL = Cf::SPL, CPW = Cf::CPW, DT = Cf::DT, TS = Cf::TS;
    constexpr int CPR = Cf::CPR, RW = Cf::RW, NST = Cf::NST, R = Cf::R, TILE = Cf::TILE;
    constexpr int NT = Sm::NT, NBC = Sm::NBC, DTP_ROW = Sm::DTP_ROW, YS_ROW = Sm::YS_ROW;
    constexpr int ROW_THREADS = Cf::ROW_THREADS, STATE_THREADS = Cf::SW * 32;
    constexpr bool BC_TMA = Sm::BC_TMA;

    extern __shared__ __align__(128) unsigned char smem[];
    T* in = reinterpret_cast<T*>(smem + Sm::kIn);           // [NST] x, delta, (z,) B, (C) of a stage
    float* bcf_all = reinterpret_cast<float*>(smem + Sm::kBC);
    float* dtp_all = reinterpret_cast<float*>(smem + Sm::kDtp);
    float* ys_all = reinterpret_cast<float*>(smem + Sm::kYs);
    T* outb = reinterpret_cast<T*>(smem + Sm::kOut);
    float* par = reinterpret_cast<float*>(smem + Sm::kPar);  // [0..DT): bias, [DT..2DT): D
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sm::kBar);
    uint64_t* prep_full = full + NST;    // row warps -> state warps: dt, dt*x, B/C of a stage
    uint64_t* prep_empty = prep_full + R;  // state warps -> row warps: that slot is consumed
    uint64_t* ys_full = prep_empty + R;  // state warps -> row warps: partial sums of a stage
    uint64_t* ys_empty = ys_full + R;    // row warps -> state warps: that slot is consumed

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t lin = blockIdx.x;  // chunk-major: ((k * batch) + b) * tiles + tile
    const int64_t tile = lin % a.tiles;
    const int64_t b = (lin / a.tiles) % a.batch;
    const int64_t k = lin / (a.tiles * a.batch);
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(a.L, t_begin + a.chunk_len);
    const int nstages = static_cast<int>((t_end - t_begin + TS - 1) / TS);
    const int64_t dbase = tile * DT;
    const bool has_z = MODE == 1 && a.z != nullptr;
    const uint32_t stage_tx =
        static_cast<uint32_t>(((has_z ? 3 : 2) * TILE + Sm::BC_ELEMS) * sizeof(T));

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(&full[i], 1);
        for (int i = 0; i < R; ++i) {
            mbar_init(&prep_full[i], ROW_THREADS);
            mbar_init(&prep_empty[i], STATE_THREADS);
            mbar_init(&ys_full[i], STATE_THREADS);
            mbar_init(&ys_empty[i], ROW_THREADS);
        }
        fence_mbar_init();
    }
    for (int i = tid; i < DT; i += Cf::THREADS) {
        const int64_t dq = dbase + i;
        const bool okq = dq < a.dim;
        par[i] = (a.delta_bias && okq) ? __ldg(a.delta_bias + dq) : 0.f;
        par[DT + i] = (MODE == 1 && a.D && okq) ? __ldg(a.D + dq) : 0.f;
    }
    __syncthreads();

    auto issue = [&](int s) {
        const int buf = s % NST;
        T* dst = in + static_cast<size_t>(buf) * Sm::STAGE_ELEMS;
        const int t = static_cast<int>(t_begin + static_cast<int64_t>(s) * TS);
        mbar_arrive_expect_tx(&full[buf], stage_tx);
        tma_load_3d(dst, &tm_x, static_cast<int>(dbase), t, static_cast<int>(b), &full[buf]);
        tma_load_3d(dst + TILE, &tm_dt, static_cast<int>(dbase), t, static_cast<int>(b), &full[buf]);
        if (has_z)
            tma_load_3d(dst + 2 * TILE, &tm_z, static_cast<int>(dbase), t, static_cast<int>(b),
                        &full[buf]);
        if constexpr (BC_TMA) {
            tma_load_3d(dst + NT * TILE, &tm_B, 0, t, static_cast<int>(b), &full[buf]);
            if constexpr (MODE == 1)
                tma_load_3d(dst + NT * TILE + TS * N, &tm_C, 0, t, static_cast<int>(b), &full[buf]);
        }
    };

    bool aborted = false;
    if (warp < RW) {
        // =================== row warps: TMA, prologue, epilogue ===================
        const int rw = warp;                 // row warp index
        int issued = 0;
        if (tid == 0)
            for (; issued < NST && issued < nstages; ++issued) issue(issued);

        // Row lane: token `lane` of a stage, channels [rw*CPR, rw*CPR + CPR).
        const int cbase = rw * CPR;
        const bool softplus_on = a.softplus != 0;
        const T* __restrict__ Bg = static_cast<const T*>(a.B);
        const T* __restrict__ Cg = static_cast<const T*>(a.C);
        constexpr int VE = 16 / sizeof(T) < N ? 16 / sizeof(T) : N;   // elements per vector
        constexpr int NVEC = NBC * TS * N / VE;                        // B/C vectors per stage
        constexpr int RUN = SPL < VE ? SPL : VE;                       // runs of one state group

        const int last = MODE == 1 ? nstages + 1 : nstages;
        for (int i = 0; i < last; ++i) {
            bool ok = true;
            if (i < nstages) {
                // ---- prologue of stage i ----
                const int buf = i % NST, slot = i % R;
                ok = mbar_wait_bounded(&full[buf], static_cast<uint32_t>((i / NST) & 1), kMaxPolls);
                if (i >= R)
                    ok = ok && mbar_wait_bounded(&prep_empty[slot],
                                                 static_cast<uint32_t>(((i / R) - 1) & 1), kMaxPolls);
                const T* xt = in + static_cast<size_t>(buf) * Sm::STAGE_ELEMS;
                const T* dlt = xt + TILE;
                const T* staged = xt + NT * TILE;
                float* bcf = bcf_all + slot * Sm::BCF;
                float* dtp = dtp_all + slot * TS * DTP_ROW;
                const int64_t ts = t_begin + static_cast<int64_t>(i) * TS;
                // B (and C) rows -> fp32 bcf[t][j][B(SPL) | C(SPL)]
                for (int idx = tid; idx < NVEC; idx += ROW_THREADS) {
                    const int which = idx / (TS * N / VE);
                    const int r = idx % (TS * N / VE);
                    const int t = r / (N / VE), n0 = (r % (N / VE)) * VE;
                    float v[VE];
                    if constexpr (BC_TMA) {
                        lds_row<VE>(staged + which * TS * N + t * N + n0, v);  // zero past the end
                    } else {
#pragma unroll
                        for (int e = 0; e < VE; ++e)
                            v[e] = ts + t < t_end
                                       ? IO<T>::ld((which ? Cg : Bg) + (b * a.L + ts + t) * N + n0 + e)
                                       : 0.f;
                    }
#pragma unroll
                    for (int e = 0; e < VE; e += RUN) {
                        const int n = n0 + e;
                        sts_f<RUN>(bcf + (t * NS + n / SPL) * 2 * SPL + which * SPL + n % SPL, &v[e]);
                    }
                }
                // dt and dt * x for token `lane`; tokens past the chunk end get
                // dt = dt*x = 0, which leaves h unchanged exactly
                {
                    float xv[CPR], dv[CPR], bv[CPR];
                    lds_row<CPR>(xt + lane * DT + cbase, xv);
                    lds_row<CPR>(dlt + lane * DT + cbase, dv);
                    lds_f<CPR>(par + cbase, bv);
                    const bool valid = ts + lane < t_end;
                    float o[2 * CPR];
#pragma unroll
                    for (int q = 0; q < CPR; ++q) {
                        float dtv = dv[q] + bv[q];
                        if (softplus_on) dtv = softplus(dtv);
                        dtv = valid ? dtv : 0.f;
                        o[2 * q] = dtv;
                        o[2 * q + 1] = dtv * xv[q];
                    }
                    sts_f<2 * CPR>(dtp + lane * DTP_ROW + 2 * cbase, o);
                }
                mbar_arrive(&prep_full[slot]);
                if constexpr (MODE == 0) {
                    // the stage's input slot is free once every row thread is done
                    if (named_bar_or(1, ROW_THREADS, !ok)) { aborted = true; break; }
                    if (tid == 0 && issued < nstages) {
                        fence_proxy_async_smem();
                        issue(issued++);
                    }
                }
            }
            if constexpr (MODE == 1) {
                if (i == 0) {
                    if (named_bar_or(1, ROW_THREADS, !ok)) { aborted = true; break; }
                } else {
                    // ---- epilogue of stage e = i - 1 ----
                    const int e = i - 1, slot = e % R, buf = e % NST;
                    ok = ok && mbar_wait_bounded(&ys_full[slot], static_cast<uint32_t>((e / R) & 1),
                                                 kMaxPolls);
                    // the output buffer this stage writes was stored by stage e - 2
                    if (tid == 0) bulk_wait_read<1>();
                    if (named_bar_or(1, ROW_THREADS, !ok)) { aborted = true; break; }
                    const T* xt = in + static_cast<size_t>(buf) * Sm::STAGE_ELEMS;
                    const T* zt = xt + 2 * TILE;
                    const float* ys = ys_all + slot * DT * NS * YS_ROW;
                    T* ot = outb + (e & 1) * TILE;
                    float xv[CPR], yv[CPR], Dq[CPR];
                    lds_row<CPR>(xt + lane * DT + cbase, xv);
                    lds_f<CPR>(par + DT + cbase, Dq);
#pragma unroll
                    for (int q = 0; q < CPR; ++q) {
                        float y = 0.f;
#pragma unroll
                        for (int jj = 0; jj < NS; ++jj) y += ys[((cbase + q) * NS + jj) * YS_ROW + lane];
                        yv[q] = fmaf(Dq[q], xv[q], y);
                    }
                    mbar_arrive(&ys_empty[slot]);
                    if (has_z) {
                        float zv[CPR];
                        lds_row<CPR>(zt + lane * DT + cbase, zv);
#pragma unroll
                        for (int q = 0; q < CPR; ++q) yv[q] *= silu(zv[q]);
                    }
                    sts_row<CPR>(ot + lane * DT + cbase, yv);
                    fence_proxy_async_smem();   // the output tile is read by the TMA store
                    named_bar_sync(1, ROW_THREADS);
                    if (tid == 0) {
                        tma_store_3d(&tm_out, static_cast<int>(dbase),
                                     static_cast<int>(t_begin + static_cast<int64_t>(e) * TS),
                                     static_cast<int>(b), ot);
                        bulk_commit();
                        // the stage's input slot is free: refill it
                        if (issued < nstages) {
                            fence_proxy_async_smem();
                            issue(issued++);
                        }
                    }
                }
            }
        }
        if (tid == 0) {
            bulk_wait_all();
            if (aborted) {
                // let the copies already in flight land before the CTA releases its smem
                for (int r = issued - NST < 0 ? 0 : issued - NST; r < issued; ++r)
                    mbar_wait_bounded(&full[r % NST], static_cast<uint32_t>((r / NST) & 1), kMaxPolls);
            }
        }
        if (aborted && lane == 0 && a.status) atomicExch(a.status, kStatusTimeout);
        return;
    }

    // =================== state warps: the recurrence ===================
    const int sw = warp - RW;
    const int c = lane / NS, j = lane % NS;
    const int col = sw * CPW + c;                // channel within the tile
    const bool ch_ok = dbase + col < a.dim;
    const int64_t d = ch_ok ? dbase + col : 0;
    float A2[SPL], h[SPL];
#pragma unroll
    for (int q = 0; q < SPL; ++q) {
        A2[q] = ch_ok ? __ldg(a.A + d * N + j * SPL + q) * kLog2e : 0.f;
        h[q] = 0.f;
    }
    if (MODE == 1 && k > 0 && ch_ok) {
        const float* hin = a.ws_H + ((b * (a.nchunks - 1) + (k - 1)) * a.dim + d) * N + j * SPL;
#pragma unroll
        for (int q = 0; q < SPL; ++q) h[q] = hin[q];
    }
    float dt_sum = 0.f;

    for (int s = 0; s < nstages; ++s) {
        const int slot = s % R;
        bool ok = mbar_wait_bounded(&prep_full[slot], static_cast<uint32_t>((s / R) & 1), kMaxPolls);
        if (MODE == 1 && s >= R)
            ok = ok && mbar_wait_bounded(&ys_empty[slot], static_cast<uint32_t>(((s / R) - 1) & 1),
                                         kMaxPolls);
        if (__any_sync(0xffffffffu, !ok)) { aborted = true; break; }
        const float* dtp = dtp_all + slot * TS * DTP_ROW;
        const float* bcf = bcf_all + slot * Sm::BCF;
        if constexpr (MODE == 1) {
            // the recurrence and this lane's partial C . h for every token of
            // the stage, kept in registers, then stored to the partial-sum slot
            float p[TS];
#pragma unroll
            for (int t = 0; t < TS; ++t) {
                const float2 dd = *reinterpret_cast<const float2*>(dtp + t * DTP_ROW + 2 * col);
                float bcv[2 * SPL];
                lds_f<2 * SPL>(bcf + (t * NS + j) * 2 * SPL, bcv);
                p[t] = state_step<SPL, true>(dd.x, dd.y, bcv, A2, h);
            }
            mbar_arrive(&prep_empty[slot]);
            float* yrow = ys_all + slot * DT * NS * YS_ROW + (sw * 32 + lane) * YS_ROW;  // row (col, j)
#pragma unroll
            for (int t4 = 0; t4 < TS; t4 += 4)
                *reinterpret_cast<float4*>(yrow + t4) =
                    make_float4(p[t4], p[t4 + 1], p[t4 + 2], p[t4 + 3]);
            mbar_arrive(&ys_full[slot]);
        } else {
#pragma unroll
            for (int t = 0; t < TS; ++t) {
                const float2 dd = *reinterpret_cast<const float2*>(dtp + t * DTP_ROW + 2 * col);
                float bv[SPL];
                lds_f<SPL>(bcf + (t * NS + j) * 2 * SPL, bv);
                dt_sum += dd.x;
                state_step<SPL, false>(dd.x, dd.y, bv, A2, h);
            }
            mbar_arrive(&prep_empty[slot]);
        }
    }
    if (aborted) {
        if (lane == 0 && a.status) atomicExch(a.status, kStatusTimeout);
        return;
    }
    if (!ch_ok) return;
    if (MODE == 0) {
        const int64_t base = (b * (a.nchunks - 1) + k) * a.dim + d;
        float* dst = a.ws_H + base * N + j * SPL;
#pragma unroll
        for (int q = 0; q < SPL; ++q) dst[q] = h[q];
        if (j == 0) a.ws_S[base] = dt_sum;
    } else if (a.final_state && k == a.nchunks - 1) {
        float* fs = a.final_state + (b * a.dim + d) * N + j * SPL;
#pragma unroll
        for (int q = 0; q < SPL; ++q) fs[q] = h[q];
    }
}

// Phase 2: one thread per (b, d, n). h_in(0) = 0 and
// h_in(k+1) = exp(A S_k) h_in(k) + H_k, written over H_k.
template <int N>
__global__ void __launch_bounds__(256) scan_carry_kernel(const ScanArgs a) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= a.batch * a.dim * N) return;
    const int64_t n = i % N;
    const int64_t d = (i / N) % a.dim;
    const int64_t b = i / (N * a.dim);
    const float A2 = __ldg(a.A + d * N + n) * kLog2e;
    float h = 0.f;
    for (int64_t k = 0; k + 1 < a.nchunks; ++k) {
        const int64_t idx = (b * (a.nchunks - 1) + k) * a.dim + d;
        h = fmaf(ex2(A2 * a.ws_S[idx]), h, a.ws_H[idx * N + n]);
        a.ws_H[idx * N + n] = h;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiled>(nullptr);
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

// [batch][L][dim] tensor, box of `box_channels` channels x TS tokens x 1 batch
// row (elements past the sequence end or the last channel read as zero).
template <typename T>
cudaError_t make_tmap(CUtensorMap* tm, const void* base, int64_t batch, int64_t L, int64_t dim,
                      int box_channels) {
    EncodeTiled fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t es = sizeof(T);
    const cuuint64_t gdim[3] = {cuuint64_t(dim), cuuint64_t(L), cuuint64_t(batch)};
    const cuuint64_t gstride[2] = {cuuint64_t(dim) * es, cuuint64_t(L) * cuuint64_t(dim) * es};
    const cuuint32_t box[3] = {cuuint32_t(box_channels), cuuint32_t(kScanStageTokens), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = fn(tm, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          3, const_cast<void*>(base), gdim, gstride, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Raise the dynamic shared-memory limit of one kernel instantiation, once per
// device (the statics are per instantiation).
template <typename T, int N, typename TC, int MODE>
cudaError_t allow_smem() {
    static std::mutex mu;
    static bool done[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(scan_kernel<T, N, TC, MODE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<T, N, TC, MODE>::kBytes);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

template <typename T, int N, typename TC>
cudaError_t launch_cfg(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    using Cf = Cfg<T, N, TC>;
    if (p.channels_per_cta != Cf::DT) return cudaErrorInvalidValue;
    CUtensorMap tx, tdt, tz, tout;
    cudaError_t e;
    if ((e = make_tmap<T>(&tx, a.x, a.batch, a.L, a.dim, Cf::DT)) != cudaSuccess) return e;
    if ((e = make_tmap<T>(&tdt, a.delta, a.batch, a.L, a.dim, Cf::DT)) != cudaSuccess) return e;
    if ((e = make_tmap<T>(&tz, a.z ? a.z : a.x, a.batch, a.L, a.dim, Cf::DT)) != cudaSuccess)
        return e;
    if ((e = make_tmap<T>(&tout, a.out, a.batch, a.L, a.dim, Cf::DT)) != cudaSuccess) return e;
    // B, C [batch][L][N]: box of N states x TS tokens (only when a row is a
    // whole number of 16-byte units; otherwise the kernel reads them directly)
    CUtensorMap tB = tx, tC = tx;
    if constexpr (Smem<T, N, TC, 1>::BC_TMA) {
        if ((e = make_tmap<T>(&tB, a.B, a.batch, a.L, N, N)) != cudaSuccess) return e;
        if ((e = make_tmap<T>(&tC, a.C, a.batch, a.L, N, N)) != cudaSuccess) return e;
    }
    const int64_t per_chunk = p.tiles * a.batch;
    if (p.nchunks > 1) {
        constexpr int sm0 = Smem<T, N, TC, 0>::kBytes;
        if ((e = allow_smem<T, N, TC, 0>()) != cudaSuccess) return e;
        scan_kernel<T, N, TC, 0>
            <<<static_cast<unsigned>(per_chunk * (p.nchunks - 1)), Cf::THREADS, sm0, s>>>(
                tx, tdt, tz, tout, tB, tC, a);
        const int64_t n = a.batch * a.dim * N;
        scan_carry_kernel<N><<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(a);
    }
    constexpr int sm1 = Smem<T, N, TC, 1>::kBytes;
    if ((e = allow_smem<T, N, TC, 1>()) != cudaSuccess) return e;
    scan_kernel<T, N, TC, 1>
        <<<static_cast<unsigned>(per_chunk * p.nchunks), Cf::THREADS, sm1, s>>>(tx, tdt, tz, tout,
                                                                                 tB, tC, a);
    return cudaGetLastError();
}

// The tile configurations by id (the same table as scan_lanes_per_channel and
// scan_tile_warps in ssm_internal.h).
using Tile0 = TileCfg<4, 4, 2>;
using Tile1 = TileCfg<8, 4, 2>;
using Tile2 = TileCfg<4, 2, 1>;
using Tile3 = TileCfg<2, 4, 2>;

template <typename T, int N>
cudaError_t launch_typed(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    switch (p.tile_cfg) {
        case 0: return launch_cfg<T, N, Tile0>(a, p, s);
        case 1: return launch_cfg<T, N, Tile1>(a, p, s);
        case 2: return launch_cfg<T, N, Tile2>(a, p, s);
        case 3: return launch_cfg<T, N, Tile3>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_n(const ScanArgs& a, const ScanPlan& p, int N, cudaStream_t s) {
    switch (N) {
        case 1: return launch_typed<T, 1>(a, p, s);
        case 2: return launch_typed<T, 2>(a, p, s);
        case 4: return launch_typed<T, 4>(a, p, s);
        case 8: return launch_typed<T, 8>(a, p, s);
        case 16: return launch_typed<T, 16>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, const ScanPlan& p, int io, int N, cudaStream_t s) {
    return io == 1 ? launch_n<__nv_bfloat16>(a, p, N, s) : launch_n<float>(a, p, N, s);
}

}  // namespace ssm
