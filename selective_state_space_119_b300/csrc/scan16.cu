// scan16.cu -- the selective scan at d_state 16 (the pages' Mamba sizes), sm_103a.
//
// Per channel (b, d) with a 16-wide diagonal fp32 state h, starting at h0 (or 0):
//   dt = softplus?(delta + bias);  h <- exp(dt A[d,:]) * h + dt B_t x;
//   y = C_t . h + D x;  out = y * silu(z)
// ("State Space Models -- Mamba, S4, and Beyond", "Mamba (S6 -- Selective
// State Space)", _selective_scan; "Mamba: State Space Models Challenge
// Transformers", "Selective Scan Algorithm" and "Mamba's Innovation:
// Selection".)
//
// Work layout. One lane owns one channel and all 16 of its states in fp32
// registers; a CTA is W warps (32 W consecutive channels) of one batch row over
// one L-chunk. Per 32-token stage, TMA (cp.async.bulk.tensor) loads the
// [32 x 32W] tiles of x, delta (and z) and the stage's B_t (and C_t) rows into
// a ring of NST shared-memory stages (mbarrier completion, bounded waits); the
// CTA converts the B / C rows to fp32 once, and every lane then reads them as
// broadcast 16-byte loads. y is written in place over the stage's x tile (each
// lane overwrites only the x value it has already read) and TMA-stored.
//
// The decay factors. For a general A, exp(dt A[d,n]) is one SFU exponential
// per state (2^(dt A log2 e)). When a channel's A row has the structure
// A[d,n] = a (n+1) -- the pages' initialisation A = -(1, 2, ..., N)
// ("State Space Models -- Mamba, S4, and Beyond", MambaBlock, A_log) -- the
// factors are the powers r, r^2, ..., r^16 of r = exp(dt a): four SFU
// exponentials (r, r^2, r^4, r^8) and eleven multiplications give all sixteen,
// no product deeper than three. Each warp tests its 32 rows once (a vote) and
// takes the matching token loop.
//
// L-chunks. The recurrence is linear in h, so the sequence can be cut into
// chunks joined by composing affine maps h -> P h + H, (P1, H1) then (P2, H2)
// = (P2 P1, P2 H1 + H2): the associative operator behind the pages' parallel
// scan ("State Space Models -- Mamba, S4, and Beyond", "Hardware-Efficient
// Scan (for Training)"). For a chunk P = exp(A S) with S its sum of dt. Two
// stream-ordered launches (no CTA waits for another CTA):
//   1. chunk state (every chunk but the last): the chunk's end state from
//      h = 0, H_n = sum_t dt_t x_t B_t[n] exp(A_n R_t) with R_t the sum of dt
//      over the chunk's tokens after t. The tokens are visited last to first,
//      so R_t is a running sum and each term is one multiply-add on the
//      weights dt_t x_t exp(A_n R_t) (for a structured row, again the powers of
//      one exponential) -- no recurrence through the states.
//   2. output: chunk k starts from h0 (or 0), composes the maps of chunks
//      0 .. k-1, then runs the recurrence over its tokens and writes y; the
//      last chunk writes final_state.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssm_tma.cuh"
#include "ssm_tmap.h"

namespace ssm {
namespace {

constexpr int kN = 16;
constexpr uint32_t kPolls = 1u << 24;      // bound on one mbarrier wait (about a second)
constexpr uint32_t kStatusTimeout = 7;     // -SSM_ERR_TIMEOUT

// Shared-memory layout of one CTA. A stage holds the x, delta (and z) tiles
// [TS][DT] and the B (and C) rows [TS][16] of TS tokens; bcf holds the fp32
// B | C rows of the stage being computed and of the next one.
template <typename T, int W, int CPL, int NST, int MODE, int TS>
struct Lay {
    static constexpr int DT = 32 * W * CPL;                  // channels per CTA
    static constexpr int TILE = TS * DT;                     // elements of a tile
    static constexpr int TILE_B = TILE * int(sizeof(T));
    static constexpr int NT = MODE == 1 ? 3 : 2;             // x, delta (, z)
    static constexpr int NBC = MODE == 1 ? 2 : 1;            // B (, C)
    static constexpr int ROW = NBC * kN;                     // floats per token in bcf
    static constexpr int ROWS_B = TS * kN * int(sizeof(T));  // bytes of one stage's B rows
    static constexpr int STAGE = NT * TILE_B + NBC * ROWS_B;
    static constexpr int kDelta = TILE_B;                    // byte offsets in a stage
    static constexpr int kZ = 2 * TILE_B;
    static constexpr int kB = NT * TILE_B;
    static constexpr int kBC = NST * STAGE;                  // [2][TS][ROW] f32
    static constexpr int kBar = kBC + 2 * TS * ROW * 4;
    static constexpr int kBytes = kBar + NST * 8;
    static_assert(TILE_B % 128 == 0 && ROWS_B % 128 == 0 && STAGE % 128 == 0,
                  "TMA destinations stay 128-byte aligned");
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
    static_assert(kScanStageTokens % TS == 0, "chunks are whole stages");
};

// CPL consecutive channels of one token row in shared memory (the kernel is
// written for CPL channels per lane; one is built).
template <typename T, int CPL> struct Row;
template <> struct Row<float, 1> {
    __device__ __forceinline__ static void ld(const float* p, float (&v)[1]) { v[0] = *p; }
    __device__ __forceinline__ static void st(float* p, const float (&v)[1]) { *p = v[0]; }
};
template <> struct Row<__nv_bfloat16, 1> {
    __device__ __forceinline__ static void ld(const __nv_bfloat16* p, float (&v)[1]) {
        v[0] = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(p)) << 16);
    }
    __device__ __forceinline__ static void st(__nv_bfloat16* p, const float (&v)[1]) {
        *p = __float2bfloat16_rn(v[0]);
    }
};
__device__ __forceinline__ void ld4(const float* p, float& a, float& b, float& c, float& d) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    a = u.x; b = u.y; c = u.z; d = u.w;
}

// The decay factors of a structured row, f[n] = 2^((n + 1) s) with s = dt a
// log2 e: four SFU exponentials and products of depth at most three.
__device__ __forceinline__ void powers16(float s, float (&f)[kN]) {
    const float r1 = ex2(s), r2 = ex2(2.f * s), r4 = ex2(4.f * s), r8 = ex2(8.f * s);
    f[0] = r1;
    f[1] = r2;
    f[2] = r1 * r2;
    f[3] = r4;
    const float2 p56 = __fmul2_rn(make_float2(r1, r2), make_float2(r4, r4));
    f[4] = p56.x;
    f[5] = p56.y;
    f[6] = f[2] * r4;
    f[7] = r8;
    const float2 r8x2 = make_float2(r8, r8);
#pragma unroll
    for (int q = 0; q < 8; q += 2) {
        const float2 u = __fmul2_rn(make_float2(f[q], f[q + 1]), r8x2);
        f[8 + q] = u.x;
        f[9 + q] = u.y;
    }
}

// The same powers, scaled: w[n] = c 2^((n + 1) s).
__device__ __forceinline__ void scaled_powers16(float c, float s, float (&w)[kN]) {
    const float g1 = ex2(s), g2 = ex2(2.f * s), g4 = ex2(4.f * s), g8 = ex2(8.f * s);
    const float2 w12 = __fmul2_rn(make_float2(c, c), make_float2(g1, g2));
    const float2 w34 = __fmul2_rn(make_float2(w12.x, c), make_float2(g2, g4));
    const float2 w56 = __fmul2_rn(w12, make_float2(g4, g4));
    const float2 w78 = __fmul2_rn(make_float2(w34.x, c), make_float2(g4, g8));
    w[0] = w12.x; w[1] = w12.y; w[2] = w34.x; w[3] = w34.y;
    w[4] = w56.x; w[5] = w56.y; w[6] = w78.x; w[7] = w78.y;
    const float2 g8x2 = make_float2(g8, g8);
#pragma unroll
    for (int q = 0; q < 8; q += 2) {
        const float2 u = __fmul2_rn(make_float2(w[q], w[q + 1]), g8x2);
        w[8 + q] = u.x;
        w[9 + q] = u.y;
    }
}

// The decay factors of a general row: f[n] = 2^(dt A[n] log2 e).
__device__ __forceinline__ void exps16(float dt, const float (&A2)[kN], float (&f)[kN]) {
#pragma unroll
    for (int q = 0; q < kN; q += 2) {
        const float2 arg = __fmul2_rn(make_float2(dt, dt), make_float2(A2[q], A2[q + 1]));
        f[q] = ex2(arg.x);
        f[q + 1] = ex2(arg.y);
    }
}

// One token of the recurrence and its readout: h <- f h + dtx B; returns C . h.
__device__ __forceinline__ float step16(const float (&f)[kN], float dtx, const float (&Bv)[kN],
                                        const float (&Cv)[kN], float (&h)[kN]) {
    const float2 dtx2 = make_float2(dtx, dtx);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kN; q += 2) {
        const float2 bx = __fmul2_rn(dtx2, make_float2(Bv[q], Bv[q + 1]));
        const float2 hn = __ffma2_rn(make_float2(f[q], f[q + 1]), make_float2(h[q], h[q + 1]), bx);
        h[q] = hn.x;
        h[q + 1] = hn.y;
        if (q < kN / 2)
            acc0 = __ffma2_rn(make_float2(Cv[q], Cv[q + 1]), hn, acc0);
        else
            acc1 = __ffma2_rn(make_float2(Cv[q], Cv[q + 1]), hn, acc1);
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// One token of the chunk-state sum: H += w B.
__device__ __forceinline__ void accum16(const float (&w)[kN], const float (&Bv)[kN], float (&H)[kN]) {
#pragma unroll
    for (int q = 0; q < kN; q += 2) {
        const float2 u = __ffma2_rn(make_float2(w[q], w[q + 1]), make_float2(Bv[q], Bv[q + 1]),
                                    make_float2(H[q], H[q + 1]));
        H[q] = u.x;
        H[q + 1] = u.y;
    }
}

template <int K>
__device__ __forceinline__ void lds_row(const float* p, float (&v)[K]) {
#pragma unroll
    for (int q = 0; q < K; q += 4) ld4(p + q, v[q], v[q + 1], v[q + 2], v[q + 3]);
}

// MODE 1: the output pass. MODE 0: the chunk-state pass (tokens last to first).
// Lane l owns the CPL consecutive channels dbase + CPL l + c, c < CPL, and all
// 16 states of each; one load of B_t (and C_t) serves all of them.
template <typename T, int W, int CPL, int NST, int TS, int MODE, bool SOFTPLUS, bool GATE>
__global__ void __launch_bounds__(32 * W, 4)
scan16_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
              const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
              const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_out,
              const ScanArgs a) {
    using Ly = Lay<T, W, CPL, NST, MODE, TS>;
    using RW = Row<T, CPL>;
    constexpr int DT = Ly::DT, ROW = Ly::ROW, THREADS = 32 * W;
    constexpr bool has_z = MODE == 1 && GATE;

    extern __shared__ __align__(128) unsigned char smem[];
    float* bcf = reinterpret_cast<float*>(smem + Ly::kBC);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Ly::kBar);

    const int tid = threadIdx.x;
    const int64_t lin = blockIdx.x;   // chunk-major: ((k * batch) + b) * tiles + tile
    const int64_t tile = lin % a.tiles;
    const int64_t b = (lin / a.tiles) % a.batch;
    const int64_t k = lin / (a.tiles * a.batch);
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(a.L, t_begin + a.chunk_len);
    const int nstages = static_cast<int>((t_end - t_begin + TS - 1) / TS);
    const int64_t dbase = tile * DT;
    const uint32_t stage_tx = static_cast<uint32_t>(
        (has_z ? 3 : 2) * Ly::TILE_B + Ly::NBC * Ly::ROWS_B);
    // the chunk-state pass visits its stages last to first
    auto stage_of = [&](int i) { return MODE == 1 ? i : nstages - 1 - i; };

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int i) {   // the i-th stage in visiting order
        const int buf = i % NST;
        unsigned char* dst = smem + static_cast<size_t>(buf) * Ly::STAGE;
        const int t = static_cast<int>(t_begin + static_cast<int64_t>(stage_of(i)) * TS);
        const int bb = static_cast<int>(b);
        mbar_arrive_expect_tx(&full[buf], stage_tx);
        tma_load_3d(dst, &tm_x, static_cast<int>(dbase), t, bb, &full[buf]);
        tma_load_3d(dst + Ly::kDelta, &tm_dt, static_cast<int>(dbase), t, bb, &full[buf]);
        if constexpr (has_z) tma_load_3d(dst + Ly::kZ, &tm_z, static_cast<int>(dbase), t, bb, &full[buf]);
        tma_load_3d(dst + Ly::kB, &tm_B, 0, t, bb, &full[buf]);
        if constexpr (MODE == 1) tma_load_3d(dst + Ly::kB + Ly::ROWS_B, &tm_C, 0, t, bb, &full[buf]);
    };
    if (tid == 0)
        for (int i = 0; i < NST && i < nstages; ++i) issue(i);

    // ---- this lane's channels ----
    const int col = tid * CPL;   // first own channel within the tile
    bool ch_ok[CPL];
    int64_t dch[CPL];
    float A2[CPL][kN], a2[CPL], bias[CPL], Dd[CPL];
    bool mine = true;   // A[d, n] = A[d, 0] (n + 1) exactly, for every own row
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        dch[c] = dbase + col + c;
        ch_ok[c] = dch[c] < a.dim;
        const int64_t ds = ch_ok[c] ? dch[c] : 0;
        const float4* ap = reinterpret_cast<const float4*>(a.A + ds * kN);
        float Arow[kN];
#pragma unroll
        for (int q = 0; q < kN / 4; ++q) {
            const float4 u = __ldg(ap + q);
            Arow[4 * q] = u.x; Arow[4 * q + 1] = u.y; Arow[4 * q + 2] = u.z; Arow[4 * q + 3] = u.w;
        }
        bool st = true;
#pragma unroll
        for (int n = 1; n < kN; ++n) st = st && (Arow[n] == Arow[0] * float(n + 1));
        mine = mine && (st || !ch_ok[c]);
#pragma unroll
        for (int n = 0; n < kN; ++n) A2[c][n] = ch_ok[c] ? Arow[n] * kLog2e : 0.f;
        a2[c] = A2[c][0];   // a log2 e (structured rows)
        bias[c] = (a.delta_bias && ch_ok[c]) ? __ldg(a.delta_bias + ds) : 0.f;
        Dd[c] = (MODE == 1 && a.D && ch_ok[c]) ? __ldg(a.D + ds) : 0.f;
    }
    const bool structured = __all_sync(0xffffffffu, mine);

    float h[CPL][kN];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
#pragma unroll
        for (int n = 0; n < kN; ++n) h[c][n] = 0.f;
        if (MODE == 1 && ch_ok[c]) {
            if (a.h0) {
                const float4* hp =
                    reinterpret_cast<const float4*>(a.h0 + (b * a.dim + dch[c]) * kN);
#pragma unroll
                for (int q = 0; q < kN / 4; ++q) {
                    const float4 u = hp[q];
                    h[c][4 * q] = u.x; h[c][4 * q + 1] = u.y; h[c][4 * q + 2] = u.z;
                    h[c][4 * q + 3] = u.w;
                }
            }
            // the state entering chunk k: h <- exp(A S_i) h + H_i over chunks 0 .. k-1
            for (int64_t i = 0; i < k; ++i) {
                const int64_t idx = (b * (a.nchunks - 1) + i) * a.dim + dch[c];
                const float S = a.ws_S[idx];
                const float4* Hp = reinterpret_cast<const float4*>(a.ws_H + idx * kN);
#pragma unroll
                for (int q = 0; q < kN / 4; ++q) {
                    const float4 u = Hp[q];
                    h[c][4 * q] = fmaf(ex2(A2[c][4 * q] * S), h[c][4 * q], u.x);
                    h[c][4 * q + 1] = fmaf(ex2(A2[c][4 * q + 1] * S), h[c][4 * q + 1], u.y);
                    h[c][4 * q + 2] = fmaf(ex2(A2[c][4 * q + 2] * S), h[c][4 * q + 2], u.z);
                    h[c][4 * q + 3] = fmaf(ex2(A2[c][4 * q + 3] * S), h[c][4 * q + 3], u.w);
                }
            }
        }
    }

    // ---- B (and C) rows of a stage -> fp32 bcf[slot][t][B | C] ----
    constexpr int VE = 16 / int(sizeof(T));               // elements per 16-byte vector
    constexpr int NVEC = Ly::NBC * TS * kN / VE;
    auto convert_bc = [&](int i) {
        const unsigned char* staged = smem + static_cast<size_t>(i % NST) * Ly::STAGE + Ly::kB;
        float* dst = bcf + (i & 1) * TS * ROW;
        for (int idx = tid; idx < NVEC; idx += THREADS) {
            const int which = idx / (TS * kN / VE);
            const int r = idx % (TS * kN / VE);
            const int t = r / (kN / VE), n0 = (r % (kN / VE)) * VE;
            const unsigned char* src = staged + (which * TS * kN + t * kN + n0) * int(sizeof(T));
            float* o = dst + t * ROW + which * kN + n0;
            if constexpr (sizeof(T) == 2) {
                const uint4 u = *reinterpret_cast<const uint4*>(src);
                *reinterpret_cast<float4*>(o) =
                    make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                                __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
                *reinterpret_cast<float4*>(o + 4) =
                    make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u),
                                __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
            } else {
                *reinterpret_cast<float4*>(o) = *reinterpret_cast<const float4*>(src);
            }
        }
    };

    bool ok = mbar_wait_bounded(&full[0], 0u, kPolls);
    convert_bc(0);
    bool aborted = __syncthreads_or(!ok);

    // chunk-state pass: dt summed over the later stages (Rb) and, within a
    // stage, over the tokens after the current one (Rl): R = Rb + Rl
    float Rb[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) Rb[c] = 0.f;

    int i = 0;
    for (; i < nstages && !aborted; ++i) {
        const int buf = i % NST;
        unsigned char* stg = smem + static_cast<size_t>(buf) * Ly::STAGE;
        T* xt = reinterpret_cast<T*>(stg) + col;
        const T* dlt = reinterpret_cast<const T*>(stg + Ly::kDelta) + col;
        const T* zt = reinterpret_cast<const T*>(stg + Ly::kZ) + col;
        const float* bc = bcf + (i & 1) * TS * ROW;
        const int64_t t0 = t_begin + static_cast<int64_t>(stage_of(i)) * TS;
        ok = i == 0 || mbar_wait_bounded(&full[buf], static_cast<uint32_t>((i / NST) & 1), kPolls);
        const int lim = static_cast<int>(t_end - t0 < TS ? t_end - t0 : TS);   // valid tokens

        // the token's x, dt (0 past the sequence end: h unchanged) and dt x
        auto prep = [&](int tl, float (&xv)[CPL], float (&dt)[CPL], float (&dtx)[CPL]) {
            float dv[CPL];
            RW::ld(xt + tl * DT, xv);
            RW::ld(dlt + tl * DT, dv);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                float v = dv[c] + bias[c];
                if constexpr (SOFTPLUS) v = softplus(v);
                dt[c] = tl < lim ? v : 0.f;
                dtx[c] = dt[c] * xv[c];
            }
        };

        if constexpr (MODE == 1) {
            // software-pipelined by one token: the next token's x, dt, dt x
            // are formed before this token's update
            float xc[CPL], dc[CPL], dxc[CPL];
            prep(0, xc, dc, dxc);
            auto token = [&](int tl, bool st_path) {
                float xn[CPL], dn[CPL], dxn[CPL];
                prep((tl + 1) & (TS - 1), xn, dn, dxn);
                float Bv[kN], Cv[kN];
                lds_row<kN>(bc + tl * ROW, Bv);
                lds_row<kN>(bc + tl * ROW + kN, Cv);
                float y[CPL], zv[CPL];
                if constexpr (has_z) RW::ld(zt + tl * DT, zv);
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    float f[kN];
                    if (st_path)
                        powers16(dc[c] * a2[c], f);
                    else
                        exps16(dc[c], A2[c], f);
                    y[c] = fmaf(Dd[c], xc[c], step16(f, dxc[c], Bv, Cv, h[c]));
                    if constexpr (has_z) y[c] *= silu(zv[c]);
                }
                RW::st(xt + tl * DT, y);   // in place over x (already read)
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    xc[c] = xn[c]; dc[c] = dn[c]; dxc[c] = dxn[c];
                }
            };
            if (structured) {
#pragma unroll 4
                for (int tl = 0; tl < TS; ++tl) token(tl, true);
            } else {
#pragma unroll 4
                for (int tl = 0; tl < TS; ++tl) token(tl, false);
            }
        } else {
            // chunk state: tokens last to first; h accumulates sum_t w_t B_t
            float Rl[CPL], sb[CPL], base[CPL][kN];
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                Rl[c] = 0.f;
                sb[c] = a2[c] * Rb[c];
            }
            auto token = [&](int tl, bool st_path) {
                float xv[CPL], dt[CPL], dtx[CPL];
                prep(tl, xv, dt, dtx);
                float Bv[kN];
                lds_row<kN>(bc + tl * ROW, Bv);
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    float w[kN];
                    if (st_path) {
                        scaled_powers16(dtx[c], fmaf(a2[c], Rl[c], sb[c]), w);
                    } else {
#pragma unroll
                        for (int q = 0; q < kN; q += 2) {
                            const float2 arg =
                                __ffma2_rn(make_float2(A2[c][q], A2[c][q + 1]),
                                           make_float2(Rl[c], Rl[c]),
                                           make_float2(base[c][q], base[c][q + 1]));
                            const float2 u = __fmul2_rn(make_float2(dtx[c], dtx[c]),
                                                        make_float2(ex2(arg.x), ex2(arg.y)));
                            w[q] = u.x;
                            w[q + 1] = u.y;
                        }
                    }
                    accum16(w, Bv, h[c]);
                    Rl[c] += dt[c];
                }
            };
            if (structured) {
#pragma unroll 4
                for (int tl = TS - 1; tl >= 0; --tl) token(tl, true);
            } else {
#pragma unroll
                for (int c = 0; c < CPL; ++c)
#pragma unroll
                    for (int n = 0; n < kN; ++n) base[c][n] = A2[c][n] * Rb[c];
#pragma unroll 4
                for (int tl = TS - 1; tl >= 0; --tl) token(tl, false);
            }
#pragma unroll
            for (int c = 0; c < CPL; ++c) Rb[c] += Rl[c];
        }

        // B / C of the next stage (its bcf half was last read during stage i - 1)
        if (i + 1 < nstages) {
            ok = ok && mbar_wait_bounded(&full[(i + 1) % NST],
                                         static_cast<uint32_t>(((i + 1) / NST) & 1), kPolls);
            convert_bc(i + 1);
        }
        if constexpr (MODE == 1) fence_proxy_async_smem();   // y is read by the TMA store
        aborted = __syncthreads_or(!ok);                      // stage i consumed by every warp
        if (tid == 0 && !aborted) {
            if constexpr (MODE == 1) {
                tma_store_3d(&tm_out, static_cast<int>(dbase), static_cast<int>(t0),
                             static_cast<int>(b), stg);
                bulk_commit();
                // the buffer is refilled once the store has read it
                bulk_wait_read<0>();
            }
            if (i + NST < nstages) {
                fence_proxy_async_smem();
                issue(i + NST);
            }
        }
    }
    if (tid == 0) bulk_wait_all();
    if (aborted) {
        if (tid == 0) {
            // let the copies already in flight land before the CTA releases its smem
            for (int r = i; r < nstages && r < i + NST; ++r)
                mbar_wait_bounded(&full[r % NST], static_cast<uint32_t>((r / NST) & 1), kPolls);
            if (a.status) atomicExch(a.status, kStatusTimeout);
        }
        return;
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        if (!ch_ok[c]) continue;
        if (MODE == 0) {
            const int64_t idx = (b * (a.nchunks - 1) + k) * a.dim + dch[c];
            float4* Hp = reinterpret_cast<float4*>(a.ws_H + idx * kN);
#pragma unroll
            for (int q = 0; q < kN / 4; ++q)
                Hp[q] = make_float4(h[c][4 * q], h[c][4 * q + 1], h[c][4 * q + 2], h[c][4 * q + 3]);
            a.ws_S[idx] = Rb[c];
        } else if (a.final_state && k == a.nchunks - 1) {
            float4* fs = reinterpret_cast<float4*>(a.final_state + (b * a.dim + dch[c]) * kN);
#pragma unroll
            for (int q = 0; q < kN / 4; ++q)
                fs[q] = make_float4(h[c][4 * q], h[c][4 * q + 1], h[c][4 * q + 2], h[c][4 * q + 3]);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <typename T, int W, int CPL, int NST, int TS, int MODE, bool SP, bool GATE>
cudaError_t allow_smem16() {
    static std::mutex mu;
    static bool done[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(scan16_kernel<T, W, CPL, NST, TS, MODE, SP, GATE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay<T, W, CPL, NST, MODE, TS>::kBytes);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

template <typename T, int W, int CPL, int NST, int TS, bool SP, bool GATE>
cudaError_t launch16_flags(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    constexpr int DT = 32 * W * CPL;
    if (p.channels_per_cta != DT) return cudaErrorInvalidValue;
    CUtensorMap tx, tdt, tz, tB, tC;
    cudaError_t e;
    if ((e = make_tmap_cached<T>(&tx, a.x, a.batch, a.L, a.dim, DT, TS)) != cudaSuccess) return e;
    if ((e = make_tmap_cached<T>(&tdt, a.delta, a.batch, a.L, a.dim, DT, TS)) != cudaSuccess) return e;
    CUtensorMap tout;
    if ((e = make_tmap_cached<T>(&tout, a.out, a.batch, a.L, a.dim, DT, TS)) != cudaSuccess) return e;
    tz = tx;
    if (GATE && (e = make_tmap_cached<T>(&tz, a.z, a.batch, a.L, a.dim, DT, TS)) != cudaSuccess)
        return e;
    if ((e = make_tmap_cached<T>(&tB, a.B, a.batch, a.L, kN, kN, TS)) != cudaSuccess) return e;
    if ((e = make_tmap_cached<T>(&tC, a.C, a.batch, a.L, kN, kN, TS)) != cudaSuccess) return e;
    const int64_t per_chunk = p.tiles * a.batch;
    if (p.nchunks > 1) {
        if ((e = allow_smem16<T, W, CPL, NST, TS, 0, SP, false>()) != cudaSuccess) return e;
        scan16_kernel<T, W, CPL, NST, TS, 0, SP, false>
            <<<static_cast<unsigned>(per_chunk * (p.nchunks - 1)), 32 * W,
               Lay<T, W, CPL, NST, 0, TS>::kBytes, s>>>(tx, tdt, tz, tB, tC, tout, a);
    }
    if ((e = allow_smem16<T, W, CPL, NST, TS, 1, SP, GATE>()) != cudaSuccess) return e;
    scan16_kernel<T, W, CPL, NST, TS, 1, SP, GATE>
        <<<static_cast<unsigned>(per_chunk * p.nchunks), 32 * W,
           Lay<T, W, CPL, NST, 1, TS>::kBytes, s>>>(tx, tdt, tz, tB, tC, tout, a);
    return cudaGetLastError();
}

template <typename T, int W, int CPL, int NST, int TS>
cudaError_t launch16_cfg(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    const bool sp = a.softplus != 0, gate = a.z != nullptr;
    if (sp)
        return gate ? launch16_flags<T, W, CPL, NST, TS, true, true>(a, p, s)
                    : launch16_flags<T, W, CPL, NST, TS, true, false>(a, p, s);
    return gate ? launch16_flags<T, W, CPL, NST, TS, false, true>(a, p, s)
                : launch16_flags<T, W, CPL, NST, TS, false, false>(a, p, s);
}

}  // namespace

cudaError_t launch_scan16(const ScanArgs& a, const ScanPlan& p, int io, cudaStream_t s) {
    // bf16: 4 warps (128 channels), a 2-stage ring; fp32 I/O: the same tile,
    // whose larger stages still fit twice
    // 4 warps (128 channels) of one channel per lane, 32-token stages, a
    // 2-stage ring: the fastest of the measured layouts (two channels per
    // lane, and 16-token stages with 4 CTAs per SM, measured slower or equal)
    constexpr int CPL = 1, W = 4, TS = 32, NST = 2;
    return io == 1 ? launch16_cfg<__nv_bfloat16, W / CPL, CPL, NST, TS>(a, p, s)
                   : launch16_cfg<float, W / CPL, CPL, NST, TS>(a, p, s);
}

}  // namespace ssm
