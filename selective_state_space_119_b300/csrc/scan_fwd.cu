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
// L-chunks. The recurrence is linear in h, so the sequence is cut into chunks
// joined by composing affine maps h -> P h + H, (P1, H1) then (P2, H2) =
// (P2 P1, P2 H1 + H2): the associative operator behind the pages' parallel
// scan ("State Space Models -- Mamba, S4, and Beyond", "Hardware-Efficient
// Scan (for Training)"; "State-space models (Mamba, S4)", "Training vs
// Inference Modes"). For a chunk P = prod_t exp(dt_t A) = exp(A sum_t dt_t), so
// only the sum of dt is kept. Three stream-ordered phases (no CTA waits for
// another CTA):
//   1. chunk state : every chunk but the last runs from h = 0 and stores its
//                    end state H and S = sum(dt)            (MODE 0)
//   2. carry       : per (b, d, n), h_in(k+1) = exp(A S_k) h_in(k) + H_k
//   3. output      : every chunk runs from its entering state, writes y; the
//                    last chunk writes final_state           (MODE 1)
//
// One CTA = one (chunk, batch row, tile of DT channels). Tokens stream through
// shared memory in stages of TS: TMA (cp.async.bulk.tensor) loads the
// [TS x DT] tiles of x, delta and z into an NST-deep mbarrier pipeline, and y
// leaves through a double-buffered [TS x DT] tile and a TMA store. Each stage
// runs three passes:
//   prologue (one thread per channel pair): dt = softplus(delta + bias) and
//            dt * x into shared memory, B_t / C_t rows converted to fp32;
//   states   (each thread: CPT channels x SPL = N / NS states, in registers):
//            h <- exp2(dt * A log2e) h + (dt x) B in packed f32x2 arithmetic,
//            and the thread's partial C . h per channel;
//   epilogue (one thread per channel pair): sum the NS partials, + D x,
//            * silu(z), round to the I/O type into the output tile.
// Sharing a channel's N states among NS / CPT threads multiplies the
// parallelism without adding exponentials; giving a thread CPT channels
// amortises its per-token loads of B_t, C_t and (dt, dt x) over more states.
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

constexpr uint32_t kMaxPolls = 1u << 24;  // bound on one mbarrier wait (seconds)
constexpr uint32_t kStatusTimeout = 7;    // -SSM_ERR_TIMEOUT

// Tile configuration: DT channels per CTA; each thread owns CPT consecutive
// channels x SPL = N / NS consecutive states, so a channel is shared by NS / CPT
// threads.
template <int DT_, int NS_, int CPT_>
struct TileCfg {
    static constexpr int DT = DT_, NS = NS_, CPT = CPT_;
};

template <typename T, int N, typename TC>
struct Cfg {
    static constexpr int DT = TC::DT;
    static constexpr int NS = TC::NS < N ? TC::NS : N;   // small N: fewer state lanes
    static constexpr int CPT = TC::CPT;
    static constexpr int SPL = N / NS;                    // states per thread
    static constexpr int TS = kScanStageTokens;           // tokens per stage
    static constexpr int NST = 4;                         // pipeline depth
    static constexpr int GROUPS = DT / CPT;               // channel groups per tile
    static constexpr int THREADS = GROUPS * NS;
    static constexpr int TILE = TS * DT;                  // elements per tile
    static_assert(N % NS == 0 && DT % CPT == 0 && DT % 2 == 0, "tile shape");
    static_assert(THREADS % (DT / 2) == 0, "prologue rows");
};

constexpr int align128(int v) { return (v + 127) & ~127; }

template <typename T, int N, typename TC, int MODE>
struct Smem {
    using C = Cfg<T, N, TC>;
    static constexpr int NT = MODE == 1 ? 3 : 2;  // tensors staged per token stage
    static constexpr int YS_ROW = C::DT + 8;      // padded rows: NS partial rows hit distinct banks
    static constexpr int kIn = 0;
    static constexpr int kDtp = align128(kIn + C::NST * NT * C::TILE * int(sizeof(T)));
    static constexpr int kYs = align128(kDtp + C::TILE * 8);
    static constexpr int kOut = align128(kYs + (MODE == 1 ? C::TS * C::NS * YS_ROW * 4 : 0));
    static constexpr int kBC = align128(kOut + (MODE == 1 ? 2 * C::TILE * int(sizeof(T)) : 0));
    static constexpr int kBar = align128(kBC + C::TS * 2 * N * 4);
    static constexpr int kFlag = kBar + C::NST * 8;
    static constexpr int kBytes = align128(kFlag + 16);
};

template <typename T>
__device__ __forceinline__ float io_ld(const T* p) { return IO<T>::ld(p); }

template <int K>
__device__ __forceinline__ void lds_vec(const float* p, float* v) {
    if constexpr (K % 4 == 0) {
#pragma unroll
        for (int i = 0; i < K; i += 4) {
            const float4 u = *reinterpret_cast<const float4*>(p + i);
            v[i] = u.x; v[i + 1] = u.y; v[i + 2] = u.z; v[i + 3] = u.w;
        }
    } else if constexpr (K == 2) {
        const float2 u = *reinterpret_cast<const float2*>(p);
        v[0] = u.x; v[1] = u.y;
    } else {
#pragma unroll
        for (int i = 0; i < K; ++i) v[i] = p[i];
    }
}

template <int K>
__device__ __forceinline__ void sts_vec(float* p, const float* v) {
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

template <typename T, int N, typename TC, int MODE>
__global__ void __launch_bounds__(Cfg<T, N, TC>::THREADS)
scan_tma_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
                const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_out,
                const ScanArgs a) {
    using Cf = Cfg<T, N, TC>;
    using Sm = Smem<T, N, TC, MODE>;
    constexpr int DT = Cf::DT, NS = Cf::NS, CPT = Cf::CPT, SPL = Cf::SPL, TS = Cf::TS;
    constexpr int NST = Cf::NST, THREADS = Cf::THREADS, TILE = Cf::TILE, NT = Sm::NT;
    constexpr int YS_ROW = Sm::YS_ROW;
    constexpr int PAIRS = DT / 2;               // prologue / epilogue: one channel pair each
    constexpr int ROW_STEP = THREADS / PAIRS;   // rows per sweep

    extern __shared__ __align__(128) unsigned char smem[];
    T* in = reinterpret_cast<T*>(smem + Sm::kIn);              // [NST][NT][TS][DT]
    float* dtp = reinterpret_cast<float*>(smem + Sm::kDtp);    // [TS][DT][2]: dt, dt*x
    float* ys = reinterpret_cast<float*>(smem + Sm::kYs);      // [TS][NS][DT+8] partial C.h
    T* outs = reinterpret_cast<T*>(smem + Sm::kOut);           // [2][TS][DT]
    float* bc = reinterpret_cast<float*>(smem + Sm::kBC);      // [TS][NS][B x SPL, C x SPL]
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Sm::kBar);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Sm::kFlag);

    const int tid = threadIdx.x;
    const int64_t lin = blockIdx.x;  // chunk-major: ((k * batch) + b) * tiles + tile
    const int64_t tile = lin % a.tiles;
    const int64_t b = (lin / a.tiles) % a.batch;
    const int64_t k = lin / (a.tiles * a.batch);
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(a.L, t_begin + a.chunk_len);
    const int nstages = static_cast<int>((t_end - t_begin + TS - 1) / TS);
    const int64_t dbase = tile * DT;
    const bool has_z = MODE == 1 && a.z != nullptr;
    const uint32_t stage_tx = static_cast<uint32_t>((has_z ? 3 : 2) * TILE * sizeof(T));

    const T* __restrict__ Bg = static_cast<const T*>(a.B);
    const T* __restrict__ Cg = static_cast<const T*>(a.C);

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        *abort_flag = 0;
    }
    __syncthreads();

    auto issue = [&](int s) {
        const int buf = s % NST;
        T* dst = in + static_cast<size_t>(buf) * NT * TILE;
        const int t = static_cast<int>(t_begin + static_cast<int64_t>(s) * TS);
        mbar_arrive_expect_tx(&bar[buf], stage_tx);
        tma_load_3d(dst, &tm_x, static_cast<int>(dbase), t, static_cast<int>(b), &bar[buf]);
        tma_load_3d(dst + TILE, &tm_dt, static_cast<int>(dbase), t, static_cast<int>(b), &bar[buf]);
        if (has_z)
            tma_load_3d(dst + 2 * TILE, &tm_z, static_cast<int>(dbase), t, static_cast<int>(b),
                        &bar[buf]);
    };
    if (tid == 0)
        for (int s = 0; s < NST && s < nstages; ++s) issue(s);

    // ---- per-thread constants ------------------------------------------------
    // state pass: channels [c0, c0 + CPT) of the tile, states [j*SPL, j*SPL + SPL)
    const int g = tid / NS, j = tid % NS;
    const int c0 = g * CPT;
    float A2[CPT][SPL], h[CPT][SPL];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const bool ok = dbase + c0 + c < a.dim;
        const int64_t d = ok ? dbase + c0 + c : 0;
#pragma unroll
        for (int q = 0; q < SPL; ++q) {
            A2[c][q] = __ldg(a.A + d * N + j * SPL + q) * kLog2e;
            h[c][q] = 0.f;
        }
        if (MODE == 1 && k > 0 && ok) {
            const float* hin = a.ws_H + ((b * (a.nchunks - 1) + (k - 1)) * a.dim + d) * N + j * SPL;
#pragma unroll
            for (int q = 0; q < SPL; ++q) h[c][q] = hin[q];
        }
    }
    float dt_sum[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) dt_sum[c] = 0.f;
    // prologue / epilogue: channel pair pc of the tile, rows prow0 + i * ROW_STEP
    const int pc = tid % PAIRS, prow0 = tid / PAIRS;
    const int64_t pd0 = dbase + 2 * pc;
    const bool p_valid = pd0 < a.dim;  // dim is even, so pd0 + 1 < dim as well
    float bias0 = 0.f, bias1 = 0.f, D0 = 0.f, D1 = 0.f;
    if (p_valid) {
        if (a.delta_bias) { bias0 = __ldg(a.delta_bias + pd0); bias1 = __ldg(a.delta_bias + pd0 + 1); }
        if (a.D) { D0 = __ldg(a.D + pd0); D1 = __ldg(a.D + pd0 + 1); }
    }

    // ---- B / C rows: prefetched into registers one stage ahead ----------------
    constexpr int NBC = (MODE == 1 ? 2 : 1) * TS * N;
    constexpr int VPT = (NBC + THREADS - 1) / THREADS;
    float bcr[VPT];
    auto load_bc = [&](int s) {
        const int64_t ts = t_begin + static_cast<int64_t>(s) * TS;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = tid + v * THREADS;
            bcr[v] = 0.f;
            if (idx < NBC) {
                const int which = idx / (TS * N), r = idx % (TS * N);
                const int t = r / N, n = r % N;
                if (ts + t < t_end) {
                    const int64_t off = (b * a.L + ts + t) * N + n;
                    bcr[v] = io_ld<T>((which ? Cg : Bg) + off);
                }
            }
        }
    };
    auto store_bc = [&]() {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int idx = tid + v * THREADS;
            if (idx < NBC) {
                const int which = idx / (TS * N), r = idx % (TS * N);
                const int t = r / N, n = r % N;
                bc[t * 2 * N + (n / SPL) * 2 * SPL + which * SPL + (n % SPL)] = bcr[v];
            }
        }
    };
    load_bc(0);

    bool aborted = false;
    int s = 0;
    for (; s < nstages; ++s) {
        const int buf = s % NST;
        const uint32_t parity = static_cast<uint32_t>((s / NST) & 1);
        const T* xt = in + static_cast<size_t>(buf) * NT * TILE;
        const T* dlt = xt + TILE;
        const T* zt = xt + 2 * TILE;
        const int64_t t0 = t_begin + static_cast<int64_t>(s) * TS;
        const int nt = static_cast<int>(t_end - t0 < TS ? t_end - t0 : TS);

        if (tid == 0 && !mbar_wait_bounded(&bar[buf], parity, kMaxPolls)) *abort_flag = 1;
        store_bc();
        __syncthreads();  // (1) tiles landed, B/C staged; previous stage fully consumed
        if (*abort_flag) { aborted = true; break; }
        mbar_wait_bounded(&bar[buf], parity, 1);  // acquire the TMA writes for this thread
        if (s + 1 < nstages) load_bc(s + 1);

        // prologue: dt and dt * x
        for (int t = prow0; t < nt; t += ROW_STEP) {
            float xv[2], dv[2];
            Vec<T, 2>::lds(xt + t * DT + 2 * pc, xv);
            Vec<T, 2>::lds(dlt + t * DT + 2 * pc, dv);
            float d0 = dv[0] + bias0, d1 = dv[1] + bias1;
            if (a.softplus) { d0 = softplus(d0); d1 = softplus(d1); }
            *reinterpret_cast<float4*>(dtp + (t * DT + 2 * pc) * 2) =
                make_float4(d0, d0 * xv[0], d1, d1 * xv[1]);
        }
        __syncthreads();  // (2) dt, dt*x ready

        // states: h <- exp2(dt A log2e) h + (dt x) B, in packed pairs of states
#pragma unroll 2
        for (int t = 0; t < nt; ++t) {
            float dd[2 * CPT];
            lds_vec<2 * CPT>(dtp + (t * DT + c0) * 2, dd);
            float bcv[2 * SPL];
            lds_vec<2 * SPL>(bc + t * 2 * N + j * 2 * SPL, bcv);
            float yp[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                const float dt = dd[2 * c], dtx = dd[2 * c + 1];
                if (MODE == 0) dt_sum[c] += dt;
                if constexpr (SPL % 2 == 0) {
                    float2 acc = make_float2(0.f, 0.f);
                    const float2 dt2 = make_float2(dt, dt), dtx2 = make_float2(dtx, dtx);
#pragma unroll
                    for (int q = 0; q < SPL; q += 2) {
                        const float2 arg = __fmul2_rn(dt2, make_float2(A2[c][q], A2[c][q + 1]));
                        const float2 dA = make_float2(ex2(arg.x), ex2(arg.y));
                        const float2 bx = __fmul2_rn(dtx2, make_float2(bcv[q], bcv[q + 1]));
                        const float2 hn = __ffma2_rn(dA, make_float2(h[c][q], h[c][q + 1]), bx);
                        h[c][q] = hn.x;
                        h[c][q + 1] = hn.y;
                        if (MODE == 1)
                            acc = __ffma2_rn(make_float2(bcv[SPL + q], bcv[SPL + q + 1]), hn, acc);
                    }
                    yp[c] = acc.x + acc.y;
                } else {
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < SPL; ++q) {
                        const float dA = ex2(dt * A2[c][q]);
                        h[c][q] = fmaf(dA, h[c][q], dtx * bcv[q]);
                        if (MODE == 1) acc = fmaf(bcv[SPL + q], h[c][q], acc);
                    }
                    yp[c] = acc;
                }
            }
            if (MODE == 1) sts_vec<CPT>(ys + (t * NS + j) * YS_ROW + c0, yp);
        }
        __syncthreads();  // (3) partial sums ready; dtp and bc free

        if (MODE == 1) {
            T* ot = outs + (s & 1) * TILE;
            for (int t = prow0; t < nt; t += ROW_STEP) {
                float y0 = 0.f, y1 = 0.f;
#pragma unroll
                for (int jj = 0; jj < NS; ++jj) {
                    const float2 u =
                        *reinterpret_cast<const float2*>(ys + (t * NS + jj) * YS_ROW + 2 * pc);
                    y0 += u.x;
                    y1 += u.y;
                }
                float xv[2];
                Vec<T, 2>::lds(xt + t * DT + 2 * pc, xv);
                float yv[2] = {fmaf(D0, xv[0], y0), fmaf(D1, xv[1], y1)};
                if (has_z) {
                    float zv[2];
                    Vec<T, 2>::lds(zt + t * DT + 2 * pc, zv);
                    yv[0] *= silu(zv[0]);
                    yv[1] *= silu(zv[1]);
                }
                Vec<T, 2>::sts(ot + t * DT + 2 * pc, yv);
            }
            fence_proxy_async_smem();
            __syncthreads();  // (4) output tile complete; input tiles of `buf` consumed
            if (tid == 0) {
                tma_store_3d(&tm_out, static_cast<int>(dbase), static_cast<int>(t0),
                             static_cast<int>(b), ot);
                bulk_commit();
                bulk_wait_read<1>();  // the store from the other output buffer is done
            }
        }
        if (tid == 0 && s + NST < nstages) {
            fence_proxy_async_smem();
            issue(s + NST);
        }
    }

    if (tid == 0) {
        bulk_wait_all();
        if (aborted) {
            // let the copies already in flight land before the CTA releases its smem
            for (int r = s; r < nstages && r < s + NST; ++r)
                mbar_wait_bounded(&bar[r % NST], static_cast<uint32_t>((r / NST) & 1), kMaxPolls);
            if (a.status) atomicExch(a.status, kStatusTimeout);
        }
    }
    if (aborted) return;

#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        if (dbase + c0 + c >= a.dim) continue;
        const int64_t d = dbase + c0 + c;
        if (MODE == 0) {
            const int64_t base = (b * (a.nchunks - 1) + k) * a.dim + d;
#pragma unroll
            for (int q = 0; q < SPL; ++q) a.ws_H[base * N + j * SPL + q] = h[c][q];
            if (j == 0) a.ws_S[base] = dt_sum[c];
        } else if (a.final_state && k == a.nchunks - 1) {
            float* fs = a.final_state + (b * a.dim + d) * N + j * SPL;
#pragma unroll
            for (int q = 0; q < SPL; ++q) fs[q] = h[c][q];
        }
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

// [batch][L][dim] tensor, box of `box_channels` channels x TS tokens x 1 batch row.
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
    e = cudaFuncSetAttribute(scan_tma_kernel<T, N, TC, MODE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<T, N, TC, MODE>::kBytes);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

template <typename T, int N, typename TC>
cudaError_t launch_cfg(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    using Cf = Cfg<T, N, TC>;
    CUtensorMap tx, tdt, tz, tout;
    cudaError_t e;
    if ((e = make_tmap<T>(&tx, a.x, a.batch, a.L, a.dim, TC::DT)) != cudaSuccess) return e;
    if ((e = make_tmap<T>(&tdt, a.delta, a.batch, a.L, a.dim, TC::DT)) != cudaSuccess) return e;
    if ((e = make_tmap<T>(&tz, a.z ? a.z : a.x, a.batch, a.L, a.dim, TC::DT)) != cudaSuccess)
        return e;
    if ((e = make_tmap<T>(&tout, a.out, a.batch, a.L, a.dim, TC::DT)) != cudaSuccess) return e;
    const int64_t per_chunk = p.tiles * a.batch;
    if (p.nchunks > 1) {
        constexpr int sm0 = Smem<T, N, TC, 0>::kBytes;
        if ((e = allow_smem<T, N, TC, 0>()) != cudaSuccess) return e;
        scan_tma_kernel<T, N, TC, 0>
            <<<static_cast<unsigned>(per_chunk * (p.nchunks - 1)), Cf::THREADS, sm0, s>>>(
                tx, tdt, tz, tout, a);
        const int64_t n = a.batch * a.dim * N;
        scan_carry_kernel<N><<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(a);
    }
    constexpr int sm1 = Smem<T, N, TC, 1>::kBytes;
    if ((e = allow_smem<T, N, TC, 1>()) != cudaSuccess) return e;
    scan_tma_kernel<T, N, TC, 1>
        <<<static_cast<unsigned>(per_chunk * p.nchunks), Cf::THREADS, sm1, s>>>(tx, tdt, tz, tout,
                                                                                 a);
    return cudaGetLastError();
}

// The tile configurations by id (see ssm_internal.h).
using Tile0 = TileCfg<64, 4, 4>;  // 1 thread per channel
using Tile1 = TileCfg<64, 4, 2>;  // 2 threads per channel
using Tile2 = TileCfg<32, 8, 2>;  // 4 threads per channel
using Tile3 = TileCfg<16, 8, 1>;  // 8 threads per channel

template <typename T, int N>
cudaError_t launch_typed(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    if constexpr (N == 16) {
        switch (p.tile_cfg) {
            case 0: return launch_cfg<T, N, Tile0>(a, p, s);
            case 1: return launch_cfg<T, N, Tile1>(a, p, s);
            case 2: return launch_cfg<T, N, Tile2>(a, p, s);
            case 3: return launch_cfg<T, N, Tile3>(a, p, s);
            default: return cudaErrorInvalidValue;
        }
    } else {
        return launch_cfg<T, N, Tile1>(a, p, s);
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
