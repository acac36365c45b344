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
// The recurrence is linear in h, so the sequence can be cut into L-chunks and
// the chunks joined by composing affine maps h -> P h + H with
// (P1, H1) then (P2, H2) = (P2 P1, P2 H1 + H2) -- the associative operator
// behind the pages' parallel scan ("State Space Models -- Mamba, S4, and
// Beyond", "Hardware-Efficient Scan (for Training)"; "State-space models
// (Mamba, S4)", "Training vs Inference Modes"). For a chunk, P = prod_t
// exp(dt_t A) = exp(A * sum_t dt_t), so only the sum of dt is stored.
//
// Three phases, all stream-ordered (no CTA waits on another CTA):
//   1. chunk_state : every chunk but the last runs its recurrence from h = 0
//                    and stores its end state H and sum(dt) S.
//   2. carry       : per (b, d, n), a short sequential pass over the chunks
//                    turns (S, H) into the state entering each chunk.
//   3. output      : every chunk runs from its entering state and writes y;
//                    the last chunk writes final_state.
// With one chunk only phase 3 runs.
//
// Layout: a CTA owns kScanThreads * kScanCPT consecutive channels of one batch
// row and one L-chunk. Each thread keeps kScanCPT channels x N states in
// registers; B_t / C_t rows (shared by every channel) are staged through
// shared memory, kStage tokens at a time, and read as broadcasts; x, delta,
// z and out are accessed as kScanCPT-wide vectors, coalesced along d.
#include <cuda_bf16.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kStage = 64;  // tokens of B / C staged in shared memory at once

enum { kModeChunkState = 0, kModeOutput = 1 };

template <typename T, int N, int CPT, int MODE>
__global__ void __launch_bounds__(kScanThreads)
scan_chunk_kernel(const ScanArgs a) {
    __shared__ float sB[kStage * N];
    __shared__ float sC[MODE == kModeOutput ? kStage * N : 1];

    const int64_t L = a.L, dim = a.dim;
    // Linear CTA index, chunk-major: ((k * batch) + b) * tiles + tile.
    const int64_t lin = blockIdx.x;
    const int64_t tile = lin % a.tiles;
    const int64_t b = (lin / a.tiles) % a.batch;
    const int64_t k = lin / (a.tiles * a.batch);
    const int64_t t_begin = k * a.chunk_len;
    const int64_t t_end = min(L, t_begin + a.chunk_len);
    const int64_t d0 = (tile * kScanThreads + threadIdx.x) * CPT;
    const bool active = d0 < dim;

    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ delta = static_cast<const T*>(a.delta);
    const T* __restrict__ Bg = static_cast<const T*>(a.B);
    const T* __restrict__ Cg = static_cast<const T*>(a.C);
    const T* __restrict__ z = static_cast<const T*>(a.z);
    T* __restrict__ out = static_cast<T*>(a.out);

    float A2[CPT][N], h[CPT][N], Dv[CPT], bias[CPT], S[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int64_t d = active ? d0 + c : 0;
#pragma unroll
        for (int n = 0; n < N; ++n) A2[c][n] = __ldg(a.A + d * N + n) * kLog2e;
        Dv[c] = a.D ? __ldg(a.D + d) : 0.f;
        bias[c] = a.delta_bias ? __ldg(a.delta_bias + d) : 0.f;
        S[c] = 0.f;
#pragma unroll
        for (int n = 0; n < N; ++n) h[c][n] = 0.f;
    }
    if (MODE == kModeOutput && k > 0 && active) {
        // State entering chunk k, left in ws_H slot k-1 by the carry phase.
        const float* hin = a.ws_H + ((b * (a.nchunks - 1) + (k - 1)) * dim + d0) * N;
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int n = 0; n < N; ++n) h[c][n] = hin[c * N + n];
    }

    for (int64_t ts = t_begin; ts < t_end; ts += kStage) {
        const int nt = static_cast<int>(t_end - ts < kStage ? t_end - ts : kStage);
        __syncthreads();  // the previous stage has been consumed
        const int64_t row = (b * L + ts) * N;
        for (int i = threadIdx.x; i < nt * N; i += kScanThreads) {
            sB[i] = IO<T>::ld(Bg + row + i);
            if (MODE == kModeOutput) sC[i] = IO<T>::ld(Cg + row + i);
        }
        __syncthreads();
        if (!active) continue;

#pragma unroll 2
        for (int tt = 0; tt < nt; ++tt) {
            const int64_t e = (b * L + ts + tt) * dim + d0;
            float xv[CPT], dt[CPT], dtx[CPT], y[CPT];
            Vec<T, CPT>::ld(x + e, xv);
            Vec<T, CPT>::ld(delta + e, dt);
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                dt[c] += bias[c];
                if (a.softplus) dt[c] = softplus(dt[c]);
                dtx[c] = dt[c] * xv[c];
                S[c] += dt[c];
                y[c] = 0.f;
            }
#pragma unroll
            for (int n = 0; n < N; ++n) {
                const float Bn = sB[tt * N + n];
                const float Cn = MODE == kModeOutput ? sC[tt * N + n] : 0.f;
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    const float dA = ex2(dt[c] * A2[c][n]);
                    h[c][n] = fmaf(dA, h[c][n], dtx[c] * Bn);
                    if (MODE == kModeOutput) y[c] = fmaf(Cn, h[c][n], y[c]);
                }
            }
            if (MODE == kModeOutput) {
#pragma unroll
                for (int c = 0; c < CPT; ++c) y[c] = fmaf(Dv[c], xv[c], y[c]);
                if (z) {
                    float zv[CPT];
                    Vec<T, CPT>::ld(z + e, zv);
#pragma unroll
                    for (int c = 0; c < CPT; ++c) y[c] *= silu(zv[c]);
                }
                Vec<T, CPT>::st(out + e, y);
            }
        }
    }

    if (!active) return;
    if (MODE == kModeChunkState) {
        const int64_t base = (b * (a.nchunks - 1) + k) * dim + d0;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
#pragma unroll
            for (int n = 0; n < N; ++n) a.ws_H[(base + c) * N + n] = h[c][n];
            a.ws_S[base + c] = S[c];
        }
    } else if (a.final_state && k == a.nchunks - 1) {
        float* fs = a.final_state + (b * dim + d0) * N;
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int n = 0; n < N; ++n) fs[c * N + n] = h[c][n];
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

template <typename T, int N>
cudaError_t launch_typed(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
    const int64_t per_chunk = p.tiles * a.batch;
    if (p.nchunks > 1) {
        scan_chunk_kernel<T, N, kScanCPT, kModeChunkState>
            <<<static_cast<unsigned>(per_chunk * (p.nchunks - 1)), kScanThreads, 0, s>>>(a);
        const int64_t n = a.batch * a.dim * N;
        scan_carry_kernel<N><<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(a);
    }
    scan_chunk_kernel<T, N, kScanCPT, kModeOutput>
        <<<static_cast<unsigned>(per_chunk * p.nchunks), kScanThreads, 0, s>>>(a);
    return cudaGetLastError();
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
