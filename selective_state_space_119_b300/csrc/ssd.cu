// ssd.cu -- Mamba-2's SSD layer on the tensor cores (tcgen05), sm_103a.
//
// The layer ("Mamba: State Space Models Challenge Transformers", "Mamba-2:
// Improved Architecture": heads of d_head channels with a d_state-wide state
// each; "State Space Models and Mamba", "Mamba 2 and Hybrid Architectures":
// the SSM recast as a structured matrix multiplication). Per batch row b and
// head hd, with one scalar decay A[hd], one step dt[b,t,hd] per token shared
// by the head's P channels and B, C rows of the head's group g:
//   h_t = exp(dt_t A) h_{t-1} + dt_t x_t B_t^T     (h: [P, N])
//   y_t = h_t C_t + D x_t
// Because the decay is a scalar per head, a chunk of Q tokens is a few dense
// products. With s_t = A * (dt_0 + ... + dt_t) inside the chunk and h_in the
// state entering it:
//   G  = C B^T                                  [Q x Q]   (K = N)
//   M  = G o (exp(s_t - s_u) dt_u)_{u <= t}     masked decay, CUDA cores
//   Y  = (M + D I) X + diag(exp(s_t)) C h_in^T [Q x P]   (K = Q, then K = N)
//   S  = (w o X)^T B,  w_u = exp(s_Q - s_u) dt_u          (K = Q)
//   h_out = exp(s_Q) h_in + S
// This kernel runs one CTA per (batch row, head) over the chunks in order,
// the state in fp32 registers, with its warps specialised. Two producer warps
// (one thread each, on two schedulers) issue the tcgen05.mma products into
// tensor memory, each group as soon as its operands are ready: the first
// requests the TMA tiles (cp.async.bulk.tensor, 128-byte swizzle) and issues
// G = C B^T once the B and C tiles have landed and Y = M X once M is in tensor
// memory; the second Y2 = C h^T once the previous chunk's epilogue has written
// h and S^T once w o X is written. Sixteen compute warps form dt
// and its cumulative sum, w o X, M and the epilogue on the CUDA cores (a thread
// owns one row of every [Q x .] accumulator, the row of its warp's TMEM lane
// quarter, and a quarter of its columns: warps w, w + 4, w + 8, w + 12 split
// them) and hand each result over through an mbarrier; they synchronise among
// themselves with a named barrier, so the producer, whose issue of products
// holds its scheduler for about as long as they take, never stalls them (the
// cumulative sum also runs on warps of the other three schedulers). D x rides
// in M's diagonal, so the X tile is read by Y alone; M goes to tensor memory
// (tcgen05.st) and is the A operand of Y = M X from there, which leaves the
// shared memory for two buffers of B and C tiles: each chunk requests the next
// chunk's as soon as its own have landed. y is staged in a tile of its own
// for its TMA store (which has a chunk's time to read it). Operands that the CUDA cores produce (M, w o X and h) are
// split into a bf16 high part and a bf16 remainder, two products each, so that
// every product carries about 16 significant bits more than one bf16 rounding
// would.
//
// Sizes: Q = 128 tokens per chunk, P = 64 (d_head), N = 128 (d_state), bf16
// x, dt, B, C, y; fp32 A, D, dt_bias, h0, final state.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssm_tc.cuh"
#include "ssm_tma.cuh"
#include "ssm_tmap.h"

namespace ssm {
namespace {

constexpr int kQ = 128;     // tokens per chunk
constexpr int kP = 64;      // channels per head
constexpr int kNs = 128;    // state width
constexpr int kComputeWarps = 16;         // warps w, w + 4, w + 8, w + 12 share TMEM lane quarter w mod 4
constexpr int kCompute = 32 * kComputeWarps;
// and two producer warps: the first issues the TMA loads, G = C B^T, Y = M X and the
// y stores; the second Y2 = C h^T and S^T = B^T (w o X), so that two threads on two
// schedulers issue products at once
constexpr int kThreads = kCompute + 64;
constexpr int kGroups = kCompute / 128;   // column groups: a thread owns 64 / kGroups columns
constexpr int kGC = kP / kGroups;         // 16 columns of P per thread
constexpr uint32_t kPolls = 1u << 24;
constexpr uint32_t kStatusTimeout = 7;

// shared memory (byte offsets from a 1024-aligned base)
constexpr int kBlk = kQ * 128;                 // one [128 rows x 64] bf16 block: 16 KB
constexpr int oC = 0;                          // C tiles of two chunks: rows t, K = n (2 blocks each)
constexpr int oB = oC + 4 * kBlk;              // B tiles of two chunks: rows u, n (2 blocks each)
constexpr int oX = oB + 4 * kBlk;              // X tile: rows u, p (1 block)
constexpr int oWh = oX + kBlk;                 // w o X high: rows u, p
constexpr int oWl = oWh + kBlk;
constexpr int oHh = oWl + kBlk;                // h high: rows n, p
constexpr int oHl = oHh + kBlk;
constexpr int oYs = oHl + kBlk;                // y staged for its TMA store: rows t, p
constexpr int oDt = oYs + kBlk;                // dt [Q] f32
constexpr int oS2 = oDt + kQ * 4;              // s log2 e [Q] f32
constexpr int oWs = oS2 + kQ * 4;              // warp partial sums [4] f32
constexpr int oBar = oWs + 64;                 // 14 mbarriers (loads, products, hand-overs)
constexpr int oTm = oBar + 112;                // TMEM base address
constexpr int kSmemUsed = oTm + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;   // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// TMEM columns: G [0, 128), Y [128, 192), Y2 [192, 256), S^T [256, 320), and M as
// the A operand of Y = M X, bf16 pairs packed into 32-bit columns (row t in lane t):
// high parts [320, 384), remainders [384, 448)
constexpr uint32_t kColG = 0, kColY = 128, kColY2 = 192, kColS = 256, kColMh = 320,
                   kColMl = 384, kTmemCols = 512;

constexpr uint32_t kIdG = tc::idesc_bf16(128, kQ, false, false);   // C (K-major) B^T (K-major)
constexpr uint32_t kIdS = tc::idesc_bf16(128, kP, true, true);     // B^T (MN-major) wX (MN-major)
constexpr uint32_t kIdY = tc::idesc_bf16(128, kP, false, true);    // M (K-major) X (MN-major)

struct SsdArgs {
    const void* x;            // [batch, L, H, 64] bf16 (rows of w o X, read directly)
    const void* dt;           // [batch, L, H] bf16
    const float* A;           // [H]
    const float* D;           // [H] or NULL
    const float* dt_bias;     // [H] or NULL
    int softplus;
    const float* h0;          // [batch, H, P, N] or NULL
    float* final_state;       // [batch, H, P, N] or NULL
    int64_t batch, L, H, G;
    unsigned int* status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// Row r of a [128 x 64] swizzled block holds 64 values; write 8 of them (one
// 16-byte chunk, columns 8c .. 8c+7) as bf16 high parts and remainders: per
// pair, the high parts rounded to bf16, widened back, and the remainder
// v - high (exact in fp32) rounded to bf16.
__device__ __forceinline__ void put8_split(unsigned char* hi, unsigned char* lo, uint32_t r,
                                           uint32_t c, const float (&v)[8]) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        hw[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
        const float2 hf = make_float2(__uint_as_float(hw[i] << 16), __uint_as_float(hw[i] & 0xffff0000u));
        const float2 l = __ffma2_rn(hf, make_float2(-1.f, -1.f), make_float2(v[2 * i], v[2 * i + 1]));
        lw[i] = pack_bf16(l.x, l.y);
    }
    const uint32_t off = tc::sw128(r, 8 * c);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes, waited for in the
// same statement.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 16 consecutive 32-bit columns of this warp's 32 TMEM lanes (one lane
// per thread).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
// Wait until this thread's tcgen05.st have completed.
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Bring a tile of a 4-D tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void prefetch_l2_4d(const CUtensorMap* tm, int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
            reinterpret_cast<uint64_t>(tm)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                            int c3, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap* tm, int c0, int c1, int c2, int c3,
                                             const void* src) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            reinterpret_cast<uint64_t>(tm)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
        : "memory");
}

// (18 warps: two of the four schedulers hold five, so at most 96 registers
// per thread fit their share of the register file)
__global__ void __launch_bounds__(kThreads, 1)
ssd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
           const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_y,
           const SsdArgs a) {
    extern __shared__ unsigned char smem_raw[];
    // the swizzled tiles need 1024-byte aligned shared-memory addresses
    const uint32_t s_raw = smem_u32(smem_raw);
    unsigned char* sm = smem_raw + (((s_raw + 1023u) & ~1023u) - s_raw);
    float* sdt = reinterpret_cast<float*>(sm + oDt);
    float* ss2 = reinterpret_cast<float*>(sm + oS2);
    float* swarp = reinterpret_cast<float*>(sm + oWs);
    // Loads (one barrier per tile and buffer), product groups (committed by
    // the producer), and the compute warps' hand-overs to the producer (one
    // arrival per compute warp). Every barrier but B, C completes once per
    // chunk (rdy_E also once before the first); the B and C tiles of chunk c go
    // to buffer c & 1, whose barriers complete once every two chunks.
    uint64_t* bar_B = reinterpret_cast<uint64_t*>(sm + oBar);   // [2]
    uint64_t* bar_C = bar_B + 2;   // [2]
    uint64_t* bar_X = bar_B + 4;
    uint64_t* bar_G = bar_B + 5;   // G = C B^T
    uint64_t* bar_S = bar_B + 6;   // S^T = B^T (w o X)
    uint64_t* bar_Y = bar_B + 7;   // Y = M X and Y2 = C h^T, issued before it
    uint64_t* bar_D = bar_B + 8;   // the abort path: every product issued has completed
    uint64_t* rdy_W = bar_B + 9;   // w o X written
    uint64_t* rdy_M = bar_B + 10;  // M stored to tensor memory
    uint64_t* rdy_E = bar_B + 11;  // epilogue done: y staged, h written, accumulators read
    uint64_t* free_Y = bar_B + 12; // the y store has read the staging tile
    uint64_t* bar_D2 = bar_B + 13; // the second producer's abort path
    uint32_t* tm_slot = reinterpret_cast<uint32_t*>(sm + oTm);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp == kComputeWarps, producer2 = warp == kComputeWarps + 1;
    const int quarter = warp & 3, grp = warp >> 2;
    const int row = 32 * quarter + lane;   // this compute thread's TMEM lane and tile row
    const int64_t b = blockIdx.x / a.H, hd = blockIdx.x % a.H;
    const int64_t g = hd / (a.H / a.G);
    const int nchunks = static_cast<int>((a.L + kQ - 1) / kQ);
    const float A2 = __ldg(a.A + hd) * kLog2e;
    const float Dh = a.D ? __ldg(a.D + hd) : 0.f;
    const float bias = a.dt_bias ? __ldg(a.dt_bias + hd) : 0.f;
    const uint32_t sbase = smem_u32(sm);
    const int gg = static_cast<int>(g), bb = static_cast<int>(b), hh = static_cast<int>(hd);

    if (producer && lane == 0) {
        for (int i = 0; i < 9; ++i) mbar_init(bar_B + i, 1);
        for (int i = 9; i < 12; ++i) mbar_init(bar_B + i, kComputeWarps);
        mbar_init(free_Y, 1);
        mbar_init(bar_D2, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tm_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tm_slot;
    bool ok = true;

    if (producer) {
        // ---------------- the producer: TMA loads and tensor-core products ----------------
        if (lane == 0) {
            // the barrier phase of each load and product group in flight, -1 for
            // none (the abort path waits for them)
            int pend_B[2] = {-1, -1}, pend_C[2] = {-1, -1};
            int pend_X = -1, pend_G = -1, pend_Y = -1;
            bool stored = false;   // a y store is in flight
            auto load_B = [&](int c) {
                const int sb = c & 1;
                mbar_arrive_expect_tx(bar_B + sb, 2 * kBlk);
                tma_load_4d(sm + oB + sb * 2 * kBlk, &tm_B, 0, gg, c * kQ, bb, bar_B + sb);
                tma_load_4d(sm + oB + sb * 2 * kBlk + kBlk, &tm_B, 64, gg, c * kQ, bb, bar_B + sb);
                pend_B[sb] = (c >> 1) & 1;
            };
            auto load_C = [&](int c) {
                const int sb = c & 1;
                mbar_arrive_expect_tx(bar_C + sb, 2 * kBlk);
                tma_load_4d(sm + oC + sb * 2 * kBlk, &tm_C, 0, gg, c * kQ, bb, bar_C + sb);
                tma_load_4d(sm + oC + sb * 2 * kBlk + kBlk, &tm_C, 64, gg, c * kQ, bb, bar_C + sb);
                pend_C[sb] = (c >> 1) & 1;
            };
            auto load_X = [&](int c) {
                mbar_arrive_expect_tx(bar_X, kBlk);
                tma_load_4d(sm + oX, &tm_x, 0, hh, c * kQ, bb, bar_X);
                pend_X = c & 1;
            };
            // chunk c's B and C tiles: wait for them, send the next chunk's to
            // the other buffer (its last readers, the products of chunk c - 1,
            // have completed) and the tiles after those into L2, then issue
            // G = C B^T (8 steps of K = 16 over the two 64-wide n blocks). G
            // needs nothing of the previous chunk's epilogue, so it is issued as
            // soon as that chunk's products have completed.
            auto tiles_and_G = [&](int c) -> bool {
                const int sb = c & 1;
                const uint32_t pb = static_cast<uint32_t>((c >> 1) & 1);
                if (!mbar_wait_bounded(bar_B + sb, pb, kPolls) || !mbar_wait_bounded(bar_C + sb, pb, kPolls))
                    return false;
                pend_B[sb] = pend_C[sb] = -1;
                tc::fence_after_sync();
                if (c + 1 < nchunks) {
                    load_B(c + 1);
                    load_C(c + 1);
                }
                if (c + 2 < nchunks) {
                    prefetch_l2_4d(&tm_B, 0, gg, (c + 2) * kQ, bb);
                    prefetch_l2_4d(&tm_B, 64, gg, (c + 2) * kQ, bb);
                    prefetch_l2_4d(&tm_C, 0, gg, (c + 2) * kQ, bb);
                    prefetch_l2_4d(&tm_C, 64, gg, (c + 2) * kQ, bb);
                    prefetch_l2_4d(&tm_x, 0, hh, (c + 1) * kQ, bb);
                }
                const uint32_t oCc = oC + sb * 2 * kBlk, oBc = oB + sb * 2 * kBlk;
#pragma unroll
                for (int k = 0; k < kNs / 16; ++k) {
                    const uint32_t off = (k >> 2) * kBlk + (k & 3) * 32;
                    tc::mma_bf16(tmem + kColG, tc::desc_sw128(sbase + oCc + off, 16, 1024),
                                 tc::desc_sw128(sbase + oBc + off, 16, 1024), kIdG, k > 0);
                }
                tc::mma_commit(bar_G);
                pend_G = c & 1;
                return true;
            };
            load_B(0);
            load_C(0);
            load_X(0);
            ok = tiles_and_G(0);
            for (int c = 0; c < nchunks && ok; ++c) {
                const uint32_t ph = static_cast<uint32_t>(c & 1);
                // Y = M X once M is in tensor memory and the X tile has landed:
                // A = M from tensor memory (K = u, 8 columns of packed pairs per
                // step of 16), B = X MN-major. Every compute warp forms M after the
                // previous chunk's epilogue, so that epilogue has staged its y by
                // then: store it (its read of the staging tile is awaited once Y
                // is issued).
                ok = mbar_wait_bounded(rdy_M, ph, kPolls) && mbar_wait_bounded(bar_X, ph, kPolls) &&
                     (c == 0 || mbar_wait_bounded(rdy_E, ph, kPolls));
                if (!ok) break;
                pend_X = -1;
                tc::fence_after_sync();
                if (c > 0) {
                    tma_store_4d(&tm_y, 0, hh, (c - 1) * kQ, bb, sm + oYs);
                    bulk_commit();
                    stored = true;
                }
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const uint32_t am = tmem + (part ? kColMl : kColMh);
#pragma unroll
                    for (int k = 0; k < kQ / 16; ++k)
                        tc::mma_bf16_tmem_a(tmem + kColY, am + 8 * k,
                                            tc::desc_sw128(sbase + oX + k * 2048, 1024, 1024), kIdY,
                                            part > 0 || k > 0);
                }
                tc::mma_commit(bar_Y);
                pend_Y = static_cast<int>(ph);
                if (c > 0) {
                    // hand the staging tile back once the store has read it
                    bulk_wait_read<0>();
                    mbar_arrive(free_Y);
                }
                // this chunk's products have completed: G and Y (issued here, in
                // order) and Y2, S (the second producer's): the X tile, the B, C
                // buffer and G's columns are free for the next
                ok = mbar_wait_bounded(bar_Y, ph, kPolls) && mbar_wait_bounded(bar_S, ph, kPolls);
                if (!ok) break;
                pend_G = pend_Y = -1;
                if (c + 1 < nchunks) {
                    load_X(c + 1);
                    ok = tiles_and_G(c + 1);
                }
            }
            // the last chunk's y, once its epilogue has staged it
            if (ok && nchunks > 0) {
                ok = mbar_wait_bounded(rdy_E, static_cast<uint32_t>(nchunks & 1), kPolls);
                if (ok) {
                    tma_store_4d(&tm_y, 0, hh, (nchunks - 1) * kQ, bb, sm + oYs);
                    bulk_commit();
                    stored = true;
                }
            }
            if (stored) bulk_wait_all();
            if (!ok) {
                // let the loads and products in flight land before the CTA
                // releases its memory (each waited for once more, bounded)
                tc::mma_commit(bar_D);
                mbar_wait_bounded(bar_D, 0u, kPolls);
                for (int s2 = 0; s2 < 2; ++s2) {
                    if (pend_B[s2] >= 0)
                        mbar_wait_bounded(bar_B + s2, static_cast<uint32_t>(pend_B[s2]), kPolls);
                    if (pend_C[s2] >= 0)
                        mbar_wait_bounded(bar_C + s2, static_cast<uint32_t>(pend_C[s2]), kPolls);
                }
                if (pend_X >= 0) mbar_wait_bounded(bar_X, static_cast<uint32_t>(pend_X), kPolls);
                if (pend_G >= 0) mbar_wait_bounded(bar_G, static_cast<uint32_t>(pend_G), kPolls);
                if (pend_Y >= 0) mbar_wait_bounded(bar_Y, static_cast<uint32_t>(pend_Y), kPolls);
            }
        }
    } else if (producer2) {
        // ---------------- the second producer: Y2 = C h^T and S^T = B^T (w o X) ----------------
        if (lane == 0) {
            for (int c = 0; c < nchunks && ok; ++c) {
                const uint32_t ph = static_cast<uint32_t>(c & 1);
                const int sb = c & 1;
                const uint32_t oCc = oC + sb * 2 * kBlk, oBc = oB + sb * 2 * kBlk;
                const uint32_t pb = static_cast<uint32_t>((c >> 1) & 1);
                // the chunk's B and C tiles (the first producer reloads a buffer
                // only after this chunk's S has completed), and h of the previous
                // chunk's epilogue (or the prologue), which has also read the
                // previous Y2 and S: Y2 = C h^T, A = C (K-major, K = n), B = h
                // MN-major (rows n)
                ok = mbar_wait_bounded(bar_B + sb, pb, kPolls) && mbar_wait_bounded(bar_C + sb, pb, kPolls) &&
                     mbar_wait_bounded(rdy_E, ph, kPolls);
                if (!ok) break;
                tc::fence_after_sync();
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const uint32_t hb = sbase + (part ? oHl : oHh);
#pragma unroll
                    for (int k = 0; k < kNs / 16; ++k) {
                        const uint32_t offa = (k >> 2) * kBlk + (k & 3) * 32;
                        tc::mma_bf16(tmem + kColY2, tc::desc_sw128(sbase + oCc + offa, 16, 1024),
                                     tc::desc_sw128(hb + k * 2048, 1024, 1024), kIdY,
                                     part > 0 || k > 0);
                    }
                }
                // S^T = B^T (w o X) once w o X is written: A = the B tile read
                // MN-major (M = n over two 64-wide blocks 16 KB apart), B = w o X
                // MN-major; K = u in steps of 16 rows; the commit covers Y2 too
                ok = mbar_wait_bounded(rdy_W, ph, kPolls);
                if (!ok) break;
                tc::fence_after_sync();
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const uint32_t wx = sbase + (part ? oWl : oWh);
#pragma unroll
                    for (int k = 0; k < kQ / 16; ++k) {
                        const uint32_t off = k * 2048;
                        tc::mma_bf16(tmem + kColS, tc::desc_sw128(sbase + oBc + off, kBlk, 1024),
                                     tc::desc_sw128(wx + off, 1024, 1024), kIdS, part > 0 || k > 0);
                    }
                }
                tc::mma_commit(bar_S);
            }
            if (!ok) {
                // let this producer's products in flight complete before the CTA
                // releases its memory
                tc::mma_commit(bar_D2);
                mbar_wait_bounded(bar_D2, 0u, kPolls);
            }
        }
    } else {
        // ---------------- the compute warps: dt, w o X, M, the epilogue ----------------
        const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;   // this warp's TMEM lanes
        // the state: thread (row n, group g) holds h[p][n] for p = 16 g .. 16 g + 15
        // (fp32) and writes it as rows n of the MN-major operand [n x p] of C h^T
        float h[kGC];
        {
            const int n = row;
#pragma unroll
            for (int i = 0; i < kGC; ++i)
                h[i] = a.h0 ? a.h0[(((b * a.H + hd) * kP) + kGC * grp + i) * kNs + n] : 0.f;
#pragma unroll
            for (int k = 0; k < kGC / 8; ++k) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = h[8 * k + i];
                put8_split(sm + oHh, sm + oHl, n, (kGC / 8) * grp + k, v);
            }
        }
        // the first chunk's C h^T reads these rows through the async proxy
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(rdy_E);

        // The cumulative sum of dt is formed by warps 1, 2, 3 and 5 (token 32 k +
        // lane in the k-th of them): not by warp 0, which shares its scheduler
        // with the producer, whose issue of tensor-core products holds it.
        const int dtw = warp == 1 ? 0 : warp == 2 ? 1 : warp == 3 ? 2 : warp == 5 ? 3 : -1;
        const int dtok = 32 * dtw + lane;
        // this thread's token of chunk c: raw dt (bf16), 0 past the sequence end
        auto load_dt = [&](int c) {
            const int64_t t = int64_t(c) * kQ + dtok;
            return t < a.L ? IO<__nv_bfloat16>::ld(static_cast<const __nv_bfloat16*>(a.dt) +
                                                    (b * a.L + t) * a.H + hd)
                           : 0.f;
        };
        float dt_next = dtw >= 0 ? load_dt(0) : 0.f;
        // this thread's part of x row `row` of chunk c (its group's 16 channels),
        // for w o X, loaded a chunk ahead
        auto load_xrow = [&](int c, uint4 (&xr)[kGC / 8]) {
            const int64_t t = int64_t(c) * kQ + row;
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(a.x) + ((b * a.L + (t < a.L ? t : 0)) * a.H + hd) * kP +
                kGC * grp);
#pragma unroll
            for (int k = 0; k < kGC / 8; ++k)
                xr[k] = t < a.L ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
        };
        uint4 xrow[kGC / 8];
        load_xrow(0, xrow);

        // Phase A of chunk c: dt (0 past the sequence end; loaded a chunk ahead),
        // s = A * cumsum(dt), one token per thread of the four dt warps, then
        // w o X (high and remainder) for S^T = B^T (w o X), then the x row of the
        // chunk after. Every compute warp passes both named barriers whatever
        // its state (a warp leaving early would hold the others there); the
        // result is this warp's: false when a wait gave up.
        float s_end = 0.f;
        auto phase_a = [&](int c, bool okw) -> bool {
            float cs = 0.f;
            if (dtw >= 0) {
                float v = 0.f;
                if (c * kQ + dtok < a.L) {
                    v = dt_next + bias;
                    if (a.softplus) v = softplus(v);
                }
                dt_next = load_dt(c + 1);
                sdt[dtok] = v;
                cs = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float u = __shfl_up_sync(0xffffffffu, cs, o);
                    if (lane >= o) cs += u;
                }
                if (lane == 31) swarp[dtw] = cs;
            }
            named_bar_sync(1, kCompute);
            if (dtw >= 0) {
                for (int w = 0; w < dtw; ++w) cs += swarp[w];
                ss2[dtok] = cs * A2;   // s_t log2 e
            }
            // (the next write of swarp is a chunk later, after several barriers)
            if (named_bar_or(1, kCompute, !okw)) return false;   // the same for every warp
            s_end = ss2[kQ - 1];
            // row u = this thread's row, columns of its group, w_u = exp(s_end -
            // s_u) dt_u, once the previous chunk's S has read the last w o X
            if (c > 0 &&
                !__all_sync(0xffffffffu, mbar_wait_bounded(bar_S, static_cast<uint32_t>((c - 1) & 1), kPolls)))
                return false;
            {
                const int u = row;
                const float w = ex2(s_end - ss2[u]) * sdt[u];
                const float2 w2 = make_float2(w, w);
#pragma unroll
                for (int k = 0; k < kGC / 8; ++k) {
                    const uint32_t wd[4] = {xrow[k].x, xrow[k].y, xrow[k].z, xrow[k].w};
                    float v[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 p = __fmul2_rn(w2, make_float2(__uint_as_float(wd[i] << 16),
                                                                    __uint_as_float(wd[i] & 0xffff0000u)));
                        v[2 * i] = p.x;
                        v[2 * i + 1] = p.y;
                    }
                    put8_split(sm + oWh, sm + oWl, u, (kGC / 8) * grp + k, v);
                }
                load_xrow(c + 1, xrow);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(rdy_W);
            return true;
        };

        // The chunks are software-pipelined: chunk c + 1's phase A runs while
        // chunk c's Y = M X computes, between chunk c's M and its epilogue.
        ok = phase_a(0, ok);
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t ph = static_cast<uint32_t>(c & 1);
            // M = G o decay o dt + D on the diagonal (so that M X carries D x),
            // row t = this thread's row, high and remainder, while S computes,
            // stored to tensor memory as the A operand of Y = M X. Warp w forms
            // the 32-column block q = w / 4 of rows 32 (w mod 4) ..: blocks
            // q > w mod 4 lie above the diagonal (zero), q < w mod 4 below it (no
            // mask). (Chunk c - 1's Y, the last reader of M, completed before its
            // epilogue.)
            ok = __all_sync(0xffffffffu, ok && mbar_wait_bounded(bar_G, ph, kPolls));
            tc::fence_after_sync();
            // this thread's s_t and s_end of chunk c, for its epilogue after the
            // next chunk's phase A has overwritten dt and s
            const float st_c = ss2[row], s_end_c = s_end;
            if (ok) {
                const int t = row;
                const float st = st_c;
                const int q = grp;
                uint32_t hw[16], lw[16];
                if (q > quarter) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) hw[i] = lw[i] = 0u;
                } else {
                    float gv[32];
                    tc::tmem_ld32(tmem + lane_base + kColG + 32 * q, gv);
                    const float2 st2 = make_float2(st, st);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const float4* dtv = reinterpret_cast<const float4*>(sdt + 32 * q + 8 * cc);
                        const float4* ssv = reinterpret_cast<const float4*>(ss2 + 32 * q + 8 * cc);
                        const float4 d0 = dtv[0], d1 = dtv[1], s0 = ssv[0], s1 = ssv[1];
                        const float du[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                        const float su[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                        float v[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 ds = __ffma2_rn(make_float2(su[2 * i], su[2 * i + 1]),
                                                         make_float2(-1.f, -1.f), st2);   // s_t - s_u
                            const float2 e = make_float2(ex2(ds.x), ex2(ds.y));
                            const float2 m = __fmul2_rn(
                                __fmul2_rn(make_float2(gv[8 * cc + 2 * i], gv[8 * cc + 2 * i + 1]),
                                           make_float2(du[2 * i], du[2 * i + 1])),
                                e);
                            v[2 * i] = m.x;
                            v[2 * i + 1] = m.y;
                        }
                        if (q == quarter) {   // the diagonal block: zero above, D on the diagonal
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int u = 32 * q + 8 * cc + i;
                                v[i] = u < t ? v[i] : (u == t ? v[i] + Dh : 0.f);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t h2 = pack_bf16(v[2 * i], v[2 * i + 1]);
                            const float2 hf = make_float2(__uint_as_float(h2 << 16),
                                                          __uint_as_float(h2 & 0xffff0000u));
                            const float2 l = __ffma2_rn(hf, make_float2(-1.f, -1.f),
                                                        make_float2(v[2 * i], v[2 * i + 1]));
                            hw[4 * cc + i] = h2;
                            lw[4 * cc + i] = pack_bf16(l.x, l.y);
                        }
                    }
                }
                tmem_st16(tmem + lane_base + kColMh + 16 * q, hw);
                tmem_st16(tmem + lane_base + kColMl + 16 * q, lw);
                tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(rdy_M);
            }
            // the next chunk's phase A, once every compute warp has read this
            // chunk's dt and s
            if (c + 1 < nchunks) {
                named_bar_sync(1, kCompute);
                ok = phase_a(c + 1, ok);
            }
            // epilogue once S and Y (and Y2) have landed: y = Y + exp(s_t) Y2 (row
            // t, the group's 16 columns) into the staging tile; state: h <-
            // exp(s_end) h + S (row n, the group's 16 p)
            // (and once the previous chunk's y store has read the staging tile)
            ok = ok && mbar_wait_bounded(bar_S, ph, kPolls) && mbar_wait_bounded(bar_Y, ph, kPolls) &&
                 (c == 0 || mbar_wait_bounded(free_Y, ph ^ 1u, kPolls));
            ok = __all_sync(0xffffffffu, ok);
            tc::fence_after_sync();
            if (ok) {
                const int t = row;
                const float et = ex2(st_c);
                float yv[kGC], y2[kGC];
                tmem_ld16(tmem + lane_base + kColY + kGC * grp, yv);
                tmem_ld16(tmem + lane_base + kColY2 + kGC * grp, y2);
#pragma unroll
                for (int k = 0; k < kGC / 8; ++k) {
                    float o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = fmaf(et, y2[8 * k + i], yv[8 * k + i]);
                    *reinterpret_cast<uint4*>(sm + oYs + tc::sw128(t, 8 * ((kGC / 8) * grp + k))) =
                        make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]),
                                   pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
                }
                const float eend = ex2(s_end_c);
                float sv[kGC];
                tmem_ld16(tmem + lane_base + kColS + kGC * grp, sv);
#pragma unroll
                for (int i = 0; i < kGC; ++i) h[i] = fmaf(eend, h[i], sv[i]);
#pragma unroll
                for (int k = 0; k < kGC / 8; ++k) {
                    float v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = h[8 * k + i];
                    put8_split(sm + oHh, sm + oHl, row, (kGC / 8) * grp + k, v);
                }
                fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(rdy_E);
            }
            // every compute warp has passed this chunk before the next one starts
            if (named_bar_or(1, kCompute, !ok)) {
                ok = false;
                break;
            }
        }
        if (ok && a.final_state) {
            const int n = row;
#pragma unroll
            for (int i = 0; i < kGC; ++i)
                a.final_state[(((b * a.H + hd) * kP) + kGC * grp + i) * kNs + n] = h[i];
        }
    }
    // every warp, both roles: a wait that gave up anywhere sets the status word
    tc::fence_before_sync();
    const bool failed = __syncthreads_or(!ok);
    tc::fence_after_sync();
    if (failed && tid == 0 && a.status) atomicExch(a.status, kStatusTimeout);
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// 4-D [batch][L][rows][64k] bf16 tensor map with a 128-byte swizzle and a box
// of 64 x 1 x 128 x 1 (rows = heads or groups; inner = channels or states).
cudaError_t make_tmap4(CUtensorMap* tm, const void* base, int64_t batch, int64_t L, int64_t rows,
                       int64_t inner) {
    EncodeTiled fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t gdim[4] = {cuuint64_t(inner), cuuint64_t(rows), cuuint64_t(L), cuuint64_t(batch)};
    const cuuint64_t gstride[3] = {cuuint64_t(inner) * 2, cuuint64_t(rows * inner) * 2,
                                   cuuint64_t(L * rows * inner) * 2};
    const cuuint32_t box[4] = {64, 1, cuuint32_t(kQ), 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gdim,
                          gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_ssd(const SsdLaunch& l, cudaStream_t s) {
    static std::mutex mu;
    static bool done[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            e = cudaFuncSetAttribute(ssd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    CUtensorMap tx, tB, tC, ty;
    if ((e = make_tmap4(&tx, l.x, l.batch, l.L, l.H, kP)) != cudaSuccess) return e;
    if ((e = make_tmap4(&ty, l.y, l.batch, l.L, l.H, kP)) != cudaSuccess) return e;
    if ((e = make_tmap4(&tB, l.B, l.batch, l.L, l.G, kNs)) != cudaSuccess) return e;
    if ((e = make_tmap4(&tC, l.C, l.batch, l.L, l.G, kNs)) != cudaSuccess) return e;
    SsdArgs a{};
    a.x = l.x; a.dt = l.dt; a.A = l.A; a.D = l.D; a.dt_bias = l.dt_bias; a.softplus = l.softplus;
    a.h0 = l.h0; a.final_state = l.final_state;
    a.batch = l.batch; a.L = l.L; a.H = l.H; a.G = l.G; a.status = l.status;
    ssd_kernel<<<static_cast<unsigned>(l.batch * l.H), kThreads, kSmemBytes, s>>>(tx, tB, tC, ty, a);
    return cudaGetLastError();
}

}  // namespace ssm
