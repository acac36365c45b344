// ssm_tc.cuh -- inline-PTX wrappers for the 5th-generation tensor cores of
// sm_100-family GPUs (tcgen05: MMA issued by one thread, operands in shared
// memory, accumulators in tensor memory), compiled here for sm_103a.
//
// Operand tiles use the 128-byte-swizzled canonical layouts that TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B: rows of 128 bytes (64 bf16), the 16-byte
// chunks of row r XOR-ed with (r mod 8), eight rows (1024 bytes) per swizzle
// atom; every tile base is 1024-byte aligned.
//   K-major operand (rows = M or N, the 64 K values of a row contiguous): the
//     8-row groups are SBO = 1024 bytes apart; K beyond 64 is a second
//     [rows x 64] block; one MMA step of K = 16 advances the start by 32 bytes.
//   MN-major operand (rows = K, the 64 M or N values of a row contiguous): the
//     8-row K groups are SBO = 1024 bytes apart and the next 64 M (or N)
//     columns are a second block LBO bytes away; one MMA step of K = 16
//     advances the start by 16 rows = 2048 bytes.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {
namespace tc {

// Byte offset of element (r, c) (c < 64, bf16) inside a [rows x 64] 128-byte
// swizzled block whose base is 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) {
    const uint32_t chunk = (c >> 3) ^ (r & 7u);
    return r * 128u + chunk * 16u + (c & 7u) * 2u;
}

// Shared-memory matrix descriptor (64 bits): start address >> 4 in [0, 14),
// leading byte offset >> 4 in [16, 30), stride byte offset >> 4 in [32, 46),
// the fixed version 1 in [46, 48), base offset 0, swizzle mode in [61, 64)
// (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B and an fp32
// accumulator: D format (1 = f32) in [4, 6), A format (1 = bf16) in [7, 10),
// B format in [10, 13), A major (1 = MN) at 15, B major at 16, N >> 3 in
// [17, 23), M >> 4 in [24, 29).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
           (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// ---- tensor memory ----
// Allocate ncols columns (a power of two, 32 .. 512) for this CTA; one warp
// executes it; the address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], issued by one thread: A in tensor memory, row
// m of the M = 128 rows in lane m, K-major, each 32-bit column two consecutive
// bf16 values (the lower one in the low half); one step of K = 16 reads 8
// columns from a_tmem.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(static_cast<uint32_t>(accumulate))
        : "memory");
}

// Arrive on an mbarrier once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
        : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per
// thread), waited for in the same statement so that no use of the registers
// can be scheduled before the load has landed.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace tc
}  // namespace ssm
