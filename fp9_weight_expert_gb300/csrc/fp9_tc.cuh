// tcgen05 (5th-generation tensor core) helpers for sm_103a: TMEM
// allocation, shared-memory operand descriptors, the f16 MMA, its commit
// to an mbarrier, and TMEM loads. Operands are K-major tiles of 16-bit
// values in the 128-byte-swizzle layout: rows of 64 values (128 bytes),
// 8-row groups of 1024 bytes, the 16-byte chunk j of row r stored at chunk
// j ^ (r mod 8).
#pragma once

#include <cstdint>

namespace fp9 {

// Byte offset of value (row, k), k < 64, in a K-major 128-byte-swizzle
// tile (tile base 1024-byte aligned).
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t k) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((((k >> 3) ^ (row & 7u)) & 7u) << 4) + (k & 7u) * 2u;
}

// Shared-memory descriptor of a K-major 128-byte-swizzle operand starting
// at shared address `addr` (the start of a 16-value K slice inside a tile
// row; tile base 1024-byte aligned): 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);  // start address / 16
    d |= static_cast<uint64_t>(1u) << 16;                // leading offset: unused for swizzled K-major
    d |= static_cast<uint64_t>(1024u >> 4) << 32;        // stride between 8-row groups / 16
    d |= static_cast<uint64_t>(1u) << 46;                // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                // 128-byte swizzle
    return d;
}

// Shared-memory descriptor of an MN-major 128-byte-swizzle operand: atoms of
// 64 MN-contiguous 16-bit values x 8 K rows (1024 bytes); `lbo` = bytes
// between atoms along MN, `sbo` = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t tc_desc_sw128_mn(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of a kind::f16 MMA: f16 A and B, f32 accumulator,
// M x N, both operands K-major (bit 16 set by the caller makes B MN-major).
__host__ __device__ constexpr uint32_t tc_idesc_f16(uint32_t M, uint32_t N) {
    return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void tc_alloc(uint32_t slot_saddr, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Makes this thread's generic-proxy shared-memory writes visible to the
// tensor core (async proxy), which reads the operands.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A * B^T for one K = 16 slice (one thread issues).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_taddr, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_taddr),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// The mbarrier at `mbar_saddr` completes one arrival when every MMA this
// thread issued before has finished.
__device__ __forceinline__ void tc_commit(uint32_t mbar_saddr) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar_saddr)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (the warp's 32
// lanes start at bits 31..16 of taddr).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// The same for 16 columns.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// D[tmem] (+)= A * B^T for one K = 16 slice with A in tensor memory: rows
// of A in lanes 0..127 from column `a_taddr`, K packed two 16-bit values per
// 32-bit column (low half the even K), 8 columns per slice.
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc, uint32_t idesc,
                                                  bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_taddr),
        "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (the warp's 32
// lanes start at bits 31..16 of taddr); tc_wait_st waits for the stores.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// fp9 -> fp16 bits for 4 consecutive weights of one body word, in column
// order: (w0, w1) and (w2, w3) as two half2 words. The 9-bit code [sign |
// body] of each weight is built in a 16-bit half by one byte permute (the
// sign bytes come from spread_sign_nibble), then shifted left by 7: the
// fp16 bits of the same value [MEMOIR-FP9].
__device__ __forceinline__ void fp9_to_half4(uint32_t word, uint32_t spread_signs, uint32_t& h01, uint32_t& h23) {
    h01 = __byte_perm(word, spread_signs, 0x5140u) * 128u;
    h23 = __byte_perm(word, spread_signs, 0x7362u) * 128u;
}

}  // namespace fp9
