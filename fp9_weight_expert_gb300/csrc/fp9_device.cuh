// Device helpers shared by the fp9 kernels (sm_103a).
//
// fp9 decode [MEMOIR-FP9] ("一鸭三吃" memoir, section "在只有 AVX2 的 N100 上，
// 我先做出了单核 MLP fp9"): the body byte eeeeemmm shifted left by 7, with
// the sign at bit 15, is an IEEE fp16 of the same value; widening that fp16
// to fp32 needs no exponent fix-up and handles +-0 and subnormals.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "fp9moe.h"

namespace fp9 {

// ---------------------------------------------------------------- status ---

__device__ __forceinline__ void record_status(int32_t* status, int32_t code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- decode ---

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t bits) {
    __half2 h = *reinterpret_cast<__half2*>(&bits);
    return __half22float2(h);
}

// Decode 16 consecutive weights: `body` holds their body bytes (byte i of
// the 16 = column i), `s16` their 16 sign bits (bit i = column i).
//
// Each 32-bit body word k holds columns 4k..4k+3. Two fp16 values are built
// per instruction pair as a half2: (4k, 4k+2) and (4k+1, 4k+3). The body
// bytes are moved to the high byte of each 16-bit half and shifted right by
// one (= body << 7 inside the half). The sign bits are moved to bits 15 and
// 31 by one multiply of the sign byte by a two-bit constant: the two
// shifted copies of the byte do not overlap, so no carry crosses them.
__device__ __forceinline__ void decode16(const uint4 body, uint32_t s16, float w[16]) {
    const uint32_t words[4] = {body.x, body.y, body.z, body.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t s8 = (k < 2) ? (s16 & 0xFFu) : (s16 >> 8);
        const int i = (k & 1) * 4;  // column of word k's first weight inside its sign byte
        uint32_t a = __byte_perm(words[k], 0u, 0x2404u) >> 1;     // cols 4k, 4k+2
        uint32_t b = (words[k] & 0xFF00FF00u) >> 1;               // cols 4k+1, 4k+3
        const uint32_t ma = s8 * ((1u << (15 - i)) + (1u << (29 - i)));
        const uint32_t mb = s8 * ((1u << (14 - i)) + (1u << (28 - i)));
        a |= ma & 0x80008000u;
        b |= mb & 0x80008000u;
        const float2 fa = half2_bits_to_float2(a);
        const float2 fb = half2_bits_to_float2(b);
        w[4 * k + 0] = fa.x;
        w[4 * k + 2] = fa.y;
        w[4 * k + 1] = fb.x;
        w[4 * k + 3] = fb.y;
    }
}

// Decode 8 consecutive weights from two body words and one sign byte.
__device__ __forceinline__ void decode8(uint32_t w0, uint32_t w1, uint32_t s8, float w[8]) {
    const uint32_t words[2] = {w0, w1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = k * 4;
        uint32_t a = __byte_perm(words[k], 0u, 0x2404u) >> 1;
        uint32_t b = (words[k] & 0xFF00FF00u) >> 1;
        a |= (s8 * ((1u << (15 - i)) + (1u << (29 - i)))) & 0x80008000u;
        b |= (s8 * ((1u << (14 - i)) + (1u << (28 - i)))) & 0x80008000u;
        const float2 fa = half2_bits_to_float2(a);
        const float2 fb = half2_bits_to_float2(b);
        w[4 * k + 0] = fa.x;
        w[4 * k + 2] = fa.y;
        w[4 * k + 1] = fb.x;
        w[4 * k + 3] = fb.y;
    }
}

// ------------------------------------------------------ mbarrier and bulk ---

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `parity` to complete, giving up after `limit_ns`
// nanoseconds or as soon as another thread of the CTA has raised *abort.
// Returns false when it gave up; then the caller records a timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 15u) == 0u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy global -> shared (no tensor map), completing `bytes` of
// transaction count on `bar`. dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// ---------------------------------------------------- programmatic launch ---

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- reductions ---

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
    return v;
}

}  // namespace fp9
