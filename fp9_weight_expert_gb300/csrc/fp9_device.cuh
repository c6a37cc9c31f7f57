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

// fp9 -> fp16 bits for pairs of weights. For 4 weights in one body word,
// their 4 sign bits are first spread to the low bit of 4 bytes (one
// multiply by a constant with bits at 0, 7, 14, 21: the shifted copies of a
// 4-bit value never overlap, so no carry crosses them). One byte permute
// then builds, in each 16-bit half, [sign byte (0 or 1)][body byte]: the
// 9-bit fp9 code s eeeee mmm. Shifting it left by 7 (a multiply by 128,
// which keeps the two halves apart because bits 9..15 of each half are 0)
// gives the fp16 bits s eeeee mmm 0000000 of the same value.
__device__ __forceinline__ uint32_t spread_sign_nibble(uint32_t nibble) {
    return (nibble * 0x00204081u) & 0x01010101u;
}

// Decode 16 consecutive weights into 8 pairs in "pair order":
// p[2k] = (w[4k], w[4k+2]) and p[2k+1] = (w[4k+1], w[4k+3]), the order in
// which each half2 is built (callers keep x and y in the same order).
// `body` holds the 16 body bytes (byte i = column i), `s16` the 16 sign
// bits (bit i = column i).
__device__ __forceinline__ void decode16_pairs(const uint4 body, uint32_t s16, float2 p[8]) {
    const uint32_t words[4] = {body.x, body.y, body.z, body.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t e = spread_sign_nibble((s16 >> (4 * k)) & 0xFu);
        p[2 * k] = half2_bits_to_float2(__byte_perm(words[k], e, 0x6240u) * 128u);      // cols 4k, 4k+2
        p[2 * k + 1] = half2_bits_to_float2(__byte_perm(words[k], e, 0x7351u) * 128u);  // cols 4k+1, 4k+3
    }
}

// Decode 8 consecutive weights (two body words, one sign byte) in column order.
__device__ __forceinline__ void decode8(uint32_t w0, uint32_t w1, uint32_t s8, float w[8]) {
    const uint32_t words[2] = {w0, w1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t e = spread_sign_nibble((s8 >> (4 * k)) & 0xFu);
        const float2 fa = half2_bits_to_float2(__byte_perm(words[k], e, 0x6240u) * 128u);
        const float2 fb = half2_bits_to_float2(__byte_perm(words[k], e, 0x7351u) * 128u);
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

// try_wait that may suspend the thread in hardware for up to `hint_ns`
// (it returns as soon as the phase completes), so waiting warps do not spin
// on the issue slots.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Wait for the phase of `parity` to complete, giving up after `limit_ns`
// nanoseconds or as soon as another thread of the CTA has raised *abort.
// Returns false when it gave up; then the caller records a timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, 2000u)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte global load with an L2 cache-eviction policy.
__device__ __forceinline__ float4 ld_global_hint(const float4* p, uint64_t policy) {
    float4 v;
    asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 prefetch of `bytes` at `src` with an L2 cache-eviction policy (a
// hint: nothing is written and nothing waits for it). src 16-byte aligned,
// bytes % 16 == 0.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(policy)
                 : "memory");
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

// ------------------------------------------------------------ stack glue ---
//
// RMSNorm of the residual stream of a stack, x = v / sqrt(mean(v^2) + eps)
// with v = h + y (unit gain), in one fixed order: 256 threads, thread t
// adds the squares of the float4s t, t + 256, ... of the row (x, y, z, w of
// each by fmaf), each warp sums its threads (warp_sum), and the 8 warp sums
// are added in warp order.
constexpr int kNormThreads = 256;

// The same scale, 1 / sqrt(mean(v^2) + eps), from a row's sum of squares
// held as n <= FP9_MAX_HIDDEN / 16 partial sums (ss[0 .. n), column
// order), added by one warp in a fixed order: lane l adds parts l, l + 32,
// ... in turn (all its loads issued first), then the xor butterfly of
// warp_sum (each step adds the same two values on both lanes). Every lane
// of every warp that calls it gets the same bits.
__device__ __forceinline__ float rms_scale_parts(const float* ss, int n, int64_t H, float eps, int lane) {
    constexpr int kPer = (FP9_MAX_HIDDEN / 16 + 31) / 32;
    float v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int i = lane + 32 * k;
        v[k] = i < n ? __ldcg(ss + i) : 0.0f;
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) s += v[k];
    s = warp_sum(s);
    return 1.0f / sqrtf(s / static_cast<float>(H) + eps);
}

// v = h + y of float4 c, read through L2 (both were written by earlier kernels).
__device__ __forceinline__ float4 residual4(const float4* h4, const float4* y4, int64_t c) {
    float4 v = __ldcg(h4 + c);
    if (y4 != nullptr) {
        const float4 d = __ldcg(y4 + c);
        v.x += d.x;
        v.y += d.y;
        v.z += d.z;
        v.w += d.w;
    }
    return v;
}

__device__ __forceinline__ float sumsq4(float4 v, float ss) {
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    return fmaf(v.w, v.w, ss);
}

// 1 / sqrt(mean + eps) from the 8 warp sums.
__device__ __forceinline__ float rms_scale(const float* warp_sums, int64_t H, float eps) {
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += warp_sums[w];
    return 1.0f / sqrtf(tot / static_cast<float>(H) + eps);
}

}  // namespace fp9
