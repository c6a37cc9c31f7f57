// fp9 codec kernels: fp32 -> fp9 planes (pack) and fp9 planes -> fp32
// (decode), plus the status strings and device queries of the library.
//
// Format [MEMOIR-FP9] ("一鸭三吃" memoir, section "在只有 AVX2 的 N100 上，我先
// 做出了单核 MLP fp9"): 1 sign bit, 5 exponent bits with bias 15, 3
// mantissa bits; the 8-bit body eeeeemmm is kept per weight and the signs of
// 8 weights are packed into one byte of a separate plane (least significant
// bit = lowest column).
#include <cuda_runtime.h>

#include <cstdint>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9moe.h"

namespace fp9 {

// Round the fp32 value with bits `xbits` (sign ignored) to the nearest fp9
// body, ties to the even mantissa, in integer arithmetic on the fp32 fields.
// Sets `range` for Inf, NaN and magnitudes that round up to 2^16 or beyond.
__device__ __forceinline__ uint32_t encode_body(uint32_t xbits, bool& range) {
    const uint32_t mag = xbits & 0x7FFFFFFFu;
    if (mag >= 0x7F800000u) {  // Inf or NaN
        range = true;
        return mag == 0x7F800000u ? 0xF8u : 0xFCu;
    }
    const int32_t E = static_cast<int32_t>(mag >> 23);  // biased fp32 exponent
    const uint32_t M = mag & 0x7FFFFFu;
    if (E >= 113) {
        // |x| >= 2^-14: fp9 exponent field e = E - 127 + 15; keep the top 3
        // mantissa bits and round on the 20 dropped ones. A carry out of the
        // mantissa moves to the next binade by plain addition.
        uint32_t code = (static_cast<uint32_t>(E - 112) << 3) | (M >> 20);
        const uint32_t rem = M & 0xFFFFFu;
        if (rem > 0x80000u || (rem == 0x80000u && (code & 1u))) code += 1u;
        if (code >= 0xF8u) {
            range = true;
            return 0xF8u;
        }
        return code;
    }
    if (E == 0) return 0u;  // fp32 zero or denormal: below 2^-126, rounds to 0
    // |x| < 2^-14: subnormal fp9, counted in units of 2^-17. The fp32
    // significand (24 bits) times 2^(E-150) over 2^-17 is sig >> (133 - E).
    const uint32_t sig = M | 0x800000u;
    const int32_t sh = 133 - E;  // >= 21
    if (sh > 24) return 0u;      // below 2^-18 (half a unit): rounds to 0
    uint32_t q = sig >> sh;
    const uint32_t rem = sig & ((1u << sh) - 1u);
    const uint32_t half = 1u << (sh - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;  // q = 8 is the smallest normal
    return q;
}

// One thread per group of 8 consecutive weights of a row.
__global__ void __launch_bounds__(256) pack_kernel(const float4* __restrict__ src, int64_t ngroups,
                                                   uint2* __restrict__ body, uint8_t* __restrict__ sign,
                                                   int32_t* status) {
    bool range = false;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < ngroups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 a = __ldcs(src + 2 * g);
        const float4 b = __ldcs(src + 2 * g + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t lo = 0, hi = 0, s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t bits = __float_as_uint(v[i]);
            const uint32_t code = encode_body(bits, range);
            if (i < 4) lo |= code << (8 * i);
            else hi |= code << (8 * (i - 4));
            s |= (bits >> 31) << i;
        }
        body[g] = make_uint2(lo, hi);
        sign[g] = static_cast<uint8_t>(s);
    }
    if (range) record_status(status, FP9_ERR_RANGE);
}

__global__ void __launch_bounds__(256) decode_kernel(const uint2* __restrict__ body,
                                                     const uint8_t* __restrict__ sign, int64_t ngroups,
                                                     float4* __restrict__ dst) {
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < ngroups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint2 b = body[g];
        float w[8];
        decode8(b.x, b.y, sign[g], w);
        dst[2 * g] = make_float4(w[0], w[1], w[2], w[3]);
        dst[2 * g + 1] = make_float4(w[4], w[5], w[6], w[7]);
    }
}

int32_t device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return n;
}

int32_t device_max_smem_optin() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return -1;
    return n;
}

static unsigned elementwise_grid(int64_t ngroups) {
    const int64_t blocks = (ngroups + 255) / 256;
    int32_t sms = device_sm_count();
    if (sms <= 0) sms = 148;
    const int64_t cap = static_cast<int64_t>(sms) * 16;
    return static_cast<unsigned>(blocks < cap ? blocks : cap);
}

}  // namespace fp9

using namespace fp9;

extern "C" fp9_status fp9_pack(const float* src, int64_t rows, int64_t cols, uint8_t* body,
                               uint8_t* sign, int32_t* d_status, void* stream) {
    FP9_CHECK_ARG(rows >= 0 && cols >= 0, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(cols % 8 == 0, FP9_ERR_SHAPE);
    if (rows == 0 || cols == 0) return FP9_OK;
    FP9_CHECK_ARG(src != nullptr && body != nullptr && sign != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(src, 16) && aligned(body, 8), FP9_ERR_ALIGN);
    const int64_t ngroups = rows * (cols / 8);
    pack_kernel<<<elementwise_grid(ngroups), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(src), ngroups, reinterpret_cast<uint2*>(body), sign, d_status);
    FP9_CUDA_TRY(cudaGetLastError());
    return FP9_OK;
}

extern "C" fp9_status fp9_decode(const uint8_t* body, const uint8_t* sign, int64_t rows, int64_t cols,
                                 float* dst, void* stream) {
    FP9_CHECK_ARG(rows >= 0 && cols >= 0, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(cols % 8 == 0, FP9_ERR_SHAPE);
    if (rows == 0 || cols == 0) return FP9_OK;
    FP9_CHECK_ARG(body != nullptr && sign != nullptr && dst != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(dst, 16) && aligned(body, 8), FP9_ERR_ALIGN);
    const int64_t ngroups = rows * (cols / 8);
    decode_kernel<<<elementwise_grid(ngroups), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint2*>(body), sign, ngroups, reinterpret_cast<float4*>(dst));
    FP9_CUDA_TRY(cudaGetLastError());
    return FP9_OK;
}

extern "C" const char* fp9_status_str(int32_t status) {
    switch (status) {
        case FP9_OK: return "FP9_OK";
        case FP9_ERR_INVALID_ARG: return "FP9_ERR_INVALID_ARG: null pointer or bad count";
        case FP9_ERR_SHAPE: return "FP9_ERR_SHAPE: a dimension breaks a layout rule";
        case FP9_ERR_ALIGN: return "FP9_ERR_ALIGN: pointer not aligned as required";
        case FP9_ERR_WORKSPACE: return "FP9_ERR_WORKSPACE: workspace too small";
        case FP9_ERR_RANGE: return "FP9_ERR_RANGE: value not representable in fp9";
        case FP9_ERR_CUDA: return "FP9_ERR_CUDA: a CUDA runtime call failed";
        case FP9_ERR_TIMEOUT: return "FP9_ERR_TIMEOUT: a bounded device wait ran out";
        default: return "FP9 unknown status";
    }
}
