// fp9 codec kernels: fp32 -> fp9 planes (pack) and fp9 planes -> fp32
// (decode), plus the status strings and device queries of the library.
//
// Format [MEMOIR-FP9] ("一鸭三吃" memoir, section "在只有 AVX2 的 N100 上，我先
// 做出了单核 MLP fp9"): 1 sign bit, 5 exponent bits with bias 15, 3
// mantissa bits; the 8-bit body eeeeemmm is kept per weight and the signs of
// 8 weights are packed into one byte of a separate plane (least significant
// bit = lowest column).
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9moe.h"

namespace fp9 {

// Round the fp32 value with bits `xbits` (sign ignored) to the nearest fp9
// body, ties to the even mantissa, in integer arithmetic on the fp32 fields.
// Sets `range` for Inf, NaN and magnitudes that round up to 2^16 or beyond.
// `tie` is for a value known more exactly than its fp32 bits: the sign of
// (exact magnitude - this magnitude). It matters only when this magnitude
// is exactly halfway between two fp9 values: then it picks the side (0:
// the even mantissa). The exact value is within half an fp32 unit of this
// one, and every fp9 midpoint is an fp32 value, so no other case moves.
__device__ __forceinline__ uint32_t encode_body(uint32_t xbits, int tie, bool& range) {
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
        if (rem > 0x80000u || (rem == 0x80000u && (tie > 0 || (tie == 0 && (code & 1u))))) code += 1u;
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
    if (rem > half || (rem == half && (tie > 0 || (tie == 0 && (q & 1u))))) q += 1u;  // q = 8: smallest normal
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
            const uint32_t code = encode_body(bits, 0, range);
            if (i < 4) lo |= code << (8 * i);
            else hi |= code << (8 * (i - 4));
            s |= (bits >> 31) << i;
        }
        body[g] = make_uint2(lo, hi);
        sign[g] = static_cast<uint8_t>(s);
    }
    if (range) record_status(status, FP9_ERR_RANGE);
}

// fp9 body of the exact product x * s, where x and s are fp32 values (x has
// at most 4 significant bits: an fp8 e4m3 value). p = x * s is rounded to
// fp32, and its error fma(x, s, -p) is exact, so p plus that error is the
// exact product; it is rounded once to fp9. The error can only matter when
// p lies exactly on an fp9 midpoint (every midpoint is an fp32 value and
// the exact product is within half an fp32 unit of p), so it is computed
// only then. Fast path: 2^-14 <= |p| < 63488, a normal fp9 that cannot
// overflow; everything else goes through encode_body.
__device__ __forceinline__ uint32_t encode_product(float x, float s, uint32_t& sign_bit, bool& range) {
    const float p = x * s;
    const uint32_t bits = __float_as_uint(p), mag = bits & 0x7FFFFFFFu;
    sign_bit = bits >> 31;
    if (mag - 0x38800000u < 0x47780000u - 0x38800000u) {
        uint32_t code = (mag >> 20) - (112u << 3);
        const uint32_t rem = mag & 0xFFFFFu;
        if (rem == 0x80000u) {
            const float d = fmaf(x, s, -p);
            const float dm = sign_bit ? -d : d;  // exact magnitude - |p|
            code += dm > 0.0f ? 1u : (dm < 0.0f ? 0u : (code & 1u));
        } else {
            code += rem > 0x80000u ? 1u : 0u;
        }
        return code;
    }
    const float d = fmaf(x, s, -p);
    const float dm = sign_bit ? -d : d;
    return encode_body(bits, (dm > 0.0f) - (dm < 0.0f), range);
}

// fp8 checkpoint -> fp9 by 128x128 scale blocks. The pages say the
// DeepSeek-V3 release is fp8 ("一鸭三吃" memoir, section "真正埋下伏笔的是内存；
// R1 之后，问题第一次被改写") with 128x128 block scales (section "先用 Qwen3 练级，
// 再让 Qwen3.5 充当高压试炼场"). Every weight of a block is its e4m3 value times
// the block's scale s, rounded once to fp9 (encode_product), so the body
// depends only on the code's magnitude: per block the CTA encodes the 128
// magnitudes |e4m3(c)| * |s| into a table indexed by the code's 7
// magnitude bits (128 bytes), then each weight is one shared-memory byte
// read. Rounding to nearest is symmetric, so the product's sign is the
// code's sign xor the scale's sign; a NaN product (a NaN code, 0 * Inf, a
// NaN scale) is the canonical NaN of the multiply, sign 0.
//
// Matrices with a ragged block (rows or cols not a multiple of 128) take
// fp8_to_fp9_kernel: grid x = block column, y = block row (a CTA walks the
// block rows blockIdx.y, + gridDim.y, ... so any row count fits the 65535
// limit), 256 threads, a thread converting kUnits units of G consecutive
// weights of a row (G = 16, or 8 when cols % 16 != 0). Matrices of whole
// blocks take fp8_to_fp9_full_kernel (below).
template <int G>
struct Fp8Block {
    static constexpr int kUnits = 128 * 128 / G / 256;  // units of G weights per thread
    uint32_t in[kUnits][G / 4];
    int64_t g[kUnits];  // unit index in the matrix (-1: none)
    float scale;
};

template <int G>
__device__ __forceinline__ void fp8_block_load(const uint8_t* __restrict__ w8, const float* __restrict__ scale,
                                               int64_t rows, int64_t cols, int64_t nbx, int64_t by,
                                               Fp8Block<G>& B) {
    const int64_t bx = blockIdx.x;
    const int64_t r0 = by * 128, c0 = bx * 128;
    B.scale = __ldg(scale + by * nbx + bx);
    const int64_t bh = rows - r0 < 128 ? rows - r0 : 128, bw = cols - c0 < 128 ? cols - c0 : 128;
    if (bh == 128 && bw == 128) {
        // a full block: 128 / G units per row, so unit threadIdx.x + 256 j
        // sits 256 G / 128 = 2 G rows below unit threadIdx.x (2 cols units)
        constexpr int kShift = G == 16 ? 3 : 4;
        const int64_t g0 =
            ((r0 + (threadIdx.x >> kShift)) * cols + c0) / G + (threadIdx.x & ((1 << kShift) - 1));
#pragma unroll
        for (int j = 0; j < Fp8Block<G>::kUnits; ++j) B.g[j] = g0 + 2 * j * cols;
    } else {
        const int per_row = static_cast<int>(bw / G);
        const int units = static_cast<int>(bh) * per_row;
#pragma unroll
        for (int j = 0; j < Fp8Block<G>::kUnits; ++j) {
            const int u = threadIdx.x + 256 * j;
            const int rr = u / per_row;
            B.g[j] = u < units ? ((r0 + rr) * cols + c0) / G + (u - rr * per_row) : -1;
        }
    }
#pragma unroll
    for (int j = 0; j < Fp8Block<G>::kUnits; ++j) {
        if (B.g[j] < 0) continue;
        if constexpr (G == 16) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4*>(w8) + B.g[j]);
            B.in[j][0] = q.x, B.in[j][1] = q.y, B.in[j][2] = q.z, B.in[j][3] = q.w;
        } else {
            const uint2 q = __ldcs(reinterpret_cast<const uint2*>(w8) + B.g[j]);
            B.in[j][0] = q.x, B.in[j][1] = q.y;
        }
    }
}

// The sign bits (bit 7 of each byte) of two code words v0, v1 as 8 bits:
// byte k of v0 at bit 24 + k, byte k of v1 at bit 28 + k. v0's signs are
// moved down to bits 8k + 3, beside v1's at 8k + 7; the multiply by
// 2^0 + 2^7 + 2^14 + 2^21 adds the copy shifted by 7 (3 - k), which takes
// 8k + 3 to 24 + k and 8k + 7 to 28 + k. All 32 shifted copies of the 8
// bits fall on distinct positions, so no carry disturbs them.
__device__ __forceinline__ uint32_t gather_signs8(uint32_t v0, uint32_t v1) {
    return ((v1 & 0x80808080u) | ((v0 >> 4) & 0x08080808u)) * 0x00204081u;
}

// Threads 0..127 write the table of a block of scale `scale`: entry c holds
// the fp9 body of |e4m3(c)| * |scale|, c < 128 (a code's magnitude bits).
// 128 bytes are one word per shared-memory bank, so a warp's lookups never
// conflict: lanes reading one magnitude (of either sign) read one word.
// Returns whether this thread's entry is an Inf or NaN body for a finite
// code: the NaN code's entry (c = 0x7F) is the NaN body whatever the scale,
// so NaN codes are looked for in the codes themselves (fp8_nan_bits).
__device__ __forceinline__ bool fp8_table_entry(uint8_t* tab, float scale) {
    bool range = false;
    if (threadIdx.x < 128) {
        // |e4m3(c)| for c < 128: the hardware conversion of the code pair
        // (c, c) to fp16, then fp32
        const __half2_raw hr =
            __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(threadIdx.x * 0x101u), __NV_E4M3);
        const float x = __low2float(*reinterpret_cast<const __half2*>(&hr));
        uint32_t sb;
        const uint8_t e = static_cast<uint8_t>(encode_product(x, fabsf(scale), sb, range));
        tab[threadIdx.x] = e;
    }
    return range && threadIdx.x != 0x7Fu;
}

// For m = the magnitude bits of four e4m3 codes (a word & 0x7F7F7F7F):
// bit 7 of a byte is set when that code is a NaN code (magnitude bits all
// ones): a byte's 7 bits plus one reach its bit 7 only then, and never
// carry into the next byte.
__device__ __forceinline__ uint32_t fp8_nan_bits(uint32_t m) { return (m + 0x01010101u) & 0x80808080u; }

// One unit of G codes (words in[0 .. G/4)) through the block's table:
// writes unit g of the body and sign planes. `sflip` is all-ones over the
// unit's sign bits when the scale is negative; `special` says a finite
// code's product overflows in this block. When that holds or the unit has
// a NaN code, each body is checked, and `hit` is set if one is Inf or NaN.
template <int G>
__device__ __forceinline__ void fp8_unit_convert(const uint32_t (&in)[G / 4], const uint8_t* tab, uint32_t sflip,
                                                 bool special, int64_t g, uint8_t* __restrict__ body,
                                                 uint8_t* __restrict__ sign, bool& hit) {
    uint32_t out[G / 4];
    uint32_t nan = 0;
#pragma unroll
    for (int w = 0; w < G / 4; ++w) {
        const uint32_t m = in[w] & 0x7F7F7F7Fu;
        nan |= fp8_nan_bits(m);
        const uint32_t b0 = tab[m & 0xFFu], b1 = tab[__byte_perm(m, 0u, 0x4441u)];
        const uint32_t b2 = tab[__byte_perm(m, 0u, 0x4442u)], b3 = tab[m >> 24];
        // the bytes do not overlap, so the adds are ors; written as
        // multiply-adds they can share the integer multiply pipe
        out[w] = (b3 * 256u + b2) * 65536u + (b1 * 256u + b0);
    }
    uint32_t sb;
    if constexpr (G == 16)
        sb = __byte_perm(gather_signs8(in[0], in[1]), gather_signs8(in[2], in[3]), 0x0073u);
    else
        sb = gather_signs8(in[0], in[1]) >> 24;
    sb ^= sflip;
    if (special || nan != 0) {
        // bytes 0xF8..0xFF (Inf 0xF8, NaN 0xFC): flag them; NaN is unsigned
#pragma unroll
        for (int w = 0; w < G / 4; ++w) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t bk = (out[w] >> (8 * k)) & 0xFFu;
                if ((bk & 0xF8u) == 0xF8u) hit = true;
                if (bk == 0xFCu) sb &= ~(1u << (4 * w + k));
            }
        }
    }
    if constexpr (G == 16) {
        __stcs(reinterpret_cast<uint4*>(body) + g, make_uint4(out[0], out[1], out[2], out[3]));
        reinterpret_cast<uint16_t*>(sign)[g] = static_cast<uint16_t>(sb);
    } else {
        __stcs(reinterpret_cast<uint2*>(body) + g, make_uint2(out[0], out[1]));
        sign[g] = static_cast<uint8_t>(sb);
    }
}

// Encodes the block's table (threads 0..127) and converts the block's units
// of this thread; returns whether any weight landed on an Inf or NaN body.
template <int G>
__device__ __forceinline__ bool fp8_block_convert(const Fp8Block<G>& B, uint8_t* tab, uint8_t* __restrict__ body,
                                                  uint8_t* __restrict__ sign) {
    __syncthreads();  // the previous block's lookups are done
    const bool range = fp8_table_entry(tab, B.scale);
    // a block with an overflowing product checks all its weights
    const bool special = __syncthreads_or(range ? 1 : 0) != 0;
    const uint32_t sflip = (__float_as_uint(B.scale) >> 31) ? (1u << G) - 1u : 0u;
    bool hit = false;
#pragma unroll
    for (int j = 0; j < Fp8Block<G>::kUnits; ++j) {
        if (B.g[j] < 0) continue;
        fp8_unit_convert<G>(B.in[j], tab, sflip, special, B.g[j], body, sign, hit);
    }
    return hit;
}

template <int G>
__global__ void __launch_bounds__(256) fp8_to_fp9_kernel(const uint8_t* __restrict__ w8,
                                                         const float* __restrict__ scale, int64_t rows,
                                                         int64_t cols, int64_t nbx, int64_t nby,
                                                         uint8_t* __restrict__ body, uint8_t* __restrict__ sign,
                                                         int32_t* status) {
    __shared__ uint8_t tab[128];
    bool hit = false;
    // a block's codes are loaded before its table is built, so they are in
    // flight meanwhile
    for (int64_t by = blockIdx.y; by < nby; by += gridDim.y) {
        Fp8Block<G> A;
        fp8_block_load<G>(w8, scale, rows, cols, nbx, by, A);
        hit |= fp8_block_convert<G>(A, tab, body, sign);
    }
    if (hit) record_status(status, FP9_ERR_RANGE);
}

// Matrices of whole 128 x 128 blocks (rows and cols multiples of 128, such
// as every DeepSeek-V3 expert matrix): a persistent grid of a few CTAs per
// SM, CTA k converting blocks k, k + gridDim.x, ... in row-major block
// order. Thread t owns the units of 16 codes at rows (t >> 3) + 32 j,
// j = 0..3, columns 16 (t & 7) .. + 15 of each block it visits. Per block:
// one barrier publishes the block's table (built during the previous
// block); the codes of the CTA's next block are loaded and its table is
// built, from a scale loaded a block earlier, before this block's lookups,
// so the loads are in flight and no warp idles at the barrier while the
// table is encoded. The table is double-buffered: the barrier that
// publishes one buffer also orders every lookup into the other (the
// previous block's) before that buffer is written again.
// Three CTAs per SM: with four, 64 registers a thread held the kernel at
// 132 against 127 us on 24 DeepSeek-V3 expert matrices; two were slower.
constexpr int kFp8FullCtasPerSm = 3;

struct Fp8Full {
    uint32_t in[4][4];  // unit j: rows (t >> 3) + 32 j
    int64_t base;       // index of unit 0's first code
    float scale;
};

__device__ __forceinline__ void fp8_full_load(const uint8_t* __restrict__ w8, int64_t cols, int64_t nbx,
                                              int64_t b, int64_t toff, Fp8Full& B) {
    const int64_t by = b / nbx, bx = b - by * nbx;
    B.base = by * 128 * cols + bx * 128 + toff;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(w8 + B.base + j * 32 * cols));
        B.in[j][0] = q.x, B.in[j][1] = q.y, B.in[j][2] = q.z, B.in[j][3] = q.w;
    }
}

__global__ void __launch_bounds__(256, kFp8FullCtasPerSm)
    fp8_to_fp9_full_kernel(const uint8_t* __restrict__ w8, const float* __restrict__ scale, int64_t cols,
                           int64_t nbx, int64_t nblocks, uint8_t* __restrict__ body, uint8_t* __restrict__ sign,
                           int32_t* status) {
    __shared__ uint8_t tab[2][128];
    const int64_t G = gridDim.x;
    const int64_t toff = static_cast<int64_t>(threadIdx.x >> 3) * cols + (threadIdx.x & 7) * 16;
    int64_t b = blockIdx.x;
    if (b >= nblocks) return;  // (the grid holds at most nblocks CTAs)
    bool hit = false;
    Fp8Full A, B;
    fp8_full_load(w8, cols, nbx, b, toff, A);
    A.scale = __ldg(scale + b);  // scales are [nby, nbx]: block b's is at b
    float s_next = b + G < nblocks ? __ldg(scale + b + G) : 0.0f;
    bool range = fp8_table_entry(tab[0], A.scale);  // the table of the block about to be published
    int p = 0;
    // block bc (codes in C) with table p; loads the next block into N
    auto step = [&](const Fp8Full& C, Fp8Full& N, int64_t bc) -> bool {
        const int64_t bn = bc + G;
        const bool more = bn < nblocks;
        if (more) {
            fp8_full_load(w8, cols, nbx, bn, toff, N);
            N.scale = s_next;
            if (bn + G < nblocks) s_next = __ldg(scale + bn + G);
        }
        // a block with an overflowing product checks all its weights
        const bool special = __syncthreads_or(range ? 1 : 0) != 0;
        if (more) range = fp8_table_entry(tab[p ^ 1], N.scale);
        const uint32_t sflip = (__float_as_uint(C.scale) >> 31) ? 0xFFFFu : 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            fp8_unit_convert<16>(C.in[j], tab[p], sflip, special, (C.base + j * 32 * cols) >> 4, body, sign, hit);
        p ^= 1;
        return more;
    };
    // two blocks per trip, A then B, so that neither is copied
    while (step(A, B, b) && step(B, A, b + G)) b += 2 * G;
    if (hit) record_status(status, FP9_ERR_RANGE);
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

extern "C" fp9_status fp9_from_fp8(const uint8_t* w8, const float* scale_inv, int64_t rows, int64_t cols,
                                   uint8_t* body, uint8_t* sign, int32_t* d_status, void* stream) {
    FP9_CHECK_ARG(rows >= 0 && cols >= 0, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(cols % 8 == 0, FP9_ERR_SHAPE);
    if (rows == 0 || cols == 0) return FP9_OK;
    FP9_CHECK_ARG(w8 != nullptr && scale_inv != nullptr && body != nullptr && sign != nullptr,
                  FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(w8, 8) && aligned(body, 8) && aligned(scale_inv, 4), FP9_ERR_ALIGN);
    const bool wide = cols % 16 == 0 && aligned(w8, 16) && aligned(body, 16) && aligned(sign, 2);
    const int64_t nbx = (cols + 127) / 128, nby = (rows + 127) / 128;
    FP9_CHECK_ARG(nbx <= 0x7FFFFFFF, FP9_ERR_SHAPE);  // one grid column per block column
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (wide && rows % 128 == 0 && cols % 128 == 0) {
        const int64_t nblocks = nbx * nby;
        int32_t sms = device_sm_count();
        if (sms <= 0) sms = 148;
        const int64_t cap = static_cast<int64_t>(sms) * kFp8FullCtasPerSm;
        fp8_to_fp9_full_kernel<<<static_cast<unsigned>(nblocks < cap ? nblocks : cap), 256, 0, st>>>(
            w8, scale_inv, cols, nbx, nblocks, body, sign, d_status);
        FP9_CUDA_TRY(cudaGetLastError());
        return FP9_OK;
    }
    const dim3 grid(static_cast<unsigned>(nbx), static_cast<unsigned>(nby < 65535 ? nby : 65535));
    if (wide)
        fp8_to_fp9_kernel<16><<<grid, 256, 0, st>>>(w8, scale_inv, rows, cols, nbx, nby, body, sign, d_status);
    else
        fp8_to_fp9_kernel<8><<<grid, 256, 0, st>>>(w8, scale_inv, rows, cols, nbx, nby, body, sign, d_status);
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
