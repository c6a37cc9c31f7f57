// fp9 SwiGLU FFN for many tokens at once (prompt prefill) on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// The pages' prefill runs the same fp9 FFN over every prompt token and is
// the part they list as furthest from the hardware's compute peak (the page
// of [MEMOIR-FP9], section "最终结果", its list of limitations: a 1481-token
// prompt prefilled at about 20 tok/s). With m tokens the FFN is a dense
// contraction, so here it runs as two GEMMs on the tensor cores:
//
//   1. gate/up: G = X W_gate^T, U = X W_up^T (both [m, inter]), with the
//      epilogue h = SiLU(G) * U written as fp16 [m, inter];
//   2. down:    y = h W_down^T = h down_t (down_t = W_down^T [inter, hidden]),
//      written as fp32 [m, hidden].
//
// fp9 is a subset of fp16 (the body byte shifted left by 7 with the sign on
// top is the fp16 of the same value, [MEMOIR-FP9]), so the weights enter the
// f16 MMA exactly. The activations x and h are rounded to fp16 (the MMA's
// operand type); products are accumulated in fp32 in tensor memory (TMEM).
//
// One CTA computes a (128 * MH) x 256 output tile:
//   gate/up: 128 intermediate rows of both gate and up (two 128-column
//            accumulators per 128 tokens);
//   down:    256 hidden columns as two 128-column halves.
// K streams through three rings of shared memory, each with its own pair of
// mbarriers (full / empty):
//   A    activation tiles, 64 K columns, loaded by TMA straight into the
//        MMA's 128-byte-swizzle K-major layout (rows past m read as zero);
//   raw  the fp9 planes of 128 K columns of both weight operands (bodies and
//        sign planes), loaded by TMA as they lie in memory;
//   B    the decoded weights of 64 K columns in the MMA's operand layout.
// Warp roles: warps 0-7 decode raw -> B (one 16-byte fp16 chunk of 8 weights
// per task) and run the epilogue; warp 8 issues the activation loads, warp
// 9 the raw weight loads (so the HBM weight stream runs ahead of the MMAs by
// up to the raw ring's depth), warp 10 one thread issues the MMAs and
// commits each A and B slot back through an mbarrier. gate/up weight rows
// are K-major; down_t tiles are MN-major (K = inter runs across rows), read
// through the transposed-B bit. Every wait is bounded: a timeout records
// FP9_ERR_TIMEOUT, raises an abort flag, and the kernel still waits for its
// own copies and MMAs before it frees TMEM and returns.
#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9_plan.h"
#include "fp9_tc.cuh"
#include "fp9moe.h"

namespace fp9 {
namespace {

constexpr int kTileRows = 128;                        // rows of one MMA tile = TMEM lanes
constexpr int kChunkK = 64;                           // K per A / B slot: 128 bytes of fp16
constexpr int kRawK = 128;                            // K per raw slot (16 sign bytes per row)
constexpr int kTileBytes = kTileRows * kChunkK * 2;   // 16 KiB: one 128 x 64 fp16 tile
constexpr int kBSlotBytes = 2 * kTileBytes;           // two weight operands
constexpr int kRawBodyBytes = 2 * kTileRows * kRawK;  // 32 KiB of fp9 bodies
constexpr int kRawSlotBytes = kRawBodyBytes + 2 * kTileRows * (kRawK / 8);  // + 4 KiB of signs
constexpr int kDecoderWarps = 8;
constexpr int kDecoderThreads = kDecoderWarps * 32;
constexpr int kActWarp = 8, kRawWarp = 9, kMmaWarp = 10;
constexpr int kThreads = 11 * 32;
constexpr int kCtlBytes = 1024;
constexpr int kSmemMax = 227 * 1024;
constexpr int kGroupM = 8;                            // M tiles per CTA-order group
constexpr uint64_t kTimeoutNs = 1000000000ull;        // 1 s per wait
constexpr int kTasks = 2 * kTileRows * kChunkK / 8 / kDecoderThreads;  // 8 decode tasks per thread per chunk
// MN-major 128-byte-swizzle operand (down_t tiles): 64 output columns x 8 K
// rows per 1024-byte atom; the two 64-column atoms of a 128-column half sit
// 1024 bytes apart, 8-row K groups 2048 bytes apart.
constexpr uint32_t kMnAtomStride = 1024;
constexpr uint32_t kMnGroupStride = 2048;

// Ring depths: the raw and B rings by tile height, the A ring takes what is
// left of the shared memory.
template <int MH>
struct Cfg {
    static constexpr int kRawSlots = MH == 1 ? 3 : 2;
    static constexpr int kBSlots = 2;
    static constexpr int kASlotBytes = MH * kTileBytes;
    static constexpr int kFixed = 1024 + kCtlBytes + kRawSlots * kRawSlotBytes + kBSlots * kBSlotBytes;
    static constexpr int kASlots = (kSmemMax - kFixed) / kASlotBytes;
    static constexpr int kSmem = kFixed + kASlots * kASlotBytes;
    static constexpr uint32_t kTmemCols = MH * 256;
    static_assert(kASlots >= 2 && kASlots <= 8, "activation ring");
};

struct Ctl {
    uint64_t a_full[8], a_empty[8];   // activation ring: TMA bytes / MMA commit
    uint64_t w_full[4], w_empty[4];   // raw ring: TMA bytes / 8 decoder warps
    uint64_t b_full[4], b_empty[4];   // decoded ring: 8 decoder warps / MMA commit
    uint64_t done;                    // every MMA of the CTA finished
    uint32_t tmem;
    int abort;
    int never;
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

// 2-D tiled tensor maps (TMA descriptors) of one launch.
struct PrefillMaps {
    CUtensorMap act;       // fp16 [m, K], box 64 x 128, 128-byte swizzle
    CUtensorMap body[2];   // gate/up: W_gate, W_up bodies, box 64 x 128; down: down_t, box 256 x 128
    CUtensorMap sign[2];   // the sign planes, box 16 x 128 (gate/up) or 32 x 128 (down)
};

struct PrefillArgs {
    int32_t m;               // tokens
    int32_t mtiles, ntiles;  // CTA tiles along tokens / output columns
    int32_t nk;              // K / 64
    int32_t wrow0;           // first weight row of the FFN in the planes
    void* out;               // gate/up: h fp16 [m, inter]; down: y fp32 [m, hidden]
    int64_t ldo;             // row stride of out (elements)
    int32_t* status;
    uint64_t timeout_ns;
};

// CTA order: groups of kGroupM token tiles walk the output tiles together,
// so the weight tiles a wave of CTAs reads are shared by up to kGroupM CTAs
// through L2.
__device__ __forceinline__ void tile_of(int L, int mtiles, int ntiles, int& mt, int& nt) {
    const int per_group = kGroupM * ntiles;
    const int g = L / per_group;
    const int first = g * kGroupM;
    const int gm = min(mtiles - first, kGroupM);
    const int r = L - g * per_group;
    mt = first + r % gm;
    nt = r / gm;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// TMA: a 2-D box of `map` at (x = inner element, y = row) into shared memory,
// completing its bytes on the mbarrier `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 8 consecutive fp9 weights (8 body bytes, one sign byte) -> one 16-byte
// chunk of fp16 in column order.
__device__ __forceinline__ uint4 decode8_half(uint2 w, uint32_t s8) {
    uint4 c;
    fp9_to_half4(w.x, spread_sign_nibble(s8 & 0xFu), c.x, c.y);
    fp9_to_half4(w.y, spread_sign_nibble((s8 >> 4) & 0xFu), c.z, c.w);
    return c;
}

// Decodes K half `h` (64 columns) of raw slot `raw` into B slot `sB`.
// Task u = t + 256 i of decoder thread t (8 per thread) is 8 weights:
//   gate/up: operand u / 1024, row (u / 8) mod 128, K columns 8 (u mod 8)
//            + [0, 8) -> chunk u mod 8 of the row in the K-major layout.
//            Raw bodies: [operand][half][row][64 B], signs [operand][row][16 B].
//   down:    K row u / 32, output columns 8 (u mod 32) + [0, 8) -> chunk of
//            the MN-major layout. Raw bodies: [K row][256 B], signs [K row][32 B].
// The 8 threads of a quarter warp write 8 chunks of one row (or one atom
// row), which the swizzle spreads over 8 bank groups; a half warp reads
// 128 contiguous raw bytes.
template <bool kDown>
__device__ __forceinline__ void decode_chunk(int t, uint32_t raw, int h, uint32_t sB) {
#pragma unroll
    for (int i = 0; i < kTasks; ++i) {
        const uint32_t u = static_cast<uint32_t>(t + kDecoderThreads * i);
        if (!kDown) {
            const uint32_t b = u >> 10, row = (u >> 3) & 127u, c = u & 7u;
            const uint2 w = ld_shared_v2(raw + b * (kTileRows * kRawK) + h * (kTileRows * 64) + row * 64u + c * 8u);
            const uint32_t s = ld_shared_u8(raw + kRawBodyBytes + b * (kTileRows * 16) + row * 16u + h * 8u + c);
            st_shared_v4(sB + b * kTileBytes + sw128_offset(row, c * 8u), decode8_half(w, s));
        } else {
            const uint32_t kr = u >> 5, c = u & 31u, rr = h * 64u + kr;
            const uint2 w = ld_shared_v2(raw + rr * 256u + c * 8u);
            const uint32_t s = ld_shared_u8(raw + kRawBodyBytes + rr * 32u + c);
            const uint32_t x = kr & 7u;
            const uint32_t dst = sB + (c >> 4) * kTileBytes + (kr >> 3) * kMnGroupStride + ((c >> 3) & 1u) * kMnAtomStride +
                                 x * 128u + (((c & 7u) ^ x) << 4);
            st_shared_v4(dst, decode8_half(w, s));
        }
    }
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ bool half2_finite(uint32_t h) {
    return ((h & 0x7C00u) != 0x7C00u) && ((h & 0x7C000000u) != 0x7C000000u);
}

// Warp-uniform bounded wait (lane 0 polls, the result is broadcast).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit, const volatile int* abort) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, limit, abort);
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void fail(Ctl& ctl, int32_t* status) {
    record_status(status, FP9_ERR_TIMEOUT);
    ctl.abort = 1;
}

template <bool kDown, int MH>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillMaps maps,
                                                              const PrefillArgs p) {
    using C = Cfg<MH>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw0 = smem_addr(smem_raw);
    const uint32_t base = (raw0 + 1023u) & ~1023u;
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw + (base - raw0));
    const uint32_t ringA = base + kCtlBytes;                           // 1024-aligned slots
    const uint32_t ringB = ringA + C::kASlots * C::kASlotBytes;
    const uint32_t ringW = ringB + C::kBSlots * kBSlotBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kASlots; ++s) {
            mbar_init(smem_addr(&ctl.a_full[s]), 1);
            mbar_init(smem_addr(&ctl.a_empty[s]), 1);
        }
        for (int s = 0; s < C::kRawSlots; ++s) {
            mbar_init(smem_addr(&ctl.w_full[s]), 1);
            mbar_init(smem_addr(&ctl.w_empty[s]), kDecoderWarps);
        }
        for (int s = 0; s < C::kBSlots; ++s) {
            mbar_init(smem_addr(&ctl.b_full[s]), kDecoderWarps);
            mbar_init(smem_addr(&ctl.b_empty[s]), 1);
        }
        mbar_init(smem_addr(&ctl.done), 1);
        ctl.abort = 0;
        ctl.never = 0;
        fence_mbar_init();
    }
    if (warp == kActWarp && lane == 0) prefetch_map(&maps.act);
    if (warp == kRawWarp && lane == 0) {
        prefetch_map(&maps.body[0]);
        prefetch_map(&maps.sign[0]);
        if (!kDown) {
            prefetch_map(&maps.body[1]);
            prefetch_map(&maps.sign[1]);
        }
    }
    if (warp == 0) tc_alloc(smem_addr(&ctl.tmem), C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;

    int mt, nt;
    tile_of(blockIdx.x, p.mtiles, p.ntiles, mt, nt);
    const int m0 = mt * kTileRows * MH;
    // output columns: 128 intermediate rows (gate/up) or 256 hidden columns (down)
    const int n0 = nt * (kDown ? 2 * kTileRows : kTileRows);
    const int nk = p.nk;

    if (warp == kActWarp) {
        // -------------------------------------------- activation loads ---
        if (lane == 0) {
            grid_dependency_wait();  // the activations come from the previous launch
            int issued = 0;
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % C::kASlots;
                if (kc >= C::kASlots &&
                    !mbar_wait_bounded(smem_addr(&ctl.a_empty[s]), ((kc / C::kASlots) + 1) & 1, p.timeout_ns, &ctl.abort)) {
                    fail(ctl, p.status);
                    break;
                }
                const uint32_t bar = smem_addr(&ctl.a_full[s]);
                mbar_arrive_expect_tx(bar, C::kASlotBytes);
#pragma unroll
                for (int mh = 0; mh < MH; ++mh)
                    tma_load_2d(ringA + s * C::kASlotBytes + mh * kTileBytes, &maps.act, kc * kChunkK,
                                m0 + mh * kTileRows, bar);
                issued = kc + 1;
            }
            // the copies this thread issued land before the CTA may exit
            for (int j = issued > C::kASlots ? issued - C::kASlots : 0; j < issued; ++j)
                (void)mbar_wait_bounded(smem_addr(&ctl.a_full[j % C::kASlots]), (j / C::kASlots) & 1, p.timeout_ns,
                                        &ctl.never);
        }
        __syncwarp();
    } else if (warp == kRawWarp) {
        // ------------------------------------------------ weight loads ---
        if (lane == 0) {
            const int nw = nk / 2;
            int issued = 0;
            for (int kw = 0; kw < nw; ++kw) {
                const int s = kw % C::kRawSlots;
                if (kw >= C::kRawSlots &&
                    !mbar_wait_bounded(smem_addr(&ctl.w_empty[s]), ((kw / C::kRawSlots) + 1) & 1, p.timeout_ns,
                                       &ctl.abort)) {
                    fail(ctl, p.status);
                    break;
                }
                const uint32_t bar = smem_addr(&ctl.w_full[s]);
                const uint32_t slot = ringW + s * kRawSlotBytes;
                mbar_arrive_expect_tx(bar, kRawSlotBytes);
                if (!kDown) {
                    const int row = p.wrow0 + n0;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        tma_load_2d(slot + b * (kTileRows * kRawK), &maps.body[b], kw * kRawK, row, bar);
                        tma_load_2d(slot + b * (kTileRows * kRawK) + kTileRows * 64, &maps.body[b], kw * kRawK + 64,
                                    row, bar);
                        tma_load_2d(slot + kRawBodyBytes + b * (kTileRows * 16), &maps.sign[b], kw * (kRawK / 8), row,
                                    bar);
                    }
                } else {
                    const int row = p.wrow0 + kw * kRawK;
                    tma_load_2d(slot, &maps.body[0], n0, row, bar);
                    tma_load_2d(slot + kRawBodyBytes, &maps.sign[0], n0 / 8, row, bar);
                }
                issued = kw + 1;
            }
            for (int j = issued > C::kRawSlots ? issued - C::kRawSlots : 0; j < issued; ++j)
                (void)mbar_wait_bounded(smem_addr(&ctl.w_full[j % C::kRawSlots]), (j / C::kRawSlots) & 1, p.timeout_ns,
                                        &ctl.never);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA ---
        if (lane == 0) {
            const uint32_t idesc = tc_idesc_f16(kTileRows, kTileRows) | (kDown ? (1u << 16) : 0u);
            for (int kc = 0; kc < nk; ++kc) {
                const int sa = kc % C::kASlots, sb = kc % C::kBSlots;
                if (!mbar_wait_bounded(smem_addr(&ctl.a_full[sa]), (kc / C::kASlots) & 1, p.timeout_ns, &ctl.abort) ||
                    !mbar_wait_bounded(smem_addr(&ctl.b_full[sb]), (kc / C::kBSlots) & 1, p.timeout_ns, &ctl.abort)) {
                    fail(ctl, p.status);
                    break;
                }
                tc_fence_after();
                const uint32_t sA = ringA + sa * C::kASlotBytes;
                const uint32_t sB = ringB + sb * kBSlotBytes;
#pragma unroll
                for (int k16 = 0; k16 < kChunkK / 16; ++k16) {
#pragma unroll
                    for (int mh = 0; mh < MH; ++mh) {
                        const uint64_t ad = tc_desc_sw128(sA + mh * kTileBytes + 32u * k16);
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const uint64_t bd =
                                kDown ? tc_desc_sw128_mn(sB + b * kTileBytes + 2u * kMnGroupStride * k16,
                                                         kMnAtomStride, kMnGroupStride)
                                      : tc_desc_sw128(sB + b * kTileBytes + 32u * k16);
                            tc_mma_f16(tmem + (mh * 2 + b) * kTileRows, ad, bd, idesc, kc > 0 || k16 > 0);
                        }
                    }
                }
                tc_commit(smem_addr(&ctl.a_empty[sa]));
                tc_commit(smem_addr(&ctl.b_empty[sb]));
            }
            tc_commit(smem_addr(&ctl.done));
            // TMEM is freed only after every MMA of this CTA has finished
            if (!mbar_wait_bounded(smem_addr(&ctl.done), 0, p.timeout_ns, &ctl.never))
                record_status(p.status, FP9_ERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- decoders ---
        const int t = threadIdx.x;
        bool ok = true;
        for (int kc = 0; kc < nk && ok; ++kc) {
            const int kw = kc >> 1, h = kc & 1;
            const int sw = kw % C::kRawSlots, sb = kc % C::kBSlots;
            if (h == 0) ok = warp_wait(smem_addr(&ctl.w_full[sw]), (kw / C::kRawSlots) & 1, p.timeout_ns, &ctl.abort);
            if (ok && kc >= C::kBSlots)
                ok = warp_wait(smem_addr(&ctl.b_empty[sb]), ((kc / C::kBSlots) + 1) & 1, p.timeout_ns, &ctl.abort);
            if (!ok) break;
            decode_chunk<kDown>(t, ringW + sw * kRawSlotBytes, h, ringB + sb * kBSlotBytes);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_addr(&ctl.b_full[sb]));
                if (h == 1) mbar_arrive(smem_addr(&ctl.w_empty[sw]));
            }
        }
        if (!ok && lane == 0) fail(ctl, p.status);
        // ----------------------------------------------------- epilogue ---
        if (warp_wait(smem_addr(&ctl.done), 0, p.timeout_ns, &ctl.abort)) {
            tc_fence_after();
            const int lq = warp & 3, sel = warp >> 2;
            const uint32_t tl = tmem + ((static_cast<uint32_t>(lq) * 32u) << 16);
            bool bad = false;  // a stored h whose fp16 is not finite
#pragma unroll
            for (int mh = 0; mh < MH; ++mh) {
                const int64_t grow = static_cast<int64_t>(m0) + mh * kTileRows + lq * 32 + lane;
                const bool valid = grow < p.m;
                if (!kDown) {
                    __half* out = static_cast<__half*>(p.out) + grow * p.ldo + n0;
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int cb = 2 * sel + c2;
                        float g[32], u[32];
                        tc_ld32(tl + (mh * 2 + 0) * kTileRows + cb * 32, g);
                        tc_ld32(tl + (mh * 2 + 1) * kTileRows + cb * 32, u);
                        uint32_t hw[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const __half2 h2 = __floats2half2_rn(silu(g[2 * i]) * u[2 * i],
                                                                 silu(g[2 * i + 1]) * u[2 * i + 1]);
                            hw[i] = *reinterpret_cast<const uint32_t*>(&h2);
                            bad = bad || (valid && !half2_finite(hw[i]));
                        }
                        if (valid) {
                            uint4* o = reinterpret_cast<uint4*>(out + cb * 32);
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                o[v] = make_uint4(hw[4 * v], hw[4 * v + 1], hw[4 * v + 2], hw[4 * v + 3]);
                        }
                    }
                } else {
                    float* out = static_cast<float*>(p.out) + grow * p.ldo + n0 + sel * kTileRows;
#pragma unroll
                    for (int cb = 0; cb < 4; ++cb) {
                        float v[32];
                        tc_ld32(tl + (mh * 2 + sel) * kTileRows + cb * 32, v);
                        if (valid) {
                            float4* o = reinterpret_cast<float4*>(out + cb * 32);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        }
                    }
                }
            }
            if (bad) record_status(p.status, FP9_ERR_RANGE);
        }
    }

    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, C::kTmemCols);
}

// x fp32 -> fp16 (round to nearest even); a value whose fp16 is not finite
// is recorded as FP9_ERR_RANGE.
__global__ void to_half_kernel(const float4* __restrict__ x, uint2* __restrict__ h, int64_t n4, int32_t* status) {
    grid_dependency_wait();
    grid_launch_dependents();
    bool finite = true;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 v = x[i];
        const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&a);
        o.y = *reinterpret_cast<const uint32_t*>(&b);
        finite = finite && half2_finite(o.x) && half2_finite(o.y);
        h[i] = o;
    }
    if (!finite) record_status(status, FP9_ERR_RANGE);
}

// ------------------------------------------------------------------ host ---

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            (void)cudaGetLastError();
    }
    return fn;
}

// A row-major 2-D map: `rows` rows of `inner` elements, `pitch` bytes apart.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner, uint64_t rows,
              uint64_t pitch, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token tiles of 128 * MH rows: MH = 2 halves the activation traffic per
// flop; MH = 1 keeps more CTAs when the grid would not fill the GPU. Picks
// the MH with fewer (waves x tile work), counting a 256-row tile as 1.8 of
// a 128-row one.
int choose_mh(int64_t m, int64_t ntiles, int sms) {
    auto waves = [&](int mh) {
        const int64_t ctas = ntiles * ((m + kTileRows * mh - 1) / (kTileRows * mh));
        return static_cast<double>((ctas + sms - 1) / sms);
    };
    return waves(2) * 1.8 <= waves(1) ? 2 : 1;
}

template <bool kDown, int MH>
cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(prefill_kernel<kDown, MH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<MH>::kSmem);
}

fp9_status ensure_attrs() {
    static bool configured[64] = {false};
    int dev = 0;
    FP9_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return FP9_ERR_CUDA;
    if (!configured[dev]) {
        if (device_max_smem_optin() < Cfg<1>::kSmem || device_max_smem_optin() < Cfg<2>::kSmem)
            return FP9_ERR_CUDA;
        FP9_CUDA_TRY((set_smem_attr<false, 1>()));
        FP9_CUDA_TRY((set_smem_attr<false, 2>()));
        FP9_CUDA_TRY((set_smem_attr<true, 1>()));
        FP9_CUDA_TRY((set_smem_attr<true, 2>()));
        configured[dev] = true;
    }
    return FP9_OK;
}

// One GEMM launch: activations act [m, K] fp16; weight rows [wrow0, ...)
// of planes with plane_rows rows of `hidden` columns (gate/up: body/sign
// [0..1] = W_gate, W_up; down: body/sign[0] = down_t).
fp9_status launch_gemm(bool down, const __half* act, int64_t m, int64_t K, const uint8_t* const body[2],
                       const uint8_t* const sign[2], int64_t plane_rows, int64_t hidden, int64_t wrow0,
                       int32_t ntiles, void* out, int64_t ldo, int32_t* status, int sms, cudaStream_t stream) {
    PrefillMaps maps;
    if (!make_map(&maps.act, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, act, static_cast<uint64_t>(K), static_cast<uint64_t>(m),
                  static_cast<uint64_t>(K) * 2, kChunkK, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B))
        return FP9_ERR_CUDA;
    for (int b = 0; b < (down ? 1 : 2); ++b) {
        if (!make_map(&maps.body[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, body[b], static_cast<uint64_t>(hidden),
                      static_cast<uint64_t>(plane_rows), static_cast<uint64_t>(hidden), down ? 2 * kTileRows : 64,
                      kTileRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map(&maps.sign[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, sign[b], static_cast<uint64_t>(hidden / 8),
                      static_cast<uint64_t>(plane_rows), static_cast<uint64_t>(hidden / 8),
                      down ? 2 * kTileRows / 8 : kRawK / 8, kTileRows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return FP9_ERR_CUDA;
    }
    if (down) {
        maps.body[1] = maps.body[0];
        maps.sign[1] = maps.sign[0];
    }
    PrefillArgs p{};
    p.m = static_cast<int32_t>(m);
    p.ntiles = ntiles;
    p.nk = static_cast<int32_t>(K / kChunkK);
    p.wrow0 = static_cast<int32_t>(wrow0);
    p.out = out;
    p.ldo = ldo;
    p.status = status;
    p.timeout_ns = kTimeoutNs;
    const int mh = choose_mh(m, ntiles, sms);
    p.mtiles = static_cast<int32_t>((m + kTileRows * mh - 1) / (kTileRows * mh));
    const int64_t ctas = static_cast<int64_t>(p.mtiles) * p.ntiles;
    if (ctas > 0x7FFFFFFF) return FP9_ERR_SHAPE;
    void (*k)(const PrefillMaps, const PrefillArgs) =
        down ? (mh == 2 ? prefill_kernel<true, 2> : prefill_kernel<true, 1>)
             : (mh == 2 ? prefill_kernel<false, 2> : prefill_kernel<false, 1>);
    const int smem = mh == 2 ? Cfg<2>::kSmem : Cfg<1>::kSmem;
    FP9_CUDA_TRY(launch_pdl(k, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), smem, stream, maps, p));
    return FP9_OK;
}

struct PrefillLayout {
    size_t off_x16 = 0, off_h = 0, total = 0;
};

PrefillLayout prefill_layout(int64_t m, int64_t hidden, int64_t inter) {
    PrefillLayout L;
    L.off_x16 = 0;
    L.off_h = align_up(sizeof(__half) * static_cast<size_t>(m) * static_cast<size_t>(hidden));
    L.total = L.off_h + align_up(sizeof(__half) * static_cast<size_t>(m) * static_cast<size_t>(inter));
    return L;
}

fp9_status check_prefill_bank(const fp9_ffn_bank* f, int64_t index) {
    FP9_CHECK_ARG(f != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(f->n >= 1 && index >= 0 && index < f->n, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(f->hidden >= 256 && f->hidden <= FP9_MAX_PREFILL_HIDDEN && f->hidden % 256 == 0, FP9_ERR_SHAPE);
    FP9_CHECK_ARG(f->inter >= 128 && f->inter <= FP9_MAX_INTER && f->inter % 128 == 0, FP9_ERR_SHAPE);
    return check_bank(*f, f->n, f->inter, f->hidden);
}

}  // namespace
}  // namespace fp9

using namespace fp9;

extern "C" size_t fp9_prefill_workspace_bytes(const fp9_ffn_bank* ffn, int64_t m) {
    if (check_prefill_bank(ffn, 0) != FP9_OK || m < 0 || m > FP9_MAX_PREFILL_TOKENS) return 0;
    return prefill_layout(m, ffn->hidden, ffn->inter).total;
}

extern "C" fp9_status fp9_ffn_prefill(const fp9_ffn_bank* ffn, int64_t index, const float* x, int64_t m,
                                      float* y, void* ws, size_t ws_bytes, int32_t* d_status, void* stream) {
    fp9_status st = check_prefill_bank(ffn, index);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(m >= 0 && m <= FP9_MAX_PREFILL_TOKENS, FP9_ERR_INVALID_ARG);
    if (m == 0) return FP9_OK;
    FP9_CHECK_ARG(x != nullptr && y != nullptr && ws != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(x, 16) && aligned(y, 16) && aligned(ws, 256), FP9_ERR_ALIGN);
    const int64_t H = ffn->hidden, I = ffn->inter;
    const PrefillLayout lay = prefill_layout(m, H, I);
    FP9_CHECK_ARG(ws_bytes >= lay.total, FP9_ERR_WORKSPACE);
    const int sms = device_sm_count();
    if (sms <= 0) return FP9_ERR_CUDA;
    st = ensure_attrs();
    if (st != FP9_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    __half* x16 = reinterpret_cast<__half*>(w + lay.off_x16);
    __half* h = reinterpret_cast<__half*>(w + lay.off_h);

    const int64_t n4 = m * H / 4;
    const int64_t blocks = (n4 + 255) / 256 < static_cast<int64_t>(sms) * 8 ? (n4 + 255) / 256 : sms * 8;
    FP9_CUDA_TRY(launch_pdl(to_half_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                            reinterpret_cast<const float4*>(x), reinterpret_cast<uint2*>(x16), n4, d_status));

    // the maps cover FFN `index` only (rows [0, inter) of its planes)
    const size_t wg = static_cast<size_t>(index) * static_cast<size_t>(I) * static_cast<size_t>(H);
    const uint8_t* gu_body[2] = {ffn->gate_body + wg, ffn->up_body + wg};
    const uint8_t* gu_sign[2] = {ffn->gate_sign + wg / 8, ffn->up_sign + wg / 8};
    st = launch_gemm(false, x16, m, H, gu_body, gu_sign, I, H, 0, static_cast<int32_t>(I / kTileRows), h, I, d_status,
                     sms, s);
    if (st != FP9_OK) return st;
    const uint8_t* d_body[2] = {ffn->down_body + wg, ffn->down_body + wg};
    const uint8_t* d_sign[2] = {ffn->down_sign + wg / 8, ffn->down_sign + wg / 8};
    return launch_gemm(true, h, m, I, d_body, d_sign, I, H, 0, static_cast<int32_t>(H / (2 * kTileRows)), y, H,
                       d_status, sms, s);
}
