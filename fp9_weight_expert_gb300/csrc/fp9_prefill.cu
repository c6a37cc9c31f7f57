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
// f16 MMA exactly: producer threads decode each weight tile into shared
// memory in the MMA's operand layout. The activations x and h are rounded to
// fp16 (the MMA's operand type); the products are accumulated in fp32 in
// tensor memory (TMEM).
//
// One CTA computes a (128 * MH) x 256 output tile:
//   gate/up: 128 intermediate rows of both gate and up (two 128-column
//            accumulators per 128 tokens);
//   down:    256 hidden columns as two 128-column halves.
// 8 producer warps stream K in chunks of 64 through a ring of stages: per
// stage the activation tile(s) (16-byte copies into the 128-byte-swizzle
// K-major layout) and the two decoded weight tiles. One elected thread of a
// ninth warp issues the MMAs and commits each stage back to the producers
// through an mbarrier. gate/up weight rows are K-major ([inter, hidden] with
// K = hidden contiguous); down_t tiles are MN-major (K = inter runs across
// rows), which the MMA reads through the transposed-B bit. Every wait is
// bounded: a timeout records FP9_ERR_TIMEOUT and the kernel still waits for
// its own MMAs before it frees TMEM and returns.
#include <cstddef>
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9_plan.h"
#include "fp9_tc.cuh"
#include "fp9moe.h"

namespace fp9 {
namespace {

constexpr int kTileRows = 128;                        // rows of one MMA tile = TMEM lanes
constexpr int kChunkK = 64;                           // K per stage: 128 bytes of fp16
constexpr int kTileBytes = kTileRows * kChunkK * 2;   // 16 KiB: one 128 x 64 fp16 tile
constexpr int kProducerWarps = 8;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kThreads = kProducerThreads + 32;       // + the MMA warp
constexpr int kCtlBytes = 1024;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kGroupM = 8;                            // M tiles per CTA-order group
constexpr uint64_t kTimeoutNs = 1000000000ull;        // 1 s per wait
// MN-major 128-byte-swizzle operand (down_t tiles): 64 output columns x 8 K
// rows per 1024-byte atom; the two 64-column atoms of a 128-column half sit
// 1024 bytes apart, 8-row K groups 2048 bytes apart.
constexpr uint32_t kMnAtomStride = 1024;
constexpr uint32_t kMnGroupStride = 2048;

template <int MH>
struct Cfg {
    static constexpr int kStageBytes = (MH + 2) * kTileBytes;
    static constexpr int kStages = (kSmemBudget - kCtlBytes - 1024) / kStageBytes;
    static constexpr int kSmem = 1024 + kCtlBytes + kStages * kStageBytes;
    static constexpr uint32_t kTmemCols = MH * 256;
    static_assert(kStages >= 3 && kStages <= 8, "stage ring");
};

struct Ctl {
    uint64_t full[8];   // producers -> MMA: stage filled (8 warp arrivals)
    uint64_t empty[8];  // MMA -> producers: stage consumed (one commit)
    uint64_t done;      // MMA -> epilogue: every accumulation finished
    uint32_t tmem;
    int abort;
    int never;
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

struct PrefillArgs {
    const __half* act;       // A operand: fp16 [m, K], row stride K
    const uint8_t* body[2];  // gate/up: W_gate, W_up; down: down_t twice
    const uint8_t* sign[2];
    int64_t hidden;          // row length of every weight plane
    int64_t K;               // contraction length (hidden, or inter for down)
    int32_t m;               // tokens
    int32_t mtiles, ntiles;  // CTA tiles along tokens / output columns
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

// 16 consecutive fp9 weights (16 body bytes, 16 sign bits) -> two 16-byte
// chunks of fp16 in column order.
__device__ __forceinline__ void decode16_half(const uint4 w, uint32_t s16, uint4& lo, uint4& hi) {
    fp9_to_half4(w.x, spread_sign_nibble(s16 & 0xFu), lo.x, lo.y);
    fp9_to_half4(w.y, spread_sign_nibble((s16 >> 4) & 0xFu), lo.z, lo.w);
    fp9_to_half4(w.z, spread_sign_nibble((s16 >> 8) & 0xFu), hi.x, hi.y);
    fp9_to_half4(w.w, spread_sign_nibble((s16 >> 12) & 0xFu), hi.z, hi.w);
}

// The fp9 weights one producer thread moves for one K chunk (16 weights per
// task, 512 tasks per operand b = j / 2):
//   gate/up: row (c mod 512) / 4 of matrix b, K columns 16 (c mod 4) + [0, 16)
//   down:    K row (c mod 512) / 8, columns 128 b + 16 (c mod 8) + [0, 16)
// with c = t + 256 j for producer thread t.
struct Loaded {
    uint4 w[4];     // fp9 bodies
    uint32_t s[4];  // their 16 sign bits
};

template <bool kDown>
__device__ __forceinline__ void load_weights(const PrefillArgs& p, int t, int64_t n0, int64_t k0, Loaded& L) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = (t + kProducerThreads * j) & 511;
        const int b = j >> 1;
        const uint8_t* body;
        const uint8_t* sign;
        if (!kDown) {
            const int64_t r = n0 + (c >> 2);
            const int64_t col = k0 + 16 * (c & 3);
            body = p.body[b] + r * p.hidden + col;
            sign = p.sign[b] + r * (p.hidden >> 3) + (col >> 3);
        } else {
            const int64_t r = k0 + (c >> 3);
            const int64_t col = n0 + 128 * b + 16 * (c & 7);
            body = p.body[0] + r * p.hidden + col;
            sign = p.sign[0] + r * (p.hidden >> 3) + (col >> 3);
        }
        L.w[j] = __ldg(reinterpret_cast<const uint4*>(body));
        L.s[j] = __ldg(reinterpret_cast<const unsigned short*>(sign));
    }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Activation tile(s) of one K chunk, copied straight into the stage's
// 128-byte-swizzle layout: MH x 128 rows x 8 chunks of 16 bytes, chunk
// c = t + 256 j of thread t (rows past m repeat row m - 1; their results
// are not stored). The 8 threads of a quarter warp copy the 8 chunks of one
// row, which the swizzle spreads over 8 bank groups.
template <int MH>
__device__ __forceinline__ void copy_act(const PrefillArgs& p, int t, int64_t m0, int64_t k0, uint32_t sA) {
#pragma unroll
    for (int j = 0; j < 4 * MH; ++j) {
        const int c = t + kProducerThreads * j;
        int64_t gr = m0 + (c >> 3);
        if (gr > p.m - 1) gr = p.m - 1;
        const uint32_t mh = static_cast<uint32_t>(c) >> 10;
        const uint32_t row = (static_cast<uint32_t>(c) >> 3) & 127u;
        cp_async16(sA + mh * kTileBytes + sw128_offset(row, (c & 7) * 8u), p.act + gr * p.K + k0 + (c & 7) * 8);
    }
}

template <bool kDown>
__device__ __forceinline__ void store_weights(const Loaded& L, int t, uint32_t sB) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t c = static_cast<uint32_t>(t + kProducerThreads * j) & 511u;
        const uint32_t tile = sB + (j >> 1) * kTileBytes;
        uint4 lo, hi;
        decode16_half(L.w[j], L.s[j], lo, hi);
        if (!kDown) {
            const uint32_t row = c >> 2, k = 16u * (c & 3u);
            st_shared_v4(tile + sw128_offset(row, k), lo);
            st_shared_v4(tile + sw128_offset(row, k + 8u), hi);
        } else {
            // K row kr holds output columns 16q..16q+15 as chunks 2q, 2q+1
            // of the 128-column half: atom q / 4, chunk positions (2q) mod 8
            // and the next, swizzled by kr mod 8. Threads with q >= 4 store
            // their second chunk first so that the 8 threads of a quarter
            // warp hit 8 different 16-byte bank groups.
            const uint32_t kr = c >> 3, q = c & 7u, x = kr & 7u;
            const uint32_t base = tile + (kr >> 3) * kMnGroupStride + (q >> 2) * kMnAtomStride + x * 128u;
            const uint32_t j0 = (2u * q) & 7u;
            const bool swap = (q & 4u) != 0;
            const uint32_t a0 = base + ((j0 ^ x) << 4), a1 = base + (((j0 + 1u) ^ x) << 4);
            st_shared_v4(swap ? a1 : a0, swap ? hi : lo);
            st_shared_v4(swap ? a0 : a1, swap ? lo : hi);
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

template <bool kDown, int MH>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const PrefillArgs p) {
    using C = Cfg<MH>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw + (base - raw));
    const uint32_t stages = base + kCtlBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_addr(&ctl.full[s]), kProducerWarps);
            mbar_init(smem_addr(&ctl.empty[s]), 1);
        }
        mbar_init(smem_addr(&ctl.done), 1);
        ctl.abort = 0;
        ctl.never = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc_alloc(smem_addr(&ctl.tmem), C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;

    int mt, nt;
    tile_of(blockIdx.x, p.mtiles, p.ntiles, mt, nt);
    const int64_t m0 = static_cast<int64_t>(mt) * kTileRows * MH;
    // output columns: 256 hidden columns (down) or 128 intermediate rows (gate/up)
    const int64_t n0 = static_cast<int64_t>(nt) * (kDown ? 2 * kTileRows : kTileRows);
    const int nk = static_cast<int>(p.K / kChunkK);

    grid_dependency_wait();  // the activations come from the previous launch
    grid_launch_dependents();

    if (warp == kProducerWarps) {
        // ---------------------------------------------------------- MMA ---
        if (lane == 0) {
            const uint32_t idesc = tc_idesc_f16(kTileRows, kTileRows) | (kDown ? (1u << 16) : 0u);
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % C::kStages;
                if (!mbar_wait_bounded(smem_addr(&ctl.full[s]), (kc / C::kStages) & 1, p.timeout_ns, &ctl.abort)) {
                    record_status(p.status, FP9_ERR_TIMEOUT);
                    ctl.abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t sA = stages + s * C::kStageBytes;
                const uint32_t sB = sA + MH * kTileBytes;
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
                tc_commit(smem_addr(&ctl.empty[s]));
            }
            tc_commit(smem_addr(&ctl.done));
            // TMEM is freed only after every MMA of this CTA has finished
            if (!mbar_wait_bounded(smem_addr(&ctl.done), 0, p.timeout_ns, &ctl.never))
                record_status(p.status, FP9_ERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- producers ---
        // Chunk kc's weights are loaded into register set kc mod kDepth and
        // its activations copied (cp.async) into its stage kDepth chunks
        // ahead; kDepth < kStages, so the stage a copy waits for was last
        // used by a chunk whose MMAs need nothing more from the producers.
        constexpr int kDepth = C::kStages - 1 < 3 ? C::kStages - 1 : 3;
        const int t = threadIdx.x;
        Loaded ring[kDepth];
#pragma unroll
        for (int i = 0; i < kDepth; ++i) {
            if (i < nk) {
                load_weights<kDown>(p, t, n0, static_cast<int64_t>(i) * kChunkK, ring[i]);
                copy_act<MH>(p, t, m0, static_cast<int64_t>(i) * kChunkK, stages + i * C::kStageBytes);
            }
            cp_async_commit();
        }
        bool ok = true;
        for (int kc0 = 0; kc0 < nk && ok; kc0 += kDepth) {
#pragma unroll
            for (int i = 0; i < kDepth; ++i) {
                const int kc = kc0 + i;
                if (kc < nk && ok) {
                    const int s = kc % C::kStages;
                    const uint32_t sA = stages + s * C::kStageBytes;
                    store_weights<kDown>(ring[i], t, sA + MH * kTileBytes);
                    cp_async_wait<kDepth - 1>();  // this thread's copies of chunk kc
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&ctl.full[s]));
                    const int kn = kc + kDepth;
                    if (kn < nk) {
                        load_weights<kDown>(p, t, n0, static_cast<int64_t>(kn) * kChunkK, ring[i]);
                        const int sn = kn % C::kStages;
                        if (kn >= C::kStages)
                            ok = warp_wait(smem_addr(&ctl.empty[sn]), ((kn / C::kStages) + 1) & 1, p.timeout_ns,
                                           &ctl.abort);
                        if (ok) copy_act<MH>(p, t, m0, static_cast<int64_t>(kn) * kChunkK, stages + sn * C::kStageBytes);
                    }
                    cp_async_commit();
                }
            }
        }
        cp_async_wait<0>();
        if (!ok && lane == 0) {
            record_status(p.status, FP9_ERR_TIMEOUT);
            ctl.abort = 1;
        }
        // ----------------------------------------------------- epilogue ---
        if (warp_wait(smem_addr(&ctl.done), 0, p.timeout_ns, &ctl.abort)) {
            tc_fence_after();
            const int lq = warp & 3, sel = warp >> 2;
            const uint32_t tl = tmem + ((static_cast<uint32_t>(lq) * 32u) << 16);
            bool bad = false;  // a stored h whose fp16 is not finite
#pragma unroll
            for (int mh = 0; mh < MH; ++mh) {
                const int64_t grow = m0 + mh * kTileRows + lq * 32 + lane;
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
                            for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        }
                    }
                }
            }
            if (bad) record_status(p.status, FP9_ERR_RANGE);
        }
    }

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

// Token tiles of 128 * MH rows: MH = 2 halves the activation traffic per
// flop; MH = 1 keeps more CTAs when the grid would not fill the GPU.
// Picks the MH with fewer (waves x tile work).
int choose_mh(int64_t m, int64_t ntiles, int sms) {
    auto cost = [&](int mh) {
        const int64_t ctas = ntiles * ((m + kTileRows * mh - 1) / (kTileRows * mh));
        return ((ctas + sms - 1) / sms) * mh;
    };
    return cost(2) <= cost(1) ? 2 : 1;
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

fp9_status launch_gemm(bool down, PrefillArgs p, int sms, cudaStream_t stream) {
    const int mh = choose_mh(p.m, p.ntiles, sms);
    p.mtiles = static_cast<int32_t>((p.m + kTileRows * mh - 1) / (kTileRows * mh));
    const int64_t ctas = static_cast<int64_t>(p.mtiles) * p.ntiles;
    if (ctas > 0x7FFFFFFF) return FP9_ERR_SHAPE;
    void (*k)(const PrefillArgs) = down ? (mh == 2 ? prefill_kernel<true, 2> : prefill_kernel<true, 1>)
                                        : (mh == 2 ? prefill_kernel<false, 2> : prefill_kernel<false, 1>);
    const int smem = mh == 2 ? Cfg<2>::kSmem : Cfg<1>::kSmem;
    FP9_CUDA_TRY(launch_pdl(k, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), smem, stream, p));
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

    const size_t wg = static_cast<size_t>(index) * static_cast<size_t>(I) * static_cast<size_t>(H);
    PrefillArgs p{};
    p.act = x16;
    p.body[0] = ffn->gate_body + wg;
    p.sign[0] = ffn->gate_sign + wg / 8;
    p.body[1] = ffn->up_body + wg;
    p.sign[1] = ffn->up_sign + wg / 8;
    p.hidden = H;
    p.K = H;
    p.m = static_cast<int32_t>(m);
    p.ntiles = static_cast<int32_t>(I / kTileRows);
    p.out = h;
    p.ldo = I;
    p.status = d_status;
    p.timeout_ns = kTimeoutNs;
    st = launch_gemm(false, p, sms, s);
    if (st != FP9_OK) return st;

    p.act = h;
    p.body[0] = p.body[1] = ffn->down_body + wg;
    p.sign[0] = p.sign[1] = ffn->down_sign + wg / 8;
    p.K = I;
    p.ntiles = static_cast<int32_t>(H / (2 * kTileRows));
    p.out = y;
    p.ldo = H;
    return launch_gemm(true, p, sms, s);
}
