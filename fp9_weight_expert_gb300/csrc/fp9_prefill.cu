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
// Warp roles: warps 0-15 decode raw -> B (one 16-byte fp16 chunk of 8
// weights per task) and, in the dense launches, run the epilogue; warp 16
// issues the activation loads, warp 17 the raw weight loads (so the HBM
// weight stream runs ahead of the MMAs by up to the raw ring's depth), warp
// 18 one thread issues the MMAs and commits each A and B slot back through
// an mbarrier. The grouped (MoE) launches are persistent (one CTA per SM
// walking the tiles); the grouped down GEMM has 4 more warps, 19-22, that
// run the epilogue of one tile while the next one's MMAs run. gate/up weight rows
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
#include "fp9_prefill.h"
#include "fp9_tc.cuh"
#include "fp9moe.h"

namespace fp9 {
namespace {

constexpr int kTileRows = 128;                        // token rows of one MMA tile = TMEM lanes
constexpr int kChunkK = 64;                           // K per A / B slot: 128 bytes of fp16
constexpr int kRawK = 128;                            // K per raw slot (16 sign bytes per row)
constexpr int kTileBytes = kTileRows * kChunkK * 2;   // 16 KiB: one 128 x 64 fp16 activation tile
constexpr int kDecoderWarps = 16;
constexpr int kDecoderThreads = kDecoderWarps * 32;
constexpr int kActWarp = kDecoderWarps, kRawWarp = kDecoderWarps + 1, kMmaWarp = kDecoderWarps + 2;
constexpr int kThreads = (kDecoderWarps + 3) * 32;
// grouped prefill_kernel: epilogue warps (a multiple of 4: one or more per
// TMEM lane quarter) besides
constexpr int kEpiWarp0 = kDecoderWarps + 3, kEpiWarps = 4;
constexpr int kGroupedThreads = (kDecoderWarps + 3 + kEpiWarps) * 32;
constexpr int kGuThreads = (kDecoderWarps + 4) * 32;   // gate/up with weights in TMEM: two MMA warps
constexpr int kCtlBytes = 1024;
constexpr int kSmemMax = 227 * 1024;
constexpr int kGroupM = 8;                            // M tiles per CTA-order group
constexpr uint64_t kTimeoutNs = 1000000000ull;        // 1 s per wait
// Weight tile of a CTA: 2 x 128 rows = one N = 256 MMA operand.
//   gate/up: 128 rows of W_gate then 128 rows of W_up, K-major with the
//            128-byte swizzle (rows 128 B apart in 8-row groups of 1024 B);
//   down:    256 output columns of down_t, MN-major with the 128-byte
//            swizzle: atoms of 64 columns x 8 K rows (1024 B), the 4 atoms
//            of a K group 1024 B apart, 8-row K groups 4096 B apart.
// One M = 128, N = 256, K = 16 MMA per 16 K columns and 128 tokens: the
// tensor core takes about as long for N = 128 as for N = 256, so the two
// operands of a tile go through one instruction.
constexpr int kNR = 128;                              // weight rows per operand
constexpr int kBTile = kNR * 128;                     // 16 KiB: one operand, 64 K columns, fp16
constexpr int kBSlot = 2 * kBTile;                    // the N = 256 operand
constexpr int kRawBody = 256 * kNR;                   // 32 KiB of bodies per raw slot
constexpr int kRawSlot = 288 * kNR;                   // + 4 KiB of signs
constexpr int kTasks = 16 * kNR / kDecoderThreads;    // 4 decode tasks of 8 weights per thread per chunk
constexpr uint32_t kMnAtomStride = 1024;
constexpr uint32_t kMnGroupStride = 4096;

// Ring depths. 128-token tiles: three activation slots, two decoded slots,
// three raw slots (two in flight while one is decoded: four 64-wide chunks
// of weights). 256-token tiles (twice the MMA time per chunk): two of each.
// Split activations (kSplit: each activation is carried as two fp16 terms,
// hi + lo, and every weight chunk meets both, so a chunk has twice the MMA
// work): 128-token tiles whose activation slot holds the hi and the lo
// tile, two slots of each ring.
template <int MH, bool kSplit = false>
struct Cfg {
    static_assert(!kSplit || MH == 1, "split activations use 128-token tiles");
    static constexpr int kASlotBytes = (kSplit ? 2 : 1) * MH * kTileBytes;
    static constexpr int kASlots = (MH == 1 && !kSplit) ? 3 : 2;
    static constexpr int kBSlots = 2;
    static constexpr int kRawSlots = (MH == 1 && !kSplit) ? 3 : 2;
    static constexpr int kSmem = 1024 + kCtlBytes + kASlots * kASlotBytes + kBSlots * kBSlot + kRawSlots * kRawSlot;
    static_assert(kSmem <= kSmemMax, "shared memory");
};

// Split layout of an fp16 activation matrix with K columns: [rows, 2K],
// each 64-column chunk c of K stored as 128 columns, its hi terms in
// [128 c, 128 c + 64) and its lo terms in [128 c + 64, 128 c + 128), where
// hi = fp16(v) and lo = fp16(v - hi) (both round to nearest even). Column
// j's hi term:
__host__ __device__ __forceinline__ int64_t split_col(int64_t j) { return ((j >> 6) << 7) + (j & 63); }

struct Ctl {
    uint64_t a_full[8], a_empty[8];   // activation ring: TMA bytes / MMA commit
    uint64_t w_full[4], w_empty[4];   // raw ring: TMA bytes / the decoder warps
    uint64_t b_full[4], b_empty[4];   // decoded ring: the decoder warps / MMA commit
    uint64_t done;                    // every MMA of the CTA finished
    uint64_t acc_full[2], acc_empty[2];  // prefill_kernel: a tile's accumulator complete / read out
    uint32_t tmem;
    int abort;
    int never;
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

// 2-D tiled tensor maps (TMA descriptors) of one launch.
struct PrefillMaps {
    CUtensorMap act;       // fp16 [rows, K], box 64 x 128, 128-byte swizzle
    CUtensorMap body[2];   // gate/up: W_gate, W_up bodies, box 64 x 128; down: down_t, box 256 x 128
    CUtensorMap sign[2];   // the sign planes, box 16 x 128 (gate/up) or 32 x 128 (down)
    CUtensorMap body_sh[2];  // grouped launches: the same for the shared-expert bank
    CUtensorMap sign_sh[2];
};

struct PrefillArgs {
    int32_t m;               // tokens (rows of act and out)
    int32_t mtiles, ntiles;  // CTA tiles along tokens / output columns
    int32_t nk;              // K / 64
    int32_t wrow0;           // first weight row of the FFN in the planes
    void* out;               // gate/up: h fp16 [m, inter]; down: y fp32 [m, hidden]
    int64_t ldo;             // row stride of out (elements)
    int32_t* status;
    uint64_t timeout_ns;
    int32_t no_copy;         // failure self-test: the weight copies are not issued
    // grouped launches (GroupTableDev): token tile -> FFN and rows
    const int32_t* g_row;
    const int32_t* g_cnt;
    const int32_t* g_mtile;
    int32_t n_groups, n_routed;
    int32_t inter;           // weight rows per FFN
    // dense down: K split into ksplit parts (whole 128-column raw chunks),
    // part s written to out + s * part_stride (the caller adds the parts)
    int32_t ksplit;
    int64_t part_stride;
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
// Task u = t + 512 i of decoder thread t (4 per thread) is 8 weights:
//   gate/up: operand u / 1024, row (u / 8) mod 128, K columns 8 (u mod 8)
//            + [0, 8) -> chunk u mod 8 of tile row 128 * operand + row.
//            Raw bodies: [operand][half][row][64 B], signs [operand][row][16 B].
//   down:    K row u / 32, output columns 8 (u mod 32) + [0, 8) -> chunk
//            u mod 8 of atom (u / 8) mod 4. Raw bodies: [K row][256 B],
//            signs [K row][32 B].
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
            const uint2 w = ld_shared_v2(raw + b * (kNR * kRawK) + h * (kNR * 64) + row * 64u + c * 8u);
            const uint32_t s = ld_shared_u8(raw + kRawBody + b * (kNR * 16) + row * 16u + h * 8u + c);
            st_shared_v4(sB + b * kBTile + sw128_offset(row, c * 8u), decode8_half(w, s));
        } else {
            const uint32_t kr = u >> 5, c = u & 31u, rr = h * 64u + kr, x = kr & 7u;
            const uint2 w = ld_shared_v2(raw + rr * 256u + c * 8u);
            const uint32_t s = ld_shared_u8(raw + kRawBody + rr * 32u + c);
            const uint32_t dst = sB + (kr >> 3) * kMnGroupStride + (c >> 3) * kMnAtomStride + x * 128u +
                                 (((c & 7u) ^ x) << 4);
            st_shared_v4(dst, decode8_half(w, s));
        }
    }
}

// SiLU with the hardware exponential (a few ulp of fp32; h is then
// rounded to fp16, 2^-11 relative, so that error does not show).
__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

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

// A CTA tile: rows [arow0, arow0 + nvalid) of act and out (rows past
// nvalid are computed but not stored), output columns from n0, weight rows
// of its FFN from wrow0 in the routed or the shared planes.
struct Tile {
    int arow0, nvalid, n0, wrow0;
    int part, c0, nc;  // K part, its first 64-column chunk and its chunks
    bool shared_bank;
};

template <bool kDown, int MH, bool kGrouped>
__device__ __forceinline__ Tile tile_at(const PrefillArgs& p, int L) {
    Tile t;
    t.shared_bank = false;
    t.part = 0;
    t.c0 = 0;
    t.nc = p.nk;
    if (kGrouped) {
        const int q = L / p.ntiles, nt = L - q * p.ntiles;
        int lo = 0, hi = p.n_groups - 1;  // the last group whose first m-tile is <= q
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.g_mtile + mid) <= q) lo = mid;
            else hi = mid - 1;
        }
        const int mt = q - __ldg(p.g_mtile + lo);
        t.arow0 = __ldg(p.g_row + lo) + mt * kTileRows;
        t.nvalid = __ldg(p.g_cnt + lo) - mt * kTileRows;
        t.shared_bank = lo >= p.n_routed;
        t.wrow0 = (t.shared_bank ? lo - p.n_routed : lo) * p.inter;
        t.n0 = nt * (kDown ? 2 * kNR : kNR);
    } else {
        // K part s of the tile: raw chunks [s R / S, (s + 1) R / S) of R
        const int per_part = p.mtiles * p.ntiles;
        t.part = L / per_part;
        L -= t.part * per_part;
        const int nraw = p.nk / 2;
        t.c0 = 2 * (t.part * nraw / p.ksplit);
        t.nc = 2 * ((t.part + 1) * nraw / p.ksplit) - t.c0;
        int mt, nt;
        tile_of(L, p.mtiles, p.ntiles, mt, nt);
        t.arow0 = mt * kTileRows * MH;
        t.nvalid = p.m - t.arow0;
        t.wrow0 = p.wrow0;
        // output columns: 128 intermediate rows (gate/up) or 256 hidden columns (down)
        t.n0 = nt * (kDown ? 2 * kNR : kNR);
    }
    return t;
}

// CTA b takes tiles b, b + gridDim.x, ... The dense launches have one CTA
// per tile, and the decoder warps read the accumulator out once the tile's
// MMAs are done. The grouped launch (MoE experts: tiles of ~50 tokens and
// K = inter, each about 20 us of work) is persistent, one CTA per SM: the
// rings run on across tiles, so the next tile's loads and decoding start
// while the current tile's last MMAs run, two TMEM accumulators alternate,
// and the epilogue warps read tile j's while the MMAs of tile j + 1 fill the
// other. Timed per CTA, a one-tile grouped CTA spent 3.7 us before its
// first MMA, 2.4 us in its epilogue and 1 us between CTAs out of 25.9.
template <bool kDown, int MH, bool kGrouped, bool kSplit>
__global__ void __launch_bounds__(kGrouped ? kGroupedThreads : kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillMaps maps, const PrefillArgs p) {
    using C = Cfg<MH, kSplit>;
    static_assert(!kGrouped || MH == 1, "grouped tiles are 128 rows");
    constexpr int kAcc = kGrouped ? 2 : 1;                // accumulators
    constexpr uint32_t kAccCols = MH * 2 * kNR;           // TMEM columns of one
    int total;
    if (kGrouped) {
        grid_dependency_wait();  // the group table comes from the previous launches
        total = __ldg(p.g_mtile + p.n_groups) * p.ntiles;
    } else {
        total = p.mtiles * p.ntiles * p.ksplit;
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw0 = smem_addr(smem_raw);
    const uint32_t base = (raw0 + 1023u) & ~1023u;
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw + (base - raw0));
    const uint32_t ringA = base + kCtlBytes;                           // 1024-aligned slots
    const uint32_t ringB = ringA + C::kASlots * C::kASlotBytes;
    const uint32_t ringW = ringB + C::kBSlots * kBSlot;
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
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(smem_addr(&ctl.acc_full[a]), 1);
            mbar_init(smem_addr(&ctl.acc_empty[a]), kEpiWarps);
        }
        mbar_init(smem_addr(&ctl.done), 1);
        ctl.abort = 0;
        ctl.never = 0;
        fence_mbar_init();
    }
    if (warp == kActWarp && lane == 0) prefetch_map(&maps.act);
    if (warp == kRawWarp && lane == 0) {
        for (int b = 0; b < (kDown ? 1 : 2); ++b) {
            prefetch_map(&maps.body[b]);
            prefetch_map(&maps.sign[b]);
            if (kGrouped) {
                prefetch_map(&maps.body_sh[b]);
                prefetch_map(&maps.sign_sh[b]);
            }
        }
    }
    if (warp == 0) tc_alloc(smem_addr(&ctl.tmem), kAcc * kAccCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;

    // Reads tile t's accumulator `acc` out (TMEM lanes 32 (warp mod 4) +
    // [0, 32): the rows of this warp's lane quarter) for the column blocks
    // first, first + step, ...: gate/up 8 blocks of 16 intermediate columns
    // (h = SiLU(g) u rounded to fp16), down 8 blocks of 32 hidden columns.
    auto read_out = [&](const Tile& t, int acc, int first, int step, bool& bad) {
        const int lq = warp & 3;
        const uint32_t tl = tmem + acc * kAccCols + ((static_cast<uint32_t>(lq) * 32u) << 16);
#pragma unroll
        for (int mh = 0; mh < MH; ++mh) {
            const int r = mh * kTileRows + lq * 32 + lane;
            const int64_t grow = static_cast<int64_t>(t.arow0) + r;
            const bool valid = r < t.nvalid;
            if (!kDown) {
                __half* out = static_cast<__half*>(p.out) + t.part * p.part_stride + grow * p.ldo;
#pragma unroll 1
                for (int cb = first; cb < kNR / 16; cb += step) {
                    float g[16], u[16];
                    tc_ld16(tl + (mh * 2 + 0) * kNR + cb * 16, g);
                    tc_ld16(tl + (mh * 2 + 1) * kNR + cb * 16, u);
                    uint32_t hw[8], lw[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float h0 = silu(g[2 * i]) * u[2 * i], h1 = silu(g[2 * i + 1]) * u[2 * i + 1];
                        const __half2 h2 = __floats2half2_rn(h0, h1);
                        hw[i] = *reinterpret_cast<const uint32_t*>(&h2);
                        bad = bad || (valid && !half2_finite(hw[i]));
                        if (kSplit) {
                            const __half2 l2 = __floats2half2_rn(h0 - __low2float(h2), h1 - __high2float(h2));
                            lw[i] = *reinterpret_cast<const uint32_t*>(&l2);
                        }
                    }
                    if (valid) {
                        const int64_t col = t.n0 + cb * 16;  // 16 columns inside one 64-column chunk
                        uint4* o = reinterpret_cast<uint4*>(out + (kSplit ? split_col(col) : col));
                        o[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        o[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                        if (kSplit) {
                            uint4* ol = reinterpret_cast<uint4*>(out + split_col(col) + 64);
                            ol[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                            ol[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int jb = first; jb < 2 * kNR / 32; jb += step) {
                    const int b = jb / (kNR / 32), cb = jb % (kNR / 32);
                    float* out =
                        static_cast<float*>(p.out) + t.part * p.part_stride + grow * p.ldo + t.n0 + b * kNR + cb * 32;
                    float v[32];
                    tc_ld32(tl + (mh * 2 + b) * kNR + cb * 32, v);
                    if (valid) {
                        float4* o = reinterpret_cast<float4*>(out);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    }
                }
            }
        }
    };

    if (warp == kActWarp) {
        // -------------------------------------------- activation loads ---
        if (lane == 0) {
            if (!kGrouped) grid_dependency_wait();  // the activations come from the previous launch
            int ka = 0;  // chunks issued, over all tiles
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
                const Tile t = tile_at<kDown, MH, kGrouped>(p, L);
                for (int kc = 0; kc < t.nc; ++kc) {
                    const int s = ka % C::kASlots;
                    if (ka >= C::kASlots && !mbar_wait_bounded(smem_addr(&ctl.a_empty[s]), ((ka / C::kASlots) + 1) & 1,
                                                               p.timeout_ns, &ctl.abort)) {
                        fail(ctl, p.status);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_addr(&ctl.a_full[s]);
                    mbar_arrive_expect_tx(bar, C::kASlotBytes);
                    if (kSplit) {  // the chunk's hi tile, then its lo tile
                        tma_load_2d(ringA + s * C::kASlotBytes, &maps.act, (t.c0 + kc) * 2 * kChunkK, t.arow0, bar);
                        tma_load_2d(ringA + s * C::kASlotBytes + kTileBytes, &maps.act,
                                    (t.c0 + kc) * 2 * kChunkK + kChunkK, t.arow0, bar);
                    } else {
#pragma unroll
                        for (int mh = 0; mh < MH; ++mh)
                            tma_load_2d(ringA + s * C::kASlotBytes + mh * kTileBytes, &maps.act,
                                        (t.c0 + kc) * kChunkK, t.arow0 + mh * kTileRows, bar);
                    }
                    ++ka;
                }
            }
            // the copies this thread issued land before the CTA may exit
            for (int j = ka > C::kASlots ? ka - C::kASlots : 0; j < ka; ++j)
                (void)mbar_wait_bounded(smem_addr(&ctl.a_full[j % C::kASlots]), (j / C::kASlots) & 1, p.timeout_ns,
                                        &ctl.never);
        }
        __syncwarp();
    } else if (warp == kRawWarp) {
        // ------------------------------------------------ weight loads ---
        if (lane == 0) {
            int kw = 0;  // raw chunks of 128 K issued, over all tiles
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
                const Tile t = tile_at<kDown, MH, kGrouped>(p, L);
                const CUtensorMap* bmap = t.shared_bank ? maps.body_sh : maps.body;
                const CUtensorMap* smap = t.shared_bank ? maps.sign_sh : maps.sign;
                for (int kr = t.c0 / 2; kr < (t.c0 + t.nc) / 2; ++kr) {
                    const int s = kw % C::kRawSlots;
                    if (kw >= C::kRawSlots &&
                        !mbar_wait_bounded(smem_addr(&ctl.w_empty[s]), ((kw / C::kRawSlots) + 1) & 1, p.timeout_ns,
                                           &ctl.abort)) {
                        fail(ctl, p.status);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_addr(&ctl.w_full[s]);
                    const uint32_t slot = ringW + s * kRawSlot;
                    mbar_arrive_expect_tx(bar, kRawSlot);
                    if (p.no_copy) {
                        // the bytes never arrive: every wait on this slot runs out
                    } else if (!kDown) {
                        const int row = t.wrow0 + t.n0;
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            tma_load_2d(slot + b * (kNR * kRawK), &bmap[b], kr * kRawK, row, bar);
                            tma_load_2d(slot + b * (kNR * kRawK) + kNR * 64, &bmap[b], kr * kRawK + 64, row, bar);
                            tma_load_2d(slot + kRawBody + b * (kNR * 16), &smap[b], kr * (kRawK / 8), row, bar);
                        }
                    } else {
                        const int row = t.wrow0 + kr * kRawK;
                        tma_load_2d(slot, &bmap[0], t.n0, row, bar);
                        tma_load_2d(slot + kRawBody, &smap[0], t.n0 / 8, row, bar);
                    }
                    ++kw;
                }
            }
            for (int j = kw > C::kRawSlots ? kw - C::kRawSlots : 0; j < kw; ++j)
                (void)mbar_wait_bounded(smem_addr(&ctl.w_full[j % C::kRawSlots]), (j / C::kRawSlots) & 1, p.timeout_ns,
                                        &ctl.never);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA ---
        if (lane == 0) {
            const uint32_t idesc = tc_idesc_f16(kTileRows, 2 * kNR) | (kDown ? (1u << 16) : 0u);
            int kg = 0;  // chunks consumed, over all tiles
            bool ok = true;
            int j = 0;
            for (int L = blockIdx.x; L < total && ok; L += gridDim.x, ++j) {
                const int nc = tile_at<kDown, MH, kGrouped>(p, L).nc;
                const int acc = j % kAcc;
                // the accumulator's previous tile has been read out
                if (j >= kAcc && !mbar_wait_bounded(smem_addr(&ctl.acc_empty[acc]), ((j / kAcc) - 1) & 1,
                                                    p.timeout_ns, &ctl.abort)) {
                    fail(ctl, p.status);
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + acc * kAccCols;
                for (int kc = 0; kc < nc; ++kc, ++kg) {
                    const int sa = kg % C::kASlots, sb = kg % C::kBSlots;
                    if (!mbar_wait_bounded(smem_addr(&ctl.a_full[sa]), (kg / C::kASlots) & 1, p.timeout_ns,
                                           &ctl.abort) ||
                        !mbar_wait_bounded(smem_addr(&ctl.b_full[sb]), (kg / C::kBSlots) & 1, p.timeout_ns,
                                           &ctl.abort)) {
                        fail(ctl, p.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = ringA + sa * C::kASlotBytes;
                    const uint32_t sB = ringB + sb * kBSlot;
#pragma unroll
                    for (int k16 = 0; k16 < kChunkK / 16; ++k16) {
                        const uint64_t bd = kDown ? tc_desc_sw128_mn(sB + 2u * kMnGroupStride * k16, kMnAtomStride,
                                                                     kMnGroupStride)
                                                  : tc_desc_sw128(sB + 32u * k16);
                        if (kSplit) {  // the hi and the lo terms into the same accumulator
                            tc_mma_f16(d, tc_desc_sw128(sA + 32u * k16), bd, idesc, kc > 0 || k16 > 0);
                            tc_mma_f16(d, tc_desc_sw128(sA + kTileBytes + 32u * k16), bd, idesc, true);
                        } else {
#pragma unroll
                            for (int mh = 0; mh < MH; ++mh) {
                                const uint64_t ad = tc_desc_sw128(sA + mh * kTileBytes + 32u * k16);
                                tc_mma_f16(d + mh * 2 * kNR, ad, bd, idesc, kc > 0 || k16 > 0);
                            }
                        }
                    }
                    tc_commit(smem_addr(&ctl.a_empty[sa]));
                    tc_commit(smem_addr(&ctl.b_empty[sb]));
                }
                if (ok) tc_commit(smem_addr(&ctl.acc_full[acc]));
            }
            tc_commit(smem_addr(&ctl.done));
            // TMEM is freed only after every MMA of this CTA has finished
            if (!mbar_wait_bounded(smem_addr(&ctl.done), 0, p.timeout_ns, &ctl.never))
                record_status(p.status, FP9_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (kGrouped && warp >= kEpiWarp0) {
        // ----------------------------------------------------- epilogue ---
        // the warps of a lane quarter take alternate column blocks
        const int eh = (warp - kEpiWarp0) >> 2;
        bool bad = false;  // a stored h whose fp16 is not finite
        int j = 0;
        for (int L = blockIdx.x; L < total; L += gridDim.x, ++j) {
            const int acc = j % kAcc;
            if (!warp_wait(smem_addr(&ctl.acc_full[acc]), (j / kAcc) & 1, p.timeout_ns, &ctl.abort)) {
                if (lane == 0) fail(ctl, p.status);
                break;
            }
            tc_fence_after();
            read_out(tile_at<kDown, MH, kGrouped>(p, L), acc, eh, kEpiWarps / 4, bad);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl.acc_empty[acc]));
        }
        if (bad) record_status(p.status, FP9_ERR_RANGE);
    } else {
        // ----------------------------------------------------- decoders ---
        const int t = threadIdx.x;
        bool ok = true;
        int nchunks = 0;  // over all of this CTA's tiles
        for (int L = blockIdx.x; L < total; L += gridDim.x) nchunks += tile_at<kDown, MH, kGrouped>(p, L).nc;
        for (int kg = 0; kg < nchunks && ok; ++kg) {
            const int kw = kg >> 1, h = kg & 1;  // every tile has an even number of chunks
            const int sw = kw % C::kRawSlots, sb = kg % C::kBSlots;
            if (h == 0) ok = warp_wait(smem_addr(&ctl.w_full[sw]), (kw / C::kRawSlots) & 1, p.timeout_ns, &ctl.abort);
            if (ok && kg >= C::kBSlots)
                ok = warp_wait(smem_addr(&ctl.b_empty[sb]), ((kg / C::kBSlots) + 1) & 1, p.timeout_ns, &ctl.abort);
            if (!ok) break;
            decode_chunk<kDown>(t, ringW + sw * kRawSlot, h, ringB + sb * kBSlot);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_addr(&ctl.b_full[sb]));
                if (h == 1) mbar_arrive(smem_addr(&ctl.w_empty[sw]));
            }
        }
        if (!ok && lane == 0) fail(ctl, p.status);
        if (!kGrouped && ok && static_cast<int>(blockIdx.x) < total) {
            // one tile per CTA: the decoder warps read it out, four per
            // lane quarter on alternate column blocks
            bool bad = false;
            if (warp_wait(smem_addr(&ctl.acc_full[0]), 0, p.timeout_ns, &ctl.abort)) {
                tc_fence_after();
                read_out(tile_at<kDown, MH, kGrouped>(p, blockIdx.x), 0, warp >> 2, 4, bad);
            } else if (lane == 0) {
                fail(ctl, p.status);
            }
            if (bad) record_status(p.status, FP9_ERR_RANGE);
        }
    }

    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, kAcc * kAccCols);
}

// ---------------------------------------------- gate/up, weights in TMEM ---
//
// The gate/up GEMM with the roles of the operands swapped: the decoded
// weights are the MMA's A operand in tensor memory (M = 128 weight rows, two
// fp16 per 32-bit column, written by the decoder warps with tcgen05.st) and
// the tokens are N (the activation tile in shared memory). The decoded
// weights never go through shared memory, which otherwise carries ~5 bytes
// of traffic per weight byte (raw in, raw out, fp16 in, fp16 out to the
// tensor core) and bounds the kernel; and the MMA's N is the tile's valid
// tokens rounded up to 16, so its work follows the tokens an FFN has.
//
// One CTA: 128 intermediate rows of W_gate and of W_up x up to 128 tokens.
// TMEM (512 columns): D_gate [0, 128), D_up [128, 256) (lane = weight row,
// column = token), then 4 slots of decoded weights of 64 K columns: gate in
// the first 32 columns, up in the next 32.
// Split activations: up to 64 tokens per tile; an activation slot holds
// the tile's hi rows (slot rows [0, 64)) and its lo rows (rows [64, 128)),
// and one MMA of N = 64 + the valid tokens rounded up to 16 takes both, so
// D column c < 64 is token c's hi part and column 64 + c its lo part
// (added in the epilogue): the same MMA count as with one fp16 term.
constexpr int kGuTokens = 128;
constexpr int kGuTokensSplit = 64;
constexpr int kGuActSlots = 4, kGuRawSlots = 4, kGuWSlots = 4;
constexpr int kGuActSlot = kGuTokens * kChunkK * 2;  // 16 KiB
constexpr int kGuSmem = 1024 + kCtlBytes + kGuActSlots * kGuActSlot + kGuRawSlots * kRawSlot;
constexpr uint32_t kGuWCol0 = 256;
static_assert(kGuSmem <= kSmemMax, "shared memory");

// Decodes the 32 weights of K half `kh` of chunk half `h` of weight row
// `row` of operand `b` in raw slot `raw` into 16 columns of half2 (low half
// the even K). Raw bodies: [operand][row][128 B] with the 128-byte swizzle
// (16-byte chunk j of row r at j ^ (r mod 8): the 8 rows a quarter warp
// reads fall in 8 bank groups); signs [operand][row][16 B].
__device__ __forceinline__ void decode_row32(uint32_t raw, uint32_t b, uint32_t row, uint32_t h, uint32_t kh,
                                             uint32_t (&r)[16]) {
    const uint32_t j0 = 4u * h + 2u * kh, x = row & 7u;
    const uint32_t rb = raw + b * (kNR * kRawK) + row * kRawK;
    uint4 v[2];
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0].x), "=r"(v[0].y), "=r"(v[0].z), "=r"(v[0].w)
                 : "r"(rb + ((j0 ^ x) << 4))
                 : "memory");
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[1].x), "=r"(v[1].y), "=r"(v[1].z), "=r"(v[1].w)
                 : "r"(rb + (((j0 + 1u) ^ x) << 4))
                 : "memory");
    uint32_t s32;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(s32) : "r"(raw + kRawBody + b * (kNR * 16) + row * 16u + 8u * h + 4u * kh)
                 : "memory");
    const uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) fp9_to_half4(w[i], spread_sign_nibble((s32 >> (4 * i)) & 0xFu), r[2 * i], r[2 * i + 1]);
}

// A grouped gate/up tile: rows [arow0, arow0 + nvalid) of act (tokens of
// one FFN), intermediate rows n0 + [0, 128) of that FFN's W_gate and W_up
// (weight rows from wrow0 in the routed or the shared planes), and the MMA's
// N: the valid tokens rounded up to 16.
struct GuTile {
    int arow0, nvalid, n0, wrow0;
    uint32_t n_mma;
    bool shared_bank;
};

// With split activations each 128-row m-tile of the group table is two
// 64-token tiles (the second one empty, nvalid <= 0, when the m-tile holds
// at most 64 tokens; every role skips empty tiles alike).
template <bool kSplit>
__device__ __forceinline__ GuTile gu_tile_at(const PrefillArgs& p, int L) {
    constexpr int kT = kSplit ? kGuTokensSplit : kGuTokens;
    constexpr int kPer = kPrefillTileRows / kT;
    GuTile t;
    const int qq = L / p.ntiles, nt = L - qq * p.ntiles;
    const int q = qq / kPer, half = qq - q * kPer;
    int lo = 0, hi = p.n_groups - 1;  // the last group whose first m-tile is <= q
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.g_mtile + mid) <= q) lo = mid;
        else hi = mid - 1;
    }
    const int mt = q - __ldg(p.g_mtile + lo);
    t.arow0 = __ldg(p.g_row + lo) + mt * kPrefillTileRows + half * kT;
    t.nvalid = __ldg(p.g_cnt + lo) - mt * kPrefillTileRows - half * kT;
    t.shared_bank = lo >= p.n_routed;
    t.wrow0 = (t.shared_bank ? lo - p.n_routed : lo) * p.inter;
    t.n0 = nt * kNR;
    const uint32_t n16 = static_cast<uint32_t>((max(min(t.nvalid, kT), 0) + 15) / 16 * 16);
    t.n_mma = kSplit ? kT + n16 : n16;
    return t;
}

// Persistent over the group table's tiles (CTA b: tiles b, b + gridDim.x,
// ...): the rings run on across tiles, so the next tile's activation and
// weight loads land while the current tile's MMAs and epilogue run. D (both
// accumulators) is read out by the decoder warps after the tile's last
// MMA; the next tile's MMAs wait until it has been (acc_empty).
template <bool kGrouped, bool kSplit>
__global__ void __launch_bounds__(kGuThreads, 1) gateup_kernel(const __grid_constant__ PrefillMaps maps,
                                                             const PrefillArgs p) {
    static_assert(kGrouped, "the gate/up kernel with weights in TMEM serves the grouped launch");
    grid_dependency_wait();  // the group table comes from the previous launches
    const int total = __ldg(p.g_mtile + p.n_groups) * p.ntiles * (kSplit ? kPrefillTileRows / kGuTokensSplit : 1);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw0 = smem_addr(smem_raw);
    const uint32_t base = (raw0 + 1023u) & ~1023u;
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw + (base - raw0));
    const uint32_t ringA = base + kCtlBytes;
    const uint32_t ringW = ringA + kGuActSlots * kGuActSlot;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGuActSlots; ++s) {
            mbar_init(smem_addr(&ctl.a_full[s]), 1);
            mbar_init(smem_addr(&ctl.a_empty[s]), 2);
        }
        for (int s = 0; s < kGuRawSlots; ++s) {
            mbar_init(smem_addr(&ctl.w_full[s]), 1);
            mbar_init(smem_addr(&ctl.w_empty[s]), kDecoderWarps);
        }
        for (int s = 0; s < kGuWSlots; ++s) {  // decoded weights in TMEM
            mbar_init(smem_addr(&ctl.b_full[s]), kDecoderWarps);
            mbar_init(smem_addr(&ctl.b_empty[s]), 2);
        }
        mbar_init(smem_addr(&ctl.acc_full[0]), 2);                 // both MMA warps' commits of a tile
        mbar_init(smem_addr(&ctl.acc_empty[0]), kDecoderWarps);    // D read out
        mbar_init(smem_addr(&ctl.done), 2);
        ctl.abort = 0;
        ctl.never = 0;
        fence_mbar_init();
    }
    if (warp == kActWarp && lane == 0) prefetch_map(&maps.act);
    if (warp == kRawWarp && lane == 0) {
        for (int b = 0; b < 2; ++b) {
            prefetch_map(&maps.body[b]);
            prefetch_map(&maps.sign[b]);
            prefetch_map(&maps.body_sh[b]);
            prefetch_map(&maps.sign_sh[b]);
        }
    }
    if (warp == 0) tc_alloc(smem_addr(&ctl.tmem), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    const int nk = p.nk;

    if (warp == kActWarp) {
        // -------------------------------------------- activation loads ---
        if (lane == 0) {
            int ka = 0;  // chunks issued, over all tiles
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
                const GuTile t = gu_tile_at<kSplit>(p, L);
                if (t.nvalid <= 0) continue;
                for (int kc = 0; kc < nk; ++kc) {
                    const int s = ka % kGuActSlots;
                    if (ka >= kGuActSlots &&
                        !mbar_wait_bounded(smem_addr(&ctl.a_empty[s]), ((ka / kGuActSlots) + 1) & 1, p.timeout_ns,
                                           &ctl.abort)) {
                        fail(ctl, p.status);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_addr(&ctl.a_full[s]);
                    mbar_arrive_expect_tx(bar, kGuActSlot);
                    if (kSplit) {  // 64 hi rows, then 64 lo rows (boxes of 64 rows)
                        tma_load_2d(ringA + s * kGuActSlot, &maps.act, kc * 2 * kChunkK, t.arow0, bar);
                        tma_load_2d(ringA + s * kGuActSlot + kGuTokensSplit * 128, &maps.act, kc * 2 * kChunkK + kChunkK,
                                    t.arow0, bar);
                    } else {
                        tma_load_2d(ringA + s * kGuActSlot, &maps.act, kc * kChunkK, t.arow0, bar);
                    }
                    ++ka;
                }
            }
            for (int j = ka > kGuActSlots ? ka - kGuActSlots : 0; j < ka; ++j)
                (void)mbar_wait_bounded(smem_addr(&ctl.a_full[j % kGuActSlots]), (j / kGuActSlots) & 1, p.timeout_ns,
                                        &ctl.never);
        }
        __syncwarp();
    } else if (warp == kRawWarp) {
        // ------------------------------------------------ weight loads ---
        if (lane == 0) {
            int kw = 0;  // raw chunks issued, over all tiles
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
                const GuTile t = gu_tile_at<kSplit>(p, L);
                if (t.nvalid <= 0) continue;
                const CUtensorMap* bmap = t.shared_bank ? maps.body_sh : maps.body;
                const CUtensorMap* smap = t.shared_bank ? maps.sign_sh : maps.sign;
                for (int kr = 0; kr < nk / 2; ++kr) {
                    const int s = kw % kGuRawSlots;
                    if (kw >= kGuRawSlots &&
                        !mbar_wait_bounded(smem_addr(&ctl.w_empty[s]), ((kw / kGuRawSlots) + 1) & 1, p.timeout_ns,
                                           &ctl.abort)) {
                        fail(ctl, p.status);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_addr(&ctl.w_full[s]);
                    const uint32_t slot = ringW + s * kRawSlot;
                    mbar_arrive_expect_tx(bar, kRawSlot);
                    const int row = t.wrow0 + t.n0;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        tma_load_2d(slot + b * (kNR * kRawK), &bmap[b], kr * kRawK, row, bar);
                        tma_load_2d(slot + kRawBody + b * (kNR * 16), &smap[b], kr * (kRawK / 8), row, bar);
                    }
                    ++kw;
                }
            }
            for (int j = kw > kGuRawSlots ? kw - kGuRawSlots : 0; j < kw; ++j)
                (void)mbar_wait_bounded(smem_addr(&ctl.w_full[j % kGuRawSlots]), (j / kGuRawSlots) & 1, p.timeout_ns,
                                        &ctl.never);
        }
        __syncwarp();
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // ---------------------------------------------------------- MMA ---
        // warp kMmaWarp issues the gate MMAs, the next warp the up MMAs (one
        // issuing thread is part of the per-instruction cost); each commits
        // its own, so every slot, acc_full and `done` take two arrivals
        const uint32_t ob = static_cast<uint32_t>(warp - kMmaWarp);
        if (lane == 0) {
            int kg = 0, j = 0;  // chunks and tiles consumed
            bool ok = true;
            for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
                const GuTile t = gu_tile_at<kSplit>(p, L);
                if (t.nvalid <= 0) continue;
                const uint32_t idesc = tc_idesc_f16(kTileRows, t.n_mma);
                // the previous tile's D has been read out
                if (j > 0 && !mbar_wait_bounded(smem_addr(&ctl.acc_empty[0]), (j - 1) & 1, p.timeout_ns, &ctl.abort)) {
                    fail(ctl, p.status);
                    break;
                }
                tc_fence_after();
                for (int kc = 0; kc < nk; ++kc, ++kg) {
                    const int sa = kg % kGuActSlots, sw = kg % kGuWSlots;
                    if (!mbar_wait_bounded(smem_addr(&ctl.a_full[sa]), (kg / kGuActSlots) & 1, p.timeout_ns,
                                           &ctl.abort) ||
                        !mbar_wait_bounded(smem_addr(&ctl.b_full[sw]), (kg / kGuWSlots) & 1, p.timeout_ns,
                                           &ctl.abort)) {
                        fail(ctl, p.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = ringA + sa * kGuActSlot;
                    const uint32_t wcol = tmem + kGuWCol0 + sw * 64u;
#pragma unroll
                    for (int k16 = 0; k16 < kChunkK / 16; ++k16) {
                        const uint64_t bd = tc_desc_sw128(sA + 32u * k16);
                        tc_mma_f16_tmem_a(tmem + ob * kNR, wcol + ob * 32u + 8u * k16, bd, idesc, kc > 0 || k16 > 0);
                    }
                    tc_commit(smem_addr(&ctl.a_empty[sa]));
                    tc_commit(smem_addr(&ctl.b_empty[sw]));
                }
                if (ok) tc_commit(smem_addr(&ctl.acc_full[0]));
                ++j;
            }
            tc_commit(smem_addr(&ctl.done));
            if (!mbar_wait_bounded(smem_addr(&ctl.done), 0, p.timeout_ns, &ctl.never))
                record_status(p.status, FP9_ERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- decoders ---
        // warp w writes TMEM lanes 32 (w mod 4) + [0, 32): weight row
        // 32 (w mod 4) + lane of operand (w / 8) (0 gate, 1 up), K half
        // (w / 4) mod 2 of each 64-wide chunk
        const uint32_t q = warp & 3, sel = warp >> 2, b = sel >> 1, kh = sel & 1;
        const uint32_t row = 32u * q + lane;
        const uint32_t tlane = tmem + ((32u * q) << 16);
        bool ok = true, bad = false;
        int kw = 0, j = 0;  // raw chunks and tiles, over all tiles
        for (int L = blockIdx.x; L < total && ok; L += gridDim.x) {
            const GuTile t = gu_tile_at<kSplit>(p, L);
            if (t.nvalid <= 0) continue;
            // both 64-wide chunks of a raw slot per iteration: two TMEM
            // stores, then one wait for their completion
            for (int kr = 0; kr < nk / 2 && ok; ++kr, ++kw) {
                const int sr = kw % kGuRawSlots;
                const int kc0 = 2 * kw, sw0 = kc0 % kGuWSlots, sw1 = (kc0 + 1) % kGuWSlots;
                ok = warp_wait(smem_addr(&ctl.w_full[sr]), (kw / kGuRawSlots) & 1, p.timeout_ns, &ctl.abort);
                if (ok && kc0 >= kGuWSlots)
                    ok = warp_wait(smem_addr(&ctl.b_empty[sw0]), ((kc0 / kGuWSlots) + 1) & 1, p.timeout_ns,
                                   &ctl.abort);
                if (ok && kc0 + 1 >= kGuWSlots)
                    ok = warp_wait(smem_addr(&ctl.b_empty[sw1]), (((kc0 + 1) / kGuWSlots) + 1) & 1, p.timeout_ns,
                                   &ctl.abort);
                if (!ok) break;
                const uint32_t raw = ringW + sr * kRawSlot;
                uint32_t r[16];
                decode_row32(raw, b, row, 0, kh, r);
                tc_st16(tlane + kGuWCol0 + sw0 * 64u + b * 32u + kh * 16u, r);
                decode_row32(raw, b, row, 1, kh, r);
                tc_st16(tlane + kGuWCol0 + sw1 * 64u + b * 32u + kh * 16u, r);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_addr(&ctl.b_full[sw0]));
                    mbar_arrive(smem_addr(&ctl.b_full[sw1]));
                    mbar_arrive(smem_addr(&ctl.w_empty[sr]));
                }
            }
            if (!ok) break;
            // ------------------------------------------------- epilogue ---
            // warp w: weight rows 32 (w mod 4) + [0, 32), tokens 32 (w / 4)
            // + [0, 32); h[token, n0 + row] = SiLU(gate) * up, 32 lanes
            // writing 32 consecutive intermediate columns of a token row
            ok = warp_wait(smem_addr(&ctl.acc_full[0]), j & 1, p.timeout_ns, &ctl.abort);
            ++j;
            if (!ok) break;
            tc_fence_after();
            const int cb = static_cast<int>(sel);
            float g[32], u[32];
            if (!kSplit) {
                tc_ld32(tlane + cb * 32, g);
                tc_ld32(tlane + kNR + cb * 32, u);
            } else if (cb < 2) {  // tokens 32 cb + [0, 32): hi part + lo part
                tc_ld32(tlane + cb * 32, g);
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    float a[16];
                    tc_ld16(tlane + kGuTokensSplit + cb * 32 + hb * 16, a);
#pragma unroll
                    for (int i = 0; i < 16; ++i) g[hb * 16 + i] += a[i];
                }
                tc_ld32(tlane + kNR + cb * 32, u);
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    float a[16];
                    tc_ld16(tlane + kNR + kGuTokensSplit + cb * 32 + hb * 16, a);
#pragma unroll
                    for (int i = 0; i < 16; ++i) u[hb * 16 + i] += a[i];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&ctl.acc_empty[0]));  // D may be overwritten now
            if (kSplit && cb >= 2) continue;
            const int64_t col = t.n0 + row;
            __half* out = static_cast<__half*>(p.out) + (kSplit ? split_col(col) : col);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int tk = cb * 32 + i;
                if (tk < t.nvalid) {
                    const float hf = silu(g[i]) * u[i];
                    const __half hv = __float2half_rn(hf);
                    bad = bad || __hisinf(hv) || __hisnan(hv);
                    __half* o = out + (static_cast<int64_t>(t.arow0) + tk) * p.ldo;
                    o[0] = hv;
                    if (kSplit) o[64] = __float2half_rn(hf - __half2float(hv));
                }
            }
        }
        if (!ok && lane == 0) fail(ctl, p.status);
        if (bad) record_status(p.status, FP9_ERR_RANGE);
    }

    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, 512);
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

// x fp32 [rows, H] -> the split layout [rows, 2H] (hi = fp16(v), lo =
// fp16(v - hi), both round to nearest even); a value whose hi is not
// finite is recorded as FP9_ERR_RANGE. H4 = H / 4; four consecutive
// columns stay inside one 64-column chunk.
__global__ void to_half_split_kernel(const float4* __restrict__ x, __half* __restrict__ h, int64_t n4, int64_t H4,
                                     int32_t* status) {
    grid_dependency_wait();
    grid_launch_dependents();
    bool finite = true;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 v = x[i];
        const int64_t r = i / H4, c = 4 * (i - r * H4);
        const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        const __half2 la = __floats2half2_rn(v.x - __low2float(a), v.y - __high2float(a));
        const __half2 lb = __floats2half2_rn(v.z - __low2float(b), v.w - __high2float(b));
        uint2 o, l;
        o.x = *reinterpret_cast<const uint32_t*>(&a);
        o.y = *reinterpret_cast<const uint32_t*>(&b);
        l.x = *reinterpret_cast<const uint32_t*>(&la);
        l.y = *reinterpret_cast<const uint32_t*>(&lb);
        finite = finite && half2_finite(o.x) && half2_finite(o.y);
        __half* dst = h + r * 8 * H4 + split_col(c);
        *reinterpret_cast<uint2*>(dst) = o;
        *reinterpret_cast<uint2*>(dst + 64) = l;
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
// the MH with fewer (waves x tile work), counting a 256-token tile as 1.8
// of a 128-token one.
int choose_mh(int64_t m, int64_t ntiles, int sms) {
    auto waves = [&](int mh) {
        const int64_t ctas = ntiles * ((m + kTileRows * mh - 1) / (kTileRows * mh));
        return static_cast<double>((ctas + sms - 1) / sms);
    };
    return waves(2) * 1.8 <= waves(1) ? 2 : 1;
}

template <bool kDown, int MH, bool kGrouped, bool kSplit>
cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(prefill_kernel<kDown, MH, kGrouped, kSplit>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<MH, kSplit>::kSmem);
}

fp9_status ensure_attrs() {
    static DeviceOnce attr;
    return attr.run([] {
        const int optin = device_max_smem_optin();
        if (optin < Cfg<1>::kSmem || optin < Cfg<2>::kSmem) return FP9_ERR_CUDA;
        if (optin < Cfg<1, true>::kSmem || optin < kGuSmem) return FP9_ERR_CUDA;
        FP9_CUDA_TRY((set_smem_attr<false, 1, false, false>()));
        FP9_CUDA_TRY((set_smem_attr<false, 2, false, false>()));
        FP9_CUDA_TRY((set_smem_attr<true, 1, false, false>()));
        FP9_CUDA_TRY((set_smem_attr<true, 2, false, false>()));
        FP9_CUDA_TRY((set_smem_attr<true, 1, true, false>()));
        FP9_CUDA_TRY((set_smem_attr<false, 1, false, true>()));
        FP9_CUDA_TRY((set_smem_attr<true, 1, false, true>()));
        FP9_CUDA_TRY((set_smem_attr<true, 1, true, true>()));
        FP9_CUDA_TRY((cudaFuncSetAttribute(gateup_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kGuSmem)));
        FP9_CUDA_TRY((cudaFuncSetAttribute(gateup_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kGuSmem)));
        return FP9_OK;
    });
}

// Tensor maps of one weight bank for a GEMM: gate/up read the bodies in
// boxes of 64 K columns x 128 rows and the signs 128 K columns at a time;
// down reads down_t in boxes of 256 output columns x 128 K rows.
bool make_weight_maps(bool down, const uint8_t* const body[2], const uint8_t* const sign[2], int64_t plane_rows,
                      int64_t hidden, CUtensorMap* bmaps, CUtensorMap* smaps) {
    for (int b = 0; b < (down ? 1 : 2); ++b) {
        if (!make_map(&bmaps[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, body[b], static_cast<uint64_t>(hidden),
                      static_cast<uint64_t>(plane_rows), static_cast<uint64_t>(hidden), down ? 2 * kNR : 64,
                      down ? kRawK : kNR, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map(&smaps[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, sign[b], static_cast<uint64_t>(hidden / 8),
                      static_cast<uint64_t>(plane_rows), static_cast<uint64_t>(hidden / 8),
                      down ? 2 * kNR / 8 : kRawK / 8, down ? kRawK : kNR, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
    }
    if (down) {
        bmaps[1] = bmaps[0];
        smaps[1] = smaps[0];
    }
    return true;
}

// Tensor maps of the W_gate and W_up planes for gate/up with weights in
// TMEM: bodies in boxes of 128 K columns x 128 rows with the 128-byte
// swizzle, signs in boxes of 16 bytes x 128 rows.
bool make_gateup_maps(const uint8_t* const body[2], const uint8_t* const sign[2], int64_t plane_rows, int64_t hidden,
                      CUtensorMap* bmaps, CUtensorMap* smaps) {
    for (int b = 0; b < 2; ++b) {
        if (!make_map(&bmaps[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, body[b], static_cast<uint64_t>(hidden),
                      static_cast<uint64_t>(plane_rows), static_cast<uint64_t>(hidden), kRawK, kNR,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&smaps[b], CU_TENSOR_MAP_DATA_TYPE_UINT8, sign[b], static_cast<uint64_t>(hidden / 8),
                      static_cast<uint64_t>(plane_rows), static_cast<uint64_t>(hidden / 8), kRawK / 8, kNR,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
    }
    return true;
}

// Activations fp16 [rows, cols] (cols = K, or 2K in the split layout),
// boxes of 64 columns x box_rows rows with the 128-byte swizzle.
bool make_act_map(CUtensorMap* map, const __half* act, int64_t rows, int64_t cols, uint32_t box_rows = kTileRows) {
    return make_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, act, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                    static_cast<uint64_t>(cols) * 2, kChunkK, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

PrefillArgs base_args(int64_t m, int64_t K, int32_t ntiles, void* out, int64_t ldo, int32_t* status) {
    PrefillArgs p{};
    p.m = static_cast<int32_t>(m);
    p.ntiles = ntiles;
    p.nk = static_cast<int32_t>(K / kChunkK);
    p.out = out;
    p.ldo = ldo;
    p.status = status;
    p.timeout_ns = kTimeoutNs;
    p.ksplit = 1;
    p.part_stride = 0;
    return p;
}

// Token-tile height (MH) and K parts of the dense down GEMM: the fewest
// rounds of CTAs times one tile's time, plus the pass that adds the parts.
// A 256-token tile of 256 columns and K takes about 2 K 256^2 / 9.2e12 s on
// one SM (the measured ~1.4 PFLOP/s over 152 SMs), a 128-token tile about
// 1 / 1.8 of that, and every CTA spends about 5 us outside its main loop
// (start and epilogue, timed per CTA); adding S parts reads S planes and
// writes one at about 6.5 TB/s. A plan replaces the one before it only when
// it is 3 % cheaper.
// Without a device (sms <= 0): one part, MH from choose_mh.
constexpr int kMaxDownSplits = 4;

struct DownPlan {
    int mh, splits;
};

DownPlan plan_down(int64_t m, int64_t H, int64_t I, int sms, bool split) {
    const int64_t ntiles = H / (2 * kNR);
    if (sms <= 0) return DownPlan{split ? 1 : choose_mh(m, ntiles, 1), 1};
    DownPlan best{1, 1};
    double best_cost = 1e300;
    for (int mh = 1; mh <= (split ? 1 : 2); ++mh) {
        const int64_t mt = (m + kTileRows * mh - 1) / (kTileRows * mh);
        for (int sp = 1; sp <= kMaxDownSplits && sp <= I / kRawK; ++sp) {
            const int64_t ctas = mt * ntiles * sp;
            const double rounds = static_cast<double>((ctas + sms - 1) / sms);
            const double tile =
                (split ? 2.0 : 1.0) * 2.0 * static_cast<double>(I) / sp * 65536.0 / 9.2e12 / (mh == 2 ? 1.0 : 1.8);
            const double sum = sp > 1 ? (sp + 1.0) * static_cast<double>(m) * static_cast<double>(H) * 4.0 / 6.5e12 : 0.0;
            const double cost = rounds * (tile + 5e-6) + sum;
            if (cost < 0.97 * best_cost) {
                best_cost = cost;
                best = DownPlan{mh, sp};
            }
        }
    }
    return best;
}

// y = the K parts of the dense down GEMM added in part order (fp32):
// parts [nparts][n4] float4, y [n4] float4.
__global__ void __launch_bounds__(256) sum_parts_kernel(const float4* __restrict__ parts, int64_t n4, int32_t nparts,
                                                        float4* __restrict__ y) {
    grid_dependency_wait();  // every part is written
    grid_launch_dependents();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 a = __ldcs(parts + i);
        for (int sp = 1; sp < nparts; ++sp) {
            const float4 b = __ldcs(parts + sp * n4 + i);
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        y[i] = a;
    }
}

// One GEMM launch: activations act [m, K] fp16; weight rows [wrow0, ...)
// of planes with plane_rows rows of `hidden` columns (gate/up: body/sign
// [0..1] = W_gate, W_up, `ncols` = inter output columns; down:
// body/sign[0] = down_t, `ncols` = hidden). A down GEMM whose plan splits K
// writes its parts to `parts` ([splits, m, ncols] fp32) and adds them into
// out (ldo == ncols) with a second launch.
fp9_status launch_gemm(bool down, bool split, const __half* act, int64_t m, int64_t K, const uint8_t* const body[2],
                       const uint8_t* const sign[2], int64_t plane_rows, int64_t hidden, int64_t wrow0, int64_t ncols,
                       void* out, int64_t ldo, float* parts, int32_t* status, int sms, cudaStream_t stream) {
    const int32_t ntiles = static_cast<int32_t>(ncols / (down ? 2 * kNR : kNR));
    PrefillMaps maps;
    if (!make_act_map(&maps.act, act, m, split ? 2 * K : K) ||
        !make_weight_maps(down, body, sign, plane_rows, hidden, maps.body, maps.sign))
        return FP9_ERR_CUDA;
    maps.body_sh[0] = maps.body_sh[1] = maps.body[0];
    maps.sign_sh[0] = maps.sign_sh[1] = maps.sign[0];
    PrefillArgs p = base_args(m, K, ntiles, out, ldo, status);
    p.wrow0 = static_cast<int32_t>(wrow0);
    const DownPlan plan = down ? plan_down(m, ncols, K, sms, split) : DownPlan{split ? 1 : choose_mh(m, ntiles, sms), 1};
    const int mh = plan.mh;
    if (plan.splits > 1) {
        if (parts == nullptr || ldo != ncols) return FP9_ERR_WORKSPACE;
        p.out = parts;
        p.ksplit = plan.splits;
        p.part_stride = m * ncols;
    }
    p.mtiles = static_cast<int32_t>((m + kTileRows * mh - 1) / (kTileRows * mh));
    const int64_t ctas = static_cast<int64_t>(p.mtiles) * p.ntiles * p.ksplit;  // one CTA per tile and K part
    if (ctas > 0x7FFFFFFF) return FP9_ERR_SHAPE;
    void (*k)(const PrefillMaps, const PrefillArgs) =
        split ? (down ? prefill_kernel<true, 1, false, true> : prefill_kernel<false, 1, false, true>)
        : down ? (mh == 2 ? prefill_kernel<true, 2, false, false> : prefill_kernel<true, 1, false, false>)
               : (mh == 2 ? prefill_kernel<false, 2, false, false> : prefill_kernel<false, 1, false, false>);
    const int smem = split ? Cfg<1, true>::kSmem : mh == 2 ? Cfg<2>::kSmem : Cfg<1>::kSmem;
    FP9_CUDA_TRY(launch_pdl(k, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), smem, stream, maps, p));
    if (plan.splits > 1) {
        const int64_t n4 = m * ncols / 4;
        const int64_t blocks = (n4 + 255) / 256 < static_cast<int64_t>(sms) * 8 ? (n4 + 255) / 256 : sms * 8;
        FP9_CUDA_TRY(launch_pdl(sum_parts_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                                reinterpret_cast<const float4*>(parts), n4, plan.splits, static_cast<float4*>(out)));
    }
    return FP9_OK;
}

struct PrefillLayout {
    size_t off_x16 = 0, off_h = 0, off_parts = 0, total = 0;
};

// x and h in the split layout (two fp16 terms per value; the one-term
// mode uses the first half of each), then the K parts of the down GEMM
// when either mode's plan splits K (sms: the device's SMs; <= 0: no split).
PrefillLayout prefill_layout(int64_t m, int64_t hidden, int64_t inter, int sms) {
    PrefillLayout L;
    L.off_x16 = 0;
    L.off_h = align_up(2 * sizeof(__half) * static_cast<size_t>(m) * static_cast<size_t>(hidden));
    L.off_parts = L.off_h + align_up(2 * sizeof(__half) * static_cast<size_t>(m) * static_cast<size_t>(inter));
    int splits = plan_down(m, hidden, inter, sms, false).splits;
    const int s2 = plan_down(m, hidden, inter, sms, true).splits;
    if (s2 > splits) splits = s2;
    L.total = L.off_parts + (splits > 1 ? align_up(sizeof(float) * static_cast<size_t>(splits) *
                                                    static_cast<size_t>(m) * static_cast<size_t>(hidden))
                                        : 0);
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

fp9_status launch_grouped_ffn(const fp9_ffn_bank& routed, const fp9_ffn_bank* shared, const GroupTableDev& tab,
                              int64_t max_mtiles, const __half* x16, __half* h, float* y, int64_t rows, bool split,
                              int32_t* status, int sms, cudaStream_t stream) {
    const int64_t H = routed.hidden, I = routed.inter;
    if (max_mtiles <= 0 || rows <= 0) return FP9_OK;
    fp9_status st = ensure_attrs();
    if (st != FP9_OK) return st;
    for (int pass = 0; pass < 2; ++pass) {
        const bool down = pass == 1;
        PrefillMaps maps;
        const uint8_t* rb[2] = {down ? routed.down_body : routed.gate_body, down ? routed.down_body : routed.up_body};
        const uint8_t* rs[2] = {down ? routed.down_sign : routed.gate_sign, down ? routed.down_sign : routed.up_sign};
        auto maps_of = [&](const uint8_t* const bb[2], const uint8_t* const ss[2], int64_t rows_, CUtensorMap* bm,
                           CUtensorMap* sm) {
            return down ? make_weight_maps(true, bb, ss, rows_, H, bm, sm) : make_gateup_maps(bb, ss, rows_, H, bm, sm);
        };
        const int64_t K = down ? I : H;
        // split gate/up tiles load 64 hi rows and 64 lo rows
        const uint32_t box_rows = (split && !down) ? kGuTokensSplit : kTileRows;
        if (!make_act_map(&maps.act, down ? h : x16, rows, split ? 2 * K : K, box_rows) ||
            !maps_of(rb, rs, routed.n * I, maps.body, maps.sign))
            return FP9_ERR_CUDA;
        if (shared != nullptr && shared->n > 0) {
            const uint8_t* sb[2] = {down ? shared->down_body : shared->gate_body,
                                    down ? shared->down_body : shared->up_body};
            const uint8_t* ss[2] = {down ? shared->down_sign : shared->gate_sign,
                                    down ? shared->down_sign : shared->up_sign};
            if (!maps_of(sb, ss, shared->n * I, maps.body_sh, maps.sign_sh)) return FP9_ERR_CUDA;
        } else {
            maps.body_sh[0] = maps.body_sh[1] = maps.body[0];
            maps.sign_sh[0] = maps.sign_sh[1] = maps.sign[0];
        }
        const int32_t ntiles = static_cast<int32_t>(down ? H / (2 * kNR) : I / kNR);
        PrefillArgs p = base_args(rows, down ? I : H, ntiles, down ? static_cast<void*>(y) : static_cast<void*>(h),
                                  down ? H : (split ? 2 * I : I), status);
        p.g_row = tab.row;
        p.g_cnt = tab.cnt;
        p.g_mtile = tab.mtile;
        p.n_groups = tab.n_groups;
        p.n_routed = tab.n_routed;
        p.inter = static_cast<int32_t>(I);
        int64_t ctas = max_mtiles * ntiles;  // an upper bound of the tiles
        if (ctas > 0x7FFFFFFF) return FP9_ERR_SHAPE;
        // a persistent grid of one CTA per SM walks the tiles
        if (ctas > sms) ctas = sms;
        void (*k)(const PrefillMaps, const PrefillArgs) =
            down ? (split ? prefill_kernel<true, 1, true, true> : prefill_kernel<true, 1, true, false>)
                 : (split ? gateup_kernel<true, true> : gateup_kernel<true, false>);
        FP9_CUDA_TRY(launch_pdl(k, dim3(static_cast<unsigned>(ctas)), dim3(down ? kGroupedThreads : kGuThreads),
                                down ? (split ? Cfg<1, true>::kSmem : Cfg<1>::kSmem) : kGuSmem, stream, maps, p));
    }
    return FP9_OK;
}

}  // namespace fp9

using namespace fp9;

extern "C" size_t fp9_prefill_workspace_bytes(const fp9_ffn_bank* ffn, int64_t m) {
    if (check_prefill_bank(ffn, 0) != FP9_OK || m < 0 || m > FP9_MAX_PREFILL_TOKENS) return 0;
    return prefill_layout(m, ffn->hidden, ffn->inter, device_sm_count()).total;
}

extern "C" fp9_status fp9_ffn_prefill(const fp9_ffn_bank* ffn, int64_t index, const float* x, int64_t m,
                                      float* y, int32_t precision, void* ws, size_t ws_bytes, int32_t* d_status,
                                      void* stream) {
    fp9_status st = check_prefill_bank(ffn, index);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(m >= 0 && m <= FP9_MAX_PREFILL_TOKENS, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(precision == FP9_PREFILL_SPLIT || precision == FP9_PREFILL_FP16, FP9_ERR_INVALID_ARG);
    const bool split = precision == FP9_PREFILL_SPLIT;
    if (m == 0) return FP9_OK;
    FP9_CHECK_ARG(x != nullptr && y != nullptr && ws != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(x, 16) && aligned(y, 16) && aligned(ws, 256), FP9_ERR_ALIGN);
    const int64_t H = ffn->hidden, I = ffn->inter;
    const int sms = device_sm_count();
    const PrefillLayout lay = prefill_layout(m, H, I, sms);
    FP9_CHECK_ARG(ws_bytes >= lay.total, FP9_ERR_WORKSPACE);
    if (sms <= 0) return FP9_ERR_CUDA;
    st = ensure_attrs();
    if (st != FP9_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    __half* x16 = reinterpret_cast<__half*>(w + lay.off_x16);
    __half* h = reinterpret_cast<__half*>(w + lay.off_h);
    float* parts = lay.total > lay.off_parts ? reinterpret_cast<float*>(w + lay.off_parts) : nullptr;

    const int64_t n4 = m * H / 4;
    const int64_t blocks = (n4 + 255) / 256 < static_cast<int64_t>(sms) * 8 ? (n4 + 255) / 256 : sms * 8;
    if (split)
        FP9_CUDA_TRY(launch_pdl(to_half_split_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                                reinterpret_cast<const float4*>(x), x16, n4, H / 4, d_status));
    else
        FP9_CUDA_TRY(launch_pdl(to_half_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                                reinterpret_cast<const float4*>(x), reinterpret_cast<uint2*>(x16), n4, d_status));

    // the maps cover FFN `index` only (rows [0, inter) of its planes)
    const size_t wg = static_cast<size_t>(index) * static_cast<size_t>(I) * static_cast<size_t>(H);
    const uint8_t* gu_body[2] = {ffn->gate_body + wg, ffn->up_body + wg};
    const uint8_t* gu_sign[2] = {ffn->gate_sign + wg / 8, ffn->up_sign + wg / 8};
    st = launch_gemm(false, split, x16, m, H, gu_body, gu_sign, I, H, 0, I, h, split ? 2 * I : I, nullptr, d_status,
                     sms, s);
    if (st != FP9_OK) return st;
    const uint8_t* d_body[2] = {ffn->down_body + wg, ffn->down_body + wg};
    const uint8_t* d_sign[2] = {ffn->down_sign + wg / 8, ffn->down_sign + wg / 8};
    return launch_gemm(true, split, h, m, I, d_body, d_sign, I, H, 0, H, y, H, parts, d_status, sms, s);
}

extern "C" fp9_status fp9_prefill_selftest_timeout(void* ws, size_t ws_bytes, int32_t* d_status, int32_t timeout_us,
                                                   void* stream) {
    FP9_CHECK_ARG(ws != nullptr && d_status != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(ws, 256), FP9_ERR_ALIGN);
    FP9_CHECK_ARG(timeout_us >= 1 && timeout_us <= 1000000, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(ws_bytes >= (static_cast<size_t>(1) << 17), FP9_ERR_WORKSPACE);
    fp9_status st = ensure_attrs();
    if (st != FP9_OK) return st;
    // one gate/up CTA: 128 tokens, hidden 256, inter 128; x (fp16) at the
    // start of ws, h after it, and the weight maps over the last 32 KiB
    // (never read: no weight copy is issued)
    constexpr int64_t H = 256, I = 128, m = 128;
    uint8_t* w = static_cast<uint8_t*>(ws);
    const __half* x16 = reinterpret_cast<const __half*>(w);
    __half* h = reinterpret_cast<__half*>(w + 65536);
    const uint8_t* planes[2] = {w + 98304, w + 98304};
    PrefillMaps maps;
    if (!make_act_map(&maps.act, x16, m, H) || !make_weight_maps(false, planes, planes, I, H, maps.body, maps.sign))
        return FP9_ERR_CUDA;
    for (int b = 0; b < 2; ++b) {
        maps.body_sh[b] = maps.body[b];
        maps.sign_sh[b] = maps.sign[b];
    }
    PrefillArgs p = base_args(m, H, 1, h, I, d_status);
    p.mtiles = 1;
    p.no_copy = 1;
    p.timeout_ns = static_cast<uint64_t>(timeout_us) * 1000ull;
    FP9_CUDA_TRY(launch_pdl(prefill_kernel<false, 1, false, false>, dim3(1), dim3(kThreads), Cfg<1>::kSmem,
                            static_cast<cudaStream_t>(stream), maps, p));
    return FP9_OK;
}
