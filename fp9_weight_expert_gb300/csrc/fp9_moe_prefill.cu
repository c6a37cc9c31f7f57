// MoE layer over many tokens at once (prompt prefill).
//
// The same layer as the decode step (router [MTP-9.2]: top_k = 8 of a
// DeepSeek-V3-style grouped sigmoid gate; FFN experts in fp9 [MEMOIR-FP9];
// routed outputs weighted, shared experts added), for m tokens. With m in
// the thousands each expert sees tens to hundreds of tokens, so the expert
// FFNs run as grouped GEMMs on the tensor cores (fp9_prefill.cu):
//
//   1. logits   [m, E] = x W_g^T in fp32 (a tiled FFMA GEMM, K split into
//               up to 8 parts added in order by the selection);
//   2. select   one warp per token: sigmoid, group scores, top groups,
//               top-k, weights (the decode router's rules and order);
//   3. rank     one CTA per expert: the rank of each (token, slot) among
//               the expert's slots, in token order (deterministic); the
//               last CTA lays out the groups (routed experts, then shared
//               experts with every token) as contiguous row ranges and
//               128-row tiles;
//   4. permute  x -> fp16 rows in group order (each token once per slot and
//               once per shared expert);
//   5. gate/up and down over the groups' tiles -> per-row FFN outputs;
//   6. combine  y[t] = sum_k w[t,k] * row(t,k) + sum_s row_s(t), in slot
//               then shared order (deterministic).
#include <cfloat>
#include <climits>
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9_plan.h"
#include "fp9_prefill.h"
#include "fp9moe.h"

namespace fp9 {

fp9_status check_layer(const fp9_moe_layer* L, int32_t bsz);

namespace {

// ------------------------------------------------------------- logits ---

constexpr int kLogitM = 128, kLogitN = 128, kLogitK = 16, kLogitThreads = 256;

// Partial logits over K part `blockIdx.z` of `splits`: part[z][t, e] = the
// sum over that part's k of x[t, k] W_g[e, k], fp32, each thread summing its
// outputs in k order; the selection adds the parts in split order. A CTA
// computes 128 tokens x 128 experts, a thread 8 x 8 of them (tokens and
// experts 4 ty / 4 tx + [0, 4) and 64 + the same), reading 4 float4 of
// shared memory per 64 multiply-adds. K runs in steps of 16,
// double-buffered; part z covers steps [z S / splits, (z + 1) S / splits)
// of the S = H / 16 steps. H % 16 == 0.
__global__ void __launch_bounds__(kLogitThreads, 2) logits_kernel(const float* __restrict__ x,
                                                                  const float* __restrict__ wr,
                                                                  float* __restrict__ part, int32_t m, int32_t E,
                                                                  int32_t H, int32_t splits) {
    __shared__ __align__(16) float xs[2][kLogitK][kLogitM + 4];
    __shared__ __align__(16) float ws[2][kLogitK][kLogitN + 4];
    grid_dependency_wait();
    grid_launch_dependents();
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int t0 = blockIdx.x * kLogitM, e0 = blockIdx.y * kLogitN;
    const int nst = H / kLogitK;
    const int s0 = static_cast<int>(static_cast<int64_t>(blockIdx.z) * nst / splits);
    const int s1 = static_cast<int>(static_cast<int64_t>(blockIdx.z + 1) * nst / splits);
    // loads: four consecutive threads read the 64 bytes of one row's k step
    // (rows tid / 4 and 64 + tid / 4 of x and of W_g)
    const int kq = tid & 3, r0 = tid >> 2;
    float4 rx[2], rw[2];
    auto load = [&](int k0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int row = r0 + 64 * j;
            rx[j] = (t0 + row < m)
                        ? __ldg(reinterpret_cast<const float4*>(x + static_cast<int64_t>(t0 + row) * H + k0) + kq)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int row = r0 + 64 * j;
            rw[j] = (e0 + row < E)
                        ? __ldg(reinterpret_cast<const float4*>(wr + static_cast<int64_t>(e0 + row) * H + k0) + kq)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int row = r0 + 64 * j;
            xs[buf][4 * kq + 0][row] = rx[j].x;
            xs[buf][4 * kq + 1][row] = rx[j].y;
            xs[buf][4 * kq + 2][row] = rx[j].z;
            xs[buf][4 * kq + 3][row] = rx[j].w;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int row = r0 + 64 * j;
            ws[buf][4 * kq + 0][row] = rw[j].x;
            ws[buf][4 * kq + 1][row] = rw[j].y;
            ws[buf][4 * kq + 2][row] = rw[j].z;
            ws[buf][4 * kq + 3][row] = rw[j].w;
        }
    };
    float acc[8][8] = {};
    if (s0 < s1) {
        load(s0 * kLogitK);
        store(0);
    }
    __syncthreads();
    for (int st = s0; st < s1; ++st) {
        const int buf = (st - s0) & 1;
        if (st + 1 < s1) load((st + 1) * kLogitK);
#pragma unroll
        for (int k = 0; k < kLogitK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&xs[buf][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&xs[buf][k][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&ws[buf][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&ws[buf][k][64 + tx * 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (st + 1 < s1) store(buf ^ 1);
        __syncthreads();
    }
    float* out = part + static_cast<int64_t>(blockIdx.z) * m * E;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = t0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        if (t >= m) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = e0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
            if (e < E) out[static_cast<int64_t>(t) * E + e] = acc[i][j];
        }
    }
}

// ------------------------------------------------------------- select ---

constexpr int kSelectWarps = 8;

// (v, i) beats (bv, bi): a larger value, or an equal value and a lower index.
__device__ __forceinline__ bool beats(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// Warp-wide best (valid, v, i): every lane gets the winner.
__device__ __forceinline__ void warp_best(bool& valid, float& v, int& i) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool ov = __shfl_xor_sync(0xFFFFFFFFu, valid, o);
        const float vv = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
        if (ov && (!valid || beats(vv, oi, v, i))) {
            valid = true;
            v = vv;
            i = oi;
        }
    }
}

struct SelectArgs {
    const float* logits;  // [splits, m, E] partial logits
    int32_t splits;
    int32_t m, E, n_groups, topk_groups, topk;
    float scale;
    int32_t* ids;         // [m, topk]
    float* wts;           // [m, topk]
    int32_t* ids_out;     // optional
    float* w_out;         // optional
};

// One warp per token: s = sigmoid(logit) (NaN -> -inf), group score = sum
// of the two largest s of the group (the one s of 1-expert groups), the
// topk_groups best groups, then the topk best experts inside them, each
// pick the best remaining (ties to the lower index): the order of a sort by
// score descending. w = s / sum(s chosen, summed in that order) * scale.
__global__ void __launch_bounds__(kSelectWarps * 32) select_kernel(const SelectArgs a) {
    extern __shared__ float s_sc[];  // [kSelectWarps][E]
    __shared__ float s_val[kSelectWarps][FP9_MAX_TOPK];
    __shared__ int32_t s_id[kSelectWarps][FP9_MAX_TOPK];
    grid_dependency_wait();
    grid_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kSelectWarps + warp;
    if (t >= a.m) return;
    const int E = a.E, G = a.n_groups, gsz = E / G;
    float* sc = s_sc + warp * E;
    for (int e = lane; e < E; e += 32) {
        float l = 0.0f;
        for (int z = 0; z < a.splits; ++z) l += __ldg(a.logits + (static_cast<int64_t>(z) * a.m + t) * E + e);
        const float s = 1.0f / (1.0f + expf(-l));
        sc[e] = (s == s) ? s : -INFINITY;
    }
    __syncwarp();
    float gscore = -INFINITY;
    if (lane < G) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int i = 0; i < gsz; ++i) {
            const float v = sc[lane * gsz + i];
            if (v > m1) {
                m2 = m1;
                m1 = v;
            } else if (v > m2) {
                m2 = v;
            }
        }
        gscore = gsz == 1 ? m1 : m1 + m2;
    }
    uint32_t kept = 0;
    bool gfree = lane < G;
    for (int r = 0; r < a.topk_groups; ++r) {
        bool valid = gfree;
        float v = gscore;
        int i = lane;
        warp_best(valid, v, i);
        kept |= 1u << i;
        if (lane == i) gfree = false;
    }
    uint32_t chosen = 0;  // bit j: expert lane + 32 j taken
    for (int k = 0; k < a.topk; ++k) {
        bool valid = false;
        float v = -INFINITY;
        int i = INT_MAX;
        for (int j = 0; lane + 32 * j < E; ++j) {
            const int e = lane + 32 * j;
            if (!((kept >> (e / gsz)) & 1u) || ((chosen >> j) & 1u)) continue;
            const float s = sc[e];
            if (!valid || beats(s, e, v, i)) {
                valid = true;
                v = s;
                i = e;
            }
        }
        warp_best(valid, v, i);
        if (lane == 0) {
            s_val[warp][k] = v;
            s_id[warp][k] = i;
        }
        if ((i & 31) == lane) chosen |= 1u << (i >> 5);
    }
    __syncwarp();
    if (lane == 0) {
        float sum = 0.0f;
        for (int k = 0; k < a.topk; ++k) sum += s_val[warp][k];
        for (int k = 0; k < a.topk; ++k) {
            const float w = s_val[warp][k] / sum * a.scale;
            const int64_t o = static_cast<int64_t>(t) * a.topk + k;
            a.ids[o] = s_id[warp][k];
            a.wts[o] = w;
            if (a.ids_out) a.ids_out[o] = s_id[warp][k];
            if (a.w_out) a.w_out[o] = w;
        }
    }
}

// --------------------------------------------------------------- rank ---

constexpr int kRankThreads = 256;

struct RankArgs {
    const int32_t* ids;   // [m, topk]
    int32_t m, topk, E, n_shared;
    int32_t* rank;        // [m, topk] rank of the slot among its expert's slots
    int32_t* cnt;         // [E + n_shared]
    int32_t* row;         // [E + n_shared]
    int32_t* mtile;       // [E + n_shared + 1]
    uint32_t* ticket;     // self-resetting last-arriver counter
};

__device__ int32_t block_scan_excl(int32_t v, int32_t& total) {
    __shared__ int32_t s_w[kRankThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    int32_t off = 0, tot = 0;
    for (int w = 0; w < kRankThreads / 32; ++w) {
        off += w < warp ? s_w[w] : 0;
        tot += s_w[w];
    }
    total = tot;
    __syncthreads();
    return off + incl - v;
}

// CTA e ranks expert e's slots in (token, slot) order; the last CTA to
// finish lays out the groups: group g (routed experts 0..E-1, then the
// shared experts, each with all m tokens) gets rows [row[g], row[g] +
// cnt[g]) and ceil(cnt[g] / 128) token tiles from mtile[g].
__global__ void __launch_bounds__(kRankThreads) rank_kernel(const RankArgs a) {
    __shared__ int s_last;
    grid_dependency_wait();
    grid_launch_dependents();
    const int e = blockIdx.x, tid = threadIdx.x;
    // thread t takes the (token, slot) pairs [t L, (t + 1) L) in order: it
    // counts its matches, one block scan gives each run's first rank, and a
    // second pass over the run writes the ranks
    const int64_t P = static_cast<int64_t>(a.m) * a.topk;
    const int64_t L = (P + kRankThreads - 1) / kRankThreads;
    const int64_t i0 = tid * L, i1 = i0 + L < P ? i0 + L : P;
    int32_t mine = 0;
    for (int64_t i = i0; i < i1; ++i) mine += __ldg(a.ids + i) == e ? 1 : 0;
    int32_t base = 0;
    int32_t r = block_scan_excl(mine, base);
    for (int64_t i = i0; i < i1 && mine > 0; ++i)
        if (__ldg(a.ids + i) == e) {
            a.rank[i] = r++;
            --mine;
        }
    if (tid == 0) {
        a.cnt[e] = base;
        __threadfence();
        s_last = (atomicInc(a.ticket, gridDim.x - 1) == gridDim.x - 1) ? 1 : 0;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    const int G = a.E + a.n_shared;
    const int per = (G + kRankThreads - 1) / kRankThreads;
    int32_t c[FP9_MAX_EXPERTS / kRankThreads + 1];
    int32_t rsum = 0, tsum = 0;
    for (int q = 0; q < per; ++q) {
        const int g = tid * per + q;
        c[q] = g < G ? (g < a.E ? __ldcg(a.cnt + g) : a.m) : 0;
        rsum += c[q];
        tsum += (c[q] + kPrefillTileRows - 1) / kPrefillTileRows;
    }
    int32_t rtot = 0, ttot = 0;
    int32_t r0 = block_scan_excl(rsum, rtot);
    int32_t m0 = block_scan_excl(tsum, ttot);
    for (int q = 0; q < per; ++q) {
        const int g = tid * per + q;
        if (g >= G) break;
        if (g >= a.E) a.cnt[g] = c[q];
        a.row[g] = r0;
        a.mtile[g] = m0;
        r0 += c[q];
        m0 += (c[q] + kPrefillTileRows - 1) / kPrefillTileRows;
    }
    if (tid == 0) a.mtile[G] = ttot;
}

// ------------------------------------------------------------ permute ---

constexpr int kRowThreads = 256;

struct PermuteArgs {
    const float* x;          // [m, H]
    const int32_t* ids;      // [m, topk]
    const int32_t* rank;     // [m, topk]
    const int32_t* row;      // [E + n_shared]
    int32_t m, H, topk, E, n_shared;
    __half* x16;             // [rows, H], or [rows, 2H] in the split layout
    int32_t* pos;            // [m, topk] the slot's row
    int32_t* status;
    int32_t split;           // 1: two fp16 terms per value (hi, lo)
};

// Token t's fp16 row goes to the row of each of its slots and to row t of
// each shared group. A value whose fp16 is not finite is a range error.
// In the split layout each value is written as hi = fp16(v) and lo =
// fp16(v - hi): 64-column chunk c of a row holds its hi terms in columns
// [128 c, 128 c + 64) and its lo terms in the next 64.
__global__ void __launch_bounds__(kRowThreads) permute_kernel(const PermuteArgs a) {
    __shared__ int32_t s_rows[FP9_MAX_TOPK + FP9_MAX_SHARED];
    grid_dependency_wait();
    grid_launch_dependents();
    const int t = blockIdx.x, tid = threadIdx.x;
    const int nr = a.topk + a.n_shared;
    if (tid < a.topk) {
        const int64_t o = static_cast<int64_t>(t) * a.topk + tid;
        const int32_t r = __ldg(a.row + __ldg(a.ids + o)) + __ldg(a.rank + o);
        s_rows[tid] = r;
        a.pos[o] = r;
    } else if (tid < nr) {
        s_rows[tid] = __ldg(a.row + a.E + (tid - a.topk)) + t;
    }
    __syncthreads();
    const int H4 = a.H / 4;
    const float4* x4 = reinterpret_cast<const float4*>(a.x) + static_cast<int64_t>(t) * H4;
    bool finite = true;
    for (int c = tid; c < H4; c += kRowThreads) {
        const float4 v = __ldg(x4 + c);
        const __half2 h0 = __floats2half2_rn(v.x, v.y), h1 = __floats2half2_rn(v.z, v.w);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&h0);
        o.y = *reinterpret_cast<const uint32_t*>(&h1);
        finite = finite && ((o.x & 0x7C00u) != 0x7C00u) && ((o.x & 0x7C000000u) != 0x7C000000u) &&
                 ((o.y & 0x7C00u) != 0x7C00u) && ((o.y & 0x7C000000u) != 0x7C000000u);
        if (a.split) {
            const __half2 l0 = __floats2half2_rn(v.x - __low2float(h0), v.y - __high2float(h0));
            const __half2 l1 = __floats2half2_rn(v.z - __low2float(h1), v.w - __high2float(h1));
            uint2 l;
            l.x = *reinterpret_cast<const uint32_t*>(&l0);
            l.y = *reinterpret_cast<const uint32_t*>(&l1);
            const int64_t col = 4 * static_cast<int64_t>(c);  // four columns inside one 64-column chunk
            const int64_t sc = ((col >> 6) << 7) + (col & 63);
            for (int r = 0; r < nr; ++r) {
                __half* dst = a.x16 + static_cast<int64_t>(s_rows[r]) * 2 * a.H + sc;
                *reinterpret_cast<uint2*>(dst) = o;
                *reinterpret_cast<uint2*>(dst + 64) = l;
            }
        } else {
            for (int r = 0; r < nr; ++r) reinterpret_cast<uint2*>(a.x16 + static_cast<int64_t>(s_rows[r]) * a.H)[c] = o;
        }
    }
    if (!finite) record_status(a.status, FP9_ERR_RANGE);
}

// ------------------------------------------------------------ combine ---

struct CombineArgs {
    const float* yrows;   // [rows, H] per-row FFN outputs
    const int32_t* pos;   // [m, topk]
    const float* wts;     // [m, topk]
    const int32_t* row;   // [E + n_shared]
    int32_t m, H, topk, E, n_shared;
    float* y;             // [m, H]
};

__global__ void __launch_bounds__(kRowThreads) moe_combine_kernel(const CombineArgs a) {
    __shared__ int32_t s_rows[FP9_MAX_TOPK + FP9_MAX_SHARED];
    __shared__ float s_w[FP9_MAX_TOPK];
    grid_dependency_wait();
    grid_launch_dependents();
    const int t = blockIdx.x, tid = threadIdx.x;
    if (tid < a.topk) {
        const int64_t o = static_cast<int64_t>(t) * a.topk + tid;
        s_rows[tid] = __ldg(a.pos + o);
        s_w[tid] = __ldg(a.wts + o);
    } else if (tid < a.topk + a.n_shared) {
        s_rows[tid] = __ldg(a.row + a.E + (tid - a.topk)) + t;
    }
    __syncthreads();
    const int H4 = a.H / 4;
    for (int c = tid; c < H4; c += kRowThreads) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < a.topk; ++k) {
            const float4 v = __ldcs(reinterpret_cast<const float4*>(a.yrows + static_cast<int64_t>(s_rows[k]) * a.H) + c);
            const float w = s_w[k];
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        for (int s = 0; s < a.n_shared; ++s) {
            const float4 v =
                __ldcs(reinterpret_cast<const float4*>(a.yrows + static_cast<int64_t>(s_rows[a.topk + s]) * a.H) + c);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        reinterpret_cast<float4*>(a.y + static_cast<int64_t>(t) * a.H)[c] = acc;
    }
}

// -------------------------------------------------------------- host ---

// K parts of the logits GEMM: about two CTAs per SM (the kernel's
// register budget), and never more parts than the workspace holds.
int64_t logit_tiles(int64_t m, int64_t E) {
    return ((m + kLogitM - 1) / kLogitM) * ((E + kLogitN - 1) / kLogitN);
}

// Parts the workspace holds: at most 32 and 1024 CTAs' worth, so that the
// partial planes take at most about 1024 / tiles x m x E floats.
int logit_split_cap(int64_t m, int64_t E, int64_t H) {
    int64_t cap = 1024 / logit_tiles(m, E);
    if (cap > 32) cap = 32;
    if (cap > H / kLogitK) cap = H / kLogitK;
    return cap < 1 ? 1 : static_cast<int>(cap);
}

int logit_splits(int64_t m, int32_t E, int64_t H, int sms) {
    int64_t s = 2 * static_cast<int64_t>(sms) / logit_tiles(m, E);
    const int cap = logit_split_cap(m, E, H);
    if (s > cap) s = cap;
    return s < 1 ? 1 : static_cast<int>(s);
}

struct MoePrefillLayout {
    size_t off_ticket = 0, off_logits = 0, off_ids = 0, off_wts = 0, off_rank = 0, off_pos = 0, off_cnt = 0,
           off_row = 0, off_mtile = 0, off_x16 = 0, off_h = 0, off_y = 0, total = 0;
    int64_t rows = 0;        // m * (topk + n_shared)
    int64_t max_mtiles = 0;  // bound on the token tiles of all groups
};

MoePrefillLayout moe_prefill_layout(const fp9_moe_layer* L, int64_t m) {
    MoePrefillLayout W;
    const int64_t E = L->n_experts, S = L->n_shared, G = E + S, K = L->topk, H = L->hidden, I = L->inter;
    W.rows = m * (K + S);
    W.max_mtiles = (m * K + kPrefillTileRows - 1) / kPrefillTileRows + E + S * ((m + kPrefillTileRows - 1) / kPrefillTileRows);
    size_t off = align_up(sizeof(uint32_t));
    W.off_logits = off;
    off = align_up(off + sizeof(float) * logit_split_cap(m, E, H) * m * E);
    W.off_ids = off;
    off = align_up(off + sizeof(int32_t) * m * K);
    W.off_wts = off;
    off = align_up(off + sizeof(float) * m * K);
    W.off_rank = off;
    off = align_up(off + sizeof(int32_t) * m * K);
    W.off_pos = off;
    off = align_up(off + sizeof(int32_t) * m * K);
    W.off_cnt = off;
    off = align_up(off + sizeof(int32_t) * G);
    W.off_row = off;
    off = align_up(off + sizeof(int32_t) * G);
    W.off_mtile = off;
    off = align_up(off + sizeof(int32_t) * (G + 1));
    // x and h in the split layout (two fp16 terms per value; the one-term
    // mode uses the first half of each)
    W.off_x16 = off;
    off = align_up(off + 2 * sizeof(__half) * W.rows * H);
    W.off_h = off;
    off = align_up(off + 2 * sizeof(__half) * W.rows * I);
    W.off_y = off;
    off = align_up(off + sizeof(float) * W.rows * H);
    W.total = off;
    return W;
}

fp9_status check_moe_prefill(const fp9_moe_layer* L, int64_t m) {
    fp9_status st = check_layer(L, 1);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(L->hidden % 256 == 0, FP9_ERR_SHAPE);
    FP9_CHECK_ARG(L->inter >= 128 && L->inter % 128 == 0, FP9_ERR_SHAPE);
    FP9_CHECK_ARG(m >= 0 && m <= FP9_MAX_PREFILL_TOKENS, FP9_ERR_INVALID_ARG);
    return FP9_OK;
}

}  // namespace
}  // namespace fp9

using namespace fp9;

extern "C" size_t fp9_moe_prefill_workspace_bytes(const fp9_moe_layer* layer, int64_t m) {
    if (check_moe_prefill(layer, m) != FP9_OK) return 0;
    return moe_prefill_layout(layer, m).total;
}

extern "C" fp9_status fp9_moe_prefill(const fp9_moe_layer* layer, const float* x, int64_t m, float* y,
                                      int32_t* ids, float* weights, int32_t precision, void* ws, size_t ws_bytes,
                                      int32_t* d_status, void* stream) {
    fp9_status st = check_moe_prefill(layer, m);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(precision == FP9_PREFILL_SPLIT || precision == FP9_PREFILL_FP16, FP9_ERR_INVALID_ARG);
    const bool split = precision == FP9_PREFILL_SPLIT;
    if (m == 0) return FP9_OK;
    FP9_CHECK_ARG(x != nullptr && y != nullptr && ws != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(x, 16) && aligned(y, 16) && aligned(ws, kAlign), FP9_ERR_ALIGN);
    const MoePrefillLayout W = moe_prefill_layout(layer, m);
    FP9_CHECK_ARG(ws_bytes >= W.total, FP9_ERR_WORKSPACE);
    const int sms = device_sm_count();
    if (sms <= 0) return FP9_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    const int32_t E = layer->n_experts, K = layer->topk, S = layer->n_shared, H = static_cast<int32_t>(layer->hidden);
    const int32_t mi = static_cast<int32_t>(m);
    float* logits = reinterpret_cast<float*>(w + W.off_logits);
    int32_t* ids_ws = reinterpret_cast<int32_t*>(w + W.off_ids);
    float* wts_ws = reinterpret_cast<float*>(w + W.off_wts);
    int32_t* rank = reinterpret_cast<int32_t*>(w + W.off_rank);
    int32_t* pos = reinterpret_cast<int32_t*>(w + W.off_pos);
    int32_t* cnt = reinterpret_cast<int32_t*>(w + W.off_cnt);
    int32_t* row = reinterpret_cast<int32_t*>(w + W.off_row);
    int32_t* mtile = reinterpret_cast<int32_t*>(w + W.off_mtile);
    __half* x16 = reinterpret_cast<__half*>(w + W.off_x16);
    __half* h = reinterpret_cast<__half*>(w + W.off_h);
    float* yrows = reinterpret_cast<float*>(w + W.off_y);

    const int splits = logit_splits(m, E, H, sms);
    FP9_CUDA_TRY(launch_pdl(logits_kernel,
                            dim3(static_cast<unsigned>((m + kLogitM - 1) / kLogitM),
                                 static_cast<unsigned>((E + kLogitN - 1) / kLogitN), static_cast<unsigned>(splits)),
                            dim3(kLogitThreads), 0, s, x, layer->w_router, logits, mi, E, H, splits));

    SelectArgs sa{logits, splits, mi, E, layer->n_groups, layer->topk_groups, K, layer->route_scale, ids_ws, wts_ws, ids,
                  weights};
    const size_t sel_smem = sizeof(float) * kSelectWarps * E;
    static DeviceOnce attr;
    const fp9_status ast = attr.run([] {
        FP9_CUDA_TRY(cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(sizeof(float) * kSelectWarps * FP9_MAX_EXPERTS)));
        return FP9_OK;
    });
    if (ast != FP9_OK) return ast;
    FP9_CUDA_TRY(launch_pdl(select_kernel, dim3(static_cast<unsigned>((m + kSelectWarps - 1) / kSelectWarps)),
                            dim3(kSelectWarps * 32), sel_smem, s, sa));

    RankArgs ra{ids_ws, mi, K, E, S, rank, cnt, row, mtile, reinterpret_cast<uint32_t*>(w + W.off_ticket)};
    FP9_CUDA_TRY(launch_pdl(rank_kernel, dim3(E), dim3(kRankThreads), 0, s, ra));

    PermuteArgs pa{x, ids_ws, rank, row, mi, H, K, E, S, x16, pos, d_status, split ? 1 : 0};
    FP9_CUDA_TRY(launch_pdl(permute_kernel, dim3(mi), dim3(kRowThreads), 0, s, pa));

    GroupTableDev tab{row, cnt, mtile, E + S, E};
    st = launch_grouped_ffn(layer->routed, S > 0 ? &layer->shared : nullptr, tab, W.max_mtiles, x16, h, yrows, W.rows,
                            split, d_status, sms, s);
    if (st != FP9_OK) return st;

    CombineArgs ca{yrows, pos, wts_ws, row, mi, H, K, E, S, y};
    FP9_CUDA_TRY(launch_pdl(moe_combine_kernel, dim3(mi), dim3(kRowThreads), 0, s, ca));
    return FP9_OK;
}
