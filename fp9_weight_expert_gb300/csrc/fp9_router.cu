// Router: fp32 logits x . W_g, sigmoid, group-limited top-k, normalised and
// scaled weights; then the job list for the fused expert kernel.
//
// The pages fix top_k = 8 experts per token ([MTP-9.2], "第 9 章 MTP1
// dual-lane overlap", section 9.2); the grouping (8 groups of 32, top-4
// groups ranked by the sum of their two best scores) is the DeepSeek-V3 gate.
//
// One launch: CTA e computes the logits of expert e for all tokens; the
// last CTA to finish (a self-resetting atomicInc ticket,
// no waiting) reads all logits back and does the selection and the job
// build.
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9_plan.h"
#include "fp9moe.h"

namespace fp9 {

constexpr int kRouterThreads = 256;
constexpr int kRouterVec = FP9_MAX_HIDDEN / 4 / kRouterThreads;  // float4 of one row per thread
constexpr int kMaxEntries = FP9_MAX_BSZ * FP9_MAX_TOPK;  // 128 (token, expert) pairs
static_assert(kMaxEntries <= kRouterThreads, "one thread per routed pair");

struct RouterArgs {
    const float* x;      // [bsz, H]: x, or h in stack mode
    const float* ss;     // stack mode: partial sums of squares of h (x = RMSNorm(h)), else NULL
    float eps;
    const float* wr;     // [E, H]
    int32_t bsz, E, H, n_groups, topk_groups, topk;
    float scale;
    int64_t I;           // intermediate size (rows per job)
    int32_t grid;        // CTAs of the fused expert kernel
    Control* ctl;
    float* logits;       // [bsz, E]
    int32_t* ids_ws;     // [bsz, topk]
    float* w_ws;         // [bsz, topk]
    int32_t* ids_out;    // optional
    float* w_out;        // optional
    Job* jobs;           // [jmax]
    int64_t* cta_row;    // [grid + 1] first row of each CTA of the fused kernel
    int32_t tpj;         // tokens per job: 1 (an MoE call) or 2
    int64_t impl_rows;   // the fused kernel's phase-0 rows (shared experts, one token per job)
};

static_assert(kMaxJobs <= kRouterThreads && kMaxEntries <= kRouterThreads, "one thread per job in the plan scan");

// Exclusive prefix sum of v over the CTA's threads (all threads call it);
// `total` gets the sum over all of them.
__device__ int32_t block_exclusive_scan(int32_t v, int tid, int32_t& total) {
    __shared__ int32_t s_warp[kRouterThreads / 32];
    const int lane = tid & 31, warp = tid >> 5;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int32_t off = 0, tot = 0;
    for (int w = 0; w < kRouterThreads / 32; ++w) {
        off += w < warp ? s_warp[w] : 0;
        tot += s_warp[w];
    }
    total = tot;
    __syncthreads();  // s_warp may be reused by the next call
    return off + incl - v;
}

// (v, i) beats (bv, bi): a larger value, or an equal value and a lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

// Selection for all tokens by the whole CTA, by ranks: a candidate's rank
// is the number of candidates that beat it (a larger score, or an equal
// score and a lower index), so the k best are the candidates of rank < k,
// each at the position of its rank (the order of a sort by score
// descending, ties to the lower index). `s` holds the [bsz, E] sigmoid
// scores (NaN replaced by -inf so that the choice stays defined).
__device__ void select_all(const RouterArgs& a, const float* s, int tid, int32_t* s_ids, float* s_wts) {
    __shared__ float s_gs[FP9_MAX_BSZ][FP9_MAX_GROUPS];
    __shared__ uint32_t s_kept[FP9_MAX_BSZ];
    __shared__ float s_sel[kMaxEntries];
    const int E = a.E, G = a.n_groups, gsize = E / G;
    // group scores: sum of the two largest members (the one member if
    // gsize == 1). The members are read from a rotated start (the groups'
    // threads then hit distinct banks), eight loads at a time.
    for (int i = tid; i < a.bsz * G; i += blockDim.x) {
        const int t = i / G, g = i % G;
        const float* grp = s + t * E + g * gsize;
        const int r0 = g % gsize;
        float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll 8
        for (int m = 0; m < gsize; ++m) {
            const int idx = m + r0 < gsize ? m + r0 : m + r0 - gsize;
            const float v = grp[idx];
            m2 = fmaxf(m2, fminf(m1, v));
            m1 = fmaxf(m1, v);
        }
        s_gs[t][g] = (gsize == 1) ? m1 : m1 + m2;
    }
    if (tid < a.bsz) s_kept[tid] = 0u;
    __syncthreads();
    for (int i = tid; i < a.bsz * G; i += blockDim.x) {
        const int t = i / G, g = i % G;
        const float v = s_gs[t][g];
        int rank = 0;
        for (int o = 0; o < G; ++o) rank += better(s_gs[t][o], o, v, g) ? 1 : 0;
        if (rank < a.topk_groups) atomicOr(&s_kept[t], 1u << g);
    }
    __syncthreads();
    for (int i = tid; i < a.bsz * E; i += blockDim.x) {
        const int t = i / E, e = i % E;
        const uint32_t kept = s_kept[t];
        if (!((kept >> (e / gsize)) & 1u)) continue;
        const float* st = s + t * E;
        const float v = st[e];
        int rank = 0;
        for (int g = 0; g < G; ++g) {
            if (!((kept >> g) & 1u)) continue;
            const float* grp = st + g * gsize;
            const int base = g * gsize;
            // the threads of a warp read the same member (a broadcast); eight
            // independent loads at a time
#pragma unroll 8
            for (int m = 0; m < gsize; ++m) rank += better(grp[m], base + m, v, e) ? 1 : 0;
        }
        if (rank < a.topk) {
            s_ids[t * a.topk + rank] = e;
            s_sel[t * a.topk + rank] = v;
        }
    }
    __syncthreads();
    if (tid < a.bsz) {  // weights: s_i / sum(s_chosen) * route_scale, summed in rank order
        const int t = tid;
        float sum = 0.0f;
        for (int k = 0; k < a.topk; ++k) sum += s_sel[t * a.topk + k];
        for (int k = 0; k < a.topk; ++k) {
            const int id = s_ids[t * a.topk + k];
            const float w = s_sel[t * a.topk + k] / sum * a.scale;
            s_wts[t * a.topk + k] = w;
            a.ids_ws[t * a.topk + k] = id;
            a.w_ws[t * a.topk + k] = w;
            if (a.ids_out) a.ids_out[t * a.topk + k] = id;
            if (a.w_out) a.w_out[t * a.topk + k] = w;
        }
    }
    __syncthreads();
}

// Warp bitonic sort of 32 (score, expert) pairs, one per lane, into the
// selection order: larger score first, equal scores by lower expert (lane 0
// holds the best). Each step keeps the better of a lane pair in the lane
// whose run and position call for it.
__device__ __forceinline__ void warp_sort_best_first(float& v, int& i, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j >= 1; j >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, j);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, j);
            const bool keep_better = ((lane & j) == 0) == ((lane & k) == 0);
            if (better(ov, oi, v, i) == keep_better) {
                v = ov;
                i = oi;
            }
        }
    }
}

// Selection when every group has 32 experts and the candidates (the best
// topk of each kept group) fit in a warp (topk_groups * topk <= 32), as in
// the DeepSeek-V3 gate (8 groups of 32, top-4 groups, top-8):
//  1. one warp per (token, group) sorts the group's 32 scores; the group
//     score is the sum of its first two; the sorted scores and their experts
//     go back to the group's slots of s / s_idx;
//  2. the kept groups by rank, as in select_all;
//  3. one warp per token sorts the first topk of each kept group; its first
//     topk lanes are the chosen experts in selection order.
// The chosen experts, their order and the weights (s_i / sum, summed in
// selection order, times route_scale) are those of select_all.
__device__ void select_g32(const RouterArgs& a, float* s, int* s_idx, int tid, int32_t* s_ids, float* s_wts) {
    __shared__ float s_gs[FP9_MAX_BSZ][FP9_MAX_GROUPS];
    __shared__ uint32_t s_kept[FP9_MAX_BSZ];
    const int E = a.E, G = a.n_groups, K = a.topk, KG = a.topk_groups, bsz = a.bsz;
    const int lane = tid & 31, warp = tid >> 5, nwarps = kRouterThreads / 32;
    for (int p = warp; p < bsz * G; p += nwarps) {
        const int t = p / G, g = p - t * G;
        float* grp = s + t * E + g * 32;
        float v = grp[lane];
        int i = g * 32 + lane;
        warp_sort_best_first(v, i, lane);
        const float v1 = __shfl_sync(0xFFFFFFFFu, v, 1);
        grp[lane] = v;
        s_idx[t * E + g * 32 + lane] = i;
        if (lane == 0) s_gs[t][g] = v + v1;
    }
    if (tid < bsz) s_kept[tid] = 0u;
    __syncthreads();
    for (int i = tid; i < bsz * G; i += blockDim.x) {
        const int t = i / G, g = i % G;
        const float v = s_gs[t][g];
        int rank = 0;
        for (int o = 0; o < G; ++o) rank += better(s_gs[t][o], o, v, g) ? 1 : 0;
        if (rank < KG) atomicOr(&s_kept[t], 1u << g);
    }
    __syncthreads();
    for (int t = warp; t < bsz; t += nwarps) {
        const uint32_t kept = s_kept[t];
        const int q = lane / K, r = lane - q * K;
        float v = -INFINITY;
        int i = INT_MAX;
        if (q < KG) {
            uint32_t m = kept;  // the q-th kept group: clear the q lowest set bits
            for (int k = 0; k < q; ++k) m &= m - 1u;
            const int g = __ffs(static_cast<int>(m)) - 1;
            v = s[t * E + g * 32 + r];
            i = s_idx[t * E + g * 32 + r];
        }
        warp_sort_best_first(v, i, lane);
        float sum = 0.0f;
        for (int k = 0; k < K; ++k) sum += __shfl_sync(0xFFFFFFFFu, v, k);
        if (lane < K) {
            const float w = v / sum * a.scale;
            s_ids[t * K + lane] = i;
            s_wts[t * K + lane] = w;
            a.ids_ws[t * K + lane] = i;
            a.w_ws[t * K + lane] = w;
            if (a.ids_out) a.ids_out[t * K + lane] = i;
            if (a.w_out) a.w_out[t * K + lane] = w;
        }
    }
    __syncthreads();
}

// Position of one-token job `tid` (sorted by expert, then token) in a job
// order that spaces the jobs of an expert chosen by several tokens k jobs
// apart, k in 1..8 chosen so that k jobs are close to a whole number of the
// fused kernel's CTA shares (J / G jobs each): then the CTAs that stream an
// expert's rows for its tokens reach each row at about the same time, and
// all but the first read of it hit in L2. The order is a k-column grid
// (position = slot * k + column): the repeated experts' groups go to the
// columns in turn, each group down one column, and the single-token jobs
// fill the other slots in order. `pos`: the job's index in its expert's
// group; `run`: the group's size. Returns -1 (keep the sorted order) when a
// group does not fit in its column. Every thread of the CTA calls it.
__device__ int32_t spaced_position(int tid, int J, int64_t G, int pos, int run) {
    __shared__ int32_t s_rsize[kMaxEntries];
    __shared__ int32_t s_grank[kMaxEntries];
    __shared__ int s_fail;
    int k = 1, best = J;
    for (int c = 1; c <= 8 && c <= J; ++c) {  // the same choice in every thread
        const int r = (c * static_cast<int>(G)) % J;  // G <= the grid: 32-bit arithmetic
        const int d = r < J - r ? r : J - r;
        if (d < best) {
            best = d;
            k = c;
        }
    }
    const bool in = tid < J;
    const int rep_start = (in && pos == 0 && run >= 2) ? 1 : 0;
    const int single = (in && run == 1) ? 1 : 0;
    int32_t nrep = 0, nsingle = 0;
    const int32_t rrank = block_exclusive_scan(rep_start, tid, nrep);
    const int32_t srank = block_exclusive_scan(single, tid, nsingle);
    if (tid == 0) s_fail = 0;
    if (rep_start) {
        s_rsize[rrank] = run;
        s_grank[tid] = rrank;
    }
    __syncthreads();
    int32_t dest = -1;
    if (in) {
        auto height = [&](int c) { return (J - c + k - 1) / k; };
        auto used = [&](int c, int upto) {  // slots of column c that repeated groups of rank < upto hold
            int u = 0;
            for (int r = c; r < upto; r += k) u += s_rsize[r];
            return u;
        };
        int col = 0, slot = 0;
        if (run >= 2) {
            const int r = s_grank[tid - pos];
            col = r % k;
            slot = used(col, r) + pos;
            if (slot >= height(col)) s_fail = 1;
        } else {
            int left = srank;
            for (col = 0; col < k; ++col) {
                const int u = used(col, nrep);
                const int free = height(col) - u;
                if (left < free) {
                    slot = u + left;
                    break;
                }
                left -= free;
            }
            if (col == k) s_fail = 1;
        }
        dest = slot * k + col;
    }
    __syncthreads();
    return s_fail ? -1 : dest;
}

// Routed job list: experts in ascending id, each with its tokens in
// ascending order, in groups of up to tpj (the shared experts need no
// routing: the fused kernel streams them on its own, before these); for
// one-token jobs at bsz >= 3, re-spaced by spaced_position. Then the
// cost-weighted split of the jobs' rows over the fused kernel's CTAs: each
// CTA's first row.
__device__ void build_jobs(const RouterArgs& a, int tid, const int32_t* s_ids, const float* s_wts) {
    __shared__ int32_t s_in[kMaxEntries];
    __shared__ int32_t s_key[kMaxEntries];
    __shared__ float s_w[kMaxEntries];
    __shared__ Job s_jobs[kMaxJobs];
    __shared__ int64_t s_u0[kMaxJobs];
    __shared__ int32_t s_cost[kMaxJobs];
    const int P = a.bsz * a.topk;
    int32_t key = INT_MAX;
    float w = 0.0f;
    if (tid < P) {
        const int t = tid / a.topk;
        key = s_ids[tid] * FP9_MAX_BSZ + t;  // unique: a token picks an expert once
        w = s_wts[tid];
        s_in[tid] = key;
    }
    __syncthreads();
    if (tid < P) {  // counting sort of the unique keys
        int rank = 0;
        for (int q = 0; q < P; ++q) rank += (s_in[q] < key) ? 1 : 0;
        s_key[rank] = key;
        s_w[rank] = w;
    }
    __syncthreads();
    int32_t is_start = 0, run = 0, pos = 0;
    int e = 0;
    if (tid < P) {  // a job starts at every tpj-th key of an expert's run
        e = s_key[tid] / FP9_MAX_BSZ;
        for (int q = tid - 1; q >= 0 && s_key[q] / FP9_MAX_BSZ == e; --q) ++pos;
        run = pos + 1;
        for (int q = tid + 1; q < P && s_key[q] / FP9_MAX_BSZ == e; ++q) ++run;
        is_start = (pos % a.tpj == 0) ? 1 : 0;
    }
    int32_t J = 0;
    int32_t before = block_exclusive_scan(is_start, tid, J);
    if (a.tpj == 1 && a.bsz >= 3) {  // J == P: job tid is key tid
        int64_t G = a.I * J;
        G = G > a.grid ? a.grid : G;
        const int32_t d = spaced_position(tid, J, G, pos, run);
        if (d >= 0) before = d;
    }
    if (is_start) {
        Job j;
        j.bank = 0;
        j.expert = e;
        j.flags = run > a.tpj ? kJobReread : 0;  // the expert's tokens fill more than one job
        j.tok[0] = s_key[tid] % FP9_MAX_BSZ;
        j.w[0] = s_w[tid];
        const bool two = a.tpj == 2 && (tid + 1 < P) && (s_key[tid + 1] / FP9_MAX_BSZ == e);
        j.ntok = two ? 2 : 1;
        j.tok[1] = two ? s_key[tid + 1] % FP9_MAX_BSZ : j.tok[0];
        j.w[1] = two ? s_w[tid + 1] : 0.0f;
        s_jobs[before] = j;
    }
    __syncthreads();
    // Work units: job j's rows start at unit I * C_j + j * gap, C_j the
    // summed row costs of the jobs before it; each CTA gets U / G units. The
    // gap between two jobs is the cost of kJobGapRows one-token rows: a CTA
    // whose range crosses a job boundary walks one more part-filled chunk
    // (a chunk never spans two jobs, and at bsz >= 2 the tokens may change
    // there: y is flushed and x staged again), and every chunk costs a
    // hand-off whatever its rows (measured: such CTAs ended 2-3 us after the
    // median), so it gets that many rows fewer. G is capped
    // so that a CTA's share is at least one row of the dearest job, which
    // leaves no CTA without a row.
    const int32_t cj = tid < J ? row_cost(s_jobs[tid].ntok) : 0;
    int32_t ctot = 0;
    const int32_t cpre = block_exclusive_scan(cj, tid, ctot);
    const int64_t gap = static_cast<int64_t>(kJobGapRows) * kRowCost1;
    const int64_t U = a.I * ctot + (J - 1) * gap;
    const int32_t cmax = (a.bsz >= 2 && a.tpj == 2) ? kRowCost2 : kRowCost1;
    int64_t G = div_nonneg(U, cmax);
    G = G > a.grid ? a.grid : (G < 1 ? 1 : G);
    if (tid < J) {
        s_u0[tid] = a.I * cpre + tid * gap;
        s_cost[tid] = cj;
        a.jobs[tid] = s_jobs[tid];
    }
    __syncthreads();
    // The fused kernel splits phase 0 evenly by rows over min(n0, grid)
    // CTAs, so they hold one row more or less of it (27 or 28 rows of the
    // DeepSeek-V3 shared expert at bsz 2). When phase 0 gives every CTA at
    // least kEvenPhase0Rows rows, phase 1 evens out the totals: CTA b's
    // first unit is its equal share of both phases less the phase-0 units
    // of the CTAs before it (taken when every CTA's share exceeds its
    // phase-0 units by a row: the first units then rise with b and end at
    // U). Otherwise each CTA gets an equal share of phase 1.
    const int64_t n0 = a.impl_rows;
    const int64_t g0 = n0 < a.grid ? n0 : a.grid;
    const int64_t T = U + n0 * kRowCost1;
    const bool even = G == a.grid && n0 >= static_cast<int64_t>(kEvenPhase0Rows) * g0 &&
                      div_nonneg(T, G) >= (div_nonneg(n0 + g0 - 1, g0) + 1) * kRowCost1;
    for (int b = tid; b <= G; b += blockDim.x) {
        // CTA b's first row: the first row whose first unit is at or past
        // the CTA's first unit (b == G: one past the last row)
        int64_t us = cta_start(b, U, G);
        if (even) {
            us = cta_start(b, T, G) - (b < g0 ? cta_start(b, n0, g0) : n0) * kRowCost1;
            us = us < 0 ? 0 : (us > U ? U : us);
        }
        int lo = 0, hi = J - 1;  // the last job starting at or before us
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (s_u0[mid] <= us) lo = mid;
            else hi = mid - 1;
        }
        int64_t r = div_nonneg(us - s_u0[lo] + s_cost[lo] - 1, s_cost[lo]);
        if (r > a.I) r = a.I;  // in the gap after job lo: the next job's first row
        a.cta_row[b] = static_cast<int64_t>(lo) * a.I + r;
    }
    if (tid == 0) {
        a.ctl->njobs = J;
        a.ctl->geff = static_cast<int32_t>(G);
    }
}

// kNorm: stack mode (a.ss set), a separate instance so that the plain
// call's code is not burdened by it.
template <bool kNorm>
__global__ void __launch_bounds__(kRouterThreads) router_kernel(const RouterArgs a) {
    extern __shared__ float s_scores[];  // [bsz, E] scores, then [bsz, E] experts, in the last CTA
    __shared__ float s_red[kRouterThreads / 32][FP9_MAX_BSZ];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e = blockIdx.x;
    const int H4 = a.H / 4;
    const float4* x4 = reinterpret_cast<const float4*>(a.x);
    const float4* w4 = reinterpret_cast<const float4*>(a.wr) + static_cast<int64_t>(e) * H4;

    // W_g is read with the L2 evict-last hint: the router weights (7.3 MB a
    // layer) stay in L2 from one step to the next while the expert weights
    // stream through it evict-first. In stack mode, where the weights of
    // many layers take turns and a row may have left L2, the CTA's row is
    // read before the wait for the kernel queued before this one (the
    // previous layer's combine), so that those loads overlap its tail: no
    // kernel of this library writes W_g, and a kernel that does not signal
    // its dependents early has completed before this one starts (the header
    // states the one case left to the caller). A plain call reads W_g after
    // the wait: with the row in L2 the early read gained nothing and
    // slowed a bsz-2 layer step by 1.1 us (its loads meet the two-token
    // combine's). x and the workspace are always read after the wait.
    const uint64_t keep = l2_evict_last_policy();
    float4 wv[kRouterVec], x0[kRouterVec];
    auto load_w = [&] {
#pragma unroll
        for (int i = 0; i < kRouterVec; ++i) {
            const int c = tid + i * kRouterThreads;
            wv[i] = c < H4 ? ld_global_hint(w4 + c, keep) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    if (kNorm) load_w();
    grid_dependency_wait();
    grid_launch_dependents();
    if (!kNorm) load_w();
#pragma unroll
    for (int i = 0; i < kRouterVec; ++i) {
        const int c = tid + i * kRouterThreads;
        x0[i] = c < H4 ? __ldg(x4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // stack mode: x = h * (1 / sqrt(mean(h^2) + eps)) of each token, the
    // scale of token t formed by warp t from the partial sums of squares
    // (the same bits as any other warp would form)
    __shared__ float s_norm[FP9_MAX_BSZ];
    static_assert(kRouterThreads / 32 >= FP9_MAX_BSZ, "a warp per token");
    constexpr bool norm = kNorm;
    if (norm) {
        const int nparts = a.H / kNormPartCols;
        if (warp < a.bsz) {
            const float sc = rms_scale_parts(a.ss + warp * nparts, nparts, a.H, a.eps, lane);
            if (lane == 0) s_norm[warp] = sc;
        }
        __syncthreads();
        const float sc = s_norm[0];
#pragma unroll
        for (int i = 0; i < kRouterVec; ++i) x0[i] = make_float4(x0[i].x * sc, x0[i].y * sc, x0[i].z * sc, x0[i].w * sc);
    }

    float acc[FP9_MAX_BSZ];
#pragma unroll
    for (int t = 0; t < FP9_MAX_BSZ; ++t) acc[t] = 0.0f;
#pragma unroll
    for (int i = 0; i < kRouterVec; ++i) {
        float v = acc[0];
        v = fmaf(wv[i].x, x0[i].x, v);
        v = fmaf(wv[i].y, x0[i].y, v);
        v = fmaf(wv[i].z, x0[i].z, v);
        v = fmaf(wv[i].w, x0[i].w, v);
        acc[0] = v;
    }
#pragma unroll
    for (int t = 1; t < FP9_MAX_BSZ; ++t) {
        if (t < a.bsz) {
            const float sc = norm ? s_norm[t] : 1.0f;
#pragma unroll
            for (int i = 0; i < kRouterVec; ++i) {
                const int c = tid + i * kRouterThreads;
                if (c < H4) {
                    float4 xv = __ldg(x4 + static_cast<int64_t>(t) * H4 + c);
                    if (norm) xv = make_float4(xv.x * sc, xv.y * sc, xv.z * sc, xv.w * sc);
                    float v = acc[t];
                    v = fmaf(wv[i].x, xv.x, v);
                    v = fmaf(wv[i].y, xv.y, v);
                    v = fmaf(wv[i].z, xv.z, v);
                    v = fmaf(wv[i].w, xv.w, v);
                    acc[t] = v;
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < FP9_MAX_BSZ; ++t) {
        if (t < a.bsz) {
            const float v = warp_sum(acc[t]);
            if (lane == 0) s_red[warp][t] = v;
        }
    }
    __syncthreads();
    if (tid < a.bsz) {
        float v = 0.0f;
        for (int w = 0; w < kRouterThreads / 32; ++w) v += s_red[w][tid];
        a.logits[tid * a.E + e] = v;
        __threadfence();  // the logit is visible before this CTA is counted
    }
    __syncthreads();
    if (tid == 0) {
        s_last = (atomicInc(&a.ctl->ticket, gridDim.x - 1) == gridDim.x - 1) ? 1 : 0;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;

    for (int i = tid; i < a.bsz * a.E; i += kRouterThreads) {
        const float l = __ldcg(a.logits + i);
        const float s = 1.0f / (1.0f + expf(-l));
        s_scores[i] = (s == s) ? s : -INFINITY;
    }
    __syncthreads();
    __shared__ int32_t s_ids[kMaxEntries];
    __shared__ float s_wts[kMaxEntries];
    if (a.E == 32 * a.n_groups && a.topk <= 32 && a.topk_groups * a.topk <= 32)
        select_g32(a, s_scores, reinterpret_cast<int*>(s_scores + a.bsz * a.E), tid, s_ids, s_wts);
    else
        select_all(a, s_scores, tid, s_ids, s_wts);
    if (a.jobs != nullptr) build_jobs(a, tid, s_ids, s_wts);
}

// Validation shared by moe_router and fp9_moe_forward (no CUDA calls).
fp9_status check_layer(const fp9_moe_layer* L, int32_t bsz) {
    FP9_CHECK_ARG(L != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(bsz >= 1 && bsz <= FP9_MAX_BSZ, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(hidden_ok(L->hidden), FP9_ERR_SHAPE);
    FP9_CHECK_ARG(L->inter >= 1 && L->inter <= FP9_MAX_INTER, FP9_ERR_SHAPE);
    FP9_CHECK_ARG(L->n_experts >= 1 && L->n_experts <= FP9_MAX_EXPERTS, FP9_ERR_SHAPE);
    FP9_CHECK_ARG(L->n_groups >= 1 && L->n_groups <= FP9_MAX_GROUPS && L->n_experts % L->n_groups == 0,
                  FP9_ERR_SHAPE);
    FP9_CHECK_ARG(L->topk_groups >= 1 && L->topk_groups <= L->n_groups, FP9_ERR_SHAPE);
    FP9_CHECK_ARG(L->topk >= 1 && L->topk <= FP9_MAX_TOPK &&
                      L->topk <= L->topk_groups * (L->n_experts / L->n_groups),
                  FP9_ERR_SHAPE);
    FP9_CHECK_ARG(L->n_shared >= 0 && L->n_shared <= FP9_MAX_SHARED, FP9_ERR_SHAPE);
    FP9_CHECK_ARG(L->route_scale == L->route_scale, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(L->w_router != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(L->w_router, 16), FP9_ERR_ALIGN);
    fp9_status st = check_bank(L->routed, L->n_experts, L->inter, L->hidden);
    if (st != FP9_OK) return st;
    if (L->n_shared > 0) {
        st = check_bank(L->shared, L->n_shared, L->inter, L->hidden);
        if (st != FP9_OK) return st;
    }
    return FP9_OK;
}

// Queues the router kernel; writes the job list when `build` is set. With
// norm.ss set, x holds h and the router routes RMSNorm(h) (stack mode).
fp9_status launch_router(const fp9_moe_layer* L, const float* x, int32_t bsz, int32_t* ids_out,
                         float* w_out, uint8_t* ws, const WsLayout& lay, bool build, cudaStream_t stream,
                         const NormIn& norm) {
    RouterArgs a;
    a.x = x;
    a.ss = norm.ss;
    a.eps = norm.eps;
    a.wr = L->w_router;
    a.bsz = bsz;
    a.E = L->n_experts;
    a.H = static_cast<int32_t>(L->hidden);
    a.n_groups = L->n_groups;
    a.topk_groups = L->topk_groups;
    a.topk = L->topk;
    a.scale = L->route_scale;
    a.ctl = reinterpret_cast<Control*>(ws);
    a.logits = reinterpret_cast<float*>(ws + lay.off_logits);
    a.ids_ws = reinterpret_cast<int32_t*>(ws + lay.off_ids);
    a.w_ws = reinterpret_cast<float*>(ws + lay.off_w);
    a.ids_out = ids_out;
    a.w_out = w_out;
    a.jobs = build ? reinterpret_cast<Job*>(ws + lay.off_jobs) : nullptr;
    a.cta_row = reinterpret_cast<int64_t*>(ws + lay.off_ctarow);
    a.I = L->inter;
    a.grid = lay.grid;
    a.tpj = 1;  // an MoE call plans one token per job
    a.impl_rows = static_cast<int64_t>(L->n_shared) * bsz * L->inter;  // one job per shared expert and token
    // scores and their experts (the fast selection sorts both in place)
    const size_t smem = 2 * sizeof(float) * bsz * L->n_experts;  // <= 64 KB
    static DeviceOnce attr;
    const fp9_status ast = attr.run([] {
        FP9_CUDA_TRY(cudaFuncSetAttribute(router_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(2 * sizeof(float) * FP9_MAX_BSZ * FP9_MAX_EXPERTS)));
        FP9_CUDA_TRY(cudaFuncSetAttribute(router_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(2 * sizeof(float) * FP9_MAX_BSZ * FP9_MAX_EXPERTS)));
        return FP9_OK;
    });
    if (ast != FP9_OK) return ast;
    if (norm.ss != nullptr)
        FP9_CUDA_TRY(launch_pdl(router_kernel<true>, dim3(L->n_experts), dim3(kRouterThreads), smem, stream, a));
    else
        FP9_CUDA_TRY(launch_pdl(router_kernel<false>, dim3(L->n_experts), dim3(kRouterThreads), smem, stream, a));
    return FP9_OK;
}

}  // namespace fp9

using namespace fp9;

extern "C" size_t fp9_moe_workspace_bytes(const fp9_moe_layer* layer, int32_t bsz) {
    if (check_layer(layer, bsz) != FP9_OK) return 0;
    const int32_t sms = device_sm_count();
    if (sms <= 0) return 0;
    return moe_layout(bsz, layer->n_experts, layer->topk, layer->hidden, expert_grid(sms, true)).total;
}

// fp9_moe_forward with host buffers: x and y go through two staging rows
// at the end of the workspace, copied in and out on the call's stream.
static size_t host_stage_bytes(int32_t bsz, int64_t hidden) {
    return align_up(sizeof(float) * static_cast<size_t>(bsz) * static_cast<size_t>(hidden));
}

extern "C" size_t fp9_moe_host_workspace_bytes(const fp9_moe_layer* layer, int32_t bsz) {
    const size_t base = fp9_moe_workspace_bytes(layer, bsz);
    if (base == 0) return 0;
    return align_up(base) + 2 * host_stage_bytes(bsz, layer->hidden);
}

extern "C" fp9_status fp9_moe_forward_host(const fp9_moe_layer* layer, const float* x_host, int32_t bsz,
                                           float* y_host, void* ws, size_t ws_bytes, int32_t* d_status,
                                           void* stream) {
    fp9_status st = check_layer(layer, bsz);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(x_host != nullptr && y_host != nullptr && ws != nullptr && x_host != y_host, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(ws, kAlign), FP9_ERR_ALIGN);
    const size_t base = fp9_moe_workspace_bytes(layer, bsz);
    FP9_CHECK_ARG(base > 0, FP9_ERR_CUDA);
    const size_t stage = host_stage_bytes(bsz, layer->hidden);
    FP9_CHECK_ARG(ws_bytes >= align_up(base) + 2 * stage, FP9_ERR_WORKSPACE);
    uint8_t* w = static_cast<uint8_t*>(ws);
    float* xd = reinterpret_cast<float*>(w + align_up(base));
    float* yd = reinterpret_cast<float*>(w + align_up(base) + stage);
    const size_t bytes = sizeof(float) * static_cast<size_t>(bsz) * static_cast<size_t>(layer->hidden);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // A page-locked y_host that the device can address (its device address
    // from cudaPointerGetAttributes, 16-byte aligned) is written by the
    // combine kernel itself: no copy back is queued after it.
    float* y_direct = nullptr;
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, y_host) == cudaSuccess) {
        if (pa.type == cudaMemoryTypeHost && pa.devicePointer != nullptr && aligned(pa.devicePointer, 16))
            y_direct = static_cast<float*>(pa.devicePointer);
    } else {
        (void)cudaGetLastError();  // an address the runtime does not know: copy back
    }
    FP9_CUDA_TRY(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s));
    st = fp9_moe_forward(layer, xd, bsz, y_direct != nullptr ? y_direct : yd, nullptr, nullptr, ws, base, d_status,
                         stream);
    if (st != FP9_OK) return st;
    if (y_direct == nullptr) FP9_CUDA_TRY(cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, s));
    return FP9_OK;
}

extern "C" fp9_status moe_router(const fp9_moe_layer* layer, const float* x, int32_t bsz, int32_t* ids,
                                 float* weights, void* ws, size_t ws_bytes, void* stream) {
    fp9_status st = check_layer(layer, bsz);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(x != nullptr && ids != nullptr && weights != nullptr && ws != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(x, 16), FP9_ERR_ALIGN);
    FP9_CHECK_ARG(aligned(ws, kAlign), FP9_ERR_ALIGN);
    const int32_t sms = device_sm_count();
    FP9_CHECK_ARG(sms > 0, FP9_ERR_CUDA);
    const WsLayout lay = moe_layout(bsz, layer->n_experts, layer->topk, layer->hidden, expert_grid(sms, true));
    FP9_CHECK_ARG(ws_bytes >= lay.total, FP9_ERR_WORKSPACE);
    return launch_router(layer, x, bsz, ids, weights, static_cast<uint8_t*>(ws), lay, false,
                         static_cast<cudaStream_t>(stream), NormIn{nullptr, 0.0f});
}
