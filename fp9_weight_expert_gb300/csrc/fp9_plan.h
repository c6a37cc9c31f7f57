// Work plan shared by the router, the fused expert kernel and the combine
// kernel: job records and the workspace layout.
//
// A job is one FFN streamed for a group of up to two tokens (the pages' bsz =
// 2 pair hits nearly disjoint expert sets, so most jobs hold one token of a
// pair; a shared expert holds both) [MTP-9.2]. An MoE call plans one token
// per job instead (tpj = 1): the jobs of an expert chosen by several tokens
// sit next to each other in the row sequence, so CTAs running side by side
// stream the same rows and all but the first read of each row hit in L2 (HBM
// bytes stay those of the union of experts), and every CTA runs the
// one-token kernel, the fastest per weight. The dense FFN keeps token pairs
// (each of its rows is streamed for both tokens at once). The jobs' intermediate rows
// are concatenated and split over the CTAs of the fused kernel: each CTA
// owns one contiguous range of (job, row) pairs, keeps y of the job's tokens
// in registers and adds it into its own fp32 partial output of each token;
// the combine kernel adds the CTAs' partials in CTA order. This is the
// single-GPU restatement of the pages' split of the FFN intermediate
// dimension over nodes with f32 partial sums [MEMOIR-COMM], [DS4-TP].
//
// The fused kernel runs two phases. Phase 0 streams the jobs that need no
// routing (the shared experts of an MoE layer, or the dense FFN), split
// evenly by rows; phase 1 streams the routed experts on the router's plan.
// Phase 0 does not wait for the router, so the router's selection runs
// while the shared expert streams.
//
// The router's split balances work, not rows: a row of a two-token job
// streams the same bytes as a one-token row but does about twice the
// multiply-adds, so rows are weighted by row_cost(ntok) units and every CTA
// gets an equal share of the units. A row belongs to the CTA whose unit
// range holds the row's first unit.
#pragma once

#include <cstddef>
#include <cstdint>

#include "fp9moe.h"

namespace fp9 {

constexpr int kTokensPerJob = 2;
// work units of one intermediate row of a job holding 1 or 2 tokens
constexpr int32_t kRowCost1 = 8, kRowCost2 = 11;
__host__ __device__ inline int32_t row_cost(int32_t ntok) { return ntok == 2 ? kRowCost2 : kRowCost1; }
// the router's split charges a CTA whose range crosses a job boundary this
// many one-token rows (the extra part-filled chunk it walks; 0, 4, 8 and 12
// were measured: 8 gave the shortest DeepSeek-V3 layer steps at bsz 1 to 8)
constexpr int32_t kJobGapRows = 8;
// the router's split evens out each CTA's total of phase-0 and phase-1 rows
// when phase 0 gives every CTA at least this many rows; with fewer, a CTA is
// done with phase 0 before the router's plan is ready, so only equal
// phase-1 shares matter (DeepSeek-V3 layer, evened against equal shares:
// bsz 1, 14 phase-0 rows, 82.3 against 81.4 us per stacked layer; bsz 2,
// 27 rows, 148.9 against 149.2; bsz 5 339.3 against 340.6)
constexpr int32_t kEvenPhase0Rows = 24;

// Job flags. kJobReread: another job of the same call streams these rows
// too (an expert chosen by several tokens, a shared expert at bsz >= 2);
// the fused kernel then reads them with the L2 evict-normal priority, so
// that the other job's reads find them in L2 although its CTAs reach the
// rows some microseconds earlier or later, while the rest of the weight
// stream is read evict-first.
constexpr int32_t kJobReread = 1;

// Stack mode of an MoE call (fp9_moe_forward_residual). The layer's input
// is x = RMSNorm(h) (unit gain), formed where it is read: the router and the
// fused kernel read h and the row's sum of squares, which the previous
// call's combine left as partial sums, one per kNormPartCols columns of each
// token's row (ss[t * H / kNormPartCols + b]); the combine adds y into h
// and writes the new partial sums.
constexpr int kNormPartCols = 16;
struct NormIn {
    const float* ss;  // partial sums of squares of h, or NULL (x is the input as given)
    float eps;
};

// the router keeps one thread per routed job
constexpr int kMaxJobs = FP9_MAX_BSZ * FP9_MAX_TOPK;  // 128

struct __align__(16) Job {
    int32_t bank;      // 0 = routed experts (or the dense FFN), 1 = shared
    int32_t expert;    // index inside the bank
    int32_t ntok;      // 1 or 2
    int32_t flags;     // kJobReread
    int32_t tok[kTokensPerJob];
    float w[kTokensPerJob];  // routing weight per token (1 for shared / dense)
};
static_assert(sizeof(Job) == 32, "Job is 32 bytes");

struct Control {
    uint32_t ticket;   // last-arriver counter of the router (self-resetting)
    int32_t njobs;     // routed jobs written by the router
    int32_t geff;      // CTAs of the fused kernel that own routed rows
    int32_t pad;
};

__host__ __device__ inline int32_t token_groups(int32_t bsz, int32_t tpj) { return (bsz + tpj - 1) / tpj; }

// Jobs of phase 0 (no routing): nexp experts of one bank for every group of
// tpj tokens (1 or 2), group-major (job j: token group j / nexp, expert
// j % nexp), so that consecutive jobs hold the same tokens.
__host__ __device__ inline Job implicit_job(int32_t j, int32_t nexp, int32_t bank, int32_t bsz, int32_t tpj) {
    Job jb;
    const int32_t p = j / nexp;
    jb.bank = bank;
    jb.expert = j - p * nexp;
    jb.flags = token_groups(bsz, tpj) > 1 ? kJobReread : 0;
    jb.tok[0] = tpj * p;
    jb.ntok = (tpj == 2 && tpj * p + 1 < bsz) ? 2 : 1;
    jb.tok[1] = jb.ntok == 2 ? jb.tok[0] + 1 : jb.tok[0];
    jb.w[0] = 1.0f;
    jb.w[1] = jb.ntok == 2 ? 1.0f : 0.0f;
    return jb;
}

constexpr size_t kAlign = 256;

inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

struct WsLayout {
    size_t off_logits = 0, off_ids = 0, off_w = 0, off_jobs = 0, off_ctarow = 0, off_mask = 0, off_partial = 0,
           total = 0;
    int32_t jmax = 0;  // largest routed job count
    int32_t grid = 0;  // CTAs of the fused kernel
};

// Partials are token-major: token t's partial of CTA b is row t * grid + b
// of a [bsz * grid, hidden] fp32 array; bit t of mask[b] says whether CTA b
// wrote it (a CTA that never held token t leaves its row unwritten).
inline size_t partial_bytes(int32_t bsz, int32_t grid, int64_t hidden) {
    return sizeof(float) * static_cast<size_t>(bsz) * grid * hidden;
}

inline WsLayout moe_layout(int32_t bsz, int32_t n_experts, int32_t topk, int64_t hidden, int32_t grid) {
    WsLayout L;
    L.jmax = bsz * topk;
    L.grid = grid;
    size_t off = align_up(sizeof(Control));
    L.off_logits = off;
    off = align_up(off + sizeof(float) * bsz * n_experts);
    L.off_ids = off;
    off = align_up(off + sizeof(int32_t) * bsz * topk);
    L.off_w = off;
    off = align_up(off + sizeof(float) * bsz * topk);
    L.off_jobs = off;
    off = align_up(off + sizeof(Job) * L.jmax);
    L.off_ctarow = off;  // [grid + 1] first (job * I + row) of each CTA in phase 1
    off = align_up(off + sizeof(int64_t) * (grid + 1));
    L.off_mask = off;
    off = align_up(off + sizeof(uint32_t) * grid);
    L.off_partial = off;
    off = align_up(off + partial_bytes(bsz, grid, hidden));
    L.total = off;
    return L;
}

inline WsLayout dense_layout(int32_t bsz, int64_t hidden, int32_t grid) {
    WsLayout L;
    L.grid = grid;
    L.off_mask = align_up(sizeof(Control));
    L.off_partial = align_up(L.off_mask + sizeof(uint32_t) * grid);
    L.total = align_up(L.off_partial + partial_bytes(bsz, grid, hidden));
    return L;
}

// CTAs of the fused kernel: one per SM. An MoE call leaves one SM free: the
// router's last CTA (which builds the plan) still holds an SM when the
// fused kernel's CTAs start, and those take the SMs in the order they free
// up, so none of them waits for the router to finish.
inline int32_t expert_grid(int32_t sms, bool moe) { return moe && sms > 1 ? sms - 1 : sms; }

// a / d for a >= 0, d > 0: a 32-bit division when both fit (a 64-bit
// division is a long emulated sequence on the GPU, and the router's plan,
// which waits on these, is on the step's critical path)
__host__ __device__ inline int64_t div_nonneg(int64_t a, int64_t d) {
    if ((static_cast<uint64_t>(a) >> 32) == 0 && (static_cast<uint64_t>(d) >> 32) == 0)
        return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(d));
    return a / d;
}

// First unit of CTA b, and the CTA that owns unit p, for n units over g
// CTAs (CTA b owns units [b*n/g, (b+1)*n/g)). With one unit per row and
// g <= n no CTA is empty.
__host__ __device__ inline int64_t cta_start(int64_t b, int64_t n, int64_t g) { return div_nonneg(b * n, g); }
__host__ __device__ inline int64_t cta_of_row(int64_t p, int64_t n, int64_t g) {
    return ((p + 1) * g - 1) / n;
}

}  // namespace fp9
