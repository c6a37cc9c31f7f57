// Work plan shared by the router, the fused expert kernel and the combine
// kernel: job records and the workspace layout.
//
// A job is one FFN streamed for a group of up to two tokens (the pages' bsz =
// 2 pair hits nearly disjoint expert sets, so most jobs hold one token of a
// pair; a shared expert holds both) [MTP-9.2]. The jobs' intermediate rows
// are concatenated and split evenly over the CTAs of the fused kernel: each
// CTA owns one contiguous range of (job, row) pairs and writes one fp32
// partial output per job it touches; the combine kernel adds them in a
// fixed order. This is the single-GPU restatement of the pages' split of
// the FFN intermediate dimension over nodes with f32 partial sums
// [MEMOIR-COMM], [DS4-TP].
#pragma once

#include <cstddef>
#include <cstdint>

#include "fp9moe.h"

namespace fp9 {

constexpr int kTokensPerJob = 2;
// the combine kernel keeps per-job data for at most this many jobs
constexpr int kMaxJobs = 256;
static_assert(FP9_MAX_SHARED * ((FP9_MAX_BSZ + 1) / 2) + FP9_MAX_BSZ * FP9_MAX_TOPK <= kMaxJobs,
              "job count bound");

struct __align__(16) Job {
    int32_t bank;      // 0 = routed experts (or the dense FFN), 1 = shared
    int32_t expert;    // index inside the bank
    int32_t ntok;      // 1 or 2
    int32_t b0;        // first CTA of the fused kernel that covers this job
    int32_t tok[kTokensPerJob];
    float w[kTokensPerJob];         // routing weight per token (1 for shared / dense)
    int32_t seg_base[kTokensPerJob];  // where this job's partials start in each token's list
    int32_t pad[2];
};
static_assert(sizeof(Job) == 48, "Job is 48 bytes");

struct Control {
    uint32_t ticket;   // last-arriver counter of the router (self-resetting)
    int32_t njobs;     // jobs written by the router
    int32_t nseg[FP9_MAX_BSZ];  // partials per token
};

constexpr size_t kAlign = 256;

inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

struct WsLayout {
    size_t off_logits = 0, off_ids = 0, off_w = 0, off_jobs = 0, off_partial = 0, total = 0;
    int32_t jmax = 0;     // largest possible job count
    int32_t maxseg = 0;   // partial slots per token
    int32_t grid = 0;     // CTAs of the fused kernel
};

// Partial outputs are stored token-major: token t's partials are the
// rows [t * maxseg, t * maxseg + nseg[t]) of a [bsz * maxseg, hidden]
// fp32 array. A token's jobs cover disjoint row ranges, so its partials
// number at most (CTAs) + (jobs holding the token).
inline WsLayout moe_layout(int32_t bsz, int32_t n_experts, int32_t topk, int32_t n_shared,
                           int64_t inter, int64_t hidden, int32_t grid) {
    WsLayout L;
    const int32_t pairs = (bsz + kTokensPerJob - 1) / kTokensPerJob;
    L.jmax = n_shared * pairs + bsz * topk;
    L.grid = grid;
    L.maxseg = grid + topk + n_shared;
    size_t off = align_up(sizeof(Control));
    L.off_logits = off;
    off = align_up(off + sizeof(float) * bsz * n_experts);
    L.off_ids = off;
    off = align_up(off + sizeof(int32_t) * bsz * topk);
    L.off_w = off;
    off = align_up(off + sizeof(float) * bsz * topk);
    L.off_jobs = off;
    off = align_up(off + sizeof(Job) * L.jmax);
    L.off_partial = off;
    off = align_up(off + sizeof(float) * static_cast<size_t>(bsz) * L.maxseg * hidden);
    L.total = off;
    return L;
}

inline WsLayout dense_layout(int32_t bsz, int64_t inter, int64_t hidden, int32_t grid) {
    WsLayout L;
    L.jmax = (bsz + kTokensPerJob - 1) / kTokensPerJob;
    L.grid = grid;
    L.maxseg = grid + 1;
    L.off_partial = align_up(sizeof(Control));
    L.total = align_up(L.off_partial + sizeof(float) * static_cast<size_t>(bsz) * L.maxseg * hidden);
    return L;
}

// First row of CTA b, and the CTA that owns row p, for n rows over g CTAs
// (CTA b owns rows [b*n/g, (b+1)*n/g); g <= n, so none is empty).
__host__ __device__ inline int64_t cta_start(int64_t b, int64_t n, int64_t g) { return b * n / g; }
__host__ __device__ inline int64_t cta_of_row(int64_t p, int64_t n, int64_t g) {
    return ((p + 1) * g - 1) / n;
}

}  // namespace fp9
