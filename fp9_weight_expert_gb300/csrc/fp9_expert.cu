// Fused fp9 expert kernel and the fixed-order combine of its partial sums.
//
// What is computed, per job (one FFN for one or two tokens) [MEMOIR-FP9]:
//   g = W_gate x,  u = W_up x,  h = SiLU(g) * u * w_route,  y += W_down h
// with every weight streamed from HBM once per call as fp9 (body byte +
// sign bit), decoded in registers by shifting the body into fp16 bits and
// widening to fp32, and all arithmetic in fp32.
//
// The pages split an FFN's intermediate dimension over 32 CPU nodes and
// sum their f32 partial outputs on the host ([MEMOIR-COMM]: "真正难的不是
// 把参数塞下，而是通信"; [MEMOIR-16]: "16 tok/s 之后"; [DS4-TP]: partial sums
// stay f32). Here the same split runs over the SMs of one GPU: the jobs'
// intermediate rows are concatenated and cut into one contiguous range per
// CTA (a persistent grid of one CTA per SM), each CTA keeps its share of y
// in registers and writes it once per job it touches, and a second kernel
// adds those partials in a fixed order.
//
// CTA layout (one per SM): warps 0..NW-1 are consumers, each thread owning
// 16 consecutive columns of the hidden dimension; warp NW is the producer,
// whose lane 0 streams chunks of kR rows of one matrix (bodies, then signs)
// with bulk copies into a ring of shared-memory stages guarded by mbarriers.
// Per chunk: gate rows, up rows (each a dot product over the hidden
// dimension, reduced across the CTA), then the down rows (an axpy into the
// thread's 16 columns of y, no reduction).
//
// Every wait is bounded (a timeout sets FP9_ERR_TIMEOUT in the status word
// and the CTA drains its copies in flight and returns).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9_plan.h"
#include "fp9moe.h"

namespace fp9 {

constexpr int kMaxRows = 8;                                     // rows per chunk (4 or 8)
constexpr int kMaxStages = 16;
constexpr int kMaxConsumerWarps = FP9_MAX_HIDDEN / 16 / 32;     // 14
constexpr int kMaxThreads = kMaxConsumerWarps * 32 + 32;        // 480
constexpr int kMaxV = 2 * kMaxRows * kTokensPerJob;             // reduced values per chunk
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;           // 1 s

struct BankPtrs {
    const uint8_t* body[3];  // gate, up, down_t
    const uint8_t* sign[3];
};

struct ExpertArgs {
    BankPtrs bank[2];        // 0: routed experts / dense FFN, 1: shared experts
    const float* x;          // [bsz, H]
    float* partial;          // token-major: [bsz * maxseg, H]
    const Job* jobs;         // MoE mode
    const Control* ctl;      // MoE mode: job count
    int32_t dense_jobs;      // > 0: dense mode, jobs are implicit
    int32_t bsz;
    int32_t H;
    int32_t maxseg;
    int64_t I;
    int32_t nstages;
    int32_t no_copy;         // self-test: the producer issues no copies
    int32_t* status;
    uint64_t timeout_ns;
};

struct SmemCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t red[2];
    int abort;
    int never;  // stays 0: a flag nobody raises
    float red_vals[2][kMaxConsumerWarps][kMaxV];
};

constexpr uint32_t kRingOffset = (sizeof(SmemCtl) + 127) / 128 * 128;

__device__ __forceinline__ Job get_job(const Job* jobs, int32_t dense_jobs, int32_t bsz, int j) {
    if (dense_jobs > 0) {
        Job jb;
        jb.bank = 0;
        jb.expert = 0;
        jb.pad[0] = jb.pad[1] = 0;
        jb.tok[0] = kTokensPerJob * j;
        jb.ntok = (kTokensPerJob * j + 1 < bsz) ? 2 : 1;
        jb.tok[1] = jb.ntok == 2 ? jb.tok[0] + 1 : jb.tok[0];
        jb.w[0] = 1.0f;
        jb.w[1] = jb.ntok == 2 ? 1.0f : 0.0f;
        jb.b0 = -1;  // computed where needed
        jb.seg_base[0] = jb.seg_base[1] = 0;  // a dense token is in exactly one job
        return jb;
    }
    return jobs[j];
}

// Rows [start, end) of the job sequence owned by CTA b. Only the first
// min(G, N) CTAs get rows, so every CTA that works owns at least one row.
struct Range {
    int64_t start, end, n, g;
};

__device__ __forceinline__ Range cta_range(int32_t J, int64_t I, int64_t grid, int64_t b) {
    Range r;
    r.n = static_cast<int64_t>(J) * I;
    r.g = r.n < grid ? r.n : grid;
    r.start = b < r.g ? cta_start(b, r.n, r.g) : 0;
    r.end = b < r.g ? cta_start(b + 1, r.n, r.g) : 0;
    return r;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Butterfly reduce-scatter of V values over a warp: returns, in lane l, the
// warp-wide sum of value (l mod V). V - 1 + log2(32 / V) shuffles.
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V], int lane) {
#pragma unroll
    for (int m = V / 2; m >= 1; m >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < m; ++i) {
            const float send = upper ? v[i] : v[i + m];
            const float keep = upper ? v[i + m] : v[i];
            v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
        }
    }
    float r = v[0];
#pragma unroll
    for (int m = V; m < 32; m <<= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, m);
    return r;
}


// The walk over a CTA's rows, one chunk of at most R rows at a time (a
// chunk never crosses a job boundary). Producer and consumers walk the
// same sequence.
struct Walk {
    int64_t pos, end, I, r0;
    int j;
    int rows;  // rows of the current chunk

    __device__ __forceinline__ void begin(const Range& rg, int64_t I_, int R) {
        I = I_;
        pos = rg.start;
        end = rg.end;
        j = static_cast<int>(pos / I);
        r0 = pos - static_cast<int64_t>(j) * I;
        set_rows(R);
    }
    __device__ __forceinline__ void set_rows(int R) {
        int r = R;
        if (I - r0 < r) r = static_cast<int>(I - r0);
        if (end - pos < r) r = static_cast<int>(end - pos);
        rows = r;
    }
    __device__ __forceinline__ bool done() const { return pos >= end; }
    // Advances past the current chunk; returns true when the next chunk
    // starts a new job.
    __device__ __forceinline__ bool next(int R) {
        pos += rows;
        r0 += rows;
        bool new_job = false;
        if (r0 == I && pos < end) {
            ++j;
            r0 = 0;
            new_job = true;
        }
        set_rows(R);
        return new_job;
    }
};

// ------------------------------------------------------------- producer ---

// Streams, per chunk c, its gate rows, its up rows, then the down rows of
// chunk c - 1 (the consumers use chunk c - 1's down rows while chunk c's
// gate/up sums are being reduced across the CTA); the last chunk's down
// rows come after the loop.
template <int R>
__device__ void producer(const ExpertArgs& a, SmemCtl& ctl, uint8_t* ring, const Range& rg,
                         uint32_t stage_bytes) {
    const uint64_t pol = l2_evict_first_policy();
    const int H = a.H;
    const uint32_t NS = static_cast<uint32_t>(a.nstages);
    uint32_t it = 0;
    bool ok = true;

    auto issue = [&](int m, const Job& job, int64_t r0, int rows) -> bool {
        const uint32_t slot = it % NS, ph = (it / NS) & 1u;
        if (!mbar_wait_bounded(smem_addr(&ctl.empty[slot]), ph ^ 1u, a.timeout_ns, &ctl.abort)) return false;
        const BankPtrs& bp = a.bank[job.bank];
        const int64_t row = static_cast<int64_t>(job.expert) * a.I + r0;
        const uint32_t bb = static_cast<uint32_t>(rows * H), sb = static_cast<uint32_t>(rows * (H / 8));
        const uint32_t full = smem_addr(&ctl.full[slot]);
        const uint32_t dst = smem_addr(ring + slot * stage_bytes);
        if (!a.no_copy) {
            mbar_arrive_expect_tx(full, bb + sb);
            bulk_g2s(dst, bp.body[m] + row * H, bb, full, pol);
            bulk_g2s(dst + R * H, bp.sign[m] + row * (H / 8), sb, full, pol);
        }
        ++it;
        return true;
    };

    Walk w;
    w.begin(rg, a.I, R);
    Job job = get_job(a.jobs, a.dense_jobs, a.bsz, w.j);
    Job pjob = job;
    int64_t pr0 = 0;
    int prows = 0;
    bool pending = false;
    while (!w.done() && ok) {
        ok = issue(0, job, w.r0, w.rows) && issue(1, job, w.r0, w.rows);
        if (ok && pending) ok = issue(2, pjob, pr0, prows);
        pjob = job;
        pr0 = w.r0;
        prows = w.rows;
        pending = true;
        if (w.next(R)) job = get_job(a.jobs, a.dense_jobs, a.bsz, w.j);
    }
    if (ok && pending) ok = issue(2, pjob, pr0, prows);
    if (!ok) {
        record_status(a.status, FP9_ERR_TIMEOUT);
        ctl.abort = 1;
        if (!a.no_copy) {  // let the copies already issued land before the CTA exits
            const uint32_t first = it > NS ? it - NS : 0u;
            for (uint32_t s = first; s < it; ++s)
                (void)mbar_wait_bounded(smem_addr(&ctl.full[s % NS]), (s / NS) & 1u, a.timeout_ns, &ctl.never);
        }
    }
}

// ------------------------------------------------------------- consumer ---

// x and y of a thread's 16 columns, per token, in the pair order of
// decode16_pairs: p[2k] = (c[4k], c[4k+2]), p[2k+1] = (c[4k+1], c[4k+3]).
template <int MT>
struct Cols {
    float2 p[MT][8];
};

struct Stages {
    uint32_t it = 0;      // stages consumed
    uint32_t red_it = 0;  // CTA reductions started
};

__device__ __forceinline__ bool wait_stage(const ExpertArgs& a, SmemCtl& ctl, const Stages& cs, uint32_t& slot) {
    const uint32_t NS = static_cast<uint32_t>(a.nstages);
    slot = cs.it % NS;
    return mbar_wait_bounded(smem_addr(&ctl.full[slot]), (cs.it / NS) & 1u, a.timeout_ns, &ctl.abort);
}

__device__ __forceinline__ void release_stage(SmemCtl& ctl, Stages& cs, uint32_t slot, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl.empty[slot]));
    ++cs.it;
}

// Partial dot products of the stage's `rows` rows with x over my 16
// columns, then their warp-level reduce-scatter into red_row[base + ...].
template <int R, int T, int MT>
__device__ __forceinline__ void gateup_rows(const uint8_t* st, int H, int rows, int c16, bool active,
                                            const Cols<MT>& x, float* red_row, int base, int lane) {
    float v[R * T];
#pragma unroll
    for (int i = 0; i < R * T; ++i) v[i] = 0.0f;
    if (active) {
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            if (rr < rows) {
                const uint4 b = *reinterpret_cast<const uint4*>(st + rr * H + c16 * 16);
                const uint32_t s16 = *reinterpret_cast<const uint16_t*>(st + R * H + rr * (H / 8) + c16 * 2);
                float2 w[8];
                decode16_pairs(b, s16, w);
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        a0 = fmaf(w[k].x, x.p[t][k].x, a0);
                        a1 = fmaf(w[k].y, x.p[t][k].y, a1);
                    }
                    v[rr * T + t] = a0 + a1;
                }
            }
        }
    }
    const float r = warp_reduce_scatter<R * T>(v, lane);
    if (lane < R * T) red_row[base + lane] = r;
}

// y[c] += h_row * W_down^T[row, c] over my 16 columns; lane (rr * T + t)
// of `hv` holds h of row rr, token t.
template <int R, int T, int MT>
__device__ __forceinline__ void down_rows(const uint8_t* st, int H, int rows, int c16, bool active, float hv,
                                          Cols<MT>& y) {
    float h[R][T];
#pragma unroll
    for (int rr = 0; rr < R; ++rr)
#pragma unroll
        for (int t = 0; t < T; ++t) h[rr][t] = __shfl_sync(0xFFFFFFFFu, hv, rr * T + t);
    if (!active) return;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        if (rr < rows) {
            const uint4 b = *reinterpret_cast<const uint4*>(st + rr * H + c16 * 16);
            const uint32_t s16 = *reinterpret_cast<const uint16_t*>(st + R * H + rr * (H / 8) + c16 * 2);
            float2 w[8];
            decode16_pairs(b, s16, w);
#pragma unroll
            for (int t = 0; t < T; ++t)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    y.p[t][k].x = fmaf(h[rr][t], w[k].x, y.p[t][k].x);
                    y.p[t][k].y = fmaf(h[rr][t], w[k].y, y.p[t][k].y);
                }
        }
    }
}

// Gate and up stages of one chunk: waits, computes, releases, and writes
// this warp's reduced values for the chunk's CTA sum. Returns false on timeout.
template <int R, int T, int MT>
__device__ __forceinline__ bool gateup_chunk(const ExpertArgs& a, SmemCtl& ctl, const uint8_t* ring,
                                             uint32_t stage_bytes, Stages& cs, int rows, int c16, bool active,
                                             const Cols<MT>& x, int warp, int lane) {
    float* red_row = ctl.red_vals[cs.red_it & 1u][warp];
#pragma unroll 1
    for (int m = 0; m < 2; ++m) {
        uint32_t slot;
        if (!wait_stage(a, ctl, cs, slot)) return false;
        gateup_rows<R, T, MT>(ring + slot * stage_bytes, a.H, rows, c16, active, x, red_row, m * R * T, lane);
        release_stage(ctl, cs, slot, lane);
    }
    if (lane == 0) mbar_arrive(smem_addr(&ctl.red[cs.red_it & 1u]));
    return true;
}

template <int R, int T, int MT>
__device__ __forceinline__ bool down_chunk(const ExpertArgs& a, SmemCtl& ctl, const uint8_t* ring,
                                           uint32_t stage_bytes, Stages& cs, int rows, int c16, bool active,
                                           float hv, Cols<MT>& y, int lane) {
    uint32_t slot;
    if (!wait_stage(a, ctl, cs, slot)) return false;
    down_rows<R, T, MT>(ring + slot * stage_bytes, a.H, rows, c16, active, hv, y);
    release_stage(ctl, cs, slot, lane);
    return true;
}

// Completes the CTA sum of chunk `red_it` and returns, in lane
// (rr * T + t), h = SiLU(g) * u * w_route for row rr, token t.
template <int R, int T>
__device__ __forceinline__ bool finish_sum(const ExpertArgs& a, SmemCtl& ctl, Stages& cs, float w0, float w1, int NW,
                                           int lane, float& hv) {
    constexpr int V = R * T;
    const uint32_t b = cs.red_it & 1u;
    if (!mbar_wait_bounded(smem_addr(&ctl.red[b]), (cs.red_it >> 1) & 1u, a.timeout_ns, &ctl.abort)) return false;
    ++cs.red_it;
    float tot = 0.0f;
    if (lane < 2 * V)
        for (int w = 0; w < NW; ++w) tot += ctl.red_vals[b][w][lane];
    const float u = __shfl_down_sync(0xFFFFFFFFu, tot, V);
    const float wt = (T == 2 && (lane & 1)) ? w1 : w0;
    hv = (lane < V) ? silu(tot) * u * wt : 0.0f;
    return true;
}

// What the consumers keep of a job: its token count, routing weights, and
// for each token the row of the partial list this CTA writes its share to
// (slot = tok * maxseg + seg_base + (b - b0)).
struct JobState {
    int ntok;
    float w0, w1;
    int slot0, slot1;
};

__device__ __forceinline__ JobState job_state(const ExpertArgs& a, const Job& job, int job_index, const Range& rg) {
    const int64_t b0 = job.b0 >= 0 ? job.b0 : cta_of_row(static_cast<int64_t>(job_index) * a.I, rg.n, rg.g);
    const int rel = static_cast<int>(static_cast<int64_t>(blockIdx.x) - b0);
    JobState js;
    js.ntok = job.ntok;
    js.w0 = job.w[0];
    js.w1 = job.w[1];
    js.slot0 = job.tok[0] * a.maxseg + job.seg_base[0] + rel;
    js.slot1 = job.tok[1] * a.maxseg + job.seg_base[1] + rel;
    return js;
}

// Writes y (this CTA's share of one job) to the job's partial slots.
template <int MT>
__device__ __forceinline__ void flush_partial(const ExpertArgs& a, int ntok, int slot0, int slot1, int c16,
                                              bool active, const Cols<MT>& y) {
    if (!active) return;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t < ntok) {
            const int slot = t == 0 ? slot0 : slot1;
            float4* dst = reinterpret_cast<float4*>(a.partial + static_cast<int64_t>(slot) * a.H + c16 * 16);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                dst[k] = make_float4(y.p[t][2 * k].x, y.p[t][2 * k + 1].x, y.p[t][2 * k].y, y.p[t][2 * k + 1].y);
        }
    }
}

template <int MT>
__device__ __forceinline__ void load_x(const ExpertArgs& a, const Job& job, int c16, bool active, Cols<MT>& x) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const bool use = active && t < job.ntok;
        const int tok = t == 0 ? job.tok[0] : job.tok[1];
        const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<int64_t>(tok) * a.H + c16 * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 xv = use ? __ldg(src + k) : make_float4(0.f, 0.f, 0.f, 0.f);
            x.p[t][2 * k] = make_float2(xv.x, xv.z);
            x.p[t][2 * k + 1] = make_float2(xv.y, xv.w);
        }
    }
}

template <int MT>
__device__ __forceinline__ void zero_cols(Cols<MT>& y) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int k = 0; k < 8; ++k) y.p[t][k] = make_float2(0.f, 0.f);
}

// Per chunk c: gate/up of c, arrive at c's CTA sum, down rows of c - 1
// (whose h is known), then wait for c's sum. x follows the gate/up job, y
// the down job; y is written out (and cleared) after the last down chunk
// of each job.
template <int R, int MT>
__device__ void consumer(const ExpertArgs& a, SmemCtl& ctl, const uint8_t* ring, const Range& rg,
                         uint32_t stage_bytes, int NW, int warp, int lane) {
    const int c16 = warp * 32 + lane;
    const bool active = c16 < a.H / 16;
    Cols<MT> x, y;
    Walk w;
    w.begin(rg, a.I, R);
    Job job = get_job(a.jobs, a.dense_jobs, a.bsz, w.j);
    load_x(a, job, c16, active, x);
    JobState js = job_state(a, job, w.j, rg);
    zero_cols(y);
    Stages cs;
    bool ok = true;
    // the chunk whose down rows are pending
    bool pending = false, p_last_of_job = false;
    int p_rows = 0, p_ntok = 1, p_slot0 = 0, p_slot1 = 0;
    float p_hv = 0.0f;

    while (!w.done()) {
        const int T = MT == 1 ? 1 : js.ntok;
        ok = (T == 2) ? gateup_chunk<R, MT, MT>(a, ctl, ring, stage_bytes, cs, w.rows, c16, active, x, warp, lane)
                      : gateup_chunk<R, 1, MT>(a, ctl, ring, stage_bytes, cs, w.rows, c16, active, x, warp, lane);
        if (!ok) break;
        if (pending) {
            ok = (p_ntok == 2)
                     ? down_chunk<R, MT, MT>(a, ctl, ring, stage_bytes, cs, p_rows, c16, active, p_hv, y, lane)
                     : down_chunk<R, 1, MT>(a, ctl, ring, stage_bytes, cs, p_rows, c16, active, p_hv, y, lane);
            if (!ok) break;
            if (p_last_of_job) {
                flush_partial(a, p_ntok, p_slot0, p_slot1, c16, active, y);
                zero_cols(y);
            }
        }
        float hv;
        ok = (T == 2) ? finish_sum<R, MT>(a, ctl, cs, js.w0, js.w1, NW, lane, hv)
                      : finish_sum<R, 1>(a, ctl, cs, js.w0, js.w1, NW, lane, hv);
        if (!ok) break;
        pending = true;
        p_rows = w.rows;
        p_ntok = T;
        p_slot0 = js.slot0;
        p_slot1 = js.slot1;
        p_hv = hv;
        p_last_of_job = w.next(R);
        if (p_last_of_job) {
            job = get_job(a.jobs, a.dense_jobs, a.bsz, w.j);
            load_x(a, job, c16, active, x);
            js = job_state(a, job, w.j, rg);
        }
    }
    if (ok && pending) {
        ok = (p_ntok == 2) ? down_chunk<R, MT, MT>(a, ctl, ring, stage_bytes, cs, p_rows, c16, active, p_hv, y, lane)
                           : down_chunk<R, 1, MT>(a, ctl, ring, stage_bytes, cs, p_rows, c16, active, p_hv, y, lane);
        if (ok) flush_partial(a, p_ntok, p_slot0, p_slot1, c16, active, y);
    }
    if (!ok) {
        record_status(a.status, FP9_ERR_TIMEOUT);
        ctl.abort = 1;
    }
}

// R: rows per chunk; MT: most tokens a job can hold (1 when bsz == 1).
template <int R, int MT>
__global__ void __launch_bounds__(kMaxThreads, 1) expert_kernel(const ExpertArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(smem);
    uint8_t* ring = smem + kRingOffset;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NW = static_cast<int>(blockDim.x / 32) - 1;
    const uint32_t stage_bytes = static_cast<uint32_t>(R * a.H / 8 * 9);

    grid_dependency_wait();  // the router's job list and x are complete
    grid_launch_dependents();
    const int32_t J = a.dense_jobs > 0 ? a.dense_jobs : a.ctl->njobs;
    const Range rg = cta_range(J, a.I, gridDim.x, blockIdx.x);
    if (rg.start >= rg.end) return;

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) {
            mbar_init(smem_addr(&ctl.full[s]), 1);
            mbar_init(smem_addr(&ctl.empty[s]), NW);
        }
        mbar_init(smem_addr(&ctl.red[0]), NW);
        mbar_init(smem_addr(&ctl.red[1]), NW);
        ctl.abort = 0;
        ctl.never = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW) {
        if (lane == 0) producer<R>(a, ctl, ring, rg, stage_bytes);
        return;
    }
    consumer<R, MT>(a, ctl, ring, rg, stage_bytes, NW, warp, lane);
}

// ------------------------------------------------------------- combine ----

struct CombineArgs {
    const float* partial;
    const Job* jobs;
    const Control* ctl;
    int32_t dense_jobs;
    int32_t bsz;
    int32_t H;
    int32_t maxseg;
    int32_t grid;  // CTAs of the expert kernel
    int64_t I;
    float* y;
};

constexpr int kCombineCols = 64;               // columns per CTA: 16 lanes x float4
constexpr int kCombineWarps = 8;
constexpr int kCombineLanes = kCombineWarps * 2;  // segment lanes: two per warp

// y[t, c] = sum of token t's partials, in list order (= job order, then
// CTA order within a job). Segment lane s (= 2 * warp + half-warp) adds
// partials s, s + 16, ...; the sixteen lane sums are then added in lane
// order.
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineArgs a) {
    __shared__ float4 red[kCombineLanes][16];
    grid_dependency_wait();  // all partials are written
    grid_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int half = lane >> 4, l16 = lane & 15;
    const int sl = warp * 2 + half;
    const int t = blockIdx.y;
    const int c = blockIdx.x * kCombineCols + l16 * 4;
    int n;
    if (a.dense_jobs > 0) {  // token t is in job t / 2 only
        const int64_t N = static_cast<int64_t>(a.dense_jobs) * a.I;
        const int64_t G = N < a.grid ? N : a.grid;
        const int64_t first = static_cast<int64_t>(t / kTokensPerJob) * a.I;
        n = static_cast<int>(cta_of_row(first + a.I - 1, N, G) - cta_of_row(first, N, G) + 1);
    } else {
        n = a.ctl->nseg[t];
    }
    const float* base = a.partial + static_cast<int64_t>(t) * a.maxseg * a.H + c;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int s = sl; s < n; s += kCombineLanes) {
        const float4 p = __ldcs(reinterpret_cast<const float4*>(base + static_cast<int64_t>(s) * a.H));
        acc.x += p.x;
        acc.y += p.y;
        acc.z += p.z;
        acc.w += p.w;
    }
    red[sl][l16] = acc;
    __syncthreads();
    if (threadIdx.x < 16) {
        float4 sum = red[0][threadIdx.x];
        for (int w = 1; w < kCombineLanes; ++w) {
            const float4 o = red[w][threadIdx.x];
            sum.x += o.x;
            sum.y += o.y;
            sum.z += o.z;
            sum.w += o.w;
        }
        reinterpret_cast<float4*>(a.y + static_cast<int64_t>(t) * a.H)[(blockIdx.x * kCombineCols) / 4 +
                                                                       threadIdx.x] = sum;
    }
}

// ------------------------------------------------------------- launches ---

static BankPtrs bank_ptrs(const fp9_ffn_bank& b) {
    BankPtrs p;
    p.body[0] = b.gate_body;
    p.body[1] = b.up_body;
    p.body[2] = b.down_body;
    p.sign[0] = b.gate_sign;
    p.sign[1] = b.up_sign;
    p.sign[2] = b.down_sign;
    return p;
}

struct LaunchShape {
    int threads;
    int nstages;
    int rows;
    size_t smem;
};

// Rows per streamed chunk: 8 unless FP9MOE_CHUNK_ROWS=4 is set (a tuning
// knob: 8 halves the per-chunk reduction cost, 4 allows twice the stages).
static int chunk_rows() {
    static int rows = 0;
    if (rows == 0) {
        const char* e = getenv("FP9MOE_CHUNK_ROWS");
        rows = (e != nullptr && atoi(e) == 4) ? 4 : 8;
    }
    return rows;
}

static fp9_status expert_shape(int32_t H, LaunchShape& s) {
    const int nw = (H / 16 + 31) / 32;
    s.threads = nw * 32 + 32;
    s.rows = chunk_rows();
    const uint32_t stage = static_cast<uint32_t>(s.rows * H / 8 * 9);
    const int32_t optin = device_max_smem_optin();
    if (optin <= 0) return FP9_ERR_CUDA;
    int ns = static_cast<int>((static_cast<int64_t>(optin) - kRingOffset) / stage);
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns < 3) return FP9_ERR_SHAPE;
    s.nstages = ns;
    s.smem = kRingOffset + static_cast<size_t>(ns) * stage;
    return FP9_OK;
}

template <int R, int MT>
static cudaError_t set_smem(size_t smem) {
    return cudaFuncSetAttribute(expert_kernel<R, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
}

static fp9_status ensure_smem_attr(size_t smem) {
    static size_t configured[64] = {0};
    int dev = 0;
    FP9_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return FP9_ERR_CUDA;
    if (configured[dev] < smem) {
        FP9_CUDA_TRY((set_smem<4, 1>(smem)));
        FP9_CUDA_TRY((set_smem<8, 1>(smem)));
        FP9_CUDA_TRY((set_smem<4, 2>(smem)));
        FP9_CUDA_TRY((set_smem<8, 2>(smem)));
        configured[dev] = smem;
    }
    return FP9_OK;
}

// Optional events bracketing each fused-kernel launch (fp9_profile_events).
static cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

// Queues the fused expert kernel and the combine kernel.
static fp9_status launch_ffn(const BankPtrs& b0, const BankPtrs& b1, const float* x, float* y, int32_t bsz,
                             int32_t H, int64_t I, uint8_t* ws, const WsLayout& lay, int32_t dense_jobs,
                             int32_t* status, cudaStream_t stream, uint64_t timeout_ns, bool no_copy,
                             bool combine) {
    LaunchShape shp;
    fp9_status st = expert_shape(H, shp);
    if (st != FP9_OK) return st;
    st = ensure_smem_attr(shp.smem);
    if (st != FP9_OK) return st;
    ExpertArgs a;
    a.bank[0] = b0;
    a.bank[1] = b1;
    a.x = x;
    a.partial = reinterpret_cast<float*>(ws + lay.off_partial);
    a.jobs = reinterpret_cast<const Job*>(ws + lay.off_jobs);
    a.ctl = reinterpret_cast<const Control*>(ws);
    a.dense_jobs = dense_jobs;
    a.bsz = bsz;
    a.H = H;
    a.maxseg = lay.maxseg;
    a.I = I;
    a.nstages = shp.nstages;
    a.no_copy = no_copy ? 1 : 0;
    a.status = status;
    a.timeout_ns = timeout_ns;
    const bool prof = g_prof_start != nullptr && g_prof_stop != nullptr;
    if (prof) FP9_CUDA_TRY(cudaEventRecord(g_prof_start, stream));
    // jobs hold two tokens only when bsz >= 2; the one-token kernel keeps
    // half the x / y registers live
    void (*kern)(const ExpertArgs) = nullptr;
    if (bsz == 1) kern = shp.rows == 8 ? expert_kernel<8, 1> : expert_kernel<4, 1>;
    else kern = shp.rows == 8 ? expert_kernel<8, 2> : expert_kernel<4, 2>;
    FP9_CUDA_TRY(launch_pdl(kern, dim3(lay.grid), dim3(shp.threads), shp.smem, stream, a));
    if (prof) FP9_CUDA_TRY(cudaEventRecord(g_prof_stop, stream));
    if (!combine) return FP9_OK;
    CombineArgs c;
    c.partial = a.partial;
    c.jobs = a.jobs;
    c.ctl = a.ctl;
    c.dense_jobs = dense_jobs;
    c.bsz = bsz;
    c.H = H;
    c.maxseg = lay.maxseg;
    c.grid = lay.grid;
    c.I = I;
    c.y = y;
    FP9_CUDA_TRY(launch_pdl(combine_kernel, dim3(H / kCombineCols, bsz), dim3(kCombineWarps * 32), 0, stream, c));
    return FP9_OK;
}

fp9_status check_layer(const fp9_moe_layer* L, int32_t bsz);
fp9_status launch_router(const fp9_moe_layer* L, const float* x, int32_t bsz, int32_t* ids_out, float* w_out,
                         uint8_t* ws, const WsLayout& lay, bool build, cudaStream_t stream);

static fp9_status check_dense(const fp9_ffn_bank* f, int32_t bsz) {
    FP9_CHECK_ARG(f != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(bsz >= 1 && bsz <= FP9_MAX_BSZ, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(hidden_ok(f->hidden), FP9_ERR_SHAPE);
    FP9_CHECK_ARG(f->inter >= 1, FP9_ERR_SHAPE);
    return check_bank(*f, 1, f->inter, f->hidden);
}

}  // namespace fp9

using namespace fp9;

extern "C" size_t fp9_dense_workspace_bytes(const fp9_ffn_bank* ffn, int32_t bsz) {
    if (check_dense(ffn, bsz) != FP9_OK) return 0;
    const int32_t sms = device_sm_count();
    if (sms <= 0) return 0;
    return dense_layout(bsz, ffn->inter, ffn->hidden, sms).total;
}

extern "C" fp9_status fp9_moe_forward(const fp9_moe_layer* layer, const float* x, int32_t bsz, float* y,
                                      int32_t* ids, float* weights, void* ws, size_t ws_bytes,
                                      int32_t* d_status, void* stream) {
    fp9_status st = check_layer(layer, bsz);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(x != nullptr && y != nullptr && ws != nullptr && x != y, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(x, 16) && aligned(y, 16), FP9_ERR_ALIGN);
    FP9_CHECK_ARG(aligned(ws, kAlign), FP9_ERR_ALIGN);
    const int32_t sms = device_sm_count();
    FP9_CHECK_ARG(sms > 0, FP9_ERR_CUDA);
    const WsLayout lay =
        moe_layout(bsz, layer->n_experts, layer->topk, layer->n_shared, layer->inter, layer->hidden, sms);
    FP9_CHECK_ARG(ws_bytes >= lay.total, FP9_ERR_WORKSPACE);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    st = launch_router(layer, x, bsz, ids, weights, w, lay, true, s);
    if (st != FP9_OK) return st;
    const BankPtrs routed = bank_ptrs(layer->routed);
    const BankPtrs shared = layer->n_shared > 0 ? bank_ptrs(layer->shared) : routed;
    return launch_ffn(routed, shared, x, y, bsz, static_cast<int32_t>(layer->hidden), layer->inter, w, lay, 0,
                      d_status, s, kDefaultTimeoutNs, false, true);
}

extern "C" fp9_status fp9_dense_ffn(const fp9_ffn_bank* ffn, const float* x, int32_t bsz, float* y, void* ws,
                                    size_t ws_bytes, int32_t* d_status, void* stream) {
    fp9_status st = check_dense(ffn, bsz);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(x != nullptr && y != nullptr && ws != nullptr && x != y, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(x, 16) && aligned(y, 16), FP9_ERR_ALIGN);
    FP9_CHECK_ARG(aligned(ws, kAlign), FP9_ERR_ALIGN);
    const int32_t sms = device_sm_count();
    FP9_CHECK_ARG(sms > 0, FP9_ERR_CUDA);
    const WsLayout lay = dense_layout(bsz, ffn->inter, ffn->hidden, sms);
    FP9_CHECK_ARG(ws_bytes >= lay.total, FP9_ERR_WORKSPACE);
    const BankPtrs p = bank_ptrs(*ffn);
    return launch_ffn(p, p, x, y, bsz, static_cast<int32_t>(ffn->hidden), ffn->inter, static_cast<uint8_t*>(ws),
                      lay, lay.jmax, d_status, static_cast<cudaStream_t>(stream), kDefaultTimeoutNs, false, true);
}

extern "C" fp9_status fp9_selftest_timeout(void* ws, size_t ws_bytes, int32_t* d_status, int32_t timeout_us,
                                           void* stream) {
    FP9_CHECK_ARG(ws != nullptr && d_status != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(ws, kAlign), FP9_ERR_ALIGN);
    FP9_CHECK_ARG(timeout_us >= 1 && timeout_us <= 1000000, FP9_ERR_INVALID_ARG);
    constexpr int32_t H = 256;
    constexpr int64_t I = 8;
    // one CTA, one dense job: x at the start of ws, partials after the layout
    WsLayout lay = dense_layout(1, I, H, 1);
    lay.off_partial = align_up(sizeof(float) * H + kAlign);
    lay.total = lay.off_partial + sizeof(float) * lay.maxseg * H;
    FP9_CHECK_ARG(ws_bytes >= lay.total && ws_bytes >= 65536, FP9_ERR_WORKSPACE);
    uint8_t* w = static_cast<uint8_t*>(ws);
    BankPtrs p;  // never dereferenced: no copies are issued
    for (int m = 0; m < 3; ++m) {
        p.body[m] = w;
        p.sign[m] = w;
    }
    return launch_ffn(p, p, reinterpret_cast<const float*>(w + kAlign), nullptr, 1, H, I, w, lay, 1, d_status,
                      static_cast<cudaStream_t>(stream), static_cast<uint64_t>(timeout_us) * 1000ull, true, false);
}

extern "C" void fp9_profile_events(void* start, void* stop) {
    g_prof_start = static_cast<cudaEvent_t>(start);
    g_prof_stop = static_cast<cudaEvent_t>(stop);
}

// ----------------------------------------------- allocation-free variant ---
//
// fp9_moe_forward_noalloc: the same router, fused expert and combine
// kernels as fp9_moe_forward, with their workspace in a fixed array of
// device memory that belongs to this library instead of a caller buffer.
// It is for callers that cannot call cudaMalloc at all: runtimes whose
// device memory is owned and capped by another framework, plugins handed
// only input and output buffers, and latency-critical paths that must not
// risk the implicit synchronisation of an allocation.
//
// The array is a file-scope __device__ object: every GPU that loads this
// library holds kNoAllocScratchBytes for it until the process exits. Host
// code may not use the array's name as a device address, so the address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) on the first call made on that device; make that first call
// before any stream capture. All calls share the array and it keeps the
// last call's contents: the control block (the router's ticket and
// counts) is cleared by every call, and calls that overlap on the GPU
// (two streams, or two host threads) race on it.

namespace fp9 {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static void* noalloc_scratch_ptr(int dev) {
    static std::mutex mu;
    static void* ptrs[64] = {nullptr};
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (ptrs[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

}  // namespace fp9

extern "C" fp9_status fp9_moe_forward_noalloc(const fp9_moe_layer* layer, const float* x, int32_t bsz, float* y,
                                              int32_t* ids, float* weights, int32_t* d_status, void* stream) {
    fp9_status st = check_layer(layer, bsz);
    if (st != FP9_OK) return st;
    FP9_CHECK_ARG(x != nullptr && y != nullptr && x != y, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(x, 16) && aligned(y, 16), FP9_ERR_ALIGN);
    const int32_t sms = device_sm_count();
    FP9_CHECK_ARG(sms > 0, FP9_ERR_CUDA);
    const WsLayout lay =
        moe_layout(bsz, layer->n_experts, layer->topk, layer->n_shared, layer->inter, layer->hidden, sms);
    // the fixed array must hold this call's workspace
    FP9_CHECK_ARG(lay.total <= kNoAllocScratchBytes, FP9_ERR_WORKSPACE);
    int dev = 0;
    FP9_CUDA_TRY(cudaGetDevice(&dev));
    uint8_t* w = static_cast<uint8_t*>(noalloc_scratch_ptr(dev));
    FP9_CHECK_ARG(w != nullptr, FP9_ERR_CUDA);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FP9_CUDA_TRY(cudaMemsetAsync(w, 0, sizeof(Control), s));
    st = launch_router(layer, x, bsz, ids, weights, w, lay, true, s);
    if (st != FP9_OK) return st;
    const BankPtrs routed = bank_ptrs(layer->routed);
    const BankPtrs shared = layer->n_shared > 0 ? bank_ptrs(layer->shared) : routed;
    return launch_ffn(routed, shared, x, y, bsz, static_cast<int32_t>(layer->hidden), layer->inter, w, lay, 0,
                      d_status, s, kDefaultTimeoutNs, false, true);
}

extern "C" size_t fp9_moe_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }
