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
// CTA layout (one per SM): NW = H / 512 consumer warps (14 for H = 7168;
// the one-token kernel rounds them up to 16) and one producer warp. The
// producer's lane 0 streams each chunk of R = NW / 2 rows as three stages,
// one per ring slot: slot 0 the gate rows, slot 1 the up rows, slot 2 the
// down rows (bodies, then signs; bulk copies completing on mbarriers).
//   gate/up: the R rows of the gate stage are cut into 2R half rows, one
//     per warp; a warp computes its half row against x (staged in shared
//     memory), so the only reduction is a 5-step warp sum; lane 0
//     publishes the sum. Then the same for the up stage.
//   down: each thread owns 16 consecutive hidden columns and keeps y for
//     them in registers: an axpy with no reduction.
// Per chunk c a warp does its gate half row (and releases the gate slot),
// its up half row (releases the up slot), arrives at c's publish barrier,
// processes the down rows of chunk c - 1 (whose h is known), then waits for
// c's barrier and forms h = SiLU(g) * u * w_route from the halves' sums.
// The producer streams gate c, up c, then down c - 1: the order in which
// the slots free up, so every refill has two phases of the chunk to land.
//
// Every wait is bounded (a timeout sets FP9_ERR_TIMEOUT in the status word
// and the CTA drains its copies in flight and returns).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9_plan.h"
#include "fp9moe.h"

namespace fp9 {

constexpr int kMaxRows = 16;                                    // rows per chunk
constexpr int kSlots = 3;                                       // gate, up, down
constexpr int kDownCols = 16;                                   // down columns per thread
constexpr int kDsv3Hidden = 7168;  // the DeepSeek-V3 hidden size: specialised kernels
constexpr int kMaxConsumerWarps = FP9_MAX_HIDDEN / kDownCols / 32;  // 14
constexpr int kMaxThreads = kMaxConsumerWarps * 32 + 32;        // 480
// One-token kernels round the consumer warps up to a multiple of 4, so that
// each of the SM's four schedulers holds as many (16 for H = 7168).
constexpr int kMaxConsumerWarps1 = (kMaxConsumerWarps + 3) / 4 * 4;
constexpr int kMaxThreads1 = kMaxConsumerWarps1 * 32 + 32;      // 544
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;           // 1 s
constexpr int kGate = 0, kUp = 1, kDown = 2;

struct BankPtrs {
    const uint8_t* body[3];  // gate, up, down_t
    const uint8_t* sign[3];
};

struct ExpertArgs {
    BankPtrs bank[2];        // 0: routed experts / dense FFN, 1: shared experts
    const float* x;          // [bsz, H]: x, or h in stack mode
    const float* ss;         // stack mode: partial sums of squares of h (x = RMSNorm(h)), else NULL
    float eps;
    const uint8_t* prefetch;  // stack mode: the next layer's router weights, read into L2 (or NULL)
    int64_t prefetch_bytes;
    float* partial;          // token-major: [bsz * gridDim.x, H]
    uint32_t* mask;          // [gridDim.x]: bit t = partial of token t written
    const Job* jobs;         // phase 1: the router's jobs
    const Control* ctl;      // phase 1: CTAs that own rows
    const int64_t* cta_row;  // phase 1: [geff + 1] first row (job * I + row) of each CTA
    int32_t impl_jobs;       // phase 0: jobs that need no routing
    int32_t impl_nexp;       // phase 0: experts of the bank (shared experts, or 1 for the dense FFN)
    int32_t impl_bank;       // phase 0: 1 (shared experts) or 0 (dense FFN)
    int32_t tpj;             // phase 0: tokens per job (1 or 2)
    int32_t routed;          // 1: phase 1 runs on the router's plan (MoE call)
    int32_t bsz;
    int32_t H;
    int64_t I;
    int32_t rows;            // R: rows per chunk
    int32_t no_copy;         // self-test: the producer issues no copies
    int32_t* status;
    uint64_t timeout_ns;
};

struct SmemCtl {
    uint64_t full[kSlots];
    uint64_t empty[kSlots];
    uint64_t pub[2];         // gate/up sums of a chunk published (double-buffered by chunk parity)
    uint64_t xbar;           // a job's x staged in shared memory
    uint64_t hfull[2];       // down helper pairs: the helper's y is in shared memory
    uint64_t hfree[2];       // ... and has been added by the owner
    int abort;
    int never;               // stays 0: a flag nobody raises
    float gu[2][2][kMaxRows][2][kTokensPerJob];  // [chunk parity][gate, up][row][half][token]
};

constexpr uint32_t kCtlBytes = (sizeof(SmemCtl) + 127) / 128 * 128;

// Shared memory: [SmemCtl][x: MT planes x 4 float4 lanes x H/16 chunks][3 stages]
__host__ __device__ inline uint32_t x_bytes(int H, int MT) { return static_cast<uint32_t>(MT * H * 4); }
__host__ __device__ inline uint32_t stage_bytes(int H, int R) { return static_cast<uint32_t>(R * H / 8 * 9); }

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// The walk over a CTA's chunks: its rows of phase 0 (the jobs that need no
// routing, split evenly by rows over the first min(G, N) CTAs), then, for an
// MoE call, its rows of phase 1 (the router's cost-weighted split). Row
// j * I + r of a phase is row r of its job j; a chunk of at most R rows
// never crosses a job boundary. Producer and consumers walk the same
// sequence; every thread that walks into phase 1 first waits for the
// router's grid, so it reads the plan only once the plan is complete.
struct Walk {
    int phase;
    int32_t pos, end, I, r0;  // rows of a phase number at most kMaxJobs * FP9_MAX_INTER < 2^31
    int j;
    int rows;  // rows of the current chunk
    Job job;

    __device__ __forceinline__ void load_job(const ExpertArgs& a) {
        job = phase == 0 ? implicit_job(j, a.impl_nexp, a.impl_bank, a.bsz, a.tpj) : a.jobs[j];
    }
    __device__ __forceinline__ void set_phase(const ExpertArgs& a, int ph) {
        phase = ph;
        int64_t s = 0, e = 0;
        const int64_t b = blockIdx.x;
        if (ph == 0) {
            const int64_t n = static_cast<int64_t>(a.impl_jobs) * I;
            const int64_t g = n < gridDim.x ? n : gridDim.x;
            if (b < g) {
                s = cta_start(b, n, g);
                e = cta_start(b + 1, n, g);
            }
        } else {
            grid_dependency_wait();  // the router's plan is complete and visible
            if (b < a.ctl->geff) {
                s = a.cta_row[b];
                e = a.cta_row[b + 1];
            }
        }
        pos = static_cast<int32_t>(s);
        end = static_cast<int32_t>(e);
        j = pos / I;
        r0 = pos - j * I;
    }
    __device__ __forceinline__ void set_rows(int R) {
        int r = R;
        if (I - r0 < r) r = I - r0;
        if (end - pos < r) r = end - pos;
        rows = r;
    }
    __device__ __forceinline__ void begin(const ExpertArgs& a, int R) {
        I = static_cast<int32_t>(a.I);
        set_phase(a, 0);
        if (pos >= end && a.routed) set_phase(a, 1);
        if (pos < end) load_job(a);
        set_rows(R);
    }
    __device__ __forceinline__ bool done() const { return pos >= end; }
    // Advances past the current chunk; returns true when the next chunk
    // starts a new job.
    __device__ __forceinline__ bool next(const ExpertArgs& a, int R) {
        pos += rows;
        r0 += rows;
        bool new_job = false;
        if (pos >= end) {
            if (phase == 0 && a.routed) {
                set_phase(a, 1);
                new_job = pos < end;
            }
        } else if (r0 == I) {
            ++j;
            r0 = 0;
            new_job = true;
        }
        if (new_job) load_job(a);
        set_rows(R);
        return new_job;
    }
};

// The gate stage and the up stage of a chunk are each R rows x 2 halves
// (columns [0, H/2) and [H/2, H)) = 2R tasks; warp w takes tasks
// k = w, w + NW, ... (row k % R, half k / R) of the gate stage, then the
// same tasks of the up stage. So every warp is done with the gate slot
// before it starts on the up slot, and the three slots are released at
// three different times per chunk (gate, up, down): each refill has two
// phases of the chunk to land in. Whether warp w reads the stages:
__device__ __forceinline__ bool reads_stages(int w, int R) { return w < 2 * R; }

// ------------------------------------------------------------- producer ---

__device__ void producer(const ExpertArgs& a, SmemCtl& ctl, uint8_t* ring) {
    const uint64_t pol_once = l2_evict_first_policy(), pol_reread = l2_evict_normal_policy();
    const int H = a.H, R = a.rows;
    const uint32_t sbytes = stage_bytes(H, R);
    uint32_t use[kSlots] = {0u, 0u, 0u};
    bool ok = true;

    auto issue = [&](int m, const Job& job, int64_t r0, int rows) -> bool {
        if (!mbar_wait_bounded(smem_addr(&ctl.empty[m]), (use[m] & 1u) ^ 1u, a.timeout_ns, &ctl.abort))
            return false;
        const BankPtrs& bp = a.bank[job.bank];
        const int64_t row = static_cast<int64_t>(job.expert) * a.I + r0;
        const uint32_t bb = static_cast<uint32_t>(rows * H), sb = static_cast<uint32_t>(rows * (H / 8));
        const uint32_t full = smem_addr(&ctl.full[m]);
        const uint32_t dst = smem_addr(ring + m * sbytes);
        const uint64_t pol = (job.flags & kJobReread) ? pol_reread : pol_once;
        if (!a.no_copy) {
            mbar_arrive_expect_tx(full, bb + sb);
            bulk_g2s(dst, bp.body[m] + row * H, bb, full, pol);
            bulk_g2s(dst + R * H, bp.sign[m] + row * (H / 8), sb, full, pol);
        }
        ++use[m];
        return true;
    };

    Walk w;
    w.begin(a, R);
    Job pjob = w.job;
    int64_t pr0 = 0;
    int prows = 0;
    bool pending = false;
    while (!w.done() && ok) {
        ok = issue(kGate, w.job, w.r0, w.rows) && issue(kUp, w.job, w.r0, w.rows);
        if (ok && pending) ok = issue(kDown, pjob, pr0, prows);
        pjob = w.job;
        pr0 = w.r0;
        prows = w.rows;
        pending = true;
        (void)w.next(a, R);
    }
    if (ok && pending) ok = issue(kDown, pjob, pr0, prows);
    if (ok && a.prefetch != nullptr) {
        // the last chunk is issued: this CTA's share of the next layer's
        // router weights goes to L2 now, shortly before that router reads it
        // (a prefetch at the kernel's start helped less: 83.2 against 83.0
        // us per stacked layer, 83.4 without)
        const int64_t slice = (a.prefetch_bytes / gridDim.x + 15) / 16 * 16;
        const int64_t b0 = static_cast<int64_t>(blockIdx.x) * slice;
        const int64_t len = a.prefetch_bytes - b0 < slice ? a.prefetch_bytes - b0 : slice;
        if (len > 0) prefetch_l2(a.prefetch + b0, static_cast<uint32_t>(len), l2_evict_last_policy());
    }
    if (!ok) {
        record_status(a.status, FP9_ERR_TIMEOUT);
        ctl.abort = 1;
        if (!a.no_copy) {  // let the copies already issued land before the CTA exits
            for (int m = 0; m < kSlots; ++m)
                if (use[m] > 0)
                    (void)mbar_wait_bounded(smem_addr(&ctl.full[m]), (use[m] - 1u) & 1u, a.timeout_ns, &ctl.never);
        }
    }
}

// ------------------------------------------------------------- consumer ---

// y of a thread's 16 columns, per token, in the pair order of
// decode16_pairs: p[2k] = (c[4k], c[4k+2]), p[2k+1] = (c[4k+1], c[4k+3]).
template <int MT>
struct Cols {
    float2 p[MT][8];
};

template <int MT>
__device__ __forceinline__ void zero_cols(Cols<MT>& y) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int k = 0; k < 8; ++k) y.p[t][k] = make_float2(0.f, 0.f);
}

__device__ __forceinline__ bool wait_full(const ExpertArgs& a, SmemCtl& ctl, int m, uint32_t use) {
    return mbar_wait_bounded(smem_addr(&ctl.full[m]), use & 1u, a.timeout_ns, &ctl.abort);
}

__device__ __forceinline__ void release(SmemCtl& ctl, int m, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl.empty[m]));
}

// Dot product of one half of a gate/up row of a stage with x: the
// 16-column chunks [half * nch / 2, (half + 1) * nch / 2); lane l takes the
// chunks l, l + 32, ... of that range. x comes from shared memory as float4
// (plane t * 4 + q holds columns 16 c + 4q .. +3 of chunk c in the order
// (0, 2, 1, 3), so consecutive lanes read consecutive 16-byte words and
// each half of the float4 pairs with one decoded weight pair of
// decode16_pairs). The multiply-adds run two at a time (packed fp32 FMA,
// each lane of it rounded like fmaf).
template <int T, int NC>
__device__ __forceinline__ void row_dot(const uint8_t* st, int H, int R, int r, int half, const float4* xs, int nch,
                                        int lane, float (&acc)[T]) {
    float2 a0[T], a1[T];
#pragma unroll
    for (int t = 0; t < T; ++t) a0[t] = a1[t] = make_float2(0.0f, 0.0f);
    const uint8_t* brow = st + r * H;
    const uint8_t* srow = st + R * H + r * (H / 8);
    auto step = [&](int c) {
        const uint4 b = *reinterpret_cast<const uint4*>(brow + c * 16);
        const uint32_t s16 = *reinterpret_cast<const uint16_t*>(srow + c * 2);
        float2 w[8];
        decode16_pairs(b, s16, w);
#pragma unroll
        for (int t = 0; t < T; ++t) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 xv = xs[(t * 4 + q) * nch + c];
                a0[t] = __ffma2_rn(w[2 * q], make_float2(xv.x, xv.y), a0[t]);
                a1[t] = __ffma2_rn(w[2 * q + 1], make_float2(xv.z, xv.w), a1[t]);
            }
        }
    };
    const int hn = nch / 2, c0 = half * hn;
    if constexpr (NC > 0) {  // every lane has NC chunks: no bounds test
#pragma unroll
        for (int i = 0; i < NC; ++i) step(c0 + lane + 32 * i);
    } else {
#pragma unroll 2
        for (int c = c0 + lane; c < c0 + hn; c += 32) step(c);
    }
#pragma unroll
    for (int t = 0; t < T; ++t) acc[t] = warp_sum((a0[t].x + a0[t].y) + (a1[t].x + a1[t].y));
}

// This warp's tasks (row halves) of the gate (m = 0) or up (m = 1) stage of
// a chunk; lane 0 publishes each half's sums into gu[par][m][row][half][token].
template <int T, int NC>
__device__ __forceinline__ void gateup_stage(SmemCtl& ctl, const uint8_t* st, int H, int R, int rows, int m,
                                             uint32_t par, const float4* xs, int nch, int warp, int NW, int lane) {
    for (int k = warp; k < 2 * R; k += NW) {
        const int r = k % R, half = k / R;
        if (r >= rows) continue;
        float acc[T];
        row_dot<T, NC>(st, H, R, r, half, xs, nch, lane, acc);
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < T; ++t) ctl.gu[par][m][r][half][t] = acc[t];
        }
    }
}

// y[c] += h_row * W_down^T[row, c] over my 16 columns; lane (rr * T + t)
// of `hv` holds h of row rr, token t.
template <int T, int MT>
__device__ __forceinline__ void down_row(const uint8_t* st, int H, int R, int rr, int cc, float hv, Cols<MT>& y) {
    float h[T];
#pragma unroll
    for (int t = 0; t < T; ++t) h[t] = __shfl_sync(0xFFFFFFFFu, hv, rr * T + t);
    const uint4 b = *reinterpret_cast<const uint4*>(st + rr * H + cc * 16);
    const uint32_t s16 = *reinterpret_cast<const uint16_t*>(st + R * H + rr * (H / 8) + cc * 2);
    float2 w[8];
    decode16_pairs(b, s16, w);
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const float2 hh = make_float2(h[t], h[t]);
#pragma unroll
        for (int k = 0; k < 8; ++k) y.p[t][k] = __ffma2_rn(hh, w[k], y.p[t][k]);
    }
}

// The down rows of a chunk: all of them (half < 0), or its first (half 0)
// or second (half 1) half, split at (rows + 1) / 2. RC > 0: a full chunk of
// RC rows is unrolled (no guards) when every lane of the warp owns columns;
// a warp with lanes past the last column takes the guarded loop, whose
// inactive lanes only join the shuffles.
template <int T, int MT, int RC>
__device__ __forceinline__ void down_stage(const uint8_t* st, int H, int R, int rows, int cc, bool active, float hv,
                                           Cols<MT>& y, int half = -1) {
    if (RC > 0 && rows == RC && __all_sync(0xFFFFFFFFu, active)) {
        if (half < 0) {
#pragma unroll
            for (int rr = 0; rr < RC; ++rr) down_row<T, MT>(st, H, R, rr, cc, hv, y);
        } else {
            const int r0 = half * ((RC + 1) / 2);
#pragma unroll
            for (int k = 0; k < RC / 2; ++k) down_row<T, MT>(st, H, R, r0 + k, cc, hv, y);
        }
        return;
    }
    const int sp = (rows + 1) / 2;
    const int lo = half == 1 ? sp : 0, hi = half == 0 ? sp : rows;
#pragma unroll 1
    for (int rr = lo; rr < hi; ++rr) {
        if (active) {
            down_row<T, MT>(st, H, R, rr, cc, hv, y);
        } else {
#pragma unroll
            for (int t = 0; t < T; ++t) (void)__shfl_sync(0xFFFFFFFFu, hv, rr * T + t);
        }
    }
}

// Adds y (this CTA's share for the tokens of `tk`) into the CTA's partial
// row of each of those tokens (row tok * G + b): the CTA's first write of a
// token stores, later ones add, so a CTA's partial of a token sums its rows
// in walk order. `written` (the same in every thread) tracks the tokens
// written so far.
template <int MT>
__device__ __forceinline__ void flush_y(const ExpertArgs& a, int ntok, int tok0, int tok1, int cc, bool active,
                                        uint32_t& written, const Cols<MT>& y) {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        if (t < ntok) {
            const int tok = t == 0 ? tok0 : tok1;
            const bool add = (written >> tok) & 1u;
            written |= 1u << tok;
            if (active) {
                float4* dst = reinterpret_cast<float4*>(
                    a.partial + (static_cast<int64_t>(tok) * gridDim.x + blockIdx.x) * a.H + cc * kDownCols);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float4 v = make_float4(y.p[t][2 * k].x, y.p[t][2 * k + 1].x, y.p[t][2 * k].y, y.p[t][2 * k + 1].y);
                    if (add) {
                        const float4 o = dst[k];
                        v.x += o.x;
                        v.y += o.y;
                        v.z += o.z;
                        v.w += o.w;
                    }
                    dst[k] = v;
                }
            }
        }
    }
}

// Stages the job's x into shared memory (plane t * 4 + q, chunk c =
// columns 16 c + 4 q + (0, 2, 1, 3) of token t), then waits until every
// consumer warp has written its share. x is read from L2 (ld.global.cg):
// in an MoE call the fused kernel reads it before its own grid-dependency
// wait, once the kernel that wrote it has completed. In stack mode x = h *
// scale, the scale formed by each warp from the partial sums of squares
// (the router's bits).
template <int MT, bool kNorm>
__device__ __forceinline__ bool stage_x(const ExpertArgs& a, SmemCtl& ctl, float4* xs, const Job& job, int nch,
                                        int tid, int NT, uint32_t& xuse, int lane) {
    const int H4 = a.H / 4;
    for (int t = 0; t < MT; ++t) {
        if (t >= job.ntok) break;
        const int tok = t == 0 ? job.tok[0] : job.tok[1];
        const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<int64_t>(tok) * a.H);
        if constexpr (kNorm) {
            // h is staged as it is and scaled in place once the warp has the
            // scale, so the loads of h and of the partial sums overlap
            for (int j = tid; j < H4; j += NT) {
                const float4 v = __ldcg(src + j);
                xs[(t * 4 + (j & 3)) * nch + (j >> 2)] = make_float4(v.x, v.z, v.y, v.w);
            }
            const int nparts = a.H / kNormPartCols;
            const float sc = rms_scale_parts(a.ss + static_cast<int64_t>(tok) * nparts, nparts, a.H, a.eps, lane);
            for (int j = tid; j < H4; j += NT) {
                float4& v = xs[(t * 4 + (j & 3)) * nch + (j >> 2)];
                v = make_float4(v.x * sc, v.y * sc, v.z * sc, v.w * sc);
            }
        } else {
            for (int j = tid; j < H4; j += NT) {
                const float4 v = __ldcg(src + j);
                xs[(t * 4 + (j & 3)) * nch + (j >> 2)] = make_float4(v.x, v.z, v.y, v.w);
            }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl.xbar));
    const bool ok = mbar_wait_bounded(smem_addr(&ctl.xbar), xuse & 1u, a.timeout_ns, &ctl.abort);
    ++xuse;
    return ok;
}

// The fixed shape of a specialised kernel: hidden size HC (0: any), its
// consumer warps (16 down columns per thread; a one-token kernel rounds
// them up to a multiple of 4, one group per scheduler, and the extra warps
// own no down columns), the 16-column chunks per lane of a half row, and its
// rows per chunk (two half rows per row: one per consumer warp, at least
// 4). For H = 7168: 14 warps and 7 rows, or 16 and 8 with one token.
template <int MT, int HC>
struct Shape {
    static constexpr int kNch = HC / 16;
    static constexpr int kNW0 = (HC / kDownCols + 31) / 32;
    static constexpr int kNW = MT == 1 ? (kNW0 + 3) / 4 * 4 : kNW0;
    static constexpr int kNC = (HC > 0 && kNch % 64 == 0) ? kNch / 64 : 0;  // chunks per lane of a half row
    static constexpr int kRows = HC > 0 ? (kNW / 2 > 4 ? kNW / 2 : 4) : 0;
};

template <int MT, int HC, bool kNorm>
__device__ void consumer(const ExpertArgs& a, SmemCtl& ctl, float4* xs, const uint8_t* ring, int NW, int warp,
                         int lane) {
    using S = Shape<MT, HC>;
    const int H = HC > 0 ? HC : a.H;
    const int R = S::kRows > 0 ? S::kRows : a.rows;
    if (S::kNW > 0) NW = S::kNW;
    const int nch = H / 16;
    // Down helpers (the one-token kernel at hidden 7168): 14 warps own the
    // 448 16-column chunks of y, and the two warps that only exist for the
    // gate/up balance take the second half of the down rows of warps 0 and
    // 1 (warp 14 + i helps warp i), adding their y into the owner's when it
    // is flushed. Warp w issues on scheduler w mod 4, so each scheduler then
    // issues 28 row units of down work per chunk instead of 32, 32, 24, 24.
    constexpr bool kHelp = MT == 1 && HC == kDsv3Hidden && S::kNW == S::kNW0 + 2 && S::kRows % 2 == 0;
    const bool helper = kHelp && warp >= S::kNW0;
    const bool helped = kHelp && warp < S::kNW - S::kNW0;
    const int cw = helper ? warp - S::kNW0 : warp;
    const int half = helper ? 1 : (helped ? 0 : -1);
    const int cc = cw * 32 + lane;
    const bool active = cc < H / kDownCols;
    const uint32_t sbytes = stage_bytes(H, R);
    const bool rd_gate = reads_stages(warp, R), rd_up = rd_gate;
    Cols<MT> y;
    zero_cols(y);
    uint32_t written = 0;  // tokens whose partial row this CTA has written
    float* hy = reinterpret_cast<float*>(const_cast<uint8_t*>(ring) + kSlots * sbytes) + (cw * 32 + lane) * 16;
    uint32_t hn = 0;  // flushes of this pair so far
    // Flushes y into the CTA's partial rows; in a helper pair the helper
    // hands its y to the owner through shared memory and the owner adds it
    // (owner rows + helper rows, a fixed order) before writing.
    auto flush = [&](int ntok, int tok0, int tok1) -> bool {
        if (helper || helped) {
            const uint32_t full = smem_addr(&ctl.hfull[cw]), free = smem_addr(&ctl.hfree[cw]);
            if (helper) {
                if (hn > 0 && !mbar_wait_bounded(free, (hn - 1) & 1u, a.timeout_ns, &ctl.abort)) return false;
#pragma unroll
                for (int k = 0; k < 8; ++k) reinterpret_cast<float2*>(hy)[k] = y.p[0][k];
                __syncwarp();
                if (lane == 0) mbar_arrive(full);
                ++hn;
                return true;
            }
            if (!mbar_wait_bounded(full, hn & 1u, a.timeout_ns, &ctl.abort)) return false;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 o = reinterpret_cast<const float2*>(hy)[k];
                y.p[0][k].x += o.x;
                y.p[0][k].y += o.y;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(free);
            ++hn;
        }
        flush_y(a, ntok, tok0, tok1, cc, active, written, y);
        return true;
    };
    Walk w;
    w.begin(a, R);
    uint32_t xuse = 0;
    bool ok = true;
    if (!w.done()) ok = stage_x<MT, kNorm>(a, ctl, xs, w.job, nch, warp * 32 + lane, NW * 32, xuse, lane);
    uint32_t c = 0;  // chunk index: uses of the gate and up slots, and the publish parity
    // the chunk whose down rows are pending (chunk c - 1) and its tokens
    bool pending = false, p_flush = false;
    int p_rows = 0, p_T = 1, p_ntok = 1, p_tok0 = 0, p_tok1 = 0;
    float p_hv = 0.0f;

    while (ok && !w.done()) {
        const int T = MT == 1 ? 1 : w.job.ntok;
        const uint32_t par = c & 1u;
        for (int m = kGate; m <= kUp && ok; ++m) {
            if (!(m == kGate ? rd_gate : rd_up)) continue;
            if (!wait_full(a, ctl, m, c)) {
                ok = false;
                break;
            }
            if (T == 2)
                gateup_stage<MT, S::kNC>(ctl, ring + m * sbytes, H, R, w.rows, m, par, xs, nch, warp, NW, lane);
            else
                gateup_stage<1, S::kNC>(ctl, ring + m * sbytes, H, R, w.rows, m, par, xs, nch, warp, NW, lane);
            release(ctl, m, lane);
        }
        if (!ok) break;
        if (lane == 0) mbar_arrive(smem_addr(&ctl.pub[par]));
        if (pending) {
            if (!wait_full(a, ctl, kDown, c - 1u)) {
                ok = false;
                break;
            }
            if (p_T == 2)
                down_stage<MT, MT, S::kRows>(ring + kDown * sbytes, H, R, p_rows, cc, active, p_hv, y);
            else
                down_stage<1, MT, S::kRows>(ring + kDown * sbytes, H, R, p_rows, cc, active, p_hv, y, half);
            release(ctl, kDown, lane);
            if (p_flush) {
                if (!flush(p_ntok, p_tok0, p_tok1)) {
                    ok = false;
                    break;
                }
                zero_cols(y);
            }
        }
        if (!mbar_wait_bounded(smem_addr(&ctl.pub[par]), (c >> 1) & 1u, a.timeout_ns, &ctl.abort)) {
            ok = false;
            break;
        }
        float hv = 0.0f;  // lane (r * T + t): h of row r, token t
        if (lane < R * T) {
            const int r = lane / T, t = lane % T;
            const float wt = t == 0 ? w.job.w[0] : w.job.w[1];
            const float g = ctl.gu[par][kGate][r][0][t] + ctl.gu[par][kGate][r][1][t];
            const float u = ctl.gu[par][kUp][r][0][t] + ctl.gu[par][kUp][r][1][t];
            hv = silu(g) * u * wt;
        }
        pending = true;
        p_rows = w.rows;
        p_T = T;
        p_hv = hv;
        p_ntok = w.job.ntok;
        p_tok0 = w.job.tok[0];
        p_tok1 = w.job.tok[1];
        p_flush = false;
        if (w.next(a, R) && (w.job.ntok != p_ntok || w.job.tok[0] != p_tok0 || w.job.tok[1] != p_tok1)) {
            // new tokens: y is flushed after this chunk's down rows; every
            // warp is past this chunk's gate/up rows, so x may change now
            p_flush = true;
            ok = stage_x<MT, kNorm>(a, ctl, xs, w.job, nch, warp * 32 + lane, NW * 32, xuse, lane);
        }
        ++c;
    }
    if (ok && pending) {
        ok = wait_full(a, ctl, kDown, c - 1u);
        if (ok) {
            if (p_T == 2)
                down_stage<MT, MT, S::kRows>(ring + kDown * sbytes, H, R, p_rows, cc, active, p_hv, y);
            else
                down_stage<1, MT, S::kRows>(ring + kDown * sbytes, H, R, p_rows, cc, active, p_hv, y, half);
            release(ctl, kDown, lane);
            ok = flush(p_ntok, p_tok0, p_tok1);
        }
    }
    if (warp == 0 && lane == 0) a.mask[blockIdx.x] = written;
    if (!ok) {
        record_status(a.status, FP9_ERR_TIMEOUT);
        ctl.abort = 1;
    }
}

// MT: most tokens a job can hold (1 when bsz == 1). HC: the hidden size
// the kernel is specialised for (0: any).
// kNorm: stack mode (x = RMSNorm(h) formed while staging; MT == 1 only).
template <int MT, int HC, bool kNorm>
__global__ void __launch_bounds__(MT == 1 ? kMaxThreads1 : kMaxThreads, 1) expert_kernel(const ExpertArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(smem);
    float4* xs = reinterpret_cast<float4*>(smem + kCtlBytes);
    uint8_t* ring = smem + kCtlBytes + (x_bytes(a.H, MT) + 127u) / 128u * 128u;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NW = static_cast<int>(blockDim.x / 32) - 1;

    // A dense call reads x, written by the kernel queued before it, so it
    // waits first. An MoE call starts while the router runs: it starts no
    // earlier than the router's CTAs have all passed their own wait for the
    // kernel that wrote x (and read the previous call's partials), and it
    // waits for the router itself before phase 1.
    if (!a.routed) grid_dependency_wait();
    grid_launch_dependents();

    if (tid == 0) {
        int gate_readers = 0, up_readers = 0;
        for (int w = 0; w < NW; ++w) {
            gate_readers += reads_stages(w, a.rows) ? 1 : 0;
            up_readers += reads_stages(w, a.rows) ? 1 : 0;
        }
        for (int m = 0; m < kSlots; ++m) mbar_init(smem_addr(&ctl.full[m]), 1);
        mbar_init(smem_addr(&ctl.empty[kGate]), gate_readers);
        mbar_init(smem_addr(&ctl.empty[kUp]), up_readers);
        mbar_init(smem_addr(&ctl.empty[kDown]), NW);
        mbar_init(smem_addr(&ctl.pub[0]), NW);
        mbar_init(smem_addr(&ctl.pub[1]), NW);
        mbar_init(smem_addr(&ctl.xbar), NW);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&ctl.hfull[i]), 1);
            mbar_init(smem_addr(&ctl.hfree[i]), 1);
        }
        ctl.abort = 0;
        ctl.never = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW) {
        if (lane == 0) producer(a, ctl, ring);
        return;
    }
    consumer<MT, HC, kNorm>(a, ctl, xs, ring, NW, warp, lane);
}

// ------------------------------------------------------------- combine ----

struct CombineArgs {
    const float* partial;  // [bsz * grid, H]
    const uint32_t* mask;  // [grid]
    int32_t H;
    int32_t grid;          // CTAs of the expert kernel
    float* y;              // [bsz, H], or NULL (stack mode)
    float* h;              // stack mode: [bsz, H] residual stream, h += y; else NULL
    float* ss;             // stack mode: [bsz, H / 16] partial sums of squares of the new h
};

constexpr int kCombineCols = 16;    // columns per CTA: 4 float4
static_assert(kCombineCols == kNormPartCols, "a combine CTA writes one partial sum of squares");
constexpr int kCombineThreads = 256;
constexpr int kCombineLanes = kCombineThreads / 4;  // partial lanes per column: 64

// y[t, c] = the sum of the expert kernel's partials of token t, in CTA
// order. Thread (lane s, float4 q) adds the partials of CTAs s, s + 64, ...
// that hold token t (all their loads in flight at once); the 64 lane sums
// are added by a fixed shuffle tree inside each warp (8 lanes per warp),
// then the 8 warps' sums in warp order. Stack mode: h += y over the CTA's
// 16 columns, and their sum of squares (float4 q = 0..3 in order) is the
// CTA's partial for the next layer's RMSNorm.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
    __shared__ float4 red[kCombineThreads / 32][4];
    const int q = threadIdx.x & 3, sl = threadIdx.x >> 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.y;
    const int c = blockIdx.x * kCombineCols + q * 4;
    const int64_t o4 = (static_cast<int64_t>(t) * a.H + c) / 4;
    // stack mode: h is read before the wait for the expert kernel, which
    // does not write it (its last writer, the previous layer's combine, was
    // complete before this layer's router passed its own wait), so that
    // load is off the path from the last partial to the new h
    float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.h != nullptr && threadIdx.x < 4) hv = __ldcg(reinterpret_cast<const float4*>(a.h) + o4);
    grid_dependency_wait();  // all partials are written
    grid_launch_dependents();
    const float* base = a.partial + static_cast<int64_t>(t) * a.grid * a.H + c;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // the written-masks and the partial rows are loaded together (one round
    // trip to L2); rows a CTA never wrote are loaded but not added
    constexpr int kPer = 4;
    for (int b0 = sl; b0 < a.grid; b0 += kCombineLanes * kPer) {
        uint32_t m[kPer];
        float4 p[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int b = b0 + k * kCombineLanes;
            m[k] = 0u;
            if (b < a.grid) {
                m[k] = __ldcg(a.mask + b);
                p[k] = __ldcs(reinterpret_cast<const float4*>(base + static_cast<int64_t>(b) * a.H));
            }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            if ((m[k] >> t) & 1u) {
                acc.x += p[k].x;
                acc.y += p[k].y;
                acc.z += p[k].z;
                acc.w += p[k].w;
            }
        }
    }
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) {  // the warp's 8 partial lanes of this float4
        acc.x += __shfl_xor_sync(0xFFFFFFFFu, acc.x, m);
        acc.y += __shfl_xor_sync(0xFFFFFFFFu, acc.y, m);
        acc.z += __shfl_xor_sync(0xFFFFFFFFu, acc.z, m);
        acc.w += __shfl_xor_sync(0xFFFFFFFFu, acc.w, m);
    }
    if (lane < 4) red[warp][q] = acc;
    __syncthreads();
    if (threadIdx.x < 4) {
        float4 sum = red[0][q];
        for (int w = 1; w < kCombineThreads / 32; ++w) {
            const float4 o = red[w][q];
            sum.x += o.x;
            sum.y += o.y;
            sum.z += o.z;
            sum.w += o.w;
        }
        if (a.y != nullptr) reinterpret_cast<float4*>(a.y)[o4] = sum;
        if (a.h != nullptr) {
            float4 v = hv;
            v.x += sum.x;
            v.y += sum.y;
            v.z += sum.z;
            v.w += sum.w;
            reinterpret_cast<float4*>(a.h)[o4] = v;
            const float s = sumsq4(v, 0.0f);
            const float s1 = __shfl_sync(0xFu, s, 1), s2 = __shfl_sync(0xFu, s, 2), s3 = __shfl_sync(0xFu, s, 3);
            if (q == 0) a.ss[static_cast<int64_t>(t) * gridDim.x + blockIdx.x] = ((s + s1) + s2) + s3;
        }
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
    int rows;
    size_t smem;
};


// Consumer warps: one thread per 16 hidden columns, rounded up to a
// multiple of 4 in the one-token kernel (16 for hidden 7168: each of the
// four schedulers then runs four warps' half rows per phase, where 14 warps
// left two schedulers with four and two with three). Rows per chunk: half
// the consumer warps (the 2R half rows of a stage give every warp one: 7,
// or 8 with one token, for hidden 7168), at least 4, and as many as fit in
// shared memory next to x.
static fp9_status expert_shape(int32_t H, int MT, LaunchShape& s) {
    int nw = (H / kDownCols + 31) / 32;
    if (MT == 1) nw = (nw + 3) / 4 * 4;  // as many consumer warps per scheduler
    s.threads = nw * 32 + 32;
    const int32_t optin = device_max_smem_optin();
    if (optin <= 0) return FP9_ERR_CUDA;
    int R = nw / 2 > 4 ? nw / 2 : 4;
    if (R > kMaxRows) R = kMaxRows;
    // the down helpers' y hand-over (one-token kernel at hidden 7168): 2 x 32 lanes x 16 floats
    const size_t helpers = (MT == 1 && H == kDsv3Hidden) ? 2 * 32 * kDownCols * sizeof(float) : 0;
    const size_t fixed = kCtlBytes + (x_bytes(H, MT) + 127u) / 128u * 128u + helpers;
    while (R > 1 && fixed + kSlots * static_cast<size_t>(stage_bytes(H, R)) > static_cast<size_t>(optin)) --R;
    if (fixed + kSlots * static_cast<size_t>(stage_bytes(H, R)) > static_cast<size_t>(optin)) return FP9_ERR_SHAPE;
    s.rows = R;
    s.smem = fixed + kSlots * static_cast<size_t>(stage_bytes(H, R));
    return FP9_OK;
}

template <int MT, int HC, bool kNorm>
static cudaError_t set_smem(int optin) {
    return cudaFuncSetAttribute(expert_kernel<MT, HC, kNorm>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}

static fp9_status ensure_smem_attr() {
    static DeviceOnce attr;
    return attr.run([] {
        const int32_t optin = device_max_smem_optin();
        if (optin <= 0) return FP9_ERR_CUDA;
        FP9_CUDA_TRY((set_smem<1, 0, false>(optin)));
        FP9_CUDA_TRY((set_smem<2, 0, false>(optin)));
        FP9_CUDA_TRY((set_smem<1, kDsv3Hidden, false>(optin)));
        FP9_CUDA_TRY((set_smem<2, kDsv3Hidden, false>(optin)));
        FP9_CUDA_TRY((set_smem<1, 0, true>(optin)));
        FP9_CUDA_TRY((set_smem<1, kDsv3Hidden, true>(optin)));
        return FP9_OK;
    });
}

// Optional events bracketing each fused-kernel launch (fp9_profile_events).
static cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

// What one fused-kernel launch streams: the bank of phase 0 (shared experts
// or the dense FFN) and, for an MoE call, the routed bank of phase 1.
struct FfnCall {
    BankPtrs routed;
    BankPtrs implicit;
    int32_t impl_nexp;   // experts of the phase-0 bank (0: none)
    int32_t impl_bank;   // 1: shared experts, 0: dense FFN
    bool moe;            // phase 1 runs on the router's plan
};

// Stack mode of a call: the input is RMSNorm(h) (norm.ss set; x points at
// h) and the combine adds y into h and writes the next partial sums of
// squares (h, ss_out set; y NULL).
struct Residual {
    NormIn norm{nullptr, 0.0f};
    float* h = nullptr;
    float* ss_out = nullptr;
    const void* prefetch = nullptr;  // the next layer's router weights (L2 prefetch)
    int64_t prefetch_bytes = 0;
};

// Queues the fused expert kernel and (when `combine`) the combine kernel.
static fp9_status launch_ffn(const FfnCall& call, const float* x, float* y, int32_t bsz, int32_t H, int64_t I,
                             uint8_t* ws, const WsLayout& lay, int32_t* status, cudaStream_t stream,
                             uint64_t timeout_ns, bool no_copy, bool combine, const Residual& res = Residual()) {
    // An MoE call plans one token per job (see the plan) and runs the
    // one-token kernel; a dense call pairs its tokens when bsz >= 2.
    const int tpj = (call.moe || bsz == 1) ? 1 : 2;
    const int MT = tpj;
    LaunchShape shp;
    fp9_status st = expert_shape(H, MT, shp);
    if (st != FP9_OK) return st;
    st = ensure_smem_attr();
    if (st != FP9_OK) return st;
    ExpertArgs a;
    a.bank[0] = call.routed;
    a.bank[1] = call.implicit;
    a.x = x;
    a.ss = res.norm.ss;
    a.eps = res.norm.eps;
    a.prefetch = static_cast<const uint8_t*>(res.prefetch);
    a.prefetch_bytes = res.prefetch_bytes;
    a.partial = reinterpret_cast<float*>(ws + lay.off_partial);
    a.mask = reinterpret_cast<uint32_t*>(ws + lay.off_mask);
    a.jobs = reinterpret_cast<const Job*>(ws + lay.off_jobs);
    a.ctl = reinterpret_cast<const Control*>(ws);
    a.cta_row = reinterpret_cast<const int64_t*>(ws + lay.off_ctarow);
    a.impl_nexp = call.impl_nexp > 0 ? call.impl_nexp : 1;
    a.impl_jobs = call.impl_nexp * token_groups(bsz, tpj);
    a.tpj = tpj;
    a.impl_bank = call.impl_bank;
    a.routed = call.moe ? 1 : 0;
    a.bsz = bsz;
    a.H = H;
    a.I = I;
    a.rows = shp.rows;
    a.no_copy = no_copy ? 1 : 0;
    a.status = status;
    a.timeout_ns = timeout_ns;
    const bool prof = g_prof_start != nullptr && g_prof_stop != nullptr;
    if (prof) FP9_CUDA_TRY(cudaEventRecord(g_prof_start, stream));
    // the DeepSeek-V3 hidden size has its own kernel with every loop bound fixed
    const bool special = H == kDsv3Hidden && shp.rows == (MT == 1 ? Shape<1, kDsv3Hidden>::kRows
                                                                   : Shape<2, kDsv3Hidden>::kRows);
    // stack mode runs only in MoE calls (MT == 1)
    const bool norm = a.ss != nullptr;
    if (norm && MT != 1) return FP9_ERR_INVALID_ARG;
    void (*kern)(const ExpertArgs) =
        special ? (norm ? expert_kernel<1, kDsv3Hidden, true>
                        : (MT == 1 ? expert_kernel<1, kDsv3Hidden, false> : expert_kernel<2, kDsv3Hidden, false>))
                : (norm ? expert_kernel<1, 0, true> : (MT == 1 ? expert_kernel<1, 0, false> : expert_kernel<2, 0, false>));
    FP9_CUDA_TRY(launch_pdl(kern, dim3(lay.grid), dim3(shp.threads), shp.smem, stream, a));
    if (prof) FP9_CUDA_TRY(cudaEventRecord(g_prof_stop, stream));
    if (!combine) return FP9_OK;
    CombineArgs c;
    c.partial = a.partial;
    c.mask = a.mask;
    c.H = H;
    c.grid = lay.grid;
    c.y = y;
    c.h = res.h;
    c.ss = res.ss_out;
    FP9_CUDA_TRY(launch_pdl(combine_kernel, dim3(H / kCombineCols, bsz), dim3(kCombineThreads), 0, stream, c));
    return FP9_OK;
}

fp9_status check_layer(const fp9_moe_layer* L, int32_t bsz);
fp9_status launch_router(const fp9_moe_layer* L, const float* x, int32_t bsz, int32_t* ids_out, float* w_out,
                         uint8_t* ws, const WsLayout& lay, bool build, cudaStream_t stream, const NormIn& norm);

static fp9_status check_dense(const fp9_ffn_bank* f, int32_t bsz) {
    FP9_CHECK_ARG(f != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(bsz >= 1 && bsz <= FP9_MAX_BSZ, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(hidden_ok(f->hidden), FP9_ERR_SHAPE);
    FP9_CHECK_ARG(f->inter >= 1 && f->inter <= FP9_MAX_INTER, FP9_ERR_SHAPE);
    return check_bank(*f, 1, f->inter, f->hidden);
}

static FfnCall moe_call(const fp9_moe_layer* layer) {
    FfnCall c;
    c.routed = bank_ptrs(layer->routed);
    c.implicit = layer->n_shared > 0 ? bank_ptrs(layer->shared) : c.routed;
    c.impl_nexp = layer->n_shared;
    c.impl_bank = 1;
    c.moe = true;
    return c;
}

}  // namespace fp9

using namespace fp9;

extern "C" size_t fp9_dense_workspace_bytes(const fp9_ffn_bank* ffn, int32_t bsz) {
    if (check_dense(ffn, bsz) != FP9_OK) return 0;
    const int32_t sms = device_sm_count();
    if (sms <= 0) return 0;
    return dense_layout(bsz, ffn->hidden, expert_grid(sms, false)).total;
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
    const WsLayout lay = moe_layout(bsz, layer->n_experts, layer->topk, layer->hidden, expert_grid(sms, true));
    FP9_CHECK_ARG(ws_bytes >= lay.total, FP9_ERR_WORKSPACE);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    st = launch_router(layer, x, bsz, ids, weights, w, lay, true, s, NormIn{nullptr, 0.0f});
    if (st != FP9_OK) return st;
    return launch_ffn(moe_call(layer), x, y, bsz, static_cast<int32_t>(layer->hidden), layer->inter, w, lay, d_status,
                      s, kDefaultTimeoutNs, false, true);
}

extern "C" fp9_status fp9_moe_forward_residual(const fp9_moe_layer* layer, const float* x, float* h, float* ss,
                                               int32_t bsz, float eps, const fp9_moe_layer* next, int32_t* ids,
                                               float* weights, void* ws, size_t ws_bytes, int32_t* d_status,
                                               void* stream) {
    fp9_status st = check_layer(layer, bsz);
    if (st != FP9_OK) return st;
    if (next != nullptr) {
        st = check_layer(next, bsz);
        if (st != FP9_OK) return st;
    }
    FP9_CHECK_ARG(h != nullptr && ss != nullptr && ws != nullptr && x != h, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(eps >= 0.0f && eps <= 1.0f, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(h, 16) && aligned(ss, 16) && (x == nullptr || aligned(x, 16)), FP9_ERR_ALIGN);
    FP9_CHECK_ARG(aligned(ws, kAlign), FP9_ERR_ALIGN);
    const int32_t sms = device_sm_count();
    FP9_CHECK_ARG(sms > 0, FP9_ERR_CUDA);
    const WsLayout lay = moe_layout(bsz, layer->n_experts, layer->topk, layer->hidden, expert_grid(sms, true));
    FP9_CHECK_ARG(ws_bytes >= lay.total, FP9_ERR_WORKSPACE);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    Residual res;
    res.norm = NormIn{x == nullptr ? ss : nullptr, eps};
    res.h = h;
    res.ss_out = ss;
    if (next != nullptr) {
        res.prefetch = next->w_router;
        res.prefetch_bytes = static_cast<int64_t>(sizeof(float)) * next->n_experts * next->hidden;
    }
    const float* in = x == nullptr ? h : x;
    st = launch_router(layer, in, bsz, ids, weights, w, lay, true, s, res.norm);
    if (st != FP9_OK) return st;
    return launch_ffn(moe_call(layer), in, nullptr, bsz, static_cast<int32_t>(layer->hidden), layer->inter, w, lay,
                      d_status, s, kDefaultTimeoutNs, false, true, res);
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
    const WsLayout lay = dense_layout(bsz, ffn->hidden, expert_grid(sms, false));
    FP9_CHECK_ARG(ws_bytes >= lay.total, FP9_ERR_WORKSPACE);
    FfnCall c;
    c.routed = c.implicit = bank_ptrs(*ffn);
    c.impl_nexp = 1;
    c.impl_bank = 0;
    c.moe = false;
    return launch_ffn(c, x, y, bsz, static_cast<int32_t>(ffn->hidden), ffn->inter, static_cast<uint8_t*>(ws), lay,
                      d_status, static_cast<cudaStream_t>(stream), kDefaultTimeoutNs, false, true);
}

extern "C" fp9_status fp9_selftest_timeout(void* ws, size_t ws_bytes, int32_t* d_status, int32_t timeout_us,
                                           void* stream) {
    FP9_CHECK_ARG(ws != nullptr && d_status != nullptr, FP9_ERR_INVALID_ARG);
    FP9_CHECK_ARG(aligned(ws, kAlign), FP9_ERR_ALIGN);
    FP9_CHECK_ARG(timeout_us >= 1 && timeout_us <= 1000000, FP9_ERR_INVALID_ARG);
    constexpr int32_t H = 256;
    constexpr int64_t I = 8;
    // one CTA, one dense job: x at the start of ws, mask and partials after it
    WsLayout lay = dense_layout(1, H, 1);
    const size_t shift = align_up(sizeof(float) * H + kAlign);
    lay.off_mask += shift;
    lay.off_partial += shift;
    lay.total += shift;
    FP9_CHECK_ARG(ws_bytes >= lay.total && ws_bytes >= 65536, FP9_ERR_WORKSPACE);
    uint8_t* w = static_cast<uint8_t*>(ws);
    FfnCall c;  // never dereferenced: no copies are issued
    for (int m = 0; m < 3; ++m) {
        c.routed.body[m] = w;
        c.routed.sign[m] = w;
    }
    c.implicit = c.routed;
    c.impl_nexp = 1;
    c.impl_bank = 0;
    c.moe = false;
    return launch_ffn(c, reinterpret_cast<const float*>(w + kAlign), nullptr, 1, H, I, w, lay, d_status,
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
// looked up with cudaGetSymbolAddress (with that device current) on the
// first call made on each device, and again on the first call after the
// device's context was replaced (cudaDeviceReset); make that first call
// before any stream capture. All calls share the array and it keeps the
// last call's contents: the control block (the router's ticket and
// counts) is cleared by every call, and calls that overlap on the GPU
// (two streams, or two host threads) race on it.

namespace fp9 {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// The current context (driver entry point looked up once; nullptr if it
// cannot be had). After cudaDeviceReset a device's primary context is a new
// one, this library's module is loaded into it again and the array gets a
// new address, so a saved address is used only in the context it was looked
// up in.
static CUcontext current_context() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        else
            (void)cudaGetLastError();
    }
    CUcontext ctx = nullptr;
    if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

// Device address of the scratch array on device `dev` (current), looked up
// with cudaGetSymbolAddress on the first call in each context of the device
// and kept; nullptr if the lookup fails.
static void* noalloc_scratch_ptr(int dev) {
    static std::mutex mu;
    static void* ptrs[64] = {nullptr};
    static CUcontext ctxs[64] = {nullptr};
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const CUcontext ctx = current_context();
    if (ptrs[dev] == nullptr || ctx == nullptr || ctx != ctxs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            (void)cudaGetLastError();
            ptrs[dev] = nullptr;
            return nullptr;
        }
        ptrs[dev] = p;
        ctxs[dev] = ctx;
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
    const WsLayout lay = moe_layout(bsz, layer->n_experts, layer->topk, layer->hidden, expert_grid(sms, true));
    // the fixed array must hold this call's workspace
    FP9_CHECK_ARG(lay.total <= kNoAllocScratchBytes, FP9_ERR_WORKSPACE);
    int dev = 0;
    FP9_CUDA_TRY(cudaGetDevice(&dev));
    uint8_t* w = static_cast<uint8_t*>(noalloc_scratch_ptr(dev));
    FP9_CHECK_ARG(w != nullptr, FP9_ERR_CUDA);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FP9_CUDA_TRY(cudaMemsetAsync(w, 0, sizeof(Control), s));
    st = launch_router(layer, x, bsz, ids, weights, w, lay, true, s, NormIn{nullptr, 0.0f});
    if (st != FP9_OK) return st;
    return launch_ffn(moe_call(layer), x, y, bsz, static_cast<int32_t>(layer->hidden), layer->inter, w, lay, d_status,
                      s, kDefaultTimeoutNs, false, true);
}

extern "C" size_t fp9_moe_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }
