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

#include "fp9_device.cuh"
#include "fp9_host.h"
#include "fp9_plan.h"
#include "fp9moe.h"

namespace fp9 {

constexpr int kR = 4;                                           // rows per chunk
constexpr int kMaxStages = 16;
constexpr int kMaxConsumerWarps = FP9_MAX_HIDDEN / 16 / 32;     // 14
constexpr int kMaxThreads = kMaxConsumerWarps * 32 + 32;        // 480
constexpr int kMaxV = 2 * kR * kTokensPerJob;                   // reduced values per chunk
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;           // 1 s

struct BankPtrs {
    const uint8_t* body[3];  // gate, up, down_t
    const uint8_t* sign[3];
};

struct ExpertArgs {
    BankPtrs bank[2];        // 0: routed experts / dense FFN, 1: shared experts
    const float* x;          // [bsz, H]
    float* partial;          // [grid * maxseg * 2, H]
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
        jb.pad0 = 0;
        jb.tok[0] = kTokensPerJob * j;
        jb.ntok = (kTokensPerJob * j + 1 < bsz) ? 2 : 1;
        jb.tok[1] = jb.ntok == 2 ? jb.tok[0] + 1 : jb.tok[0];
        jb.w[0] = 1.0f;
        jb.w[1] = jb.ntok == 2 ? 1.0f : 0.0f;
        return jb;
    }
    return jobs[j];
}

__device__ __forceinline__ int64_t min3(int64_t a, int64_t b, int64_t c) {
    const int64_t m = a < b ? a : b;
    return m < c ? m : c;
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

__device__ __forceinline__ void load_row16(const uint8_t* st, int H, int rr, int c16, uint4& body,
                                           uint32_t& s16) {
    body = *reinterpret_cast<const uint4*>(st + rr * H + c16 * 16);
    s16 = *reinterpret_cast<const uint16_t*>(st + kR * H + rr * (H / 8) + c16 * 2);
}

// ------------------------------------------------------------- producer ---

__device__ void producer(const ExpertArgs& a, SmemCtl& ctl, uint8_t* ring, int64_t start, int64_t end,
                         uint32_t stage_bytes) {
    const uint64_t pol = l2_evict_first_policy();
    const int H = a.H;
    const int64_t I = a.I;
    const uint32_t NS = static_cast<uint32_t>(a.nstages);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t pos = start; pos < end && ok;) {
        const int j = static_cast<int>(pos / I);
        const int64_t r0 = pos - static_cast<int64_t>(j) * I;
        const int rows = static_cast<int>(min3(kR, I - r0, end - pos));
        const Job job = get_job(a.jobs, a.dense_jobs, a.bsz, j);
        const BankPtrs& bp = a.bank[job.bank];
        const int64_t row = static_cast<int64_t>(job.expert) * I + r0;
        const uint32_t bb = static_cast<uint32_t>(rows * H), sb = static_cast<uint32_t>(rows * (H / 8));
        for (int m = 0; m < 3; ++m) {
            const uint32_t slot = it % NS, ph = (it / NS) & 1u;
            if (!mbar_wait_bounded(smem_addr(&ctl.empty[slot]), ph ^ 1u, a.timeout_ns, &ctl.abort)) {
                ok = false;
                break;
            }
            const uint32_t full = smem_addr(&ctl.full[slot]);
            const uint32_t dst = smem_addr(ring + slot * stage_bytes);
            if (!a.no_copy) {
                mbar_arrive_expect_tx(full, bb + sb);
                bulk_g2s(dst, bp.body[m] + row * H, bb, full, pol);
                bulk_g2s(dst + kR * H, bp.sign[m] + row * (H / 8), sb, full, pol);
            }
            ++it;
        }
        pos += rows;
    }
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

struct ConsumerState {
    uint32_t it = 0;      // stages consumed
    uint32_t red_it = 0;  // CTA reductions done
};

// One chunk of `rows` rows for a job of T tokens. Returns false on timeout.
template <int T>
__device__ __forceinline__ bool run_chunk(const ExpertArgs& a, SmemCtl& ctl, const uint8_t* ring,
                                          uint32_t stage_bytes, ConsumerState& cs, int rows, int c16,
                                          bool active, const Job& job, const float (&xr)[kTokensPerJob][16],
                                          float (&yr)[kTokensPerJob][16], int NW, int warp, int lane) {
    constexpr int V = 2 * kR * T;
    const int H = a.H;
    const uint32_t NS = static_cast<uint32_t>(a.nstages);
    float v[V];
#pragma unroll
    for (int i = 0; i < V; ++i) v[i] = 0.0f;

    // gate (m = 0) and up (m = 1): partial dot products over my 16 columns
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const uint32_t slot = cs.it % NS, ph = (cs.it / NS) & 1u;
        if (!mbar_wait_bounded(smem_addr(&ctl.full[slot]), ph, a.timeout_ns, &ctl.abort)) return false;
        const uint8_t* st = ring + slot * stage_bytes;
        if (active) {
#pragma unroll
            for (int rr = 0; rr < kR; ++rr) {
                if (rr < rows) {
                    uint4 b;
                    uint32_t s16;
                    load_row16(st, H, rr, c16, b, s16);
                    float w[16];
                    decode16(b, s16, w);
#pragma unroll
                    for (int t = 0; t < T; ++t) {
                        float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            p0 = fmaf(w[i], xr[t][i], p0);
                            p1 = fmaf(w[i + 1], xr[t][i + 1], p1);
                        }
                        v[m * kR * T + rr * T + t] = p0 + p1;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl.empty[slot]));
        ++cs.it;
    }

    // CTA-wide sums of the 2 * kR * T values, in a fixed order
    const float r = warp_reduce_scatter<V>(v, lane);
    const uint32_t b = cs.red_it & 1u, rph = (cs.red_it >> 1) & 1u;
    if (lane < V) ctl.red_vals[b][warp][lane] = r;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl.red[b]));
    if (!mbar_wait_bounded(smem_addr(&ctl.red[b]), rph, a.timeout_ns, &ctl.abort)) return false;
    ++cs.red_it;
    float tot = 0.0f;
    if (lane < V)
        for (int w = 0; w < NW; ++w) tot += ctl.red_vals[b][w][lane];
    const float u = __shfl_down_sync(0xFFFFFFFFu, tot, kR * T);
    float hv = 0.0f;
    const float wt = (T == 2 && (lane & 1)) ? job.w[1] : job.w[0];
    if (lane < kR * T) hv = silu(tot) * u * wt;
    float h[kR][T];
#pragma unroll
    for (int rr = 0; rr < kR; ++rr)
#pragma unroll
        for (int t = 0; t < T; ++t) h[rr][t] = __shfl_sync(0xFFFFFFFFu, hv, rr * T + t);

    // down rows: y[c] += h_row * W_down^T[row, c] over my 16 columns
    {
        const uint32_t slot = cs.it % NS, ph = (cs.it / NS) & 1u;
        if (!mbar_wait_bounded(smem_addr(&ctl.full[slot]), ph, a.timeout_ns, &ctl.abort)) return false;
        const uint8_t* st = ring + slot * stage_bytes;
        if (active) {
#pragma unroll
            for (int rr = 0; rr < kR; ++rr) {
                if (rr < rows) {
                    uint4 bb;
                    uint32_t s16;
                    load_row16(st, H, rr, c16, bb, s16);
                    float w[16];
                    decode16(bb, s16, w);
#pragma unroll
                    for (int t = 0; t < T; ++t)
#pragma unroll
                        for (int i = 0; i < 16; ++i) yr[t][i] = fmaf(h[rr][t], w[i], yr[t][i]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl.empty[slot]));
        ++cs.it;
    }
    return true;
}

__device__ __forceinline__ void flush_partial(const ExpertArgs& a, const Job& job, int64_t seg, int c16,
                                              bool active, const float (&yr)[kTokensPerJob][16]) {
    if (!active) return;
#pragma unroll
    for (int t = 0; t < kTokensPerJob; ++t) {
        if (t < job.ntok) {
            float4* dst = reinterpret_cast<float4*>(
                a.partial + ((static_cast<int64_t>(blockIdx.x) * a.maxseg + seg) * kTokensPerJob + t) * a.H +
                c16 * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = make_float4(yr[t][4 * q], yr[t][4 * q + 1], yr[t][4 * q + 2], yr[t][4 * q + 3]);
        }
    }
}

__device__ void consumer(const ExpertArgs& a, SmemCtl& ctl, const uint8_t* ring, int64_t start, int64_t end,
                         uint32_t stage_bytes, int NW, int warp, int lane) {
    const int H = a.H;
    const int64_t I = a.I;
    const int c16 = warp * 32 + lane;
    const bool active = c16 < H / 16;
    float xr[kTokensPerJob][16], yr[kTokensPerJob][16];
    Job job;
    job.ntok = 0;
    int cur = -1;
    int64_t seg = 0;
    const int64_t job0 = start / I;
    ConsumerState cs;
    bool ok = true;
    for (int64_t pos = start; pos < end;) {
        const int j = static_cast<int>(pos / I);
        const int64_t r0 = pos - static_cast<int64_t>(j) * I;
        const int rows = static_cast<int>(min3(kR, I - r0, end - pos));
        if (j != cur) {
            if (cur >= 0) flush_partial(a, job, seg, c16, active, yr);
            cur = j;
            job = get_job(a.jobs, a.dense_jobs, a.bsz, j);
            seg = j - job0;
#pragma unroll
            for (int t = 0; t < kTokensPerJob; ++t) {
                const bool use = active && t < job.ntok;
                const int tok = t == 0 ? job.tok[0] : job.tok[1];
                const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<int64_t>(tok) * H + c16 * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 xv = use ? __ldg(src + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xr[t][4 * q] = xv.x;
                    xr[t][4 * q + 1] = xv.y;
                    xr[t][4 * q + 2] = xv.z;
                    xr[t][4 * q + 3] = xv.w;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) yr[t][i] = 0.0f;
            }
        }
        ok = (job.ntok == 2)
                 ? run_chunk<2>(a, ctl, ring, stage_bytes, cs, rows, c16, active, job, xr, yr, NW, warp, lane)
                 : run_chunk<1>(a, ctl, ring, stage_bytes, cs, rows, c16, active, job, xr, yr, NW, warp, lane);
        if (!ok) break;
        pos += rows;
    }
    if (ok) {
        if (cur >= 0) flush_partial(a, job, seg, c16, active, yr);
    } else {
        record_status(a.status, FP9_ERR_TIMEOUT);
        ctl.abort = 1;
    }
}

__global__ void __launch_bounds__(kMaxThreads, 1) expert_kernel(const ExpertArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(smem);
    uint8_t* ring = smem + kRingOffset;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NW = static_cast<int>(blockDim.x / 32) - 1;
    const uint32_t stage_bytes = static_cast<uint32_t>(kR * a.H / 8 * 9);

    grid_dependency_wait();  // no-op unless launched as a programmatic dependent
    const int32_t J = a.dense_jobs > 0 ? a.dense_jobs : a.ctl->njobs;
    const int64_t N = static_cast<int64_t>(J) * a.I, G = gridDim.x;
    const int64_t start = cta_start(blockIdx.x, N, G), end = cta_start(blockIdx.x + 1, N, G);
    if (start >= end) return;

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
        if (lane == 0) producer(a, ctl, ring, start, end, stage_bytes);
        return;
    }
    consumer(a, ctl, ring, start, end, stage_bytes, NW, warp, lane);
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

constexpr int kCombineWarps = 8;

// y[t, c] = sum over the jobs holding token t, in job order, and over the
// CTAs covering each job, in CTA order, of their partials. Warp w adds the
// segments w, w + 8, ...; the eight warp sums are added in warp order.
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineArgs a) {
    __shared__ float4 red[kCombineWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.y;
    const int c = blockIdx.x * 128 + lane * 4;
    const int32_t J = a.dense_jobs > 0 ? a.dense_jobs : a.ctl->njobs;
    const int64_t N = static_cast<int64_t>(J) * a.I, G = a.grid;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int64_t idx = 0;
    for (int j = 0; j < J; ++j) {
        const Job job = get_job(a.jobs, a.dense_jobs, a.bsz, j);
        for (int q = 0; q < job.ntok; ++q) {
            if ((q == 0 ? job.tok[0] : job.tok[1]) != t) continue;
            const int64_t first_row = static_cast<int64_t>(j) * a.I;
            const int64_t b0 = cta_of_row(first_row, N, G);
            const int64_t b1 = cta_of_row(first_row + a.I - 1, N, G);
            const int64_t skip = ((warp - idx) % kCombineWarps + kCombineWarps) % kCombineWarps;
            for (int64_t b = b0 + skip; b <= b1; b += kCombineWarps) {
                const int64_t k = j - cta_start(b, N, G) / a.I;
                const float4 p = __ldcs(reinterpret_cast<const float4*>(
                    a.partial + ((b * a.maxseg + k) * kTokensPerJob + q) * a.H + c));
                acc.x += p.x;
                acc.y += p.y;
                acc.z += p.z;
                acc.w += p.w;
            }
            idx += b1 - b0 + 1;
        }
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float4 s = red[0][lane];
        for (int w = 1; w < kCombineWarps; ++w) {
            const float4 o = red[w][lane];
            s.x += o.x;
            s.y += o.y;
            s.z += o.z;
            s.w += o.w;
        }
        reinterpret_cast<float4*>(a.y + static_cast<int64_t>(t) * a.H)[c / 4] = s;
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
    size_t smem;
};

static fp9_status expert_shape(int32_t H, LaunchShape& s) {
    const int nw = (H / 16 + 31) / 32;
    s.threads = nw * 32 + 32;
    const uint32_t stage = static_cast<uint32_t>(kR * H / 8 * 9);
    const int32_t optin = device_max_smem_optin();
    if (optin <= 0) return FP9_ERR_CUDA;
    int ns = static_cast<int>((static_cast<int64_t>(optin) - kRingOffset) / stage);
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns < 2) return FP9_ERR_SHAPE;
    s.nstages = ns;
    s.smem = kRingOffset + static_cast<size_t>(ns) * stage;
    return FP9_OK;
}

static fp9_status ensure_smem_attr(size_t smem) {
    static size_t configured[64] = {0};
    int dev = 0;
    FP9_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return FP9_ERR_CUDA;
    if (configured[dev] < smem) {
        FP9_CUDA_TRY(cudaFuncSetAttribute(expert_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem)));
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
    expert_kernel<<<lay.grid, shp.threads, shp.smem, stream>>>(a);
    FP9_CUDA_TRY(cudaGetLastError());
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
    combine_kernel<<<dim3(H / 128, bsz), kCombineWarps * 32, 0, stream>>>(c);
    FP9_CUDA_TRY(cudaGetLastError());
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
    lay.total = lay.off_partial + sizeof(float) * lay.maxseg * kTokensPerJob * H;
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
