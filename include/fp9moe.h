/*
 * fp9moe.h -- C ABI of the fp9 FFN/MoE decode-step library (libfp9moe.so).
 *
 * The library computes the decode-time FFN/MoE step of a DeepSeek-V3-class
 * model whose expert weights are stored in the fp9 format, on one GB300
 * (sm_103a) GPU, with hand-written CUDA kernels.
 *
 * Sources of the method:
 *   [MEMOIR-FP9]  "一鸭三吃：我把评测鸭变成了满血 DeepSeek-V3.2 推理系统"
 *                 (judgeduck.ai/duck-llm/zh/memoir.html), section
 *                 "在只有 AVX2 的 N100 上，我先做出了单核 MLP fp9": the fp9
 *                 format (1 sign bit, 5 exponent bits with the fp16 bias 15,
 *                 3 mantissa bits), stored as an 8-bit body byte per weight
 *                 plus a sign plane of 8 signs per byte, decoded by shifting
 *                 the body into fp16 bits and widening to fp32.
 *   [MEMOIR-COMM] same page, section "真正难的不是把参数塞下，而是通信": the
 *                 FFN is split tensor-parallel and f32 partial sums are added.
 *   [MEMOIR-16]   same page, section "16 tok/s 之后": the MoE forward and its
 *                 reduce of partial sums.
 *   [MTP-9.2]     "第 9 章 MTP1 dual-lane overlap"
 *                 (judgeduck.ai/duck-llm/zh/09-mtp1-dual-lane-overlap.html),
 *                 section 9.2: top_k = 8; a bsz = 2 pair reads two nearly
 *                 disjoint expert sets.
 *   [DS4-TP]      "ds4.c 学习笔记 — 张量并行"
 *                 (ds4-learning.pages.dev/glossary/tensor-parallelism.html),
 *                 section "形态一：Mac-to-Mac 张量并行": f32 partial sums, at
 *                 most 8 rows per verify batch.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must point to memory of the current
 *     CUDA device; the caller owns all memory. The library allocates no
 *     memory (the one exception is the fixed array that
 *     fp9_moe_forward_noalloc uses, a static device object of the library)
 *     and does not synchronise (the one exception is a host-buffer call
 *     with pageable memory, see fp9_moe_forward_host): work is queued on
 *     `stream` (a cudaStream_t; NULL means the legacy default stream).
 *   - Argument checks run on the host before anything is queued and are
 *     returned synchronously. A failed launch returns FP9_ERR_CUDA.
 *   - Conditions found on the device (a value out of fp9 range, a bounded
 *     wait that ran out) are recorded in *d_status, a device int32 the
 *     caller zeroes; the first error wins. d_status may be NULL, in which
 *     case they are not reported.
 *   - Matrices are row-major. An fp9 matrix [rows, cols] is two planes:
 *       body [rows, cols] uint8, byte = eeeeemmm;
 *       sign [rows, cols/8] uint8, the sign of column c in bit (c mod 8) of
 *       byte c/8 (least significant bit first); cols % 8 == 0.
 *   - Calls that share a workspace must not overlap in time (use one
 *     workspace per stream).
 */
#ifndef FP9MOE_H
#define FP9MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp9_status {
    FP9_OK = 0,
    FP9_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, bad count      */
    FP9_ERR_SHAPE = 2,       /* a dimension breaks a layout rule            */
    FP9_ERR_ALIGN = 3,       /* a pointer is not aligned as required        */
    FP9_ERR_WORKSPACE = 4,   /* the workspace is too small                  */
    FP9_ERR_RANGE = 5,       /* device: a value is not representable in fp9 */
    FP9_ERR_CUDA = 6,        /* a CUDA runtime call failed                  */
    FP9_ERR_TIMEOUT = 7      /* device: a bounded wait ran out              */
} fp9_status;

/* Limits of this implementation. */
#define FP9_MAX_BSZ 8          /* tokens per call ([DS4-TP]: 8 verify rows) */
#define FP9_MAX_HIDDEN 7168    /* hidden size H; H % 128 == 0              */
#define FP9_MAX_EXPERTS 1024   /* routed experts per layer                  */
#define FP9_MAX_GROUPS 32      /* router groups                             */
#define FP9_MAX_TOPK 16        /* experts chosen per token                  */
#define FP9_MAX_SHARED 8       /* shared experts per layer                  */
#define FP9_MAX_INTER 4194304  /* intermediate size I (2^22)                */

/*
 * A bank of n SwiGLU FFNs of equal shape, each three fp9 matrices of
 * [inter, hidden]: gate, up and down_t = W_down^T (so that one
 * intermediate row's down weights are contiguous). Each plane pointer is a
 * device pointer to n contiguous matrices:
 *   gate_body, up_body, down_body: [n, inter, hidden]      uint8
 *   gate_sign, up_sign, down_sign: [n, inter, hidden / 8]  uint8
 * All six must be 16-byte aligned. For FFN k, y = W_down (SiLU(W_gate x) *
 * (W_up x)) [MEMOIR-FP9].
 */
typedef struct fp9_ffn_bank {
    int64_t n;
    int64_t inter;
    int64_t hidden;
    const uint8_t* gate_body;
    const uint8_t* gate_sign;
    const uint8_t* up_body;
    const uint8_t* up_sign;
    const uint8_t* down_body;
    const uint8_t* down_sign;
} fp9_ffn_bank;

/*
 * One MoE layer (host struct; its pointers are device pointers).
 * Router: s = sigmoid(w_router x) over n_experts (w_router fp32
 * [n_experts, hidden], 16-byte aligned); the experts form n_groups equal
 * groups; a group scores the sum of its two largest s (its one s if groups
 * have one expert); the topk_groups best groups are kept, then the topk
 * best experts inside them (ties go to the lower index), with weights
 * s_i / sum(s_chosen) * route_scale. top_k = 8 is the pages' value
 * [MTP-9.2]; the grouping is the DeepSeek-V3 gate.
 * Output: y = sum_k w_k FFN_{id_k}(x) + sum of the shared FFNs (weight 1).
 * routed.n must equal n_experts and shared.n must equal n_shared; both
 * banks share the layer's hidden and inter.
 * In fp9_moe_forward_residual the router starts reading w_router before
 * it waits for the kernel queued just before it on the stream, when that
 * kernel lets dependents start early (programmatic dependent launch): no
 * kernel of this library writes w_router, and any other kernel has
 * completed first unless it signals its dependents early itself; such a
 * kernel must not write w_router right before a call.
 */
typedef struct fp9_moe_layer {
    int64_t hidden;
    int64_t inter;
    int32_t n_experts;
    int32_t n_groups;
    int32_t topk_groups;
    int32_t topk;
    int32_t n_shared;
    float route_scale;
    const float* w_router;
    fp9_ffn_bank routed;
    fp9_ffn_bank shared;
} fp9_moe_layer;

/*
 * fp9_pack: encode an fp32 matrix to fp9 planes [MEMOIR-FP9].
 *   src  device fp32 [rows, cols], 16-byte aligned.
 *   body device uint8 [rows, cols]; sign device uint8 [rows, cols / 8].
 *   Rounds to nearest, ties to the even mantissa, directly from fp32;
 *   keeps subnormals and the sign of zero. |x| >= 63488, Inf and NaN are
 *   stored as e = 31 codes (Inf: body 0xF8, NaN: body 0xFC) and recorded
 *   as FP9_ERR_RANGE in *d_status.
 *   Needs cols % 8 == 0 (FP9_ERR_SHAPE); rows, cols >= 0 (0 is a no-op).
 */
fp9_status fp9_pack(const float* src, int64_t rows, int64_t cols,
                    uint8_t* body, uint8_t* sign, int32_t* d_status, void* stream);

/*
 * fp9_from_fp8: convert an fp8 block-scaled checkpoint matrix to fp9 planes.
 * The pages say the DeepSeek-V3 release is fp8 (about 688 GB; the page of
 * [MEMOIR-FP9], section "真正埋下伏笔的是内存；R1 之后，问题第一次被改写")
 * with the 128x128 block-scale format also used by Qwen3's fp8 checkpoints
 * (same page, section "先用 Qwen3 练级，再让 Qwen3.5 充当高压试炼场"); fp9
 * stores no scale.
 *   w8        device uint8 [rows, cols]: fp8 e4m3 bytes (bias 7, no
 *             infinities, S.1111.111 = NaN), 8-byte aligned.
 *   scale_inv device fp32 [ceil(rows/128), ceil(cols/128)]: the scale of
 *             each 128x128 block (row-major; edge blocks cover what is left).
 *   body, sign as in fp9_pack (body 8-byte aligned). cols % 8 == 0.
 *   Each weight e4m3(w8[r, c]) * scale_inv[r/128, c/128] is rounded once,
 *   from the exact product, to the nearest fp9 (ties to the even mantissa),
 *   as fp9_pack rounds an fp32 value; magnitudes >= 63488 and NaN are
 *   recorded as FP9_ERR_RANGE in *d_status (stored as Inf / NaN codes).
 */
fp9_status fp9_from_fp8(const uint8_t* w8, const float* scale_inv, int64_t rows,
                        int64_t cols, uint8_t* body, uint8_t* sign,
                        int32_t* d_status, void* stream);

/*
 * fp9_decode: fp9 planes -> fp32 [rows, cols], bit-exact: each value is
 * the IEEE fp16 with bits (body << 7 | sign << 15), widened [MEMOIR-FP9].
 *   body, sign as in fp9_pack (device); dst device fp32 [rows, cols],
 *   16-byte aligned. cols % 8 == 0.
 */
fp9_status fp9_decode(const uint8_t* body, const uint8_t* sign, int64_t rows,
                      int64_t cols, float* dst, void* stream);

/*
 * Workspace sizes (bytes) for moe_router / fp9_moe_forward and for
 * fp9_dense_ffn at batch bsz, on the current device. Return 0 when the
 * arguments are invalid or the device cannot be queried. A workspace must
 * be 256-byte aligned and zeroed once after allocation; every call leaves
 * its internal counter at zero again.
 */
size_t fp9_moe_workspace_bytes(const fp9_moe_layer* layer, int32_t bsz);
size_t fp9_dense_workspace_bytes(const fp9_ffn_bank* ffn, int32_t bsz);

/*
 * moe_router: routing only.
 *   x device fp32 [bsz, hidden]; ids device int32 [bsz, topk] in
 *   descending score order; weights device fp32 [bsz, topk]. 1 <= bsz <=
 *   FP9_MAX_BSZ. Logits are fp32 dot products.
 */
fp9_status moe_router(const fp9_moe_layer* layer, const float* x, int32_t bsz,
                      int32_t* ids, float* weights, void* ws, size_t ws_bytes,
                      void* stream);

/*
 * fp9_moe_forward: y = MoE(x) for one layer, at 1 <= bsz <= FP9_MAX_BSZ.
 *   x, y device fp32 [bsz, hidden], 16-byte aligned (y may not alias x).
 *   ids / weights: optional device outputs of the routing (NULL to skip).
 *   An expert chosen by several tokens is one job per token; its rows are
 *   read with the L2 evict-normal priority, so the repeated reads mostly
 *   hit in L2 (every other weight is read once, evict-first); partial sums over intermediate slices stay fp32 and
 *   are added in a fixed order, so results are deterministic for a given
 *   device ([MEMOIR-COMM], [MEMOIR-16], [DS4-TP]).
 */
fp9_status fp9_moe_forward(const fp9_moe_layer* layer, const float* x,
                           int32_t bsz, float* y, int32_t* ids, float* weights,
                           void* ws, size_t ws_bytes, int32_t* d_status,
                           void* stream);

/*
 * fp9_moe_forward_residual: one layer step of a stack of MoE layers with the
 * glue between layers folded into the layer's own kernels ("第 9 章 MTP1
 * dual-lane overlap", section 9.5: stage 0 of a decode layer holds the
 * layernorm and the residual add). Per token t:
 *   in[t] = x[t] if x is given, else h[t] / sqrt(mean(h[t]^2) + eps)
 *           (RMSNorm with unit gain, mean(h[t]^2) from the partial sums
 *           in ss[t]);
 *   h[t] += MoE(in[t]) of `layer`, as fp9_moe_forward computes it;
 *   ss[t, b] = the sum of the squares of the new h[t, 16 b .. 16 b + 15],
 *           b = 0 .. hidden / 16 - 1 (the next call's norm).
 * A stack calls it once per layer: the first layer with x = RMSNorm(h)
 * (fp9_residual_rmsnorm(h, NULL, x)), the others with x = NULL; after the
 * last, fp9_residual_rmsnorm(h, NULL, x_out) gives the normed output. No x
 * is stored between layers: the router and the fused kernel scale h where
 * they read it, and the combine kernel writes h and ss, so a layer step is
 * three kernels instead of four. The partial sums and their total are added
 * in fixed orders (deterministic for a device); the router and the fused
 * kernel form the same scale bit for bit.
 *   x      device fp32 [bsz, hidden] or NULL; may not alias h.
 *   h      device fp32 [bsz, hidden], updated in place.
 *   ss     device fp32 [bsz, hidden / 16]: read when x is NULL, rewritten.
 *   eps    0 <= eps <= 1.
 *   next   the stack's next layer, or NULL: its router weights are read
 *          into L2 (a prefetch hint, issued by the expert kernel's CTAs
 *          once they have issued their last weight copies), so that the
 *          next call's router finds them there even when many layers are
 *          resident. Checked like `layer`.
 *   layer, bsz, ids, weights, ws, ws_bytes (fp9_moe_workspace_bytes),
 *   d_status, stream: as fp9_moe_forward. x, h, ss 16-byte aligned.
 *   Errors: as fp9_moe_forward.
 */
fp9_status fp9_moe_forward_residual(const fp9_moe_layer* layer, const float* x,
                                    float* h, float* ss, int32_t bsz, float eps,
                                    const fp9_moe_layer* next, int32_t* ids,
                                    float* weights, void* ws, size_t ws_bytes,
                                    int32_t* d_status, void* stream);

/*
 * fp9_moe_forward_host: fp9_moe_forward with x and y in host memory, for a
 * caller that holds its activations on the host (one call per layer step
 * instead of a copy, the forward and a copy). This is an interface of this
 * library only; the pages have no counterpart.
 *   x_host, y_host: host fp32 [bsz, hidden]. With page-locked memory both
 *   transfers are asynchronous and the call returns at once. With a pageable
 *   y_host the call is synchronous: the copy of y back to pageable memory
 *   returns only once it is done, i.e. after the whole forward (a pageable
 *   x_host only makes the copy of x finish before the call returns). Queued
 *   on `stream`: the copy of x into the workspace, the forward, and the copy
 *   of y back, except for a page-locked y_host that the device can address
 *   (cudaPointerGetAttributes gives it a device address, 16-byte aligned),
 *   which the forward's last kernel writes directly. y_host holds the result
 *   once the stream has reached that point (synchronise the stream, or wait
 *   on an event recorded after the call).
 *   ws: device, >= fp9_moe_host_workspace_bytes(layer, bsz), 256-byte
 *   aligned: fp9_moe_forward's workspace followed by two staging rows.
 *   Errors: as fp9_moe_forward; FP9_ERR_CUDA if a copy cannot be queued.
 */
fp9_status fp9_moe_forward_host(const fp9_moe_layer* layer,
                                const float* x_host, int32_t bsz,
                                float* y_host, void* ws, size_t ws_bytes,
                                int32_t* d_status, void* stream);
size_t fp9_moe_host_workspace_bytes(const fp9_moe_layer* layer, int32_t bsz);

/*
 * fp9_dense_ffn: y = FFN(x) for a dense fp9 SwiGLU FFN (ffn->n == 1), as in
 * the model's first layers: the page of [MEMOIR-FP9], section "在只有 AVX2 的
 * N100 上，我先做出了单核 MLP fp9", where the fp9 MLP first ran as one dense
 * SwiGLU MLP on a single core (gate, up, SiLU(gate) * up, down).
 *   x, y   device fp32 [bsz, hidden], 16-byte aligned, y may not alias x;
 *          1 <= bsz <= FP9_MAX_BSZ.
 *   ffn    host struct (device planes), n == 1; hidden % 128 == 0 and
 *          hidden <= FP9_MAX_HIDDEN, 1 <= inter <= FP9_MAX_INTER
 *          (FP9_ERR_SHAPE otherwise).
 *   ws     device, >= fp9_dense_workspace_bytes(ffn, bsz), 256-byte aligned.
 *   The weights are streamed once per call for each pair of tokens; the
 *   arithmetic is the decode step's (fp32 products and sums, partials over
 *   intermediate slices added in a fixed order: deterministic for a device).
 *   Errors: argument checks as above (synchronous); FP9_ERR_TIMEOUT in
 *   *d_status if a bounded wait runs out.
 */
fp9_status fp9_dense_ffn(const fp9_ffn_bank* ffn, const float* x, int32_t bsz,
                         float* y, void* ws, size_t ws_bytes, int32_t* d_status,
                         void* stream);

/*
 * Precision of the prefill entry points (their `precision` argument). The
 * fp9 weights are exact in fp16 (body << 7 | sign << 15 is their fp16,
 * [MEMOIR-FP9]), so only the activations x and h = SiLU(W_gate x) *
 * (W_up x) are rounded to the MMA's fp16 operand type:
 *   FP9_PREFILL_SPLIT (0, the default): each activation is carried as two
 *     fp16 terms, hi = fp16(v) and lo = fp16(v - hi) (22 significant bits),
 *     and every weight meets both in fp32-accumulated MMAs; y agrees with
 *     the exact FFN within 2e-4 * max|y| per token row, as the decode path
 *     does. It takes about twice the MMA work of the dense kernels.
 *   FP9_PREFILL_FP16 (1, opt-in): one fp16 term per activation; y differs
 *     from the exact FFN by about the fp16 unit roundoff (2^-11) relative
 *     to sum |terms|, which misses that rule (relative L2 error about
 *     4e-4); faster.
 */
#define FP9_PREFILL_SPLIT 0
#define FP9_PREFILL_FP16 1

/*
 * fp9_ffn_prefill: y = FFN_k(x) for m tokens at once (prompt prefill), on
 * the tensor cores. The pages run the same fp9 FFN over every prompt token
 * and list their prefill kernel as far below the hardware's compute peak
 * (the page of [MEMOIR-FP9], section "最终结果", its list of limitations);
 * with m tokens the FFN is two dense GEMMs (gate/up with SwiGLU, then down).
 *   ffn    host struct of a bank (device planes); k in [0, ffn->n) selects
 *          the FFN (e.g. the dense FFN, or one expert of a bank).
 *   x      device fp32 [m, hidden]; y device fp32 [m, hidden]; both
 *          16-byte aligned. y may alias x (x is read, as fp16, before y
 *          is written). 0 <= m <= FP9_MAX_PREFILL_TOKENS
 *          (m = 0 is a no-op).
 *   Shape: hidden % 256 == 0 (256 <= hidden <= FP9_MAX_PREFILL_HIDDEN),
 *          inter % 128 == 0 (inter <= FP9_MAX_INTER), else FP9_ERR_SHAPE.
 *   precision  FP9_PREFILL_SPLIT (default) or FP9_PREFILL_FP16, see above;
 *          any other value is FP9_ERR_INVALID_ARG.
 *   ws     device, >= fp9_prefill_workspace_bytes(ffn, m), 256-byte aligned
 *          (holds x and h = SiLU(W_gate x) * (W_up x) as fp16 terms, and
 *          for small m the down GEMM's partial outputs: it then splits K
 *          into up to 4 parts and adds them in part order, so y is still
 *          deterministic).
 *   Arithmetic: products of the exact fp16 weights and the fp16 activation
 *   terms are accumulated in fp32 (tensor memory). An x or h whose fp16 is
 *   not finite (|v| >= 65520, Inf, NaN) is recorded as FP9_ERR_RANGE in
 *   *d_status.
 */
#define FP9_MAX_PREFILL_TOKENS 1048576
#define FP9_MAX_PREFILL_HIDDEN 32768
fp9_status fp9_ffn_prefill(const fp9_ffn_bank* ffn, int64_t k, const float* x,
                           int64_t m, float* y, int32_t precision, void* ws,
                           size_t ws_bytes, int32_t* d_status, void* stream);

/* Workspace bytes of fp9_ffn_prefill for m tokens on the current device
 * (0 if the arguments are invalid), for either precision: x and h as two
 * fp16 terms each, plus fp32 partial outputs when the down GEMM splits K
 * for this m on this device's SM count (small m), so query it on the
 * device that will run the call. */
size_t fp9_prefill_workspace_bytes(const fp9_ffn_bank* ffn, int64_t m);

/*
 * fp9_moe_prefill: y = MoE(x) for m tokens at once (prompt prefill): the
 * layer of fp9_moe_forward, with the expert FFNs on the tensor cores. The
 * router is the decode step's (fp32 logits, then the same selection rules
 * and weight formula); each token's slots are grouped by expert, every
 * expert with tokens runs its FFN once over all of them as a GEMM (the
 * arithmetic of fp9_ffn_prefill, in the chosen `precision`), and y[t] =
 * sum_k w[t,k] FFN_{id[t,k]}(x[t]) + sum_s FFN_shared_s(x[t]) is added in
 * slot, then shared-expert order (deterministic for a device).
 *   layer  as for fp9_moe_forward, plus hidden % 256 == 0 and inter % 128
 *          == 0 (FP9_ERR_SHAPE).
 *   x, y   device fp32 [m, hidden], 16-byte aligned, y may not alias x;
 *          0 <= m <= FP9_MAX_PREFILL_TOKENS (0 is a no-op).
 *   ids, weights  optional device outputs [m, topk] (NULL to skip).
 *   precision  FP9_PREFILL_SPLIT (default) or FP9_PREFILL_FP16.
 *   ws     device, >= fp9_moe_prefill_workspace_bytes(layer, m), 256-byte
 *          aligned, zeroed once after allocation (its counter resets
 *          itself). It holds the routing, and x, h and the per-expert
 *          outputs of every (token, expert) pair: about
 *          m * (topk + n_shared) * (8 * hidden + 4 * inter) bytes.
 *   A token value or h whose fp16 is not finite is FP9_ERR_RANGE.
 */
fp9_status fp9_moe_prefill(const fp9_moe_layer* layer, const float* x,
                           int64_t m, float* y, int32_t* ids, float* weights,
                           int32_t precision, void* ws, size_t ws_bytes,
                           int32_t* d_status, void* stream);

/* Workspace bytes of fp9_moe_prefill for m tokens (0 if invalid). */
size_t fp9_moe_prefill_workspace_bytes(const fp9_moe_layer* layer, int64_t m);

/*
 * fp9_residual_rmsnorm: stack glue between layers, per token t:
 *   h[t] += y[t] (skipped when y is NULL);
 *   x_out[t] = h[t] / sqrt(mean(h[t]^2) + eps)   (unit gain).
 * The pages keep the layernorm and the residual add on the GPU side of each
 * decode layer ("第 9 章 MTP1 dual-lane overlap", section 9.5: stage 0 of a
 * layer holds them); between two MoE layers of a stack the step is
 * h <- h + MoE(RMSNorm(h)).
 *   h, y, x_out device fp32 [bsz, hidden], 16-byte aligned, hidden % 4 == 0;
 *   h is updated in place; x_out may not alias h or y. 1 <= bsz <=
 *   FP9_MAX_BSZ, eps >= 0. The sum of squares is added in a fixed order.
 *   Errors: FP9_ERR_INVALID_ARG / FP9_ERR_SHAPE / FP9_ERR_ALIGN (synchronous).
 */
fp9_status fp9_residual_rmsnorm(float* h, const float* y, float* x_out,
                                int32_t bsz, int64_t hidden, float eps,
                                void* stream);

/*
 * fp9_selftest_timeout: failure-detection check. Launches the fused expert
 * kernel on a small dense problem with its weight copies switched off, so
 * every consumer wait runs out after timeout_us microseconds; the kernel
 * records FP9_ERR_TIMEOUT in *d_status and returns with the context
 * intact. ws: device, >= 64 KiB, 256-byte aligned (used as x and scratch).
 */
fp9_status fp9_selftest_timeout(void* ws, size_t ws_bytes, int32_t* d_status,
                                int32_t timeout_us, void* stream);

/*
 * fp9_prefill_selftest_timeout: failure-detection check of the prefill
 * kernels' bounded waits. Launches one gate/up CTA of fp9_ffn_prefill (128
 * tokens, hidden 256, inter 128) with its weight copies switched off, so
 * every wait on the weights runs out after timeout_us microseconds; the
 * kernel records FP9_ERR_TIMEOUT in *d_status, waits (bounded) for its own
 * copies and MMAs, frees its tensor memory and returns with the context
 * intact. ws: device, >= 128 KiB, 256-byte aligned (scratch); timeout_us in
 * [1, 1000000].
 */
fp9_status fp9_prefill_selftest_timeout(void* ws, size_t ws_bytes,
                                        int32_t* d_status, int32_t timeout_us,
                                        void* stream);

/*
 * fp9_moe_forward_noalloc: fp9_moe_forward for callers that cannot
 * allocate device memory (a runtime whose device memory is owned and
 * capped by another framework, a plugin handed only its input and output
 * buffers, a latency-critical path that must not risk the synchronisation
 * of an allocation). The pages have no counterpart: this is an interface
 * of this library only.
 *   Same arguments and results as fp9_moe_forward without ws / ws_bytes.
 *   The workspace is a fixed array of fp9_moe_noalloc_scratch_bytes()
 *   (16 MiB) of device memory inside the library, held by every GPU that
 *   loads it until the process exits; no memory is allocated by the call.
 *   A call whose workspace would not fit returns FP9_ERR_WORKSPACE (the
 *   DeepSeek-V3 layer fits up to bsz 3 on a 152-SM GPU).
 *   The first call on a device looks up the array's device address on
 *   that device (cudaGetSymbolAddress), and so does the first call after
 *   the device's context was replaced (cudaDeviceReset): make that call
 *   before any stream capture.
 *   Every call clears the control block it needs zeroed. All calls share
 *   the one array, so calls that overlap on the GPU (other streams, other
 *   host threads) race: serialise them.
 */
fp9_status fp9_moe_forward_noalloc(const fp9_moe_layer* layer, const float* x,
                                   int32_t bsz, float* y, int32_t* ids,
                                   float* weights, int32_t* d_status,
                                   void* stream);

/* Size in bytes of the fixed scratch array of fp9_moe_forward_noalloc. */
size_t fp9_moe_noalloc_scratch_bytes(void);

/*
 * fp9_profile_events: tracing hook. When both events (cudaEvent_t handles
 * created by the caller) are non-NULL, every later launch of the fused
 * expert kernel records `start` just before and `stop` just after itself,
 * on its own stream, so the caller can time that kernel alone; NULL, NULL
 * turns this off. Process-wide setting, not thread-safe.
 */
void fp9_profile_events(void* start, void* stop);

/* Human-readable name of a status code (static string). */
const char* fp9_status_str(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* FP9MOE_H */
