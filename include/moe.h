/*
 * moe.h -- C ABI of the GB300 (sm_103a) forward pass of one Mixture-of-Experts
 * FFN layer: router, top-k gating, count / prefix-sum / permute dispatch,
 * grouped SwiGLU expert GEMMs over ragged per-expert row counts, and the
 * inverse permutation with the gate-weighted sum.
 *
 *   y = sum_{i in top-k(r(x))} g_i(x) * FFN_i(x)
 *       (Moebius reading notes, "MoE（混合专家）架构回顾", eq. (1))
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are DEVICE pointers (memory of the current CUDA device) unless a
 *   comment says otherwise.  The caller owns every buffer; the library never
 *   allocates, frees, synchronises or copies to the host inside a compute
 *   call.  All compute calls are asynchronous on `stream`.
 * - Tensors are dense and row-major; `bf16` is IEEE bfloat16 stored as
 *   uint16_t.  Every device pointer must be 16-byte aligned.
 * - Shapes: T tokens, H hidden size, E routed experts, k experts per token,
 *   I expert intermediate size.  Limits: 1 <= T <= 2^20, 1 <= k <= min(E, 32),
 *   1 <= E <= 512, T*k <= 2^24, 64 <= H <= 16384 and H % 64 == 0,
 *   64 <= I <= 32768 and I % 64 == 0.
 * - Errors: arguments are validated on the host before anything is launched;
 *   a bad argument returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED_SHAPE /
 *   MOE_ERR_WORKSPACE_TOO_SMALL and launches nothing.  A failed launch returns
 *   MOE_ERR_CUDA.  Conditions only the device can see (an expert id out of
 *   range, a pipeline wait that ran out of time) are latched in a status word
 *   at the start of the workspace and read with moe_get_device_status(); the
 *   kernels never trap.
 * - Deliberate departures from the first sketch of this interface: the
 *   dispatch call writes no permuted copy of x (moe_grouped_swiglu_ffn
 *   gathers the rows it needs into its workspace), moe_combine takes no
 *   separate shared-expert output (those rows ride in out_perm[T*k:]), and
 *   out_perm is fp16 rather than bf16 (11 significant bits for the k-row sum).
 * - Workspace: one caller-allocated device buffer of moe_workspace_size(desc)
 *   bytes (256-byte aligned) serves every call made with that descriptor;
 *   initialise its status word once with moe_workspace_init().  Calls that
 *   share a workspace must be ordered on one stream.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* identical to cudaStream_t */
typedef struct CUevent_st *moe_event_t;   /* identical to cudaEvent_t  */

typedef int32_t moe_status_t;
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,         /* NULL / misaligned pointer, bad enum        */
  MOE_ERR_UNSUPPORTED_SHAPE = -2,   /* a size outside the limits above            */
  MOE_ERR_WORKSPACE_TOO_SMALL = -3, /* ws_bytes < moe_workspace_size(desc)        */
  MOE_ERR_CUDA = -4,                /* a CUDA runtime / launch error              */
  MOE_ERR_DEVICE_CHECK = -5,        /* invalid metadata (expert id, offsets) or an
                                       expert output beyond fp16 range            */
  MOE_ERR_TIMEOUT = -6,             /* a bounded device pipeline wait ran out     */
  MOE_ERR_UNSUPPORTED_DEVICE = -7   /* current device is not compute capability 10.3 */
};

/*
 * Gating variants (CS349D lecture 8 notes, section 1.2 "MoE 层的结构"):
 *  TOPK_SOFTMAX          keep the k largest logits, softmax over them; the k
 *                        weights sum to 1 (Shazeer, Mixtral).
 *  SOFTMAX_TOPK          softmax over all E logits, keep the k largest
 *                        probabilities without renormalising; sum < 1
 *                        (DeepSeek-V2).
 *  SOFTMAX_TOPK_RENORM   as SOFTMAX_TOPK, divided by the sum of the kept k
 *                        (Qwen3 layers); equal to TOPK_SOFTMAX in exact
 *                        arithmetic, since softmax keeps the order.
 *  SIGMOID_BIAS_RENORM   affinity a = sigmoid(s); select the k largest of
 *                        a + b with a per-expert bias b that only changes the
 *                        selection; weight a_i / sum of selected a
 *                        (DeepSeek-V3).
 * Selection is decided on float32 keys; equal keys go to the lower expert
 * index; slot j of a token is its j-th best expert.
 */
enum {
  MOE_GATE_TOPK_SOFTMAX = 0,
  MOE_GATE_SOFTMAX_TOPK = 1,
  MOE_GATE_SOFTMAX_TOPK_RENORM = 2,
  MOE_GATE_SIGMOID_BIAS_RENORM = 3
};

/* Layer shape.  has_shared_expert adds one expert every token passes through
 * with weight 1 (CS349D lecture 8 notes, section 1.2, "专家的粒度": 256 routed
 * experts plus 1 shared expert). */
typedef struct {
  int32_t T, H, E, k, I;
  int32_t gating;            /* MOE_GATE_* */
  int32_t has_shared_expert; /* 0 or 1 */
} moe_layer_desc_t;

/* Layer weights (device, read-only, owned by the caller).
 *  w_router   [E,H] fp32, router s = W_r x ("MoE推理优化全景指南",
 *             "从 Dense FFN 到专家集合").
 *  sel_bias   [E] fp32 selection-only bias; required for
 *             SIGMOID_BIAS_RENORM, ignored (may be NULL) otherwise.
 *  w13        [E,2I,H] bf16: rows [0,I) gate projection, rows [I,2I) up
 *             projection of each expert's SwiGLU MLP (Moebius reading notes,
 *             eq. (2); Moebius paper, "Weights Resharding").
 *  w2         [E,H,I] bf16 down projection.
 *  w13_shared [2I,H] bf16 and w2_shared [H,I] bf16: the shared expert;
 *             required iff has_shared_expert. */
typedef struct {
  const float *w_router;
  const float *sel_bias;
  const void *w13;
  const void *w2;
  const void *w13_shared;
  const void *w2_shared;
} moe_layer_weights_t;

/* Layer weights with FP8 expert matrices (moe_layer_forward_fp8): the router
 * and selection bias as in moe_layer_weights_t; every expert matrix as E4M3
 * codes (one byte per weight, same shape and order as the bf16 tensors) with
 * one int8 block exponent s per 128 x 128 block (weight = code * 2^s),
 * written by moe_quantize_fp8:
 *  w13        [E,2I,H] E4M3;  w13_scale [E,2,ceil(I/128),ceil(H/128)] int8
 *             (the gate half's blocks, then the up half's)
 *  w2         [E,H,I] E4M3;   w2_scale [E,ceil(H/128),ceil(I/128)] int8
 *  w13_shared [2I,H] / w13_shared_scale [2,ceil(I/128),ceil(H/128)] and
 *  w2_shared [H,I] / w2_shared_scale [ceil(H/128),ceil(I/128)]: required iff
 *             has_shared_expert. */
typedef struct {
  const float *w_router;
  const float *sel_bias;
  const void *w13;
  const int8_t *w13_scale;
  const void *w2;
  const int8_t *w2_scale;
  const void *w13_shared;
  const int8_t *w13_shared_scale;
  const void *w2_shared;
  const int8_t *w2_shared_scale;
} moe_layer_weights_fp8_t;

/* Byte offsets (from the workspace base) of the buffers moe_layer_forward
 * leaves in the workspace, for inspection after the stream has synchronised.
 * R = T*k + (has_shared_expert ? T : 0) permuted rows. */
typedef struct {
  size_t status;       /* int32 status word                             */
  size_t logits;       /* [T,E] fp32 router logits                       */
  size_t topk_ids;     /* [T,k] int32                                    */
  size_t topk_w;       /* [T,k] fp32 gate weights                        */
  size_t gap;          /* [T] fp32 top-k boundary gap                     */
  size_t counts;       /* [E] int32                                      */
  size_t offsets;      /* [E+1] int32                                    */
  size_t perm_src;     /* [T*k] int32                                    */
  size_t inv_pos;      /* [T*k] int32                                    */
  size_t w_perm;       /* [T*k] fp32 gate weight in permuted order        */
  size_t x_perm;       /* [R,H] bf16 tokens grouped by expert             */
  size_t h;            /* [R,I] bf16 SiLU(gate)*up                        */
  size_t out_perm;     /* [R,H] fp16 gate-weighted expert outputs         */
  size_t plan;         /* int32 tile plan of the grouped GEMMs, nseg =
                        * E (+1 with a shared expert) segments:
                        * [0, nseg]            first permuted row of each
                        *                      segment, then R
                        * [nseg+1, 2(nseg+1))  gate/up tile prefix sum
                        * [2(nseg+1), 3(nseg+1)) down tile prefix sum
                        * 3(nseg+1) + 0 / 1    K blocks (of 64) per split-K
                        *                      piece, gate/up / down
                        * 3(nseg+1) + 2 / 3    pipeline layout, gate/up /
                        *                      down: 0 = narrow, 1 = wide,
                        *                      2 = thin (every segment has
                        *                      at most 16 rows), 3 = medium
                        *                      (down only: at most 64), 4 =
                        *                      pair (down only: 256 W2 rows
                        *                      by <= 128 token rows), 5 = thin
                        *                      pair (down only) */
  size_t total;        /* == moe_workspace_size(desc)                     */
} moe_workspace_layout_t;

/* Number of events moe_layer_forward records when given an event array:
 * before routing, after routing, after dispatch, after the gather, after the
 * gate/up GEMM, after the down GEMM, after the combine. */
#define MOE_STAGE_EVENTS 7

/* ----------------------------------------------------------------- host -- */

/* Workspace bytes every call below needs for this descriptor (worst case over
 * all routings).  Host only; 0 if the descriptor is invalid. */
size_t moe_workspace_size(const moe_layer_desc_t *d);

/* Fill *out with the workspace layout of this descriptor.  Host only. */
moe_status_t moe_workspace_layout(const moe_layer_desc_t *d, moe_workspace_layout_t *out);

/* Clear the workspace's status block (async on stream): the status word and
 * the arrival counters the small-batch router, the split-K GEMM pieces and
 * the persistent decode layer use (each returns to zero by itself when its
 * kernel completes).  Call once
 * after allocating a workspace, and again after a call reported
 * MOE_ERR_TIMEOUT or MOE_ERR_CUDA. */
moe_status_t moe_workspace_init(void *workspace, size_t ws_bytes, moe_stream_t stream);

/* Synchronise `stream`, read the status word, optionally clear it.  Returns
 * MOE_OK, MOE_ERR_DEVICE_CHECK or MOE_ERR_TIMEOUT (device conditions latched
 * since the last clear) or MOE_ERR_CUDA.  *raw (may be NULL) receives the
 * status bits. */
moe_status_t moe_get_device_status(void *workspace, size_t ws_bytes, moe_stream_t stream,
                                   int32_t clear, int32_t *raw);

/* Static text for a status code. */
const char *moe_status_string(moe_status_t s);

/* Check of the failure reporting the pipelined kernels rely on: launches one
 * thread that waits, with the same bounded wait as the GEMM and router
 * pipelines, on a barrier that nothing completes.  After about one second the
 * wait gives up and latches bit 6 in the workspace status word (the kernel
 * then returns; the context stays usable), so a following
 * moe_get_device_status returns MOE_ERR_TIMEOUT.  Asynchronous on `stream`;
 * MOE_ERR_INVALID_ARG for a NULL, unaligned or too small workspace. */
moe_status_t moe_check_bounded_wait(void *workspace, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------ compute -- */

/*
 * moe_route -- router and top-k gating.
 * Router s = W_r x ("MoE推理优化全景指南", section "从 Dense FFN 到专家集合");
 * top-k and gate weights per the variant d->gating (CS349D lecture 8 notes,
 * section 1.2).
 *   x            [T,H] bf16 hidden states
 *   w_router     [E,H] fp32;  sel_bias [E] fp32 (SIGMOID_BIAS_RENORM only)
 *   logits       [T,E] fp32 out: router logits, fp32 FMA accumulation
 *   topk_ids     [T,k] int32 out, topk_w [T,k] fp32 out (slot order: best first)
 *   boundary_gap [T] fp32 out or NULL: selection key of the k-th best expert
 *                minus that of the (k+1)-th (0 when k == E); gaps below 1e-5
 *                mark near-ties whose selection rounding can decide.
 * Uses the workspace's router scratch.
 */
moe_status_t moe_route(const moe_layer_desc_t *d, const void *x, const float *w_router,
                       const float *sel_bias, float *logits, int32_t *topk_ids, float *topk_w,
                       float *boundary_gap, void *workspace, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_build_dispatch -- count / prefix sum / permute by expert
 * ("MoE推理优化全景指南", section "Dispatch 并不是一次普通 all-to-all":
 * histogram, each expert's offset from the prefix sum, tokens permuted into
 * contiguous per-expert segments).
 *   topk_ids  [T,k] int32 in; assignment a = t*k + j
 *   topk_w    [T,k] fp32 in or NULL
 *   counts    [E] int32 out: assignments per expert
 *   offsets   [E+1] int32 out: offsets[e] = sum of counts[<e], offsets[E] = T*k
 *   perm_src  [T*k] int32 out: position p -> assignment a; expert e owns
 *             positions [offsets[e], offsets[e+1]) in ascending token order
 *   inv_pos   [T*k] int32 out: assignment a -> position p (inverse of perm_src)
 *   w_perm    [T*k] fp32 out or NULL: topk_w in permuted order (needs topk_w)
 * Bit-exact and deterministic (no atomics decide positions).  An id outside
 * [0,E) latches MOE_ERR_DEVICE_CHECK in the status word; its assignment is
 * dropped from the layout, and the outputs are then not meaningful.
 */
moe_status_t moe_build_dispatch(const moe_layer_desc_t *d, const int32_t *topk_ids,
                                const float *topk_w, int32_t *counts, int32_t *offsets,
                                int32_t *perm_src, int32_t *inv_pos, float *w_perm,
                                void *workspace, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_grouped_swiglu_ffn -- the experts' SwiGLU FFNs as grouped GEMMs over the
 * ragged per-expert row counts ("MoE推理优化全景指南", section
 * "Expert GEMM 为什么经常不够大": one scheduled GEMM over [m_i, hidden] @ W_i
 * for all experts; expert shapes from Moebius reading notes eq. (2)).
 *   h_p      = SiLU(W_gate,e x_t) * (W_up,e x_t)      (gate/up GEMM + epilogue)
 *   out_p    = w_perm[p] * (W_down,e h_p)              (down GEMM + epilogue)
 * for every position p of expert e's segment, x_t the token at p.
 *   x            [T,H] bf16
 *   perm_src     [T*k] int32, offsets [E+1] int32 (from moe_build_dispatch)
 *   w_perm       [T*k] fp32 or NULL (NULL: unweighted outputs)
 *   w13, w2      routed expert weights; w13_shared / w2_shared required iff
 *                d->has_shared_expert (run as one more segment of all T tokens
 *                with weight 1, stored in rows [T*k, T*k+T) of out_perm)
 *   out_perm     [R,H] fp16 out, R = T*k + (shared ? T : 0).  fp16 carries
 *                11 significant bits -- 8x finer than bf16 -- so the k rows a
 *                token sums stay accurate; an element beyond +-65504 is
 *                clamped and latches MOE_ERR_DEVICE_CHECK in the status word.
 * Uses the workspace for x_perm, h and the tile plan.  Experts with no rows
 * read no weights.
 */
moe_status_t moe_grouped_swiglu_ffn(const moe_layer_desc_t *d, const void *x,
                                    const int32_t *perm_src, const int32_t *offsets,
                                    const float *w_perm, const void *w13, const void *w2,
                                    const void *w13_shared, const void *w2_shared,
                                    void *out_perm, void *workspace, size_t ws_bytes,
                                    moe_stream_t stream);

/*
 * moe_combine -- inverse permutation and gate-weighted sum
 * ("MoE推理优化全景指南", section "一个 token 为什么要跨 GPU", last step
 * "inverse permutation + weighted sum", and section "Dispatch 并不是一次普通
 * all-to-all": restore the original token order and apply the routing weights).
 *   y[t,:] = sum_j wt(t,j) * out_perm[inv_pos[t*k+j],:]  (+ out_perm[T*k+t,:]
 *            when d->has_shared_expert)
 *   wt(t,j) = topk_w[t*k+j], or 1 when topk_w is NULL (weights already applied
 *            by moe_grouped_swiglu_ffn)
 *   out_perm [R,H] fp16 (as written by moe_grouped_swiglu_ffn)
 *   y        [T,H] bf16 out; sums in fp32 in slot order, rounded once.
 */
moe_status_t moe_combine(const moe_layer_desc_t *d, const void *out_perm, const int32_t *inv_pos,
                         const float *topk_w, void *y, moe_stream_t stream);

/*
 * moe_layer_forward -- the whole layer (Moebius reading notes eq. (1)): route,
 * dispatch, grouped SwiGLU FFN with the gate weights applied in the down-GEMM
 * epilogue, combine.  One stream, no host synchronisation; intermediates stay
 * in the workspace (moe_workspace_layout).
 *   x [T,H] bf16 in, y [T,H] bf16 out.
 *   stage_events: NULL, or MOE_STAGE_EVENTS cudaEvent_t handles recorded on
 *   `stream` at the stage boundaries (for per-stage timing).
 */
moe_status_t moe_layer_forward(const moe_layer_desc_t *d, const moe_layer_weights_t *w,
                               const void *x, void *y, void *workspace, size_t ws_bytes,
                               moe_stream_t stream, moe_event_t const *stage_events);

/* Execution paths of moe_layer_forward_ex. */
enum {
  MOE_PATH_AUTO = 0,        /* the persistent layer where it applies, else the chain */
  MOE_PATH_KERNEL_CHAIN = 1,/* route, dispatch, gather, two GEMMs, combine: one
                               launch per stage, linked by programmatic
                               dependent launch */
  MOE_PATH_PERSISTENT = 2,  /* one cooperative launch for the whole layer */
  MOE_PATH_CHAIN_ONE_SM = 3 /* the kernel chain with one-SM GEMM tiles only: no
                               CTA-pair tiles for prefill batches */
};

/*
 * moe_layer_forward_ex -- moe_layer_forward with a choice of execution path.
 * Both paths compute the same layer (Moebius reading notes eq. (1)) and
 * leave the same routing metadata, h and out_perm in the workspace.
 *
 * The persistent path runs the layer as phases and tile tasks of one
 * cooperative kernel with one CTA per SM, the single-kernel MoE layer of the
 * CS349D lecture 8 notes (section 6, "FlashMoE"): router logits, a bounded
 * grid barrier, top-k gating and the counting dispatch (repeated in every
 * CTA), the gate/up and down GEMM tiles with the K steps of all tiles split
 * evenly over the CTAs (a down tile of expert e starts once every gate/up
 * tile of e has written its h rows), a second grid barrier and the combine.
 * It removes the per-stage launches that dominate decode batches.  It takes
 * shapes with T <= 16 and H >= 256 (MOE_ERR_UNSUPPORTED_SHAPE otherwise when
 * requested explicitly); x_perm is not written (the gate/up tiles read x
 * directly).  Every cross-CTA wait gives up after about one second and
 * latches a timeout (MOE_ERR_TIMEOUT from moe_get_device_status); call
 * moe_workspace_init before the next use of that workspace.
 * MOE_PATH_AUTO takes the persistent path for those shapes.
 *
 * In the kernel chain, prefill-sized batches run the expert GEMMs on CTA
 * pairs: a cluster of two CTAs on two SMs computes tiles of 256 weight rows by
 * up to 256 token rows with tcgen05.mma.cta_group::2, each CTA holding half
 * of both operands.  Gate/up takes pairs from T*k >= 256*E, down from
 * T*k >= 64*E when I >= 2048 (else 256*E); H must be a multiple of 256 and I
 * of 128.
 * MOE_PATH_CHAIN_ONE_SM runs the chain with one-SM tiles at every size; the
 * two give results within rounding of each other (the K order of the fp32
 * accumulation is the same; tile shapes differ).
 *   path: MOE_PATH_*; anything else returns MOE_ERR_INVALID_ARG.
 *   stage_events (as moe_layer_forward): with the persistent path the first
 *   event is recorded before the launch and all others after it.
 */
moe_status_t moe_layer_forward_ex(const moe_layer_desc_t *d, const moe_layer_weights_t *w,
                                  const void *x, void *y, void *workspace, size_t ws_bytes,
                                  moe_stream_t stream, moe_event_t const *stage_events,
                                  int32_t path);

/*
 * FP8 expert weights ("MoE推理优化全景指南", section "量化与 offload 并非独立开关",
 * "专家权重量化": FP8 cuts the expert weights' capacity and bandwidth; the
 * scale layout is the implementation's choice).  Format: OCP FP8 E4M3 codes
 * with one power-of-two scale per block of 128 rows x 128 columns of each
 * matrix.  Because the scale is a power of two, code * 2^s is exact in bf16:
 * the FP8 layer computes the bf16 layer over the dequantised weights, with
 * half the weight bytes to stream.
 *
 * moe_quantize_fp8 -- quantise n bf16 matrices w [n][rows][K] to E4M3 codes q
 * [n][rows][K] and block exponents scale_exp [n][ceil(rows/128)][ceil(K/128)]:
 * s = the smallest integer with max|w| / 2^s <= 448 over the block (0 for an
 * all-zero block), code = round-to-nearest-even of w / 2^s, saturating at
 * +-448.  For W13 [E,2I,H] pass n = 2E, rows = I; for W2 [E,H,I] n = E,
 * rows = H.  Limits: n, rows >= 1, 64 <= K, K % 64 == 0; w and q 16-byte
 * aligned (MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED_SHAPE otherwise).
 * Asynchronous on `stream`; the caller owns every buffer.
 */
moe_status_t moe_quantize_fp8(const void *w, int32_t n, int32_t rows, int32_t K, void *q,
                              int8_t *scale_exp, moe_stream_t stream);

/*
 * moe_layer_forward_fp8 -- the layer forward (Moebius reading notes eq. (1))
 * with FP8 expert weights (moe_layer_weights_fp8_t).  The weight copies
 * stream E4M3 codes; converter warps turn them into fp16 values (times the
 * block scale, exact in fp16) and store them into TMEM, where the tensor
 * cores read the weight operand; the token rows are fp16 (x converted on the
 * way into x_perm, h written in fp16).  Decode batches (T <= 16, H >= 256)
 * run the persistent single-kernel layer of moe_layer_forward_ex; larger
 * batches the kernel chain (route, dispatch, fp16 gather, FP8 gate/up and
 * down GEMMs, combine).  An h or gate-weighted value beyond fp16's range is
 * saturated and latches MOE_ERR_DEVICE_CHECK.  Other arguments as
 * moe_layer_forward.
 */
moe_status_t moe_layer_forward_fp8(const moe_layer_desc_t *d, const moe_layer_weights_fp8_t *w,
                                   const void *x, void *y, void *workspace, size_t ws_bytes,
                                   moe_stream_t stream);

/*
 * Capacity limit ("MoE推理优化全景指南", section "Capacity、padding 与 token
 * dropping": C = ceil(capacity factor x N_a / E); an expert takes at most C
 * assignments and the rest are dropped; CS349D lecture 8 notes, section 1.4:
 * a dropped (token, expert) pair contributes 0 to the token's output).
 * Inference engines are dropless (moe_layer_forward); these calls reproduce
 * the capacity-limited layer of training systems, with a bounded number of
 * rows per expert.
 *
 * moe_expert_capacity -- C = ceil(cf * T * k / E) for cf = cf_num / cf_den,
 * in exact integer arithmetic (host only; 0 for a non-positive argument or
 * cf_num, cf_den above 2^30).
 */
int32_t moe_expert_capacity(int64_t cf_num, int64_t cf_den, int32_t T, int32_t k, int32_t E);

/*
 * moe_layer_forward_capacity -- the layer with at most `capacity` assignments
 * per routed expert: of each expert's assignments the first `capacity` in
 * token order are kept, the rest dropped (weight 0; the kept gate weights are
 * not renormalised).  The shared expert is never limited.  Kernel chain path;
 * the workspace then holds the kept layout: counts = kept rows per expert,
 * offsets over the kept rows (offsets[E] = kept assignments), perm_src over
 * them (-1 past offsets[E]), inv_pos = -1 for a dropped assignment, and the
 * shared expert's rows at [offsets[E], offsets[E] + T) of x_perm, h and
 * out_perm.  capacity >= 1 (MOE_ERR_INVALID_ARG otherwise); other arguments as
 * moe_layer_forward.
 */
moe_status_t moe_layer_forward_capacity(const moe_layer_desc_t *d, const moe_layer_weights_t *w,
                                        const void *x, void *y, int32_t capacity,
                                        void *workspace, size_t ws_bytes, moe_stream_t stream);

/* Check of the persistent layer's grid barrier: a two-CTA cooperative launch
 * waits at that barrier sized for three CTAs.  Both waits give up after about
 * one second and latch MOE_ERR_TIMEOUT's bit 7 in the status word; the kernel
 * returns and the context stays usable.  Call moe_workspace_init afterwards
 * (the barrier's arrival count is left behind).  Asynchronous on `stream`;
 * MOE_ERR_INVALID_ARG for a NULL, unaligned or too small workspace. */
moe_status_t moe_check_bounded_grid_wait(void *workspace, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_build_dispatch_noalloc -- moe_build_dispatch for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is an
 * integration aid, not a step of the method.
 *
 * Who needs it: a caller with no way to get a scratch buffer, such as a plugin
 * inside a host framework that owns the whole device-memory budget and gives
 * its extensions no allocator, or a latency-critical path that must not call
 * cudaMalloc because the call can synchronise the device.  Such a caller
 * cannot provide the workspace moe_build_dispatch needs.
 *
 * What it does: the same count / prefix sum / permute with the same results
 * (bit for bit) as moe_build_dispatch; arguments as there, minus the
 * workspace.  Its scratch lives in one fixed array of
 * MOE_NOALLOC_SCRATCH_BYTES in this library's device memory, which every GPU
 * that loads the library holds until the process exits.  The call allocates
 * nothing and calls no allocating routine.
 *   device_status  [1] int32 out or NULL: after the call, the status bits of
 *                  this dispatch (bit 0 set: an expert id outside [0,E) was
 *                  seen; its assignment was dropped from the layout).
 * Limit: with N = T*k assignments, nblk = ceil(N / chunk) blocks where
 *   chunk = max(256, 256 * ceil(ceil(N / 1024) / 256)), the call needs
 *   256 + 8 * nblk * E bytes; a larger batch returns MOE_ERR_UNSUPPORTED_SHAPE
 *   and launches nothing.  (E = 128: every T*k; E = 256: T*k <= 131072;
 *   E = 512: T*k <= 65536.)
 * Set-up: the first call on each device looks up the array's device address
 *   (with that device current); make that first call before any stream
 *   capture.  Under CUDA's lazy module loading that first lookup can load
 *   this library's device code and reserve the array's device memory (the
 *   runtime's doing, once per device); from then on no call reserves
 *   memory.  The address is cached per device, so after cudaDeviceReset the
 *   library must be reloaded before this entry point is used again.
 * Sharing: every call uses the same array and it keeps the last call's
 *   contents (the call clears what must start at zero).  Calls whose work
 *   overlaps on the GPU -- e.g. on two streams with no ordering between
 *   them -- race on the array and give wrong results; order them on one
 *   stream.
 */
#define MOE_NOALLOC_SCRATCH_BYTES ((1u << 20) + 256u) /* 1 MiB of tables + status slot */
moe_status_t moe_build_dispatch_noalloc(const moe_layer_desc_t *d, const int32_t *topk_ids,
                                        const float *topk_w, int32_t *counts, int32_t *offsets,
                                        int32_t *perm_src, int32_t *inv_pos, float *w_perm,
                                        int32_t *device_status, moe_stream_t stream);

/*
 * moe_reshard_ep_to_tp_pack -- the local permute of an expert-weight switch
 * from expert parallelism to tensor parallelism (Moebius, section 3.1 "Weights
 * Resharding" and Figure 4: EP -> TP packs each rank's complete experts into
 * one contiguous chunk per peer, so that one all-to-all delivers every peer
 * its shard of every expert already in the TP layout).  Under EP a rank owns
 * E_local complete experts; under TP each of the P ranks owns an I/P slice of
 * the intermediate dimension of every expert.
 *   w13        [E_local, 2I, H] bf16 in (rows [0,I) gate, [I,2I) up)
 *   w2         [E_local, H, I] bf16 in
 *   w13_chunks [P, E_local, 2I/P, H] bf16 out: chunk p of expert e holds gate
 *              rows [p*I/P, (p+1)*I/P), then up rows [I + p*I/P,
 *              I + (p+1)*I/P): a W13 of intermediate size I/P, gate first
 *   w2_chunks  [P, E_local, H, I/P] bf16 out: columns [p*I/P, (p+1)*I/P)
 *              of every row of W2
 * Either tensor may be skipped by passing NULL for both its input and its
 * output.  Every element is copied once (a pure permutation: bit-exact).
 * Limits: 1 <= P <= I, I % P == 0, (I/P) % 8 == 0, H % 8 == 0, E_local >= 1,
 * and each tensor below 2^35 bytes; otherwise MOE_ERR_UNSUPPORTED_SHAPE.
 * Pointers 16-byte aligned and the outputs not overlapping the inputs
 * (MOE_ERR_INVALID_ARG otherwise).  Asynchronous on `stream`; the caller
 * owns every buffer.
 */
moe_status_t moe_reshard_ep_to_tp_pack(int32_t E_local, int32_t H, int32_t I, int32_t P,
                                       const void *w13, const void *w2, void *w13_chunks,
                                       void *w2_chunks, moe_stream_t stream);

/*
 * moe_reshard_tp_to_ep_unpack -- the inverse local permute (TP -> EP:
 * Moebius, same section -- the all-to-all first delivers, from every peer q,
 * q's shard of this rank's E_local experts; the local permute then
 * interleaves the shards into complete experts).  Inputs in the chunk layout
 * of moe_reshard_ep_to_tp_pack (chunk index = the peer the shard came from),
 * outputs in the EP layout; the same limits.  unpack(pack(W)) == W exactly.
 */
moe_status_t moe_reshard_tp_to_ep_unpack(int32_t E_local, int32_t H, int32_t I, int32_t P,
                                         const void *w13_chunks, const void *w2_chunks,
                                         void *w13, void *w2, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
