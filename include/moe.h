/*
 * moe.h -- C ABI of the single-GPU MoE layer path for GB300 (sm_103a).
 *
 * The path ("gating -> dispatch -> experts -> combine") is the runtime MoE
 * execution path described in "第十五章：多节点大模型推理" section 4.1/4.3 and
 * in the token trace page, hop 4 ("dispatch to two experts"), with the
 * group-limited routing of the "ep-deploy" handbook page (section "EPLB 与路由
 * 约束") and the gate_up-fused, masked expert GEMM of the MoE-TP/EP comparison
 * on "推理INFRA方法论-02-parallelism".  On one GPU the all-to-all of those pages
 * becomes a permutation into expert-contiguous rows and back.
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer owned by the caller, except
 *    the shape struct and the `bytes`/`status` out-parameters, which are host
 *    pointers.  The library never allocates or frees device memory.
 *  - Tensors are dense and row-major.  bf16 means IEEE bfloat16 (uint16 bit
 *    pattern).  Pointers to bf16/fp32 tensors must be 16-byte aligned; the
 *    workspace must be 256-byte aligned.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) and runs asynchronously.  Host-side validation returns a status
 *    synchronously before anything is enqueued; MOE_ERR_CUDA means a launch
 *    failed (cudaGetLastError()).
 *  - Errors detected on the device (an expert id out of range, masked_m >
 *    M_max, a bounded wait that timed out) are OR-ed into a status word at
 *    the start of the workspace and read with moe_get_device_status().
 *    Kernels never trap; a timed-out wait returns and leaves the context
 *    usable.
 *  - T == 0 is a valid no-op returning MOE_OK.
 *  - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

/* Router score function. */
typedef enum {
  /* s'_e = sigmoid(l_e) + bias_scale * bias_e selects; weights are the
   * selected sigmoid(l) renormalised to sum 1 (bias only selects). */
  MOE_SCORE_SIGMOID_BIAS = 0,
  /* softmax over the logits; the top-k of softmax equals the top-k of the
   * logits; weights are the selected softmax values renormalised. */
  MOE_SCORE_SOFTMAX = 1
} moe_score_t;

/* Problem statement: T tokens of hidden size d, E experts in G equal groups,
 * keep topk_group groups, route each token to k experts; each expert is a
 * SwiGLU FFN of width inter. */
typedef struct {
  int32_t T;
  int32_t d;
  int32_t E;
  int32_t G;
  int32_t topk_group;
  int32_t k;
  int32_t inter;
  int32_t score;    /* moe_score_t */
  float bias_scale; /* 0.15 in the routing simulation of the ep-deploy page */
} moe_shape_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misalignment */
  MOE_ERR_UNSUPPORTED = 2, /* valid shape the kernels do not handle */
  MOE_ERR_WORKSPACE = 3,   /* workspace too small or misaligned */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  MOE_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out */
  MOE_ERR_OVERFLOW = 6     /* masked_m[e] > M_max (rows beyond are ignored) */
} moe_status_t;

typedef enum { MOE_LAYOUT_CONTIGUOUS = 0, MOE_LAYOUT_MASKED = 1 } moe_layout_t;

/* What happens to assignments past an expert's capacity ("第十五章" section
 * 4.3, overflow table): dropped (they add nothing to the output), or run in a
 * second round on the same expert after the first. */
typedef enum { MOE_OVERFLOW_DROP = 0, MOE_OVERFLOW_SECOND_ROUND = 1 } moe_overflow_t;

/* Shape limits (MOE_ERR_INVALID_ARG beyond them unless noted):
 *   E % G == 0, 1 <= topk_group <= G <= 32, 1 <= k <= min(32, topk_group*E/G),
 *   E <= 1024, d % 8 == 0, T*k < 2^31.
 * Expert FFN additionally needs d % 64 == 0 and inter % 64 == 0
 * (MOE_ERR_UNSUPPORTED otherwise). */

/* Human-readable name of a status. Never NULL. */
const char *moe_status_string(moe_status_t status);

/* Bytes of workspace that moe_route, moe_dispatch, moe_expert_ffn
 * (contiguous layout) and moe_layer need for `shape`. */
moe_status_t moe_workspace_size(const moe_shape_t *shape, size_t *bytes);

/* Bytes of workspace for moe_expert_ffn / moe_expert_gate_up /
 * moe_expert_down with the given layout (M_max is ignored for the contiguous
 * layout, where the rows are T*k). */
moe_status_t moe_expert_ffn_workspace_size(const moe_shape_t *shape, int32_t layout,
                                           int32_t M_max, size_t *bytes);

/* Prepares a fresh workspace (async): clears the device status word and the
 * flags the expert FFN's down GEMM uses between CTAs (zero at rest, and left
 * zero by every call that completes).  Call once before the workspace's
 * first use. */
moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronises `stream`, returns the OR of device-side errors recorded in the
 * workspace since the last call (as the highest-numbered status found), and
 * clears the word.  When the word was not zero it also clears the down
 * GEMM's flags (a launch that stopped at a timed-out wait can leave them
 * raised), so the workspace is ready for the next call, a replayed graph
 * included.  The only entry point that blocks the host. */
moe_status_t moe_get_device_status(void *ws, size_t ws_bytes, moe_stream_t stream,
                                   moe_status_t *status);

/*
 * Gating ("第十五章" 4.1: the model's gating picks the top-k logical experts
 * from the hidden state; "ep-deploy" page: group-limited top-k).
 *   x      [T,d]  bf16     token hidden states
 *   w_r    [d,E]  bf16     router weight
 *   bias   [E]    fp32     per-expert selection bias (NULL for softmax)
 *   topk_ids [T,k] int32   out: experts, descending selection score, ties to
 *                          the lower index
 *   topk_w   [T,k] fp32    out: combine weights (sum to 1 per token)
 *   logits   [T,E] fp32    out, optional (NULL): router logits
 * Logits are fp32 sums of exact bf16 products in a fixed order (lane l of 32
 * owns the 8-element chunks c with c mod 32 == l and sums them in order; the
 * 32 lane sums are combined by an xor butterfly), and sigmoid/exp use a
 * fixed Cody-Waite + Taylor evaluation, so ids are reproducible bit-exactly.
 * With logits == NULL, d % 64 == 0, d <= 16384 and E % 64 == 0 the call is
 * screened, with the same outputs: the logits are first taken on the tensor
 * cores, where every accumulation chain is 8 MMAs long; each score gets an
 * interval that holds its fixed-order value, from the bound
 *   |l_tc - l_fixed| <= alpha(d) * ||x_t||_2 * ||w_e||_2
 * (alpha is about 8e-5 at d = 7168; it covers the fixed order's own
 * rounding and tensor-core accumulation whose every MMA errs by up to 2^-17
 * of the magnitudes it adds, 64 units in the last place); every expert whose
 * selection (or whose group's keep decision) the intervals leave open gets
 * its fixed-order logit, and the selection is made on those.  Every selected
 * expert is among them, so its weight and order come from fixed-order
 * logits.  The outputs equal the fixed-order ones for any finite input, with
 * no margin or data-dependent condition; moe_route_refined_count reports how
 * many fixed-order logits a call computed.
 */
moe_status_t moe_route(const moe_shape_t *shape, const void *x, const void *w_r,
                       const float *bias, int32_t *topk_ids, float *topk_w,
                       float *logits, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * The scoring + group-limited selection half of moe_route on given logits
 * [T,E] fp32 (same outputs).  Needs no workspace.
 */
moe_status_t moe_route_from_logits(const moe_shape_t *shape, const float *logits,
                                   const float *bias, int32_t *topk_ids, float *topk_w,
                                   moe_stream_t stream);

/*
 * Group-limited top-k alone ("ep-deploy" page, section "EPLB 与路由约束": a
 * group's score is the sum of its two best expert scores, the topk_group best
 * groups are kept, the k best experts inside them are chosen) on given fp32
 * scores [T,E].  Group sums are fp32.  Ties go to the lower index.
 */
moe_status_t moe_group_topk(const moe_shape_t *shape, const float *scores,
                            int32_t *topk_ids, moe_stream_t stream);

/*
 * Dispatch as a permutation ("第十五章" 3.4: dispatch sends each token's
 * activation to its k experts; single GPU: expert-contiguous rows).
 *   topk_ids [T,k] int32  expert of each assignment a = t*k + j
 *   x        [T,d] bf16   (may be NULL to compute indices only)
 *   counts   [E]   int32  out: assignments per expert (sum T*k)
 *   offsets  [E+1] int32  out: exclusive prefix sum of counts
 *   src_token [T*k] int32 out: token of each permuted row
 *   dest     [T*k] int32  out: permuted row of each assignment
 *   x_perm   [T*k,d] bf16 out (ignored if x is NULL): x_perm[dest[a]] = x[a/k]
 * Order inside an expert is stable in a (a counting sort); no atomics-order
 * dependence.  Ids outside [0,E) set MOE_ERR_INVALID_ARG on the device.
 */
moe_status_t moe_dispatch(const moe_shape_t *shape, const int32_t *topk_ids,
                          const void *x, int32_t *counts, int32_t *offsets,
                          int32_t *src_token, int32_t *dest, void *x_perm, void *ws,
                          size_t ws_bytes, moe_stream_t stream);

/*
 * Expert SwiGLU FFN as grouped GEMMs on the tensor cores (the "DeepGEMM
 * masked, gate_up fused" kernel of the MoE-TP/EP comparison page, rebuilt for
 * tcgen05): per expert e, h = silu(X_e Wg_e^T) * (X_e Wu_e^T) (bf16), then
 * y = h Wd_e^T (fp32).
 *   layout MOE_LAYOUT_CONTIGUOUS: x_in [T*k, d] bf16, rows of expert e are
 *       [offsets[e], offsets[e+1]) (seg = offsets, [E+1]); y_out [T*k, d].
 *   layout MOE_LAYOUT_MASKED: x_in [E, M_max, d] bf16, rows [0, masked_m[e])
 *       of slab e are valid (seg = masked_m, [E]); y_out [E, M_max, d]; rows
 *       past masked_m are not written.
 *   w_gate_up [E, 2*inter, d] bf16 (rows 0..inter-1 gate, inter.. up)
 *   w_down    [E, d, inter] bf16
 *   y_out     fp32
 * Experts with no rows cost nothing (their weights are not read).
 * The down GEMM is a persistent grid; when its last wave is short, two CTA
 * pairs share each of its tiles (K halves) through flags in the workspace.
 * The half that reaches its epilogue first stores, the other adds; the only
 * wait is the adder's, on a half that is already storing, so the launch does
 * not need its pairs to be resident together (kernels on other streams may
 * hold SMs).  The wait is bounded all the same (a timeout sets
 * MOE_ERR_TIMEOUT).  Results do not depend on timing: either order gives the
 * same fp32 sum.  Each call clears the flags before the down GEMM runs, so
 * calls captured in a CUDA graph may be replayed.
 */
moe_status_t moe_expert_ffn(const moe_shape_t *shape, int32_t layout, const void *x_in,
                            const int32_t *seg, int32_t M_max, const void *w_gate_up,
                            const void *w_down, float *y_out, void *ws, size_t ws_bytes,
                            moe_stream_t stream);

/* First half of moe_expert_ffn: h_out = silu(X Wg^T) * (X Wu^T), bf16,
 * [rows, inter] in the same layout as x_in. */
moe_status_t moe_expert_gate_up(const moe_shape_t *shape, int32_t layout,
                                const void *x_in, const int32_t *seg, int32_t M_max,
                                const void *w_gate_up, void *h_out, void *ws,
                                size_t ws_bytes, moe_stream_t stream);

/* Second half: y_out = h Wd^T, fp32, [rows, d] in the same layout as h_in. */
moe_status_t moe_expert_down(const moe_shape_t *shape, int32_t layout, const void *h_in,
                             const int32_t *seg, int32_t M_max, const void *w_down,
                             float *y_out, void *ws, size_t ws_bytes,
                             moe_stream_t stream);

/*
 * Combine (token trace page, hop 4: y = p5 E5(x) + p27 E27(x)):
 *   y[t] = sum_{j<k} topk_w[t,j] * y_perm[dest[t*k+j]]   (fp32, j ascending)
 *   y_perm [T*k, d] fp32, dest [T*k] int32, topk_w [T,k] fp32, y [T,d] bf16.
 */
moe_status_t moe_combine(const moe_shape_t *shape, const float *y_perm,
                         const int32_t *dest, const float *topk_w, void *y,
                         moe_stream_t stream);

/*
 * The whole layer: route -> dispatch -> gate_up+SwiGLU -> down -> combine,
 * all on `stream`, no host synchronisation, intermediates in the workspace.
 * With d a multiple of 256 (moe_layer_yperm_row_bytes then 2*d + d/32), the
 * down GEMM keeps its rows in a compact form: each group of
 * 32 columns as fp16 values scaled by a power of two (the group's largest
 * magnitude just under 2^15) and one byte for that exponent, a rounding of
 * at most 2^-11 of the group's largest value; the combine restores each
 * value exactly from that form before its fp32 sum.  Elsewhere the rows stay
 * fp32, as moe_expert_ffn writes them.
 *   x [T,d] bf16, w_r [d,E] bf16, bias [E] fp32 (NULL for softmax),
 *   w_gate_up [E,2*inter,d] bf16, w_down [E,d,inter] bf16, y [T,d] bf16 out,
 *   topk_ids [T,k] int32 / topk_w [T,k] fp32 / counts [E] int32: optional
 *   copies of the routing and the per-expert counts (NULL to skip).
 *   stage_events: NULL, or 6 cudaEvent_t handles (host array) recorded on
 *   `stream` before the router, after the router, after dispatch, after the
 *   gate_up GEMM, after the down GEMM and after combine (per-stage timing).
 */
moe_status_t moe_layer(const moe_shape_t *shape, const void *x, const void *w_r,
                       const float *bias, const void *w_gate_up, const void *w_down,
                       void *y, int32_t *topk_ids, float *topk_w, int32_t *counts,
                       void *ws, size_t ws_bytes, void *const *stage_events,
                       moe_stream_t stream);

/*
 * moe_dispatch without a workspace, for callers that cannot allocate device
 * memory: a serving runtime that reserves all of HBM up front and hands out
 * no further buffers, plain C code with no device allocator of its own, or
 * code on a path where cudaMalloc/cudaFree (which may synchronise the
 * device) are not allowed.  The pages have no counterpart; it is a
 * convenience of this library.
 *   Arguments and outputs are those of moe_dispatch minus the workspace.
 *   The per-chunk expert histograms live in a 1 MiB device array inside the
 *   library (every GPU that loads the library holds it until exit), which
 *   limits ceil(T*k / c) * E to 262144 entries, c being the assignments per
 *   chunk (128 up to T*k = 32768, 512 beyond; so T*k <= 524288 at E = 256);
 *   larger shapes return MOE_ERR_UNSUPPORTED.  Nothing is allocated.
 *   The first call on a device looks up the array's device address (no
 *   allocation) and caches it with the id of the device's current context;
 *   a call that finds another context current (after cudaDeviceReset, say)
 *   looks it up again.  Make the first call on a device, and the first
 *   after such a reset, before any stream capture.
 *   All calls share the array: calls that overlap on the GPU race; calls
 *   ordered on one stream are safe, and nothing needs clearing between them.
 *   Out-of-range ids are skipped (their counts are missing from `counts`)
 *   but, with no workspace, not reported in a status word.
 */
moe_status_t moe_dispatch_noalloc(const moe_shape_t *shape, const int32_t *topk_ids,
                                  const void *x, int32_t *counts, int32_t *offsets,
                                  int32_t *src_token, int32_t *dest, void *x_perm,
                                  moe_stream_t stream);

/*
 * Dispatch onto physical expert copies ("ep-deploy" handbook page, section
 * "EPLB 与路由约束": hot experts are copied and placed; "第十五章" section 4.3:
 * the gating picks logical experts and the system sends each assignment to
 * one of the expert's equivalent copies, the less loaded one).
 *   phys_expert [P] int32 (device): the logical expert held by each physical
 *     slot, in placement order (moe_eplb_plan's gpu_slots: GPU g holds slots
 *     g*P/G .. (g+1)*P/G - 1).  1 <= P <= 65536.
 *   The r-th assignment (in increasing a = t*k + j) of logical expert e,
 *   which has n_rep copies, goes to its copy r mod n_rep, copies counted in
 *   slot order -- at every step the copy with the fewest rows so far, ties
 *   to the first; an expert's copies thus differ by at most one row.
 * Outputs (device, caller-owned): counts_phys [P], offsets_phys [P+1]
 *   (exclusive scan in slot order, so the rows of a GPU's slots are one
 *   contiguous range: the send buffer of an expert-parallel dispatch),
 *   dest [T*k] (row of each assignment; -1 for an id outside [0,E) or an
 *   expert with no copy), src_token [T*k] (token of each row), x_perm
 *   [T*k, d] bf16 rows (NULL x to skip the gather).  Rows are contiguous per
 *   slot and stable in a inside a slot.  With one copy per expert in expert
 *   order the outputs are moe_dispatch's.
 * Workspace: moe_dispatch_replicated_workspace_size bytes.  A routed expert
 *   with no copy, or a slot holding an id outside [0,E), is reported as
 *   MOE_ERR_INVALID_ARG in the status word.
 */
moe_status_t moe_dispatch_replicated_workspace_size(const moe_shape_t *shape,
                                                    int32_t num_physical, size_t *bytes);
moe_status_t moe_dispatch_replicated(const moe_shape_t *shape, int32_t num_physical,
                                     const int32_t *phys_expert, const int32_t *topk_ids,
                                     const void *x, int32_t *counts_phys, int32_t *offsets_phys,
                                     int32_t *src_token, int32_t *dest, void *x_perm, void *ws,
                                     size_t ws_bytes, moe_stream_t stream);

/*
 * Capacity variant ("第十五章：多节点大模型推理" section 4.3, "Capacity Factor"):
 * each expert takes at most C assignments per batch.
 *
 * moe_expert_capacity returns C = ceil(c * T * k / E) (evaluated in double;
 * the page's example T = 5600, k = 16, E = 896, c = 1.2 gives 120), or -1
 * for T < 0, k < 1, E < 1 or c not finite and >= 0.
 */
int32_t moe_expert_capacity(int32_t T, int32_t k, int32_t E, double c);

/*
 * Dispatch with capacity C >= 0.  Assignments a = t*k + j of each expert are
 * taken in increasing a; the first C keep a padded row e*C + r (r = rank at
 * the expert); later ones go, by `overflow`, to row
 * E*C + ovf_offsets[e] + (r - C) (MOE_OVERFLOW_SECOND_ROUND) or nowhere
 * (MOE_OVERFLOW_DROP: dest = -1).
 * Outputs (device, caller-owned): counts [E] = n_e, kept [E] = min(n_e, C),
 *   ovf_offsets [E+1] = exclusive prefix sum of n_e - kept[e],
 *   dest [T*k] int32, src_row [E*C + T*k] int32 (token of each used row;
 *   other entries are not written), x_rows [(E*C + T*k), d] bf16 (NULL to
 *   skip the gather; rows not used are not written).  The padded rows
 *   [0, E*C) form the masked layout of moe_expert_ffn with masked_m = kept,
 *   M_max = C; the overflow rows are contiguous with offsets ovf_offsets.
 * Workspace: as moe_dispatch.  E*C + T*k must be < 2^31.
 */
moe_status_t moe_dispatch_capacity(const moe_shape_t *shape, int32_t capacity,
                                   int32_t overflow, const int32_t *topk_ids, const void *x,
                                   int32_t *counts, int32_t *kept, int32_t *ovf_offsets,
                                   int32_t *dest, int32_t *src_row, void *x_rows, void *ws,
                                   size_t ws_bytes, moe_stream_t stream);

/* Workspace bytes for moe_layer_capacity with this shape and capacity. */
moe_status_t moe_layer_capacity_workspace_size(const moe_shape_t *shape, int32_t capacity,
                                               size_t *bytes);

/*
 * The layer with capacity C: route, capacity dispatch, the expert FFN over
 * the padded rows (masked layout, M_max = C), with MOE_OVERFLOW_SECOND_ROUND
 * a second expert FFN over the overflow rows, then the combine over the
 * assignments that have a row (dropped ones add nothing; weights are not
 * renormalised).  Where the expert GEMMs stream their weights (fewer than
 * 256 rows per expert on average) the two rounds run as one launch per GEMM,
 * each expert's padded rows then its overflow rows, so every weight is read
 * once.  Arguments as moe_layer; kept [E] (optional) receives min(n_e, C).
 * With the second round the output is the uncapped layer's.
 */
moe_status_t moe_layer_capacity(const moe_shape_t *shape, int32_t capacity, int32_t overflow,
                                const void *x, const void *w_r, const float *bias,
                                const void *w_gate_up, const void *w_down, void *y,
                                int32_t *counts, int32_t *kept, void *ws, size_t ws_bytes,
                                moe_stream_t stream);

/*
 * FP8 quantization (e4m3 with fp32 block scales; the "ep-deploy" page's
 * cost model dispatches FP8 with scales, 7168 + 224 bytes per token, and
 * "推理INFRA方法论-02-parallelism" measures the FP8 grouped expert GEMM):
 *   s = 2^e, e the smallest integer >= -127 with amax <= 448 * 2^e for
 *   the block's largest magnitude amax (1 when the block is all zeros, 2^127
 *   when amax is not finite): a power of two, which the FP8 GEMM hands to the
 *   tensor cores as an 8-bit exponent;
 *   q = e4m3(x / s) (exact division), round to nearest even, saturating at
 *   448.
 * moe_quantize_fp8_rows: x [rows, cols] bf16 -> q [rows, cols] e4m3 codes,
 *   scales [rows, cols/128] fp32 (one per row and 128 columns).
 * moe_quantize_fp8_blocks: w [mats, rows, cols] bf16 -> q [mats, rows, cols],
 *   scales [mats, rows/128, cols/128] (one per 128 x 128 block).
 * rows (blocks: rows too) and cols must be multiples of 128 (rows of the
 * row form: any); all pointers device, 16-byte aligned.
 */
moe_status_t moe_quantize_fp8_rows(const void *x, int64_t rows, int32_t cols, void *q,
                                   float *scales, moe_stream_t stream);
moe_status_t moe_quantize_fp8_blocks(const void *w, int32_t mats, int32_t rows, int32_t cols,
                                     void *q, float *scales, moe_stream_t stream);

/*
 * FP8 expert FFN: moe_expert_ffn with e4m3 operands and block scales.
 *   x_q [rows, d] e4m3 codes, x_scale [rows, d/128] fp32 (per row and 128
 *   columns, as moe_quantize_fp8_rows); w_gate_up_q [E, 2*inter, d] and
 *   w_down_q [E, d, inter] e4m3 codes with w_*_scale [E, rows/128, cols/128]
 *   fp32 (per 128 x 128 block, as moe_quantize_fp8_blocks); seg, M_max and
 *   the layouts as moe_expert_ffn; y_out [rows, d] fp32.
 *   The tensor cores apply both scales of each 128-column k-block
 *   themselves (block-scaled MMAs, the scales as 8-bit exponents) and
 *   accumulate in fp32; h = silu(g) * u is rounded to bf16 and quantized per
 *   row and 128 columns (in the gate_up epilogue where the tiles allow), and
 *   multiplied by w_down the same way.  Every scale
 *   must be a power of two in [2^-127, 2^127], as the quantizers above make
 *   them; any other value sets MOE_ERR_INVALID_ARG in the device status
 *   (and the affected outputs are undefined).
 *   d and inter must be multiples of 128 (MOE_ERR_UNSUPPORTED otherwise).
 */
moe_status_t moe_expert_ffn_fp8_workspace_size(const moe_shape_t *shape, int32_t layout,
                                               int32_t M_max, size_t *bytes);
moe_status_t moe_expert_ffn_fp8(const moe_shape_t *shape, int32_t layout, const void *x_q,
                                const float *x_scale, const int32_t *seg, int32_t M_max,
                                const void *w_gate_up_q, const float *w_gate_up_scale,
                                const void *w_down_q, const float *w_down_scale, float *y_out,
                                void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * The layer with FP8 experts: route (from bf16 x, as moe_layer), quantize x
 * per row and 128 columns, dispatch the FP8 rows with their scales (the
 * "ep-deploy" page's FP8 dispatch: d + 4*d/128 bytes per row), the FP8
 * expert FFN, and the combine (fp32 sums, from the compact rows where d is
 * a multiple of 256, as moe_layer).  Weights as
 * moe_expert_ffn_fp8; y [T,d] bf16; counts [E] optional.
 */
moe_status_t moe_layer_fp8_workspace_size(const moe_shape_t *shape, size_t *bytes);
moe_status_t moe_layer_fp8(const moe_shape_t *shape, const void *x, const void *w_r,
                           const float *bias, const void *w_gate_up_q,
                           const float *w_gate_up_scale, const void *w_down_q,
                           const float *w_down_scale, void *y, int32_t *counts, void *ws,
                           size_t ws_bytes, moe_stream_t stream);

/*
 * Expert placement planner ("ep-deploy" handbook page, section "EPLB 与路由约束",
 * host code, no GPU): places num_experts logical experts, given their loads
 * (load [E] host doubles, >= 0), on num_gpus GPUs as num_physical physical
 * experts (num_physical - E redundant copies).
 *   num_nodes > 0 (hierarchical): the expert groups (E / num_groups
 *   consecutive experts) are packed onto the nodes by group load, the same
 *   number per node, so no group spans nodes; inside each node, copies are
 *   added one at a time to the expert with the largest load per copy (equal:
 *   the one first in the node's order) until the node has num_physical/nodes
 *   physical experts; these (weight load / copies) are packed onto the
 *   node's GPUs.  num_nodes = 0 (global): the cluster is one node.
 *   Packing: heaviest item first (equal: lower index), into the lightest
 *   pack with room (equal: lower pack index); every pack gets the same count.
 * Outputs (host, caller-owned): gpu_slots [num_physical], GPU g holding the
 *   logical experts gpu_slots[g * P/G .. (g+1) * P/G) (P = num_physical,
 *   G = num_gpus); replicas [E] copies per expert.
 * Errors: MOE_ERR_INVALID_ARG when E % num_groups, num_groups % nodes,
 *   num_gpus % nodes or num_physical % num_gpus is not zero, num_physical < E,
 *   or a load is negative or not finite.
 */
moe_status_t moe_eplb_plan(const double *load, int32_t num_experts, int32_t num_groups,
                           int32_t num_nodes, int32_t num_gpus, int32_t num_physical,
                           int32_t *gpu_slots, int32_t *replicas);

/*
 * Number of kernels moe_layer launches per call for this shape (for launch
 * accounting).
 */
int32_t moe_layer_launch_count(const moe_shape_t *shape);

/*
 * Bytes of one routed row of moe_layer's down-GEMM output as the combine
 * reads it: 4*d (fp32 rows) or 2*d + d/32 (the compact rows); 0 for an
 * invalid shape.  For byte accounting.
 */
int64_t moe_layer_yperm_row_bytes(const moe_shape_t *shape);

/*
 * (token, expert) pairs whose fixed-order logit the last screened routing in
 * `ws` (moe_route without logits, moe_layer, moe_layer_capacity,
 * moe_layer_fp8 of this shape) computed -- at least T*k, since every
 * selected expert is refined: copies one int32 to device memory `count` on
 * `stream` (asynchronous); -1 when the shape is not screened.
 */
moe_status_t moe_route_refined_count(const moe_shape_t *shape, const void *ws, size_t ws_bytes,
                                     int32_t *count, moe_stream_t stream);

/*
 * A prepared copy of a router weight for the screened path, so that screened
 * calls skip making it (about 3.7 MB read and written, two launches, at
 * d = 7168, E = 256).
 *   moe_router_prep_size: bytes of the copy for this shape (E*d*2 rounded up
 *     to 256, plus E*4 rounded up to 256; depends on d and E only);
 *     MOE_ERR_UNSUPPORTED when the shape is not screened.
 *   moe_router_prepare: writes the copy of w_r [d,E] (transposed to [E,d],
 *     then the norm of every expert's weight column) into `prep`, device
 *     memory the caller owns (256-byte aligned, prep_bytes >= the size),
 *     asynchronously on `stream`, and records `prep` for the pointer w_r.
 *     Every later screened call (moe_route without logits, moe_layer,
 *     moe_layer_capacity, moe_layer_fp8) whose w_r is this pointer and whose
 *     d and E match reads the copy instead of making one.  Up to 64 weights
 *     can be recorded (MOE_ERR_UNSUPPORTED beyond).  Preparing the same w_r
 *     again replaces its record.
 *   moe_router_release: drops the record of w_r (no-op if none).
 * The record follows the pointer, not the contents: call moe_router_prepare
 * again after changing the weight in place, and moe_router_release before
 * freeing the weight or `prep` (an allocator may hand the same address to
 * another tensor).  `prep` must stay valid while recorded.
 */
moe_status_t moe_router_prep_size(const moe_shape_t *shape, size_t *bytes);
moe_status_t moe_router_prepare(const moe_shape_t *shape, const void *w_r, void *prep,
                                size_t prep_bytes, moe_stream_t stream);
moe_status_t moe_router_release(const void *w_r);

/*
 * Self-test of the bounded wait used by every device-side spin: launches one
 * CTA that waits on a barrier nobody completes, gives up after `limit_ns`
 * nanoseconds and records MOE_ERR_TIMEOUT in the workspace status word.
 */
moe_status_t moe_selftest_wait_timeout(void *ws, size_t ws_bytes, uint64_t limit_ns,
                                       moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
