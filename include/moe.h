/*
 * moe.h -- C ABI of the group-limited MoE layer forward on GB300 (sm_103a).
 *
 * The layer is the one described in the article
 *   "InternLumina-U2中256个专家的路由秘密：分组受限Top-K、Expert Bias与Fused MoE详解"
 * (called "the routing page" below):
 *   - an fp32 linear router followed by an element-wise sigmoid (section 二, step 1);
 *   - group-limited top-k: the experts are cut in order into n_group groups, a
 *     group scores the sum of its two best scores, the topk_group best groups
 *     survive and the top k of their experts are chosen (section 二, step 2);
 *   - expert_bias is added to the scores for choosing only (section 三);
 *   - the weights are the chosen unbiased scores over (their sum + eps), times
 *     routed_scaling_factor (section 二, step 3);
 *   - every chosen expert is a SwiGLU FFN whose gate, up and down weights are
 *     stacked per expert (section 四); one shared expert is always added
 *     (section 五); expert hit counts are kept (section 六).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; all
 *     tensors are dense, row-major, with no padding between rows.
 *   - bf16 tensors are passed as their 16-bit patterns (moe_bf16).
 *   - The caller owns every buffer, including the workspace.  The library
 *     never allocates or frees device memory and never synchronises the stream
 *     (moe_get_status excepted).  Work is enqueued on `stream`, a cudaStream_t
 *     passed as void* (NULL = the legacy default stream); outputs are ready
 *     when that stream reaches the point of the call.
 *   - Every entry point validates its arguments first and returns a negative
 *     MOE_ERR_* code without launching anything when they are wrong.  It never
 *     truncates or clamps silently.  MOE_ERR_CUDA means a launch failed; the
 *     CUDA error is left for the caller to read with cudaGetLastError().
 *   - Faults found on the device (non-finite logits, an expert index out of
 *     range, a wait that ran out) never trap: the kernel records a bit in the
 *     workspace's status word, skips the offending item, and returns.  Read
 *     and clear the word with moe_get_status().
 *   - Workspaces are 256-byte aligned blocks of moe_workspace_bytes() bytes.
 *     Call moe_workspace_init() once after allocating one.  Two calls that use
 *     the same workspace must not run concurrently.
 *   - Pointers handed to the tensor-core kernels must be 16-byte aligned
 *     (MOE_ERR_MISALIGNED otherwise).
 *
 * Supported shapes (MOE_ERR_UNSUPPORTED_SHAPE otherwise): E == 32 * n_group
 * with 1 <= n_group <= 8 (one expert per lane per group in the routing warp),
 * 1 <= topk_group <= n_group, 1 <= k <= min(32, 32 * topk_group), E % 128 == 0
 * for the router GEMM, H % 256 == 0, I % 128 == 0, Is == I, 1 <= T <= 2^24.
 */
#ifndef GLR_MOE_H
#define GLR_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* bf16 bit pattern */

/* Layer configuration (routing page, section 一, hyper-parameter table):
 * T tokens, hidden size H, E routed experts in n_group groups of which
 * topk_group survive, k experts per token, expert FFN inner size I, shared
 * expert inner size Is, routed_scaling_factor rsf (2.5) and the normaliser's
 * eps (1e-20, section 二 step 3). */
typedef struct moe_cfg {
    int32_t T, H, E, n_group, topk_group, k, I, Is;
    float rsf, eps;
} moe_cfg;

/* return codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)
#define MOE_ERR_UNSUPPORTED_SHAPE (-2)
#define MOE_ERR_MISALIGNED (-3)
#define MOE_ERR_WORKSPACE_TOO_SMALL (-4)
#define MOE_ERR_CUDA (-5)
#define MOE_ERR_DEVICE_STATUS (-6)
#define MOE_ERR_TIMEOUT (-7)
#define MOE_ERR_UNSUPPORTED_DEVICE (-8)

/* bits of the device status word */
#define MOE_STATUS_NONFINITE_LOGIT 1   /* a logit, score or bias was NaN/inf     */
#define MOE_STATUS_BAD_EXPERT_INDEX 2  /* topk_idx held an id outside [0, E)     */
#define MOE_STATUS_TIMEOUT 4           /* a bounded device wait ran out          */
#define MOE_STATUS_COUNT_MISMATCH 8    /* bucketed rows != k*T (follows from 2)  */

/* workspace kinds */
#define MOE_WS_ROUTE 0
#define MOE_WS_FORWARD 1
#define MOE_WS_BACKWARD 2

/* Bytes of workspace that moe_route (which = MOE_WS_ROUTE) or moe_forward
 * (which = MOE_WS_FORWARD) needs for this configuration; 0 if the
 * configuration is invalid or unsupported.  Host only, no CUDA call. */
size_t moe_workspace_bytes(const moe_cfg *cfg, int which);

/* Clears the status word and the bookkeeping header of a freshly allocated
 * workspace (an asynchronous memset on `stream`). */
int moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Router of the routing page, section 二 steps 1-3 and section 三, for T tokens.
 *   hidden       [T, H] bf16
 *   W_router     [E, H] fp32 (the router is computed to fp32 accuracy: the
 *                weight is split into three bf16 parts whose products with
 *                the bf16 hidden state are exact, accumulated in fp32)
 *   expert_bias  [E] fp32, or NULL for zero; used for choosing only
 *   topk_idx     [T, k] int32 out: chosen experts in order of (biased score
 *                desc, index asc); ties go to the lower index
 *   topk_w       [T, k] fp32 out: s / (sum of the k chosen s + eps) * rsf,
 *                s the unbiased sigmoid scores
 *   expert_counts[E] int32 out: hits per expert over the T tokens (section 六)
 *   aux_P        [E] fp32 out or NULL: mean over tokens of each expert's
 *                score divided by the token's score sum
 *   aux_loss     [1] fp32 out or NULL: E * sum_i (counts_i / (k T)) * P_i,
 *                the load-balancing loss of the pitfalls page ("MoE 负载均衡
 *                Loss 别忘加" of the InternLumina-U2 training-pitfalls article)
 *   ws           workspace of moe_workspace_bytes(cfg, MOE_WS_ROUTE) bytes
 * Deterministic: the same inputs give bit-identical outputs. */
int moe_route(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router,
              const float *expert_bias, int32_t *topk_idx, float *topk_w,
              int32_t *expert_counts, float *aux_P, float *aux_loss,
              void *ws, size_t ws_bytes, void *stream);

/* One-time preparation of the router weight for moe_route_prepared: writes
 * its exact bf16 x 3 split, W_split [3, E, H] bf16 (hi, mid, lo with
 * hi + mid + lo == W_router for every normal fp32 value), on `stream`.
 * W_router [E, H] fp32 (4-byte aligned), W_split 16-byte aligned, owned by
 * the caller.  The routing page computes the router in fp32 (section 二 step
 * 1); this is how the tensor-core path stays fp32-exact.  The split has no
 * counterpart on the page: it moves the per-call split of moe_route out of the
 * step. */
int moe_prepare_router(const moe_cfg *cfg, const float *W_router, moe_bf16 *W_split, void *stream);

/* moe_route with the weight prepared by moe_prepare_router: same outputs,
 * bit for bit, as moe_route(cfg, hidden, W_router, ...).  W_router is still
 * read for small T (<= 32 tokens run on the CUDA cores with the fp32 weight);
 * W_split must hold moe_prepare_router(W_router) (a stale split gives the
 * logits of the weight it was made from).  expert_counts is cleared with an
 * asynchronous memset on `stream`. */
int moe_route_prepared(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router,
                       const moe_bf16 *W_split, const float *expert_bias, int32_t *topk_idx,
                       float *topk_w, int32_t *expert_counts, float *aux_P, float *aux_loss,
                       void *ws, size_t ws_bytes, void *stream);

/* The first half of moe_route alone: logits [T, E] fp32 = hidden . W_router^T
 * (routing page, section 二 step 1).  Same arguments and workspace. */
int moe_router_logits(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router,
                      float *logits, void *ws, size_t ws_bytes, void *stream);

/* The second half of moe_route alone: selection, weights, counts and the
 * balance loss from given fp32 logits [T, E] (routing page, section 二 steps
 * 1-3, section 三).  Same outputs and workspace as moe_route; non-finite
 * logits set MOE_STATUS_NONFINITE_LOGIT. */
int moe_route_from_logits(const moe_cfg *cfg, const float *logits, const float *expert_bias,
                          int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                          float *aux_P, float *aux_loss, void *ws, size_t ws_bytes, void *stream);

/* The sigmoid scores the selecting kernels rank (routing page, section 二
 * step 1): scores[i] = 1 / (1 + exp(-logits[i])) in fp32, computed with the
 * very device function those kernels use (an fp32 exponential, then an
 * IEEE round-to-nearest reciprocal of 1 + exp(-L); not correctly rounded as
 * a whole).  For measuring that function against an exact sigmoid.
 * logits, scores: n fp32 values on the device, 4-byte aligned (may alias). */
int moe_router_scores(const float *logits, float *scores, int64_t n, void *stream);

/* Expert stage of the routing page, sections 四 and 五:
 *   out[t] = bf16( sum_j topk_w[t,j] * FFN_{topk_idx[t,j]}(hidden[t])
 *                  + FFN_shared(hidden[t]) (+ residual[t]) )
 * with FFN(x) = down( silu(gate x) * up x ), silu(z) = z / (1 + exp(-z)); the
 * products run on tensor cores with bf16 operands and fp32 accumulation; the
 * SwiGLU intermediate and each expert's output row are stored as bf16; the
 * weighted sum is fp32 and rounded once.
 *   hidden          [T, H] bf16
 *   W_gate_up       [E, 2I, H] bf16: per expert, rows [0, I) are gate_proj and
 *                   rows [I, 2I) are up_proj (each [I, H], the page's
 *                   [256, 512, 2048] stacks)
 *   W_down          [E, I, H] bf16: down_proj as the page stacks it,
 *                   expert output = intermediate[1, I] @ W_down[e]
 *   shared_gate_up  [2Is, H] bf16, same layout as one expert of W_gate_up
 *   shared_down     [Is, H] bf16
 *   topk_idx        [T, k] int32 (any order; an id outside [0, E) is skipped
 *                   and sets MOE_STATUS_BAD_EXPERT_INDEX)
 *   topk_w          [T, k] fp32
 *   residual        [T, H] bf16 or NULL: added before the final rounding
 *                   (a decoder layer's residual connection)
 *   out             [T, H] bf16 out (may alias residual, not hidden)
 *   ws              workspace of moe_workspace_bytes(cfg, MOE_WS_FORWARD) bytes
 * Tokens are bucketed by expert in a stable order (the "sort tokens into
 * buckets" inference path of section 四), so outputs are deterministic. */
int moe_forward(const moe_cfg *cfg, const moe_bf16 *hidden, const moe_bf16 *W_gate_up,
                const moe_bf16 *W_down, const moe_bf16 *shared_gate_up, const moe_bf16 *shared_down,
                const int32_t *topk_idx, const float *topk_w, const moe_bf16 *residual,
                moe_bf16 *out, void *ws, size_t ws_bytes, void *stream);

/* The whole layer in one call: moe_route followed by moe_forward, on one
 * workspace of moe_layer_workspace_bytes(cfg, flags) bytes
 * (moe_workspace_init() once after allocating it).  Arguments as in those two
 * calls; W_split is moe_prepare_router's output or NULL (then the router
 * weight is split inside the call); topk_idx, topk_w, expert_counts and the
 * optional aux_P [E] / aux_loss [1] (the balance loss, as in moe_route; NULL
 * to skip) are outputs here.  flags = 0 gives the same outputs, bit for bit,
 * as the two calls; because one call owns both halves, its routing kernel
 * also writes the expert stage's bucketing histogram (per 16-token chunk,
 * hits per expert), so the expert stage skips that pass.
 *
 * flags = MOE_LAYER_FUSED_ROUTER (for E = 256 experts in n_group = 8 groups
 * with k <= 8, H <= 8192; other shapes ignore it): the router's tensor-core
 * kernel also does the rest of routing and the bucketing of section 四.
 * After its own token tiles, each CTA takes finished tiles from a queue,
 * selects their tokens' experts (the same arithmetic and tie rules as
 * moe_route, so the outputs are identical bit for bit), claims each pair's
 * row in its expert's bucket with one integer atomic per expert and tile, and
 * bulk-copies the hidden rows there.  Bucket e then starts at row e T of a
 * larger activation matrix in the workspace (E T rows of H bf16: 34 GB at
 * T = 32768, H = 2048), and the order of rows inside a bucket depends on
 * scheduling; no row's result does, and the combine adds every token's rows in
 * a fixed order, so out is deterministic and equal to the unfused path's.
 * On a GB300 this path measures slower than the unfused kernels (its
 * selection runs on 8 warps per SM and its row copies follow the
 * multiplications), so it is not the default.  It forms no balance loss:
 * aux_P / aux_loss must be NULL with it.
 *
 * flags = MOE_LAYER_FUSED_COMBINE (where the down GEMM runs on CTA pairs:
 * T >= 24576, k <= 8, without MOE_LAYER_FUSED_ROUTER; ignored otherwise):
 * the shared expert's down projection runs after the routed experts' and
 * forms the combine of section 五 in its epilogue (the routing page, section
 * 四's "fused" MoE), so the shared rows never go through memory and the
 * combine is not a launch of its own.  The sum is the combine's, term for
 * term, so out is identical bit for bit to flags = 0.  On a GB300 it measures
 * slower (the GEMM's epilogue warps keep fewer row loads in flight than the
 * combine kernel), so it is not the default.  Unknown flags return
 * MOE_ERR_INVALID_ARG. */
#define MOE_LAYER_FUSED_ROUTER 1
#define MOE_LAYER_FUSED_COMBINE 2
size_t moe_layer_workspace_bytes(const moe_cfg *cfg, int flags);
int moe_layer(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router, const moe_bf16 *W_split,
              const float *expert_bias, const moe_bf16 *W_gate_up, const moe_bf16 *W_down,
              const moe_bf16 *shared_gate_up, const moe_bf16 *shared_down, const moe_bf16 *residual,
              int32_t *topk_idx, float *topk_w, int32_t *expert_counts, float *aux_P, float *aux_loss,
              moe_bf16 *out, int flags, void *ws, size_t ws_bytes, void *stream);

/* Backward of moe_forward for fixed routing (the training step of the layer;
 * the routing page trains the layer but prints no backward: these are the
 * gradients of the forward above, the bf16 rounding of the intermediate
 * passed through as the identity).  Given d_out [T, H] bf16 = dL/d out:
 *   d_hidden        [T, H] bf16 out: dL/d hidden through the experts and the
 *                   shared expert (the residual's own identity path is not
 *                   added; the router's contribution is not included)
 *   dW_gate_up      [E, 2I, H] fp32 out, dW_down [E, I, H] fp32 out,
 *   d_shared_gate_up [2I, H] fp32 out, d_shared_down [I, H] fp32 out: the
 *                   weight gradients summed over the T tokens (overwritten)
 *   d_topk_w        [T, k] fp32 out: <d_out[t], expert_{topk_idx[t,j]}(hidden[t])>
 * Other arguments as moe_forward; I % 256 == 0; workspace of
 * moe_workspace_bytes(cfg, MOE_WS_BACKWARD) bytes.  Deterministic. */
int moe_backward(const moe_cfg *cfg, const moe_bf16 *hidden, const moe_bf16 *W_gate_up,
                 const moe_bf16 *W_down, const moe_bf16 *shared_gate_up, const moe_bf16 *shared_down,
                 const int32_t *topk_idx, const float *topk_w, const moe_bf16 *d_out,
                 moe_bf16 *d_hidden, float *dW_gate_up, float *dW_down, float *d_shared_gate_up,
                 float *d_shared_down, float *d_topk_w, void *ws, size_t ws_bytes, void *stream);

/* Dense SwiGLU MLP: the first decoder layer of the model on the routing page
 * ("first_k_dense_replace = 1", section 五: layer 0 is an ordinary MLP, the
 * 19 layers after it are MoE).  The page gives the layer neither a formula
 * nor a size; this takes the experts' form with its own intermediate size I:
 *   out[t] = bf16( down( silu(gate x[t]) * up x[t] ) (+ residual[t]) )
 * run on the grouped tensor-core GEMMs with a single weight group.
 *   hidden     [T, H] bf16, H % 256 == 0
 *   W_gate_up  [2I, H] bf16: rows [0, I) gate, [I, 2I) up; I % 128 == 0
 *   W_down     [I, H] bf16: out = a[1, I] @ W_down
 *   residual   [T, H] bf16 or NULL; out [T, H] bf16 (may alias residual)
 *   ws         workspace of moe_dense_workspace_bytes(T, H, I) bytes
 *              (moe_workspace_init() once after allocating it) */
size_t moe_dense_workspace_bytes(int32_t T, int32_t H, int32_t I);
int moe_dense_ffn(int32_t T, int32_t H, int32_t I, const moe_bf16 *hidden, const moe_bf16 *W_gate_up,
                  const moe_bf16 *W_down, const moe_bf16 *residual, moe_bf16 *out, void *ws,
                  size_t ws_bytes, void *stream);

/* ---- Expert parallelism -------------------------------------------------
 * The InternLumina-U2 training-pitfalls article, section "专家并行（EP）怎么
 * 切": the stacked expert weights are sharded along their first (expert)
 * dimension over R ranks, rank r holding experts [r E/R, (r + 1) E/R) of
 * W_gate_up and W_down; the router, the bias and the shared expert are
 * replicated.  A rank's forward then runs, with two all-to-all exchanges of
 * rows between the ranks (done by the caller, e.g. torch.distributed):
 *   moe_route                      its own tokens' routing;
 *   moe_ep_dispatch                the rows to send, grouped by destination;
 *   (all-to-all: counts, rows, expert ids)
 *   moe_expert_rows                the received rows through the local experts;
 *   (all-to-all back, into the first k T rows of a [k T + T, H] buffer)
 *   moe_dense_ffn                  the shared expert into that buffer's last T rows;
 *   moe_combine                    the weighted sum, as moe_forward's.
 * Each row's expert output does not depend on where the row is computed and
 * the combine adds in moe_forward's order, so the result equals moe_forward's
 * bit for bit. */

/* Groups the (token, j) pairs by the rank that holds their expert
 * (topk_idx / (E / ranks)), stably (ascending (token, j) within a rank):
 *   send_counts [ranks]   rows for each destination rank;
 *   x_send [k T, H] bf16  the hidden row of every pair, in that order (rank
 *                         0's rows first);
 *   e_send [k T] int32    the pair's expert as an id local to its rank;
 *   slot_of [T, k] int32  the row of pair (t, j) in x_send (its results come
 *                         back to the same row), -1 for an expert id outside
 *                         [0, E) (flagged in the workspace's status word).
 * Needs E % ranks == 0, ranks <= 256, H % 8 == 0; the workspace is
 * moe_ep_dispatch_workspace_bytes(cfg, ranks) bytes (moe_workspace_init()
 * once).  Device pointers, asynchronous on `stream`. */
size_t moe_ep_dispatch_workspace_bytes(const moe_cfg *cfg, int32_t ranks);
int moe_ep_dispatch(const moe_cfg *cfg, int32_t ranks, const moe_bf16 *hidden, const int32_t *topk_idx,
                    int32_t *send_counts, moe_bf16 *x_send, int32_t *e_send, int32_t *slot_of, void *ws,
                    size_t ws_bytes, void *stream);

/* The expert stage for a set of rows that each name their expert:
 *   y[i] = bf16( down_e( silu(gate_e x[i]) * up_e x[i] ) ),  e = expert[i],
 * unweighted, with the weights of E = cfg->E local experts (W_gate_up
 * [E, 2I, H], W_down [E, I, H], as moe_forward's; cfg->H and cfg->I as
 * there; cfg->T, k and the shared expert are not used).  The rows are
 * bucketed by expert and run through the same grouped tensor-core GEMMs as
 * moe_forward's, so y[i] equals moe_forward's row for the same pair bit for
 * bit.  rows may be 0 (nothing launched); an expert id outside [0, E) gives a
 * zero row and sets the status word.  The workspace is
 * moe_expert_rows_workspace_bytes(cfg, rows) bytes (moe_workspace_init()
 * once; a workspace sized for more rows serves fewer). */
size_t moe_expert_rows_workspace_bytes(const moe_cfg *cfg, int32_t rows);
int moe_expert_rows(const moe_cfg *cfg, int32_t rows, const moe_bf16 *x, const int32_t *expert,
                    const moe_bf16 *W_gate_up, const moe_bf16 *W_down, moe_bf16 *y, void *ws, size_t ws_bytes,
                    void *stream);

/* moe_forward's last step on rows computed elsewhere (routing page, section
 * 五: the shared expert added directly):
 *   out[t] = bf16( sum_j topk_w[t,j] Y[slot_of[t,j]] + Y[shared_row0 + t]
 *                  (+ residual[t]) ),
 * in fp32, j in order, then the shared row, then the residual.  Y [y_rows, H]
 * bf16; slot_of [T, k] (-1 or a row at or past y_rows: the pair is skipped);
 * topk_w [T, k] fp32; residual [T, H] or NULL; out [T, H] (may alias
 * residual).  Needs shared_row0 + T <= y_rows, H % 8 == 0. */
int moe_combine(const moe_cfg *cfg, const moe_bf16 *Y, int64_t y_rows, int64_t shared_row0, const int32_t *slot_of,
                const float *topk_w, const moe_bf16 *residual, moe_bf16 *out, void *stream);

/* Router without caller-provided scratch (no counterpart on the pages: it is
 * an interface convenience, not part of the method).  Same computation,
 * outputs and determinism as moe_route, but the scratch that moe_route keeps
 * in its workspace (the split router weight, the logits, the balance-loss
 * partials) lives in one array inside this library, so the caller supplies
 * only inputs and outputs.  It is meant for callers that cannot allocate
 * device memory on the call path: plug-in hosts whose operator interface
 * hands over input and output tensors but no allocator, runtimes that own
 * every byte of device memory and give none to their plug-ins, and
 * latency-sensitive loops where a cudaMalloc would synchronise the device.
 * This entry point itself never calls cudaMalloc, cudaFree or any allocating
 * library routine.
 *
 * The array is a static __device__ buffer of MOE_ROUTE_STATIC_SCRATCH_BYTES
 * (40 MiB), held on every GPU that loads the library until the process exits.
 * That covers T up to 32768 tokens at E = 256, H = 2048 (more for smaller E
 * or H); larger configurations are rejected with MOE_ERR_UNSUPPORTED_SHAPE
 * before anything is launched.  The array has its own address in every CUDA
 * context; the first call in a context (per device, and again after a device
 * reset or in a context the host created itself) looks that address up with
 * the context current, so make that first call before any stream capture.
 * Every call on a device shares the one array: calls whose work overlaps on
 * the GPU (other streams, other threads) race and must be serialised by the
 * caller.  Each call clears the status word it uses; status_out (a DEVICE
 * pointer, or NULL) receives that call's MOE_STATUS_* bits in stream order,
 * and is written only when the call returns MOE_OK (on an error return it
 * keeps whatever it held). */
#define MOE_ROUTE_STATIC_SCRATCH_BYTES (40u << 20)
int moe_route_static(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router,
                     const float *expert_bias, int32_t *topk_idx, float *topk_w,
                     int32_t *expert_counts, float *aux_P, float *aux_loss,
                     int32_t *status_out, void *stream);

/* Training-side feedback after a routing step (routing page, section 三: the
 * bias of cold experts is raised and that of overloaded experts lowered so
 * that tokens drift to idle experts; section 六: per-expert hit totals are
 * kept).  The page gives no formula; this is a sign step around the balanced
 * load k T / E:
 *   expert_bias[e] += gamma  if expert_counts[e] < k T / E,
 *                     -gamma if expert_counts[e] > k T / E, unchanged if equal;
 *   totals[e]      += expert_counts[e].
 * expert_counts [E] int32 (moe_route's output), expert_bias [E] fp32 or NULL,
 * totals [E] int64 or NULL (device pointers, updated in place on `stream`). */
int moe_expert_feedback(const moe_cfg *cfg, const int32_t *expert_counts, float gamma, float *expert_bias,
                        int64_t *totals, void *stream);

/* Decoder-layer pre-norm for stacking MoE layers (the routing page, §五,
 * builds its MoE blocks into decoder layers but does not describe their norm):
 *   out[t] = bf16( x[t] / sqrt(mean_h x[t,h]^2 + eps) )  (unit weight, fp32)
 * x, out [T, H] bf16 (may alias), H % 8 == 0, 16-byte aligned. */
int moe_rmsnorm(int32_t T, int32_t H, const moe_bf16 *x, moe_bf16 *out, float eps, void *stream);

/* Waits for `stream`, then copies the workspace's status word (MOE_STATUS_*
 * bits, OR-ed over every call since the last reset) to *status (a HOST
 * pointer); clears it when reset != 0.  Returns MOE_OK, or MOE_ERR_CUDA. */
int moe_get_status(void *ws, size_t ws_bytes, void *stream, int32_t *status, int reset);

/* Number of kernels the last successful moe_route / moe_route_prepared /
 * moe_prepare_router / moe_forward / moe_layer / moe_route_from_logits /
 * moe_router_logits call on this thread enqueued (memsets not counted). */
int moe_last_launch_count(void);

/* Kernel timing.  moe_profile_enable(1): every kernel the library launches
 * is bracketed by two CUDA events recorded on its stream (a few microseconds
 * of overhead per launch, no synchronisation; the events also keep a kernel
 * from starting before the previous one has ended).  moe_profile_enable(2):
 * per stage -- the routing and bucketing kernels of a call (router GEMM,
 * selection, balance-loss reduction, histogram, scan, scatter) are timed as
 * one interval, kernel id MOE_KERNEL_STAGE_ROUTE_PERMUTE, and every other
 * kernel on its own; events are recorded only where the stage changes.
 * moe_profile_enable(0) stops.  moe_profile_read() waits for the recorded
 * events, folds them into per-kernel totals and returns the total
 * milliseconds and interval count of `kernel_id` (0 <= kernel_id <
 * MOE_KERNEL_COUNT), clearing them when reset != 0. */
#define MOE_KERNEL_COUNT 19
#define MOE_KERNEL_STAGE_ROUTE_PERMUTE 18
int moe_profile_enable(int on);
int moe_profile_read(int kernel_id, double *total_ms, int32_t *launches, int reset);
const char *moe_kernel_name(int kernel_id);

/* Fault injection for tests of the failure path (no counterpart on the pages).
 * The next `launches` grouped gate/up GEMM launches made by moe_forward, in
 * this process, run with their TMA producer withholding every load and a
 * 50 ms wait limit: the MMA lane's first wait runs out, the kernel winds down
 * (copies drained, TMEM freed) and sets MOE_STATUS_TIMEOUT; the call's output
 * is then meaningless, but the CUDA context stays usable.  0 cancels. */
int moe_debug_inject_timeout(int launches);

/* Static description of a return code. */
const char *moe_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* GLR_MOE_H */
