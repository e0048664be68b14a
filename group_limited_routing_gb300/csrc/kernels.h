// Internal interface between the C-ABI layer (api.cu) and the kernels.
// Not installed; the public contract is include/moe.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace glr {

// ---- programmatic dependent launch ------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation and starts with pdl_wait(), which returns once the kernel
// before it in the stream has completed and its writes are visible -- before
// any global memory is touched.  No kernel triggers its dependents early, so
// the next kernel is launched when this one finishes, but its launch
// processing and (for the GEMMs) its prologue overlap this one's teardown.
// (Triggering at the start of each CTA was measured slower: the dependents'
// waiting CTAs then sit beside the running ones.)  Since every kernel waits,
// completion stays ordered along the whole stream.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- routing arithmetic shared by every kernel that selects experts ---------
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Sigmoid score of a router logit (routing page, section 二 step 1),
// s = 1 / (1 + exp(-L)), in a dozen fp32 instructions without branches, and
// the same bits in every selecting kernel.  exp(-L) = 2^(-L log2 e): the
// product with log2 e (split into its fp32 value and the remainder) is formed
// as a rounded part a plus its residual r, the residual found with one FMA
// (the FMA form of the error-free product, Ogita, Rump and Oishi 2005); the
// hardware's 2^a is then scaled by 2^r ~ 1 + r ln 2, and 1 / (1 + e) is the
// hardware reciprocal refined by one Newton-Raphson step.  L is clamped at
// -87 so that 1 + e stays finite (the clamp moves s by less than 2e-38).  Not
// correctly rounded: the test suite measures its distance from an exact
// sigmoid.
__device__ __forceinline__ float router_sigmoid(float L)
{
    constexpr float LOG2E_HI = 1.44269502162933349609375f;   // log2(e) rounded to fp32
    constexpr float LOG2E_LO = 1.925963033500011e-08f;       // log2(e) - LOG2E_HI
    constexpr float LN2 = 0.693147180559945309f;
    const float x = fmaxf(L, -87.0f);
    const float a = -x * LOG2E_HI;
    float r = fmaf(-x, LOG2E_HI, -a);                         // (-x) LOG2E_HI - a, exactly
    r = fmaf(-x, LOG2E_LO, r);
    float e = ex2_approx(a);
    e = fmaf(e, r * LN2, e);
    const float d = 1.0f + e;
    const float y = rcp_approx(d);
    return fmaf(y, fmaf(-d, y, 1.0f), y);
}

// Order-preserving map of fp32 onto uint32 (for non-NaN values): a > b as
// floats exactly when key(a) > key(b), so a float maximum is an integer one.
// +0 and -0 get neighbouring keys; the scores compared (sigmoid + bias, and
// sums of two of them) are never -0.
__device__ __forceinline__ uint32_t fkey(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float fkey_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ---- sizes shared by the host layer and the kernels -------------------------
constexpr int ROUTE_CHUNK = 32;    // tokens per block of the routing kernel (4 per warp) ...
constexpr int ROUTE_CHUNK_SMALL = 8;  // ... and for T <= ROUTE_SMALL_T (1 per warp, 4x the blocks)
constexpr int ROUTE_SMALL_T = 8192;
inline int route_chunk(int T) { return T <= ROUTE_SMALL_T ? ROUTE_CHUNK_SMALL : ROUTE_CHUNK; }
constexpr int PERM_CHUNK = 16;     // tokens per block of the bucketing kernels
constexpr int GEMM_BM = 128;       // tensor-core tile rows (tokens)
constexpr int GEMM_BK = 64;        // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int MAX_GROUPS = 8;      // routing warp: one expert per lane per group

// status bits (mirror include/moe.h)
constexpr int ST_NONFINITE = 1;
constexpr int ST_BAD_INDEX = 2;
constexpr int ST_TIMEOUT = 4;
constexpr int ST_COUNT_MISMATCH = 8;

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
    int status;      // OR of ST_* bits
    int num_mtiles;  // m-tiles of the grouped GEMMs (written on the device)
    int tile_ctr[2]; // claim counters of the two weight-gradient launches (zeroed on the device)
    int fin_ticket;  // blocks of the balance-loss reduction done (back to zero at its end)
    int num_ptiles;  // 256-row pair tiles of the CTA-pair grouped GEMM (written on the device)
    int num_ptiles_routed;  // the routed buckets' pair tiles among them (they come first)
    int pad[57];
};

// The _SMALL kinds are the grouped GEMMs for T <= GEMM_SMALL_T (decode): every
// bucket then has at most T rows, so only GEMM_SMALL_T A rows are loaded per
// stage and the smem this frees goes to a deeper weight ring.
// Backward kinds: GK_GATE_UP_BWD recomputes the gate/up products (storing
// G, U and the weighted intermediate); GK_DGRAD_DOWN is d(intermediate) =
// dOut_perm . W_down^T with the SwiGLU backward in its epilogue; GK_WGRAD is
// a per-expert weight gradient (M = features, N = hidden, K = the expert's
// bucket rows, both operands MN-major).
// GK_ROUTER_PAIR is the 256-expert router on CTA pairs (tiles of 256 tokens,
// each CTA loading half of the weight parts; grid = 2 x the pairs).
// GK_DOWN_PAIR is the grouped down GEMM on CTA pairs: 256-row pair tiles of
// one bucket, each CTA loading its 128 A rows and half of the W_down columns.
// GK_DOWN_COMBINE is the shared expert's down GEMM with the combine in its
// epilogue: per 128-token tile and 256 hidden columns, the shared rows'
// output plus the weighted sum of each token's routed rows, written to the
// layer output.
// GK_ROUTER_FUSED is the 256-expert router whose epilogue also selects the
// experts, claims every pair's row in its expert's bucket and copies the
// hidden rows there (routing and bucketing in one launch).
enum GemmKind {
    GK_ROUTER = 0, GK_GATE_UP = 1, GK_DOWN = 2, GK_GATE_UP_SMALL = 3, GK_DOWN_SMALL = 4,
    GK_GATE_UP_BWD = 5, GK_DGRAD_DOWN = 6, GK_WGRAD = 7, GK_ROUTER_WIDE = 8, GK_ROUTER_FUSED = 9,
    GK_ROUTER_PAIR = 10, GK_DOWN_PAIR = 11, GK_DOWN_COMBINE = 12
};
constexpr int FUSED_MAX_K = 8;      // experts per token the fused router selects at most
constexpr int GEMM_SMALL_T = 16;
constexpr int BWD_ROW_ALIGN = 64;   // backward buckets start on 64-row boundaries (K blocks of the weight gradients)

// Parameters of the tensor-core GEMM kernels.  Tensor maps live in the
// kernel's parameter space (__grid_constant__), so TMA reads them in place.
struct GemmParams {
    CUtensorMap tmA0;   // router: hidden; gate_up: X_perm; down: intermediate
    CUtensorMap tmA1;   // gate_up: hidden (shared-expert rows)
    CUtensorMap tmB0;   // router: W split [3E, H]; gate_up: W_gate_up [E*2I, H]; down: W_down [E*I, H]
    CUtensorMap tmB1;   // gate_up: shared_gate_up [2I, H]; down: shared_down [I, H]
    CUtensorMap tmOut;  // grouped: the output, boxes of 64 columns x 32 rows (TMA stores)
    void *out;          // router: logits fp32 [T, E]; gate_up: intermediate bf16; down: Y bf16
    const int4 *mtiles; // grouped: {group, first row, rows, 0} (pair kinds: the 256-row pair tiles)
    const int *num_mtiles;
    int num_tiles_static; // router: tiles known on the host
    int n_tiles;          // n-tiles per m-tile
    int kblocks;          // K / GEMM_BK (router: per K part)
    int ksplit;           // router: K parts per tile (0 or 1: none); part kp writes out + kp * part_stride
    long long part_stride; // router: floats between the K parts' logits
    int T, E, I, H, kT;
    int ld_out;           // output row stride in elements
    int *status;
    // backward kinds
    const float *w_perm;  // routing weight of every bucket row (1 for shared rows)
    uint16_t *gu_out;     // GK_GATE_UP_BWD: G and U, bf16 [rows, 2I] (32-row interleaved)
    uint16_t *aw_out;     // GK_GATE_UP_BWD: bf16(w * bf16(silu(G) * U)) [rows, I]
    const uint16_t *gu_in; // GK_DGRAD_DOWN: G and U
    uint16_t *dgu_out;    // GK_DGRAD_DOWN: dG and dU, bf16 [rows, 2I]
    float *dw_part;       // GK_DGRAD_DOWN: per (row, n-tile) partial dot products [kT_padded, n_tiles]
    const int2 *eoff;     // GK_WGRAD: per expert (first bucket row, padded rows); entry E = shared
    void *out_shared;     // GK_WGRAD: the shared expert's gradient
    int wg_fm, wg_fn;     // GK_WGRAD: feature blocks (128) and hidden blocks (256) per expert
    int b_row_shared;     // GK_WGRAD: first B row of the shared expert, or -1 to use its A rows
    // fault injection for tests: when set, the producer issues no loads, so
    // the first wait of the MMA lane runs out after wait_limit_ns
    int inject_withhold;
    int *tile_ctr;        // GK_WGRAD: tiles claimed so far (zero at launch)
    unsigned long long wait_limit_ns;
    // GK_ROUTER_FUSED (E = 256 in 8 groups, one token tile per tile, no K split;
    // out: the logits [T, 256] fp32, read back by the post phase)
    const float *bias;        // expert_bias [E], or NULL
    int32_t *idx_out;         // topk_idx [T, k]
    float *w_out;             // topk_w [T, k]
    int32_t *counts;          // expert_counts [E], zero at launch; also the buckets' fill levels
    int32_t *slot_local;      // [T, k] row of each pair inside its expert's bucket
    int *ready;               // [token tiles] epilogue warps done storing the tile's logits (zero at launch)
    int *unit_ctr;            // the post phase's tile queue (zero at launch)
    const uint16_t *hidden;   // [T, H], the rows copied into the buckets
    uint16_t *xperm;          // [E * T, H]: expert e's bucket starts at row e * T
    int topk_group, k;
    float rsf, eps;
    // grouped gate/up: routed m-tiles read their A rows from the tile list's
    // fourth field (the bucket layout above) instead of the second
    int cap_rows;
    // GK_DOWN_COMBINE: out[t] = bf16(Y_shared[t] + sum_j w[t,j] Y[slot_of[t,j]]
    // (+ residual[t])) for the tile's tokens; out is `out`, ld_out = H
    const uint16_t *cmb_y;      // the routed rows [kT, H]
    const int32_t *cmb_slot;    // slot_of [T, k]
    const float *cmb_w;         // topk_w [T, k]
    const uint16_t *cmb_res;    // residual [T, H] or NULL
    int cmb_k;
    // router kinds, scored output (no K split): when set, `out` receives the
    // sigmoid scores s = router_sigmoid(logit) instead of the logits, and
    // gscore [T, E / 32, 2] every group's two best biased scores s + bias
    // (bias = `bias` or zero; a tie for the top counts twice; the group score
    // is their fp32 sum); non-finite logits set ST_NONFINITE
    float *gscore;
};

// Smem bytes a GEMM kind needs (stages + alignment slack + barriers).
int gemm_smem_bytes(int kind);
int gemm_tmem_cols(int kind);

cudaError_t launch_gemm(int kind, const GemmParams &p, int grid, cudaStream_t s);

// W (fp32) -> hi/mid/lo bf16 parts [3][E][H]; also zeroes counts[E] when given.
cudaError_t launch_split_router(const float *W, uint16_t *W3, int E, int H, int32_t *counts, cudaStream_t s);

// Small-T router logits on the CUDA cores (fp32 W read as is); clears counts.
constexpr int ROUTER_SIMT_MAX_T = 32;   // decode sizes; the tensor-core path wins above
cudaError_t launch_router_simt(const uint16_t *x, const float *W, int T, int E, int H, float *logits,
                               int32_t *counts, cudaStream_t s);

// scores[i] = router_sigmoid(logits[i]) (n > 0)
cudaError_t launch_router_scores(const float *logits, float *scores, long long n, cudaStream_t s);

// counts[E] must be zero (or hold counts to add to) before the launch.
// logits: nparts partial-sum buffers of [T, E], part_stride floats apart (the
// router GEMM's K parts; 1 part: plain logits), nparts <= ROUTER_MAX_KSPLIT
constexpr int ROUTER_MAX_KSPLIT = 4;
cudaError_t launch_route_select(const float *logits, int nparts, long long part_stride, const float *bias, int T,
                                int E, int n_group, int topk_group, int k, float rsf, float eps, int32_t *idx,
                                float *w, int32_t *counts, float *ppart, int *status, int *fin_ticket,
                                cudaStream_t s);

// The same selection from the router GEMM's scored output (sigmoid scores
// [T, E] and every group's two best biased scores [T, E / 32, 2]), for 8
// groups of 32 with 4 kept; same
// outputs, bit for bit.  chunk_hist (nullable): per PERM_CHUNK-token chunk
// hits per expert, [E][ceil(T / PERM_CHUNK)] (the bucketing histogram).
cudaError_t launch_route_select_scored(const float *scores, const float *gscore, const float *bias, int T, int E,
                                       int k, float rsf, float eps, int32_t *idx, float *w, int32_t *counts,
                                       float *ppart, int *status, int *fin_ticket, int32_t *chunk_hist,
                                       cudaStream_t s);
// tokens per block of the routing kernels when they also write the bucketing
// histogram (whole PERM_CHUNK chunks per block)
inline int route_chunk_hist(int T) { return T <= ROUTE_SMALL_T ? PERM_CHUNK : 2 * PERM_CHUNK; }

// part: at least ROUTE_FIN_BLOCKS x E floats of scratch; ticket: an int that is
// zero when the launch starts (the routing kernel before it clears it)
constexpr int ROUTE_FIN_BLOCKS = 32;
cudaError_t launch_route_finalize(const int32_t *counts, const float *ppart, int nchunk, int T, int E, int k,
                                  float *part, int *ticket, float *aux_P, float *aux_loss, cudaStream_t s);

cudaError_t launch_bucket_hist(const int32_t *idx, int T, int E, int k, int32_t *hist, int *status,
                               cudaStream_t s);

// hist [E][nchunk] -> per-chunk starts inside each bucket (relative); sizes[E]
// (and the same into sizes2[E] when given)
cudaError_t launch_bucket_scan(int32_t *hist, int nchunk, int E, int32_t *sizes, cudaStream_t s,
                               int32_t *sizes2 = nullptr);

// ptiles (nullable): also the 256-row pair-tile list (hdr->num_ptiles);
// with_shared = false: no shared-expert group in the tile lists
cudaError_t launch_bucket_scatter(const int32_t *idx, const uint16_t *x, const int32_t *chunk_base,
                                  const int32_t *sizes, int T, int H, int E, int k, int32_t *slot_of,
                                  uint16_t *x_perm, int4 *mtiles, WsHeader *hdr, cudaStream_t s,
                                  int4 *ptiles = nullptr, bool with_shared = true);

// expert parallelism: the destination rank of every pair, the received
// rows' local expert ids, and a gather of bf16 rows by slot
cudaError_t launch_ep_dest(const int32_t *idx, long long n, int E, int per_rank, int32_t *dest, cudaStream_t s);
cudaError_t launch_ep_local_ids(const int32_t *idx, const int32_t *slot_of, long long n, int per_rank,
                                int32_t *e_send, cudaStream_t s);
cudaError_t launch_rows_gather(const uint16_t *rows, const int32_t *slot_of, int n, int H, uint16_t *out,
                               cudaStream_t s);

// T <= BUCKET_SMALL_MAX_T: hist, scan and scatter in one launch (same outputs)
constexpr int BUCKET_SMALL_MAX_T = 32;
// (m-tiles of at most mt rows)
cudaError_t launch_bucket_small(const int32_t *idx, const uint16_t *x, int T, int H, int E, int k, int mt,
                                int32_t *sizes, int32_t *slot_of, uint16_t *x_perm, int4 *mtiles, WsHeader *hdr,
                                cudaStream_t s);

// m-tile list of a dense MLP: T tokens in tiles of mt rows, group 0
cudaError_t launch_dense_tiles(int T, int mt, int4 *mtiles, WsHeader *hdr, cudaStream_t s);

// out[t] = bf16( sum_j w[t,j] Y[slot_of[t,j]] + Y[shared_row0 + t] (+ residual[t]) );
// w == NULL means every weight is 1; shared_row0 < 0 means k*T.  With `offs`,
// slot_of holds rows inside each expert's bucket and the Y row of pair (t, j)
// is offs[idx[t,j]] + slot_of[t,j] (a pair whose expert is not in [0, E) is
// skipped).
// y_rows >= 0: Y's row count; pair rows at or past it are skipped like -1.
cudaError_t launch_combine(const uint16_t *Y, const int32_t *slot_of, const float *w, const uint16_t *residual,
                           int T, int H, int k, uint16_t *out, cudaStream_t s, long long shared_row0 = -1,
                           const int32_t *idx = nullptr, const int32_t *offs = nullptr, int E = 0,
                           long long y_rows = -1);

// After the fused router: bucket offsets (exclusive scan of the E bucket
// sizes) into offs[E + 1] and the m-tile list of the grouped GEMMs, whose
// routed m-tiles read their A rows at e * T + r (the fused router's buckets).
cudaError_t launch_bucket_tiles(const int32_t *sizes, int T, int E, int k, int4 *mtiles, WsHeader *hdr,
                                int32_t *offs, cudaStream_t s);

// backward bucketing: as launch_bucket_scatter, buckets on BWD_ROW_ALIGN rows,
// plus dOut rows and routing weights per bucket row and the bucket table eoff
cudaError_t launch_bucket_scatter_bwd(const int32_t *idx, const uint16_t *x, const int32_t *chunk_base,
                                      const int32_t *sizes, int T, int H, int E, int k, int32_t *slot_of,
                                      uint16_t *x_perm, int4 *mtiles, WsHeader *hdr, const uint16_t *dout,
                                      const float *w, uint16_t *do_perm, float *w_perm, int2 *eoff, int shared_base,
                                      cudaStream_t s);
cudaError_t launch_zero_pad(const int2 *eoff, const int32_t *sizes, int T, int E, int H, int I, uint16_t *x_perm,
                            uint16_t *do_perm, uint16_t *aw, uint16_t *dgu, int *tile_ctr, cudaStream_t s);
cudaError_t launch_dw_reduce(const int32_t *slot_of, const float *dw_part, int n, int ntiles, float *dw,
                             cudaStream_t s);

cudaError_t launch_expert_feedback(const int32_t *counts, int E, int T, int k, float gamma, float *bias,
                                   long long *totals, cudaStream_t s);

cudaError_t launch_rmsnorm(const uint16_t *x, uint16_t *out, int T, int H, float eps, cudaStream_t s);

}  // namespace glr
