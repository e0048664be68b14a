// Routing kernels of the MoE layer forward (SIMT, sm_103a).
//
// Follows the article "InternLumina-U2中256个专家的路由秘密：分组受限Top-K、Expert
// Bias与Fused MoE详解" (the routing page):
//   section 二 step 1  sigmoid scores of the fp32 router logits;
//   section 二 step 2  group-limited top-k (group score = sum of the group's two
//                      best scores, keep topk_group groups, top-k of their experts);
//   section 三         expert_bias is added for choosing only;
//   section 二 step 3  w = s / (sum of the chosen s + eps) * routed_scaling_factor;
//   section 六         per-expert hit counts;
// and the load-balancing loss E * sum_i f_i * P_i of the InternLumina-U2
// training-pitfalls article (section "MoE 负载均衡 Loss 别忘加").
//
// Kernels, in the order a forward runs them:
//   split_router_kernel        fp32 router weight -> exact bf16 hi/mid/lo parts
//                              for the tensor-core router GEMM (once per model);
//   router_simt_kernel         decode-size router logits on the CUDA cores,
//                              one block per expert, fp32 weight as is;
//   route_select_kernel<G>     scores, group-limited top-k, weights and hit
//                              counts, one warp per token, any n_group <= 8;
//   route_select_sorted_kernel the same selection specialised for 4 of 8 groups;
//   route_finalize_kernel      balance loss from the per-chunk score sums,
//                              several blocks, the last one to finish combines;
//   expert_feedback_kernel     expert-bias update and running hit totals.
// Router logits may arrive as several K parts (a split-K router GEMM); the
// selection kernels add the parts in part order before the sigmoid.
//
// Ties go to the lower index at both levels; the k experts come out in order of
// (biased score desc, index asc).  Everything is deterministic: per-block
// histograms and score sums are reduced in a fixed order, never with float
// atomics.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "kernels.h"
#include "route_token.cuh"

namespace glr {

// ---------------------------------------------------------------------------
// W (fp32) -> hi, mid, lo (bf16) with hi + mid + lo == W exactly for normal
// values: each part is the bf16 rounding of what the previous parts left.
// Layout of W3: [3][E][H].
// The same launch also clears `counts` (E entries) for the routing kernel
// that follows it on the stream.
__global__ void split_router_kernel(const float *__restrict__ W, uint16_t *__restrict__ W3, int n,
                                    int32_t *__restrict__ counts, int E)
{
    pdl_wait();
    if (blockIdx.x == 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            counts[e] = 0;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float w = W[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
        W3[i] = __bfloat16_as_ushort(hi);
        W3[n + i] = __bfloat16_as_ushort(mid);
        W3[2 * n + i] = __bfloat16_as_ushort(lo);
    }
}

cudaError_t launch_split_router(const float *W, uint16_t *W3, int E, int H, int32_t *counts, cudaStream_t s)
{
    const int n = E * H;
    const int blocks = min((n + 255) / 256, 4096);
    const cudaError_t le = launch_pdl(split_router_kernel, dim3(blocks), dim3(256), 0, s, W, W3, n, counts,
                                      counts ? E : 0);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// Router logits for small T (decode) on the CUDA cores, fp32 weight as is.
// One block per expert: thread i takes 8 consecutive hidden columns
// (i * 8 + 2048 q), loads that piece of the expert's weight row once and of
// every token's hidden row, and forms each token's partial dot product with
// fused multiply-adds in column order; the 256 partials of a token are then
// added by a butterfly inside each warp and the 8 warp sums in warp order.
// With a block per expert the weight stream (E H fp32, read once) is spread
// over the whole GPU.  Block 0 also clears `counts` for the routing kernel
// that follows.
constexpr int SIMT_THREADS = 256;

__global__ void __launch_bounds__(SIMT_THREADS) router_simt_kernel(const uint16_t *__restrict__ x,
                                                                   const float *__restrict__ W, int T, int E, int H,
                                                                   float *__restrict__ logits,
                                                                   int32_t *__restrict__ counts)
{
    pdl_wait();
    __shared__ float red[SIMT_THREADS / 32][ROUTER_SIMT_MAX_T];
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (e == 0 && counts)
        for (int i = threadIdx.x; i < E; i += blockDim.x)
            counts[i] = 0;
    float acc[ROUTER_SIMT_MAX_T];
#pragma unroll
    for (int t = 0; t < ROUTER_SIMT_MAX_T; ++t)
        acc[t] = 0.0f;
    const float *wrow = W + (size_t)e * H;
    for (int c = threadIdx.x * 8; c < H; c += SIMT_THREADS * 8) {
        const float4 w0 = __ldg(reinterpret_cast<const float4 *>(wrow + c));
        const float4 w1 = __ldg(reinterpret_cast<const float4 *>(wrow + c + 4));
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int t0 = 0; t0 < ROUTER_SIMT_MAX_T; t0 += 8) {    // 8 tokens' pieces in flight at a time
            if (t0 < T) {
                uint4 xv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (t0 + u < T)
                        xv[u] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + u) * H + c));
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (t0 + u < T) {
                        const uint32_t q[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            acc[t0 + u] = fmaf(__uint_as_float(q[h] << 16), wv[2 * h], acc[t0 + u]);
                            acc[t0 + u] = fmaf(__uint_as_float(q[h] & 0xffff0000u), wv[2 * h + 1], acc[t0 + u]);
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < ROUTER_SIMT_MAX_T; ++t) {
        if (t < T) {
            float a = acc[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                a += __shfl_xor_sync(0xffffffffu, a, off);
            if (lane == 0)
                red[warp][t] = a;
        }
    }
    __syncthreads();
    if (threadIdx.x < T) {
        float a = 0.0f;
#pragma unroll
        for (int w = 0; w < SIMT_THREADS / 32; ++w)
            a += red[w][threadIdx.x];
        logits[(size_t)threadIdx.x * E + e] = a;
    }
}

cudaError_t launch_router_simt(const uint16_t *x, const float *W, int T, int E, int H, float *logits,
                               int32_t *counts, cudaStream_t s)
{
    if (T > ROUTER_SIMT_MAX_T || H % 8 != 0)
        return cudaErrorInvalidValue;
    const cudaError_t le = launch_pdl(router_simt_kernel, dim3(E), dim3(SIMT_THREADS), 0, s, x, W, T, E, H, logits,
                                      counts);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// The routing kernels' sigmoid over a flat array (a diagnostic: the scores
// the selection ranks, for comparison with an exact sigmoid).
__global__ void router_scores_kernel(const float *__restrict__ L, float *__restrict__ s, long long n)
{
    pdl_wait();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        s[i] = router_sigmoid(L[i]);
}

cudaError_t launch_router_scores(const float *L, float *s, long long n, cudaStream_t st)
{
    const long long blocks = std::min<long long>((n + 255) / 256, 152 * 8);
    const cudaError_t le = launch_pdl(router_scores_kernel, dim3((unsigned)blocks), dim3(256), 0, st, L, s, n);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// Logit (t, e) when the router GEMM wrote it in `nparts` K parts (partial sums
// over consecutive K ranges, part p at logits + p * part_stride): their sum in
// part order, so the result does not depend on scheduling.
__device__ __forceinline__ float load_logit(const float *__restrict__ logits, size_t off, int nparts,
                                            long long part_stride)
{
    if (nparts == 1)
        return __ldg(logits + off);
    float v[ROUTER_MAX_KSPLIT];
#pragma unroll
    for (int q = 0; q < ROUTER_MAX_KSPLIT; ++q)          // every part's load in flight at once
        v[q] = (q < nparts) ? __ldg(logits + (size_t)q * part_stride + off) : 0.0f;
    float L = v[0];
#pragma unroll
    for (int q = 1; q < ROUTER_MAX_KSPLIT; ++q)
        if (q < nparts)
            L += v[q];
    return L;
}

// One warp per token (route_token): lane l holds experts 32*j + l for
// j < n_group, so every load of a logits row is a run of 128-byte coalesced
// accesses.
//
// Block: 8 warps, `chunk` tokens (route_chunk(T)).  Hits per expert go to a shared-memory
// histogram and then to `counts` with integer atomics (exact, order-free).
// With `ppart`, the block also writes per-expert sums of the token-normalised
// scores of its chunk for the balance loss.
template <int G>
__global__ void __launch_bounds__(256) route_select_kernel(
    const float *__restrict__ logits, int nparts, long long part_stride, const float *__restrict__ bias, int T,
    int chunk, int TG, int K, float rsf, float eps,
    int32_t *__restrict__ idx_out, float *__restrict__ w_out, int32_t *__restrict__ counts,
    float *__restrict__ ppart, int *__restrict__ status, int *__restrict__ fin_ticket)
{
    pdl_wait();
    constexpr int E = 32 * G;
    constexpr unsigned FULL = 0xffffffffu;
    __shared__ int sh_hist[E];
    __shared__ float sh_p[8][E];
    if (fin_ticket && blockIdx.x == 0 && threadIdx.x == 0)
        *fin_ticket = 0;                           // for the balance-loss reduction that follows

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        sh_hist[e] = 0;

    float bias_r[G];
#pragma unroll
    for (int j = 0; j < G; ++j)
        bias_r[j] = bias ? bias[32 * j + lane] : 0.0f;
    float pacc[G];
#pragma unroll
    for (int j = 0; j < G; ++j)
        pacc[j] = 0.0f;
    __syncthreads();

    bool nonfinite = false;
    const int t0 = blockIdx.x * chunk;
    const int t1 = min(T, t0 + chunk);
    for (int t = t0 + warp; t < t1; t += 8) {
        float L[G], s[G];
#pragma unroll
        for (int j = 0; j < G; ++j)
            L[j] = load_logit(logits, (size_t)t * E + 32 * j + lane, nparts, part_stride);
        int my_e;
        float my_w;
        route_token<G>(L, bias_r, lane, TG, K, rsf, eps, s, my_e, my_w, nonfinite);
        if (lane < K) {
            idx_out[(size_t)t * K + lane] = my_e;
            w_out[(size_t)t * K + lane] = my_w;
            atomicAdd(&sh_hist[my_e], 1);
        }

        if (ppart) {
            float tot = 0.0f;
#pragma unroll
            for (int j = 0; j < G; ++j)
                tot += s[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                tot += __shfl_xor_sync(FULL, tot, off);
            const float inv = 1.0f / tot;
#pragma unroll
            for (int j = 0; j < G; ++j)
                pacc[j] += s[j] * inv;
        }
    }
    if (__any_sync(FULL, nonfinite) && lane == 0)
        atomicOr(status, ST_NONFINITE);

    if (ppart) {
#pragma unroll
        for (int j = 0; j < G; ++j)
            sh_p[warp][32 * j + lane] = pacc[j];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (sh_hist[e])
            atomicAdd(&counts[e], sh_hist[e]);      // integer sums: the result is order-free
        if (ppart) {
            float v = 0.0f;
            for (int q = 0; q < 8; ++q)
                v += sh_p[q][e];
            ppart[(size_t)blockIdx.x * E + e] = v;
        }
    }
}

// The same selection for the page's setting (topk_group of n_group groups
// kept, instantiated for 4 of 8), with far fewer instructions per token:
//  * after the group stage every lane has exactly TG candidates (its experts
//    in the kept groups); it sorts them once by (key desc, group asc), so a
//    top-k round is two warp reductions plus a shift of the winning lane's
//    list instead of a scan over all its groups;
//  * the token's keys and unbiased scores go to a per-warp shared-memory row
//    (index = expert id), from which the kept groups' keys and each round's
//    winning score are read by index;
//  * the next token's logits are loaded before the current one is processed.
// Results are identical to route_select_kernel's: same score formula, same
// group scores and ranking, same winner per round (max key, then lowest
// expert id), the same sequential sum for the normaliser.
template <int G, int TG>
__global__ void __launch_bounds__(256, 5) route_select_sorted_kernel(
    const float *__restrict__ logits, int nparts, long long part_stride, const float *__restrict__ bias, int T,
    int chunk, int K, float rsf, float eps,
    int32_t *__restrict__ idx_out, float *__restrict__ w_out, int32_t *__restrict__ counts,
    float *__restrict__ ppart, int *__restrict__ status, int *__restrict__ fin_ticket)
{
    pdl_wait();
    constexpr int E = 32 * G;
    constexpr unsigned FULL = 0xffffffffu;
    if (fin_ticket && blockIdx.x == 0 && threadIdx.x == 0)
        *fin_ticket = 0;                           // for the balance-loss reduction that follows
    __shared__ int sh_hist[E];
    __shared__ float sh_p[8][E];
    __shared__ float sh_s[8][E];       // per warp: the current token's unbiased scores, by expert
    __shared__ uint32_t sh_k[8][E];    // per warp: its biased-score keys, by expert
    __shared__ float sh_bias[E];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    bool nonfinite = false;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        sh_hist[e] = 0;
        const float b = bias ? bias[e] : 0.0f;
        nonfinite |= !isfinite(b);
        sh_bias[e] = b;
    }
    // per-warp sums of the token-normalised scores (balance loss), by expert
#pragma unroll
    for (int j = 0; j < G; ++j)
        sh_p[warp][32 * j + lane] = 0.0f;
    __syncthreads();

    const int t0 = blockIdx.x * chunk;
    const int t1 = min(T, t0 + chunk);
    float Ln[G];
    if (t0 + warp < t1) {
#pragma unroll
        for (int j = 0; j < G; ++j)
            Ln[j] = load_logit(logits, (size_t)(t0 + warp) * E + 32 * j + lane, nparts, part_stride);
    }
    for (int t = t0 + warp; t < t1; t += 8) {
        float L[G];
#pragma unroll
        for (int j = 0; j < G; ++j)
            L[j] = Ln[j];
        if (t + 8 < t1) {
#pragma unroll
            for (int j = 0; j < G; ++j)
                Ln[j] = load_logit(logits, (size_t)(t + 8) * E + 32 * j + lane, nparts, part_stride);
        }
        float s[G];
        uint32_t kk[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            nonfinite |= !(fabsf(L[j]) <= 3.402823466e38f);   // NaN or +-inf
            s[j] = router_sigmoid(L[j]);                        // section 二 step 1
            kk[j] = fkey(s[j] + sh_bias[32 * j + lane]);       // section 三: choose on s + bias
            sh_s[warp][32 * j + lane] = s[j];
            sh_k[warp][32 * j + lane] = kk[j];
        }

        // group score = top-1 + top-2 of the group's biased scores (a tie for
        // the top counts twice)
        float g[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const uint32_t m1 = __reduce_max_sync(FULL, kk[j]);
            const uint32_t m2o = __reduce_max_sync(FULL, kk[j] < m1 ? kk[j] : 0u);
            const uint32_t m2 = (__popc(__ballot_sync(FULL, kk[j] == m1)) > 1) ? m1 : m2o;
            g[j] = fkey_value(m1) + fkey_value(m2);
        }

        // keep the TG best groups (ties to the lower group index)
        float gl = g[0];
#pragma unroll
        for (int j = 1; j < G; ++j)
            if (lane == j)
                gl = g[j];
        int rank = 0;
#pragma unroll
        for (int i = 0; i < G; ++i)
            rank += (g[i] > gl || (g[i] == gl && i < lane)) ? 1 : 0;
        uint32_t keep = __ballot_sync(FULL, lane < G && rank < TG) & ((1u << G) - 1u);
        __syncwarp();                                   // the warp's row of keys and scores is written

        // this lane's candidates in ascending group order, then sorted by key
        // (descending) with adjacent exchanges that swap only on a strictly
        // larger key, so equal keys keep the lower group first
        uint32_t ck[TG];
        int cj[TG];
#pragma unroll
        for (int i = 0; i < TG; ++i) {
            const int j = __ffs(keep) - 1;
            keep &= keep - 1u;
            cj[i] = j;
            ck[i] = sh_k[warp][32 * j + lane];
        }
#pragma unroll
        for (int i = 1; i < TG; ++i) {
#pragma unroll
            for (int q = i; q > 0; --q) {
                if (ck[q] > ck[q - 1]) {
                    const uint32_t tk = ck[q];
                    ck[q] = ck[q - 1];
                    ck[q - 1] = tk;
                    const int tj = cj[q];
                    cj[q] = cj[q - 1];
                    cj[q - 1] = tj;
                }
            }
        }

        // top-K: each round takes the largest head key, ties to the lowest expert id
        float den = 0.0f;
        int my_e = -1;
        float my_s = 0.0f;
        for (int r = 0; r < K; ++r) {
            const uint32_t wk = __reduce_max_sync(FULL, ck[0]);
            const uint32_t cand = (ck[0] == wk) ? (uint32_t)(32 * cj[0] + lane) : 0xffffffffu;
            const uint32_t we = __reduce_min_sync(FULL, cand);
            if (cand == we) {                              // the winning lane drops its head
#pragma unroll
                for (int i = 0; i + 1 < TG; ++i) {
                    ck[i] = ck[i + 1];
                    cj[i] = cj[i + 1];
                }
                ck[TG - 1] = 0u;
            }
            const float sw = sh_s[warp][we];              // the winner's unbiased score
            den += sw;                                    // sequential, in output order
            if (lane == r) {
                my_e = (int)we;
                my_s = sw;
            }
        }
        den += eps;
        if (lane < K) {
            idx_out[(size_t)t * K + lane] = my_e;
            w_out[(size_t)t * K + lane] = (my_s / den) * rsf;   // section 二 step 3
            atomicAdd(&sh_hist[my_e], 1);
        }

        if (ppart) {
            float tot = 0.0f;
#pragma unroll
            for (int j = 0; j < G; ++j)
                tot += s[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                tot += __shfl_xor_sync(FULL, tot, off);
            const float inv = 1.0f / tot;
#pragma unroll
            for (int j = 0; j < G; ++j)
                sh_p[warp][32 * j + lane] += s[j] * inv;
        }
        __syncwarp();                                   // row reads done before the next token's writes
    }
    if (__any_sync(FULL, nonfinite) && lane == 0)
        atomicOr(status, ST_NONFINITE);

    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (sh_hist[e])
            atomicAdd(&counts[e], sh_hist[e]);      // integer sums: the result is order-free
        if (ppart) {
            float v = 0.0f;
            for (int q = 0; q < 8; ++q)
                v += sh_p[q][e];
            ppart[(size_t)blockIdx.x * E + e] = v;
        }
    }
}

// The same selection from the router GEMM's scored output: the sigmoid scores
// s [T, E] and every group's score [T, G] were formed in the GEMM's epilogue
// (router_epilogue_tile), with the same router_sigmoid and the same fp32
// additions, so nothing of the selection changes.  Per token (one warp) the
// kernel reads the 8 group scores, keeps the TG best (ties to the lower
// group), reads only the kept groups' scores (one coalesced row piece each)
// and runs the top-K rounds of route_select_sorted_kernel on them; the
// winner's unbiased score travels with its candidate, so no shared-memory
// row is needed.  With `ppart` every score of the token is read for the
// balance-loss sums (same order of additions as the other kernels).  With
// `chunk_hist` the block (chunk = 16 or 32 tokens) also writes the hits per
// expert of each PERM_CHUNK-token chunk, [E][nchunk_perm].
template <int G, int TG>
__global__ void __launch_bounds__(256) route_select_scored_kernel(
    const float *__restrict__ scores, const float *__restrict__ gscore, const float *__restrict__ bias, int T,
    int chunk, int K, float rsf, float eps, int32_t *__restrict__ idx_out, float *__restrict__ w_out,
    int32_t *__restrict__ counts, float *__restrict__ ppart, int *__restrict__ status, int *__restrict__ fin_ticket,
    int32_t *__restrict__ chunk_hist, int nchunk_perm)
{
    pdl_wait();
    constexpr int E = 32 * G;
    constexpr unsigned FULL = 0xffffffffu;
    constexpr int NQ = 2;                          // PERM_CHUNK chunks per block at most
    if (fin_ticket && blockIdx.x == 0 && threadIdx.x == 0)
        *fin_ticket = 0;                           // for the balance-loss reduction that follows
    __shared__ int sh_hist[NQ][E];
    __shared__ float sh_p[8][E];
    __shared__ float sh_bias[E];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    bool nonfinite = false;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const float b = bias ? bias[e] : 0.0f;
        nonfinite |= !isfinite(b);
        sh_bias[e] = b;
#pragma unroll
        for (int q = 0; q < NQ; ++q)
            sh_hist[q][e] = 0;
    }
    if (ppart) {
#pragma unroll
        for (int j = 0; j < G; ++j)
            sh_p[warp][32 * j + lane] = 0.0f;
    }
    __syncthreads();

    const int t0 = blockIdx.x * chunk;
    const int t1 = min(T, t0 + chunk);
    static_assert(G % 2 == 0, "group score pairs are read as float4");
    // the token's groups' two best scores (every lane reads the same row of
    // 2 G floats); the next token's row is loaded before the current token is
    // processed; the group score is their sum
    float4 gn[G / 2];
    if (t0 + warp < t1) {
#pragma unroll
        for (int v = 0; v < G / 2; ++v)
            gn[v] = __ldg(reinterpret_cast<const float4 *>(gscore + (size_t)(t0 + warp) * 2 * G) + v);
    }
    for (int t = t0 + warp; t < t1; t += 8) {
        float g[G];
#pragma unroll
        for (int v = 0; v < G / 2; ++v) {
            g[2 * v] = gn[v].x + gn[v].y;
            g[2 * v + 1] = gn[v].z + gn[v].w;
        }
        if (t + 8 < t1) {
#pragma unroll
            for (int v = 0; v < G / 2; ++v)
                gn[v] = __ldg(reinterpret_cast<const float4 *>(gscore + (size_t)(t + 8) * 2 * G) + v);
        }
        float gl = g[0];
#pragma unroll
        for (int j = 1; j < G; ++j)
            if (lane == j)
                gl = g[j];
        int rank = 0;
#pragma unroll
        for (int i = 0; i < G; ++i)
            rank += (g[i] > gl || (g[i] == gl && i < lane)) ? 1 : 0;
        uint32_t keep = __ballot_sync(FULL, lane < G && rank < TG) & ((1u << G) - 1u);

        // this lane's candidates (its expert of each kept group), ascending
        // group, then sorted by key (descending), equal keys keep the lower
        // group; the candidates' groups are packed 8 bits each into cjp
        // (entry i in bits 8i), so dropping the head is one shift
        uint32_t ck[TG];
        int cj[TG];
        const float *srow = scores + (size_t)t * E + lane;
#pragma unroll
        for (int i = 0; i < TG; ++i) {
            const int j = __ffs(keep) - 1;
            keep &= keep - 1u;
            cj[i] = j;
            ck[i] = fkey(__ldg(srow + 32 * j) + sh_bias[32 * j + lane]);   // section 三: choose on s + bias
        }
#pragma unroll
        for (int i = 1; i < TG; ++i) {
#pragma unroll
            for (int q = i; q > 0; --q) {
                if (ck[q] > ck[q - 1]) {
                    const uint32_t tk = ck[q];
                    ck[q] = ck[q - 1];
                    ck[q - 1] = tk;
                    const int tj = cj[q];
                    cj[q] = cj[q - 1];
                    cj[q - 1] = tj;
                }
            }
        }
        uint32_t cjp = 0;
#pragma unroll
        for (int i = 0; i < TG; ++i)
            cjp |= (uint32_t)cj[i] << (8 * i);

        // top-K: each round takes the largest head key, ties to the lowest expert id
        int my_e = -1;
        for (int r = 0; r < K; ++r) {
            const uint32_t wk = __reduce_max_sync(FULL, ck[0]);
            const uint32_t cand = (ck[0] == wk) ? (((cjp & 0xffu) << 5) | (uint32_t)lane) : 0xffffffffu;
            const uint32_t we = __reduce_min_sync(FULL, cand);
            if (cand == we) {                              // the winning lane drops its head
#pragma unroll
                for (int i = 0; i + 1 < TG; ++i)
                    ck[i] = ck[i + 1];
                ck[TG - 1] = 0u;
                cjp >>= 8;
            }
            if (lane == r)
                my_e = (int)we;
        }
        // the winners' unbiased scores; the normaliser adds them in output order
        const float my_s = (lane < K) ? __ldg(scores + (size_t)t * E + my_e) : 0.0f;
        float den = 0.0f;
        for (int r = 0; r < K; ++r)
            den += __shfl_sync(FULL, my_s, r);
        den += eps;
        if (lane < K) {
            idx_out[(size_t)t * K + lane] = my_e;
            w_out[(size_t)t * K + lane] = (my_s / den) * rsf;   // section 二 step 3
            atomicAdd(&sh_hist[(t - t0) / PERM_CHUNK][my_e], 1);
        }

        if (ppart) {
            float sj[G];
#pragma unroll
            for (int j = 0; j < G; ++j)
                sj[j] = __ldg(srow + 32 * j);
            float tot = 0.0f;
#pragma unroll
            for (int j = 0; j < G; ++j)
                tot += sj[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                tot += __shfl_xor_sync(FULL, tot, off);
            const float inv = 1.0f / tot;
#pragma unroll
            for (int j = 0; j < G; ++j)
                sh_p[warp][32 * j + lane] += sj[j] * inv;
        }
    }
    if (__any_sync(FULL, nonfinite) && lane == 0)
        atomicOr(status, ST_NONFINITE);

    __syncthreads();
    const int q0 = t0 / PERM_CHUNK;
    const int nq = (t1 - t0 + PERM_CHUNK - 1) / PERM_CHUNK;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int tot = 0;
#pragma unroll
        for (int q = 0; q < NQ; ++q)
            tot += sh_hist[q][e];
        if (counts && tot)
            atomicAdd(&counts[e], tot);              // integer sums: the result is order-free
        if (chunk_hist) {
            for (int q = 0; q < nq; ++q)
                chunk_hist[(size_t)e * nchunk_perm + q0 + q] = sh_hist[q][e];   // [expert][chunk]
        }
        if (ppart) {
            float v = 0.0f;
            for (int q = 0; q < 8; ++q)
                v += sh_p[q][e];
            ppart[(size_t)blockIdx.x * E + e] = v;
        }
    }
}

// The same selection with four threads per token (no balance-loss sums, k <=
// 8): lanes 4i .. 4i + 3 of a warp take token i, a block of 128 threads 32
// tokens (two bucketing chunks).
//  * Each lane ranks two of the token's eight group scores; the quad ORs its
//    lanes' bits into the kept-group mask (TG best groups, ties to the lower
//    group).
//  * Lane q takes the q-th kept group (ascending) and runs its 32 experts in
//    ascending id order through an 8-entry list kept in descending order of
//    biased score: an expert moves ahead of an entry only when strictly
//    larger, so equal scores keep the lower id first.
//  * Two merge steps (lanes q ^ 1, then q ^ 2) combine the quad's lists: the
//    better of A[p] and B[7 - p] for every p is the top half of a bitonic
//    sequence, which three compare-exchange stages sort -- "better" meaning a
//    larger biased score, or an equal one with a lower expert id.
// The result is the warp kernels' (biased score desc, id asc) order, and the
// weights use the same sequential normaliser, so the outputs agree bit for
// bit.  Every lane holds the merged list; lane q writes entries 2q, 2q + 1.
__device__ __forceinline__ bool sel_better(float va, int ea, float vb, int eb)
{
    return va > vb || (va == vb && (unsigned)ea < (unsigned)eb);
}

__device__ __forceinline__ void sel_cas(float &va, int &ea, float &vb, int &eb)
{
    // after the call (va, ea) is the better of the two
    const bool sw = sel_better(vb, eb, va, ea);
    const float tv = va;
    const int te = ea;
    va = sw ? vb : va;
    ea = sw ? eb : ea;
    vb = sw ? tv : vb;
    eb = sw ? te : eb;
}

// merges this lane's sorted list with the one of lane ^ mask (both lanes end
// with the same sorted top 8)
__device__ __forceinline__ void sel_merge(float (&v)[8], int (&e)[8], int lane, int mask)
{
    float ov[8];
    int oe[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        ov[p] = __shfl_xor_sync(0xffffffffu, v[p], mask);
        oe[p] = __shfl_xor_sync(0xffffffffu, e[p], mask);
    }
    const bool lower = (lane & mask) == 0;   // the list of the lower lane plays A in both lanes
    float a[8], b[8];
    int ae[8], be[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        a[p] = lower ? v[p] : ov[p];
        ae[p] = lower ? e[p] : oe[p];
        b[p] = lower ? ov[p] : v[p];
        be[p] = lower ? oe[p] : e[p];
    }
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const bool ta = sel_better(a[p], ae[p], b[7 - p], be[7 - p]);
        v[p] = ta ? a[p] : b[7 - p];
        e[p] = ta ? ae[p] : be[7 - p];
    }
#pragma unroll
    for (int d = 4; d > 0; d >>= 1)
#pragma unroll
        for (int p = 0; p < 8; ++p)
            if ((p & d) == 0)
                sel_cas(v[p], e[p], v[p + d], e[p + d]);
}

template <int G, int TG>
__global__ void __launch_bounds__(128) route_select_quad_kernel(
    const float *__restrict__ scores, const float *__restrict__ gscore, const float *__restrict__ bias, int T,
    int K, float rsf, float eps, int32_t *__restrict__ idx_out, float *__restrict__ w_out,
    int32_t *__restrict__ counts, int *__restrict__ status, int32_t *__restrict__ chunk_hist, int nchunk_perm)
{
    pdl_wait();
    constexpr int E = 32 * G;
    constexpr int GP = 33;
    static_assert(G == 8 && TG == 4, "four kept groups, one per lane of a quad");
    static_assert(2 * PERM_CHUNK == 32, "a block is two bucketing chunks");
    __shared__ float sb[G * GP];
    __shared__ int sh_hist[2][E];
    __shared__ float sbq[128 * 33];              // per lane: its kept group's 32 scores
    const int tid = threadIdx.x, lane = tid & 31;
    const int q = tid & 3;
    bool nonfinite = false;
    for (int e = tid; e < E; e += blockDim.x) {
        const float b = bias ? bias[e] : 0.0f;
        nonfinite |= !isfinite(b);
        sb[(e >> 5) * GP + (e & 31)] = b;
        sh_hist[0][e] = 0;
        sh_hist[1][e] = 0;
    }
    __syncthreads();
    const int tl = tid >> 2;                      // the token's place in the block
    const int t0 = blockIdx.x * 32;
    const int t = t0 + tl;
    const bool valid = t < T;

    // the token's groups' two best biased scores; group score = their sum
    float m1[G], m2[G], g[G];
#pragma unroll
    for (int v2 = 0; v2 < G / 2; ++v2) {
        const float4 x = valid ? __ldg(reinterpret_cast<const float4 *>(gscore + (size_t)t * 2 * G) + v2)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        m1[2 * v2] = x.x;
        m2[2 * v2] = x.y;
        m1[2 * v2 + 1] = x.z;
        m2[2 * v2 + 1] = x.w;
    }
#pragma unroll
    for (int i = 0; i < G; ++i)
        g[i] = m1[i] + m2[i];
    // kept groups: this lane ranks groups 2q and 2q + 1
    uint32_t keep = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int j = 2 * q + h;
        float gj = g[0];
#pragma unroll
        for (int i = 1; i < G; ++i)
            gj = (i == j) ? g[i] : gj;
        int rank = 0;
#pragma unroll
        for (int i = 0; i < G; ++i)
            rank += (g[i] > gj || (g[i] == gj && i < j)) ? 1 : 0;
        keep |= (rank < TG) ? (1u << j) : 0u;
    }
    keep |= __shfl_xor_sync(0xffffffffu, keep, 1);
    keep |= __shfl_xor_sync(0xffffffffu, keep, 2);
    // a floor under the token's 8th-best score: the kept groups hold 2 TG >= 8
    // scores at or above the smallest of their top-2, so nothing below it can
    // be chosen (TG = 4, k <= 8)
    float floor8 = 3.402823466e38f;
#pragma unroll
    for (int i = 0; i < G; ++i)
        floor8 = ((keep >> i) & 1u) ? fminf(floor8, m2[i]) : floor8;

    // this lane's kept group: the q-th set bit of keep
    uint32_t kk = keep;
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (i < q)
            kk &= kk - 1u;
    const int j = valid ? __ffs(kk) - 1 : 0;
    const float4 *s4 = reinterpret_cast<const float4 *>(scores + (size_t)(valid ? t : 0) * E + 32 * j);
    // the group's scores into this lane's shared-memory row (the weights
    // below read them back from there), and the bits of those whose biased
    // score is at or above the floor
    float *brow = sbq + (size_t)tid * 33;
    uint32_t cand = 0;
#pragma unroll
    for (int i4 = 0; i4 < 8; ++i4) {
        const float4 sv = valid ? __ldg(s4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float sc[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float b = sc[u] + sb[j * GP + 4 * i4 + u];   // section 三: choose on s + bias
            brow[4 * i4 + u] = sc[u];
            cand |= (valid && b >= floor8) ? (1u << (4 * i4 + u)) : 0u;
        }
    }
    __syncwarp();

    // this lane's candidates in ascending id order through an 8-entry list in
    // descending order of biased score: a candidate enters when it beats the
    // last entry and moves up past every strictly smaller one, so equal
    // scores keep the lower id first (empty entries: most negative float, id -1)
    float v[8];
    int ev[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        v[p] = -3.402823466e38f;
        ev[p] = -1;
    }
    while (cand) {
        const int i = __ffs(cand) - 1;
        cand &= cand - 1u;
        const float b = brow[i] + sb[j * GP + i];         // the same fp32 sum as above
        const int id = 32 * j + i;
        const bool in = b > v[7];
        v[7] = in ? b : v[7];
        ev[7] = in ? id : ev[7];
#pragma unroll
        for (int p = 7; p > 0; --p) {
            const bool up = v[p] > v[p - 1];
            const float tv = v[p - 1];
            const int te = ev[p - 1];
            v[p - 1] = up ? v[p] : tv;
            ev[p - 1] = up ? ev[p] : te;
            v[p] = up ? tv : v[p];
            ev[p] = up ? te : ev[p];
        }
    }
    sel_merge(v, ev, lane, 1);
    sel_merge(v, ev, lane, 2);

    // weights from the unbiased scores, normaliser in output order (section 二
    // step 3); the score of expert e sits in the row of the quad lane that
    // handled its group (group g is the lane's kept group when g is the
    // lane's-index-th set bit of keep)
    const float *qrows = sbq + (size_t)(tid & ~3) * 33;
    float sw[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int e = ev[p];
        sw[p] = (valid && p < K && e >= 0) ? qrows[__popc(keep & ((1u << (e >> 5)) - 1u)) * 33 + (e & 31)] : 0.0f;
    }
    float den = 0.0f;
#pragma unroll
    for (int p = 0; p < 8; ++p)
        if (p < K)
            den += sw[p];
    den += eps;
    if (valid) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = 2 * q + h;
            float wp = sw[0];
            int ep = ev[0];
#pragma unroll
            for (int i = 1; i < 8; ++i) {
                wp = (i == p) ? sw[i] : wp;
                ep = (i == p) ? ev[i] : ep;
            }
            if (p < K) {
                idx_out[(size_t)t * K + p] = ep;
                w_out[(size_t)t * K + p] = (wp / den) * rsf;
                if (ep >= 0)
                    atomicAdd(&sh_hist[tl / PERM_CHUNK][ep], 1);
            }
        }
    }
    if (__any_sync(0xffffffffu, nonfinite) && lane == 0)
        atomicOr(status, ST_NONFINITE);
    __syncthreads();
    const int nq = (min(T, t0 + 32) - t0 + PERM_CHUNK - 1) / PERM_CHUNK;
    for (int e = tid; e < E; e += blockDim.x) {
        const int a = sh_hist[0][e], b = sh_hist[1][e];
        if (counts && a + b)
            atomicAdd(&counts[e], a + b);            // integer sums: the result is order-free
        if (chunk_hist) {
            chunk_hist[(size_t)e * nchunk_perm + 2 * blockIdx.x] = a;
            if (nq > 1)
                chunk_hist[(size_t)e * nchunk_perm + 2 * blockIdx.x + 1] = b;
        }
    }
}

cudaError_t launch_route_select_scored(const float *scores, const float *gscore, const float *bias, int T, int E,
                                       int k, float rsf, float eps, int32_t *idx, float *w, int32_t *counts,
                                       float *ppart, int *status, int *fin_ticket, int32_t *chunk_hist,
                                       cudaStream_t s)
{
    if (E != 256)
        return cudaErrorInvalidValue;
    if (!ppart && k <= 8) {
        // four threads per token, 32 tokens (two bucketing chunks) per block
        const int blocks = (T + 31) / 32;
        const int nchunk_perm = (T + PERM_CHUNK - 1) / PERM_CHUNK;
        const cudaError_t le = launch_pdl(route_select_quad_kernel<8, 4>, dim3(blocks), dim3(128), 0, s, scores,
                                          gscore, bias, T, k, rsf, eps, idx, w, counts, status, chunk_hist,
                                          nchunk_perm);
        if (le != cudaSuccess)
            return le;
        return cudaPeekAtLastError();
    }
    const int chunk = route_chunk_hist(T);          // whole bucketing chunks per block
    const int blocks = (T + chunk - 1) / chunk;
    const int nchunk_perm = (T + PERM_CHUNK - 1) / PERM_CHUNK;
    const cudaError_t le = launch_pdl(route_select_scored_kernel<8, 4>, dim3(blocks), dim3(256), 0, s, scores,
                                      gscore, bias, T, chunk, k, rsf, eps, idx, w, counts, ppart, status, fin_ticket,
                                      chunk_hist, nchunk_perm);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

cudaError_t launch_route_select(const float *logits, int nparts, long long part_stride, const float *bias, int T,
                                int E, int n_group, int topk_group, int k, float rsf, float eps, int32_t *idx,
                                float *w, int32_t *counts, float *ppart, int *status, int *fin_ticket,
                                cudaStream_t s)
{
    const int chunk = route_chunk(T);
    const int blocks = (T + chunk - 1) / chunk;
#define GLR_ROUTE_CASE(GG)                                                                                   \
    case GG: {                                                                                               \
        const cudaError_t le = launch_pdl(route_select_kernel<GG>, dim3(blocks), dim3(256), 0, s, logits,      \
                                          nparts, part_stride, bias, T, chunk, topk_group, k, rsf, eps, idx, w,  \
                                          counts, ppart, status, fin_ticket);                                    \
        if (le != cudaSuccess)                                                                               \
            return le;                                                                                       \
        break;                                                                                               \
    }
    if (n_group == 8 && topk_group == 4) {
        const cudaError_t le = launch_pdl(route_select_sorted_kernel<8, 4>, dim3(blocks), dim3(256), 0, s, logits,
                                          nparts, part_stride, bias, T, chunk, k, rsf, eps, idx, w, counts, ppart,
                                          status, fin_ticket);
        if (le != cudaSuccess)
            return le;
        return cudaPeekAtLastError();
    }
    switch (n_group) {
        GLR_ROUTE_CASE(1)
        GLR_ROUTE_CASE(2)
        GLR_ROUTE_CASE(3)
        GLR_ROUTE_CASE(4)
        GLR_ROUTE_CASE(5)
        GLR_ROUTE_CASE(6)
        GLR_ROUTE_CASE(7)
        GLR_ROUTE_CASE(8)
    default: return cudaErrorInvalidValue;
    }
#undef GLR_ROUTE_CASE
    (void)E;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// Balance loss (only when asked for): P[e] = sum over chunks of ppart[c][e] / T
// and aux = E * sum_e counts[e] / (k T) * P[e].  Block b adds a fixed run of
// chunk rows (thread e takes expert e, so every row is one coalesced load) and
// stores its partial sums; the last block to finish (a ticket in the
// workspace header, cleared by the routing kernel that runs just before)
// adds the partials in block order in double and forms P and the loss.  Every sum runs in a fixed order,
// so the result is reproducible bit for bit; no block ever waits for another.
constexpr int FIN_BLOCKS = ROUTE_FIN_BLOCKS;

__global__ void __launch_bounds__(256) route_finalize_kernel(const int32_t *__restrict__ counts,
                                                             const float *__restrict__ ppart, int nchunk,
                                                             int rows_per_block, int T, int E, int K,
                                                             float *__restrict__ part, int *__restrict__ ticket,
                                                             float *__restrict__ aux_P, float *__restrict__ aux_loss)
{
    pdl_wait();
    __shared__ int s_last;
    __shared__ double red[8];
    const int e = threadIdx.x;                      // blockDim.x == 256 >= E
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r0 = blockIdx.x * rows_per_block;
    const int r1 = min(nchunk, r0 + rows_per_block);
    if (e < E) {
        float v = 0.0f;
#pragma unroll 8
        for (int r = r0; r < r1; ++r)
            v += ppart[(size_t)r * E + e];
        part[(size_t)blockIdx.x * E + e] = v;
    }
    __threadfence();                                // partials visible before the ticket
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = (atomicAdd(ticket, 1) == (int)gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    double contrib = 0.0;
    if (e < E) {
        double psum = 0.0;
#pragma unroll 8
        for (int b = 0; b < (int)gridDim.x; ++b)
            psum += (double)__ldcg(part + (size_t)b * E + e);
        const double P = psum / (double)T;
        if (aux_P)
            aux_P[e] = (float)P;
        contrib = (double)counts[e] / ((double)K * (double)T) * P;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        contrib += __shfl_xor_sync(0xffffffffu, contrib, off);
    if (lane == 0)
        red[warp] = contrib;
    __syncthreads();
    if (threadIdx.x == 0) {
        if (aux_loss) {
            double a = 0.0;
            for (int w = 0; w < 8; ++w)
                a += red[w];
            *aux_loss = (float)((double)E * a);
        }
        *ticket = 0;                                // ready for the next call on this workspace
    }
}

cudaError_t launch_route_finalize(const int32_t *counts, const float *ppart, int nchunk, int T, int E, int k,
                                  float *part, int *ticket, float *aux_P, float *aux_loss, cudaStream_t s)
{
    if (E > 256 || nchunk < 1)
        return cudaErrorInvalidValue;
    const int rows = (nchunk + FIN_BLOCKS - 1) / FIN_BLOCKS;
    const int blocks = (nchunk + rows - 1) / rows;
    const cudaError_t le = launch_pdl(route_finalize_kernel, dim3(blocks), dim3(256), 0, s, counts, ppart, nchunk,
                                      rows, T, E, k, part, ticket, aux_P, aux_loss);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// Expert-bias feedback and hit tracking (training side of the routing page:
// section 三, cold experts up and hot experts down; section 六, running hit
// totals).  bias[e] += +gamma / -gamma / 0 as counts[e] is below / above /
// at the balanced load k T / E; totals[e] += counts[e].
__global__ void expert_feedback_kernel(const int32_t *__restrict__ counts, int E, double mean, float gamma,
                                       float *__restrict__ bias, long long *__restrict__ totals)
{
    pdl_wait();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E)
        return;
    const int c = counts[e];
    if (totals)
        totals[e] += c;
    if (bias) {
        const float step = ((double)c < mean) ? gamma : (((double)c > mean) ? -gamma : 0.0f);
        bias[e] = bias[e] + step;
    }
}

cudaError_t launch_expert_feedback(const int32_t *counts, int E, int T, int k, float gamma, float *bias,
                                   long long *totals, cudaStream_t s)
{
    const cudaError_t le = launch_pdl(expert_feedback_kernel, dim3((E + 255) / 256), dim3(256), 0, s, counts, E,
                                      (double)k * T / E, gamma, bias, totals);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

}  // namespace glr
