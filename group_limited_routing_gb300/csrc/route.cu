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
// Ties go to the lower index at both levels; the k experts come out in order of
// (biased score desc, index asc).  Everything is deterministic: per-block
// histograms and score sums are reduced in a fixed order, never with float
// atomics.
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.h"

namespace glr {

// ---------------------------------------------------------------------------
// W (fp32) -> hi, mid, lo (bf16) with hi + mid + lo == W exactly for normal
// values: each part is the bf16 rounding of what the previous parts left.
// Layout of W3: [3][E][H].
__global__ void split_router_kernel(const float *__restrict__ W, uint16_t *__restrict__ W3, int n)
{
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

cudaError_t launch_split_router(const float *W, uint16_t *W3, int E, int H, cudaStream_t s)
{
    const int n = E * H;
    const int blocks = min((n + 255) / 256, 4096);
    split_router_kernel<<<blocks, 256, 0, s>>>(W, W3, n);
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// (value desc, index asc) ordering with an explicit "no candidate" state
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib)
{
    return ib < 0 || (ia >= 0 && (va > vb || (va == vb && ia < ib)));
}

// One warp per token.  Lane l holds experts 32*j + l for j < n_group, so each
// group lives in one register index across the 32 lanes, and every load of a
// logits row is a run of 128-byte coalesced accesses.
//
// Block: 8 warps, ROUTE_CHUNK tokens; writes its per-expert hit histogram and
// (optionally) per-expert sums of the token-normalised scores for the chunk.
template <int G>
__global__ void __launch_bounds__(256) route_select_kernel(
    const float *__restrict__ logits, const float *__restrict__ bias, int T, int TG, int K, float rsf, float eps,
    int32_t *__restrict__ idx_out, float *__restrict__ w_out, int32_t *__restrict__ hist, float *__restrict__ ppart,
    int *__restrict__ status)
{
    constexpr int E = 32 * G;
    __shared__ int sh_hist[E];
    __shared__ float sh_p[8][E];

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
    const int t0 = blockIdx.x * ROUTE_CHUNK;
    const int t1 = min(T, t0 + ROUTE_CHUNK);
    for (int t = t0 + warp; t < t1; t += 8) {
        const float *row = logits + (size_t)t * E;
        float s[G], b[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float L = __ldg(row + 32 * j + lane);
            nonfinite |= !isfinite(L) || !isfinite(bias_r[j]);
            s[j] = 1.0f / (1.0f + expf(-L));          // section 二 step 1
            b[j] = s[j] + bias_r[j];                  // section 三: choose on s + bias
        }

        // group score = top-1 + top-2 of the biased scores of the group
        float g[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float m1 = b[j], m2 = -INFINITY;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float o1 = __shfl_xor_sync(0xffffffffu, m1, off);
                const float o2 = __shfl_xor_sync(0xffffffffu, m2, off);
                const float hi = fmaxf(m1, o1), lo = fminf(m1, o1);
                m2 = fmaxf(lo, fmaxf(m2, o2));
                m1 = hi;
            }
            g[j] = m1 + m2;
        }

        // keep the TG best groups (ties to the lower group index)
        uint32_t keep = 0;
#pragma unroll
        for (int j = 0; j < G; ++j) {
            int rank = 0;
#pragma unroll
            for (int i = 0; i < G; ++i)
                rank += (g[i] > g[j] || (g[i] == g[j] && i < j)) ? 1 : 0;
            keep |= (rank < TG ? 1u : 0u) << j;
        }

        // top-K of the surviving experts, K rounds of warp arg-max
        uint32_t taken = 0;
        float den = 0.0f;
        int my_e = -1;
        float my_s = 0.0f;
        for (int r = 0; r < K; ++r) {
            float bv = -INFINITY;
            int be = -1;
#pragma unroll
            for (int j = 0; j < G; ++j)
                if (((keep >> j) & 1u) && !((taken >> j) & 1u) && better(b[j], 32 * j + lane, bv, be)) {
                    bv = b[j];
                    be = 32 * j + lane;
                }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (better(ov, oe, bv, be)) {
                    bv = ov;
                    be = oe;
                }
            }
            // every lane now holds the same winner be (>= 0: 32*TG >= K survivors)
            const int wj = be >> 5, wl = be & 31;
            float sw = 0.0f;
#pragma unroll
            for (int j = 0; j < G; ++j)
                if (j == wj)
                    sw = s[j];
            sw = __shfl_sync(0xffffffffu, sw, wl);
            if (lane == wl)
                taken |= 1u << wj;
            den += sw;                                // sequential, in output order
            if (lane == r) {
                my_e = be;
                my_s = sw;
            }
        }
        den += eps;
        if (lane < K) {
            idx_out[(size_t)t * K + lane] = my_e;
            w_out[(size_t)t * K + lane] = (my_s / den) * rsf;   // section 二 step 3
            atomicAdd(&sh_hist[my_e], 1);                       // integer: order-free
        }

        if (ppart) {
            float tot = 0.0f;
#pragma unroll
            for (int j = 0; j < G; ++j)
                tot += s[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                tot += __shfl_xor_sync(0xffffffffu, tot, off);
            const float inv = 1.0f / tot;
#pragma unroll
            for (int j = 0; j < G; ++j)
                pacc[j] += s[j] * inv;
        }
    }
    if (__any_sync(0xffffffffu, nonfinite) && lane == 0)
        atomicOr(status, ST_NONFINITE);

    if (ppart) {
#pragma unroll
        for (int j = 0; j < G; ++j)
            sh_p[warp][32 * j + lane] = pacc[j];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        hist[(size_t)blockIdx.x * E + e] = sh_hist[e];
        if (ppart) {
            float v = 0.0f;
            for (int q = 0; q < 8; ++q)
                v += sh_p[q][e];
            ppart[(size_t)blockIdx.x * E + e] = v;
        }
    }
}

cudaError_t launch_route_select(const float *logits, const float *bias, int T, int E, int n_group, int topk_group,
                                int k, float rsf, float eps, int32_t *idx, float *w, int32_t *hist, float *ppart,
                                int *status, cudaStream_t s)
{
    const int blocks = (T + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
#define GLR_ROUTE_CASE(GG)                                                                                  \
    case GG:                                                                                                \
        route_select_kernel<GG><<<blocks, 256, 0, s>>>(logits, bias, T, topk_group, k, rsf, eps, idx, w,   \
                                                       hist, ppart, status);                                \
        break;
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
// counts[e] = sum over chunks of hist[c][e]; P[e] = sum of ppart[c][e] / T;
// aux = E * sum_e counts[e] / (k T) * P[e].  One block of 1024 threads: four
// threads per expert each take a fixed quarter of the chunks; all sums run
// in a fixed order, so the result is reproducible bit for bit.
__global__ void __launch_bounds__(1024) route_finalize_kernel(const int32_t *__restrict__ hist,
                                                              const float *__restrict__ ppart, int nchunk, int T,
                                                              int E, int K, int32_t *__restrict__ counts,
                                                              float *__restrict__ aux_P, float *__restrict__ aux_loss)
{
    __shared__ long long sc[4][256];
    __shared__ double sp[4][256];
    __shared__ double red[1024];
    const int e = threadIdx.x & 255, q = threadIdx.x >> 8;
    long long c = 0;
    double pv = 0.0;
    if (e < E) {
        for (int ch = q; ch < nchunk; ch += 4) {
            c += hist[(size_t)ch * E + e];
            if (ppart)
                pv += (double)ppart[(size_t)ch * E + e];
        }
    }
    sc[q][e] = c;
    sp[q][e] = pv;
    __syncthreads();
    double contrib = 0.0;
    if (q == 0 && e < E) {
        const long long tot = sc[0][e] + sc[1][e] + sc[2][e] + sc[3][e];
        counts[e] = (int32_t)tot;
        const double P = (sp[0][e] + sp[1][e] + sp[2][e] + sp[3][e]) / (double)T;
        if (aux_P)
            aux_P[e] = (float)P;
        contrib = (double)tot / ((double)K * (double)T) * P;
    }
    red[threadIdx.x] = contrib;
    __syncthreads();
    for (int off = 512; off > 0; off >>= 1) {
        if (threadIdx.x < off)
            red[threadIdx.x] += red[threadIdx.x + off];
        __syncthreads();
    }
    if (threadIdx.x == 0 && aux_loss)
        *aux_loss = (float)((double)E * red[0]);
}

cudaError_t launch_route_finalize(const int32_t *hist, const float *ppart, int nchunk, int T, int E, int k,
                                  int32_t *counts, float *aux_P, float *aux_loss, cudaStream_t s)
{
    route_finalize_kernel<<<1, 1024, 0, s>>>(hist, ppart, nchunk, T, E, k, counts, aux_P, aux_loss);
    return cudaPeekAtLastError();
}

}  // namespace glr
