// One token's group-limited top-k selection by one warp (SIMT, sm_103a),
// shared by the routing kernel (route.cu) and the fused router's epilogue
// (gemm.cu), so that both give the same bits.
//
// Routing article "InternLumina-U2中256个专家的路由秘密：分组受限Top-K、Expert
// Bias与Fused MoE详解":
//   section 二 step 1  s = sigmoid(logit);
//   section 三         the choice is made on s + expert_bias;
//   section 二 step 2  group score = the group's two best biased scores, the
//                      TG best groups survive, the K best of their experts win;
//   section 二 step 3  w = s / (sum of the K chosen s + eps) * rsf.
// Lane l holds experts 32 j + l for j < G, so each group lives in one register
// index across the 32 lanes; group maxima and the K arg-max rounds are warp
// reductions (redux) on order-preserving integer keys.  Ties go to the lower
// group and to the lower expert; the K experts come out in order of (biased
// score desc, expert asc), and the normaliser is summed in that order.
#pragma once

#include "kernels.h"

namespace glr {

// L: this lane's logits of experts 32 j + lane; bias_r: their biases.
// Out: s (the scores), and for lane r < K the r-th chosen expert (my_e) and
// its weight (my_w); nonfinite is OR-ed with any non-finite logit or bias.
template <int G>
__device__ __forceinline__ void route_token(const float (&L)[G], const float (&bias_r)[G], int lane, int TG, int K,
                                            float rsf, float eps, float (&s)[G], int &my_e, float &my_w,
                                            bool &nonfinite)
{
    constexpr unsigned FULL = 0xffffffffu;
    float b[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        nonfinite |= !isfinite(L[j]) || !isfinite(bias_r[j]);
        s[j] = router_sigmoid(L[j]);
        b[j] = s[j] + bias_r[j];
    }

    // group score = top-1 + top-2 of the biased scores of the group
    float g[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const uint32_t u = fkey(b[j]);
        const uint32_t m1 = __reduce_max_sync(FULL, u);
        const int first = __ffs(__ballot_sync(FULL, u == m1)) - 1;
        const uint32_t m2 = __reduce_max_sync(FULL, lane == first ? 0u : u);   // best of the others
        g[j] = fkey_value(m1) + fkey_value(m2);
    }

    // keep the TG best groups (ties to the lower group index): lane j < G
    // ranks group j, one ballot collects the verdicts
    float gl = g[0];
#pragma unroll
    for (int j = 1; j < G; ++j)
        if (lane == j)
            gl = g[j];
    int rank = 0;
#pragma unroll
    for (int i = 0; i < G; ++i)
        rank += (g[i] > gl || (g[i] == gl && i < lane)) ? 1 : 0;
    const uint32_t keep = __ballot_sync(FULL, lane < G && rank < TG) & ((1u << G) - 1u);

    // top-K of the surviving experts: K rounds of (max key, then lowest index)
    uint32_t kb[G];
#pragma unroll
    for (int j = 0; j < G; ++j)
        kb[j] = fkey(b[j]);
    uint32_t avail = keep;   // this lane's candidates not yet taken, by group
    float den = 0.0f;
    my_e = -1;
    float my_s = 0.0f;
    for (int r = 0; r < K; ++r) {
        uint32_t bk = 0;
        int bj = -1;
#pragma unroll
        for (int j = 0; j < G; ++j) {
            if (((avail >> j) & 1u) && (bj < 0 || kb[j] > bk)) {   // ascending j: ties keep the lower index
                bk = kb[j];
                bj = j;
            }
        }
        const uint32_t wk = __reduce_max_sync(FULL, bj >= 0 ? bk : 0u);
        const uint32_t we = __reduce_min_sync(FULL, (bj >= 0 && bk == wk) ? (uint32_t)(32 * bj + lane) : 0xffffffffu);
        const int wl = (int)(we & 31u), wj = (int)(we >> 5);
        float sl = 0.0f;
#pragma unroll
        for (int j = 0; j < G; ++j)
            if (j == bj)
                sl = s[j];
        const float sw = __shfl_sync(FULL, sl, wl);   // the winner's unbiased score
        if (lane == wl)
            avail &= ~(1u << wj);
        den += sw;                                    // sequential, in output order
        if (lane == r) {
            my_e = (int)we;
            my_s = sw;
        }
    }
    den += eps;
    my_w = (my_s / den) * rsf;
}

}  // namespace glr
