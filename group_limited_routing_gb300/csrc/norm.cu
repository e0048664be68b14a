// Pre-norm of a decoder layer for stacking MoE layers: out[t] = bf16( x[t] /
// sqrt(mean_h x[t,h]^2 + eps) ), unit weight, fp32 arithmetic.  The routing
// article ("InternLumina-U2中256个专家的路由秘密…", §五) builds its MoE blocks
// into decoder layers but does not describe their norm; an RMS norm in front
// of the MoE block with a residual around it is the usual decoder layer and
// keeps a 19-layer stack of random-weight layers finite.
#include <cuda_bf16.h>

#include "kernels.h"

namespace glr {

// One warp per token row; H % 8 == 0 (16-byte vectors).
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ out,
                                                      int T, int H, float eps)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= T)
        return;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)row * H);
    uint4 *orow = reinterpret_cast<uint4 *>(out + (size_t)row * H);
    const int nv = H / 8;
    float ss = 0.0f;
    for (int v = lane; v < nv; v += 32) {
        const uint4 q = xr[v];
        const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(p2[i]);
            ss += f.x * f.x + f.y * f.y;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = 1.0f / sqrtf(ss / (float)H + eps);
    for (int v = lane; v < nv; v += 32) {
        const uint4 q = xr[v];
        const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&q);
        uint4 o;
        uint32_t *op = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(p2[i]);
            __nv_bfloat162 b = __floats2bfloat162_rn(f.x * inv, f.y * inv);
            op[i] = *reinterpret_cast<uint32_t *>(&b);
        }
        orow[v] = o;
    }
}

cudaError_t launch_rmsnorm(const uint16_t *x, uint16_t *out, int T, int H, float eps, cudaStream_t s)
{
    const int blocks = (T + 7) / 8;
    const cudaError_t le = launch_pdl(rmsnorm_kernel, dim3(blocks), dim3(256), 0, s, x, out, T, H, eps);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

}  // namespace glr
