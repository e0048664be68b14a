// Tensor-core GEMMs of the MoE layer forward on sm_103a (tcgen05 + TMEM + TMA).
//
// One persistent, warp-specialised kernel template serves three products:
//   GK_ROUTER   logits[T, E] = hidden[T, H] . W^T in fp32 accuracy: W (fp32)
//               is pre-split into hi + mid + lo bf16 parts, every product of a
//               bf16 hidden value with a bf16 part is exact, and the three
//               MMAs accumulate into one fp32 TMEM accumulator.  (Routing
//               article "InternLumina-U2中256个专家的路由秘密…", section 二 step 1:
//               the router linear layer runs in fp32.)
//   GK_GATE_UP  per expert bucket: G = X_e . Wgate^T, U = X_e . Wup^T, written
//               as bf16( silu(G) * U )  (section 四: SwiGLU experts stacked as
//               3D weights; the shared expert of section 五 is the last group).
//   GK_DOWN     per expert bucket: Y = intermediate_e . W_down[e], W_down
//               stacked [E, I, H] as on the page (an MN-major B operand).
//
// Roles (192 threads, one CTA per SM):
//   warp 0, one lane : TMA producer, fills a STAGES-deep ring of smem stages
//   warp 1           : allocates TMEM; one lane issues tcgen05.mma and commits
//   warps 2..5       : epilogue, TMEM -> registers -> global; warp w reads TMEM
//                      lanes 32*(w%4) .. +31 (the lane quadrant it may access)
// Two TMEM accumulators let the epilogue of one tile overlap the MMAs of the
// next.  Tiles are 128 rows x BN columns; CTAs walk the tile list round-robin.
//
// Every wait is bounded (see ptx.cuh).  When one runs out the CTA sets an
// abort flag, every role leaves its loop, the producer waits (bounded) for its
// TMA copies in flight, the MMA lane drains its MMAs, TMEM is freed and the
// status word gets MOE_STATUS_TIMEOUT.  Nothing traps.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace glr {

template <int KIND>
struct GemmCfg;

template <>
struct GemmCfg<GK_ROUTER> {
    static constexpr int BN = 128;                     // experts per tile
    static constexpr int NB = 3;                       // W parts: hi, mid, lo
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_PART = BN * GEMM_BK * 2;    // 16 KB per part
    static constexpr int B_BYTES = NB * B_PART;
    static constexpr int STAGES = 3;
    static constexpr int TMEM_COLS = 256;              // 2 accumulators x 128
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, false, false);
};

template <>
struct GemmCfg<GK_GATE_UP> {
    static constexpr int BN = 256;                     // 128 gate + 128 up columns
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_HALF = 128 * GEMM_BK * 2;   // 16 KB
    static constexpr int B_BYTES = BN * GEMM_BK * 2;
    static constexpr int STAGES = 4;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, false, false);
};

template <>
struct GemmCfg<GK_DOWN> {
    static constexpr int BN = 256;                     // hidden columns per tile
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_ATOM = 64 * GEMM_BK * 2;    // 64 N x 64 K box, 8 KB
    static constexpr int B_BYTES = BN * GEMM_BK * 2;
    static constexpr int STAGES = 4;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, false, true);
};

template <int KIND>
struct GemmLayout {
    using C = GemmCfg<KIND>;
    static constexpr int STAGE_BYTES = C::A_BYTES + C::B_BYTES;
    static constexpr int NBARS = 2 * C::STAGES + 5;    // full, empty, tfull x2, tempty x2, fin
    static constexpr int SMEM = C::STAGES * STAGE_BYTES + 1024 /*align*/ + NBARS * 8 + 16;
};

struct TileInfo {
    int group;    // expert id, E for the shared expert
    int a_row;    // first A row (TMA coordinate)
    int out_row;  // first output row
    int rows;     // valid rows (<= 128)
    int nt;       // n-tile index
    int shared;
};

template <int KIND>
__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, int tile)
{
    TileInfo ti;
    ti.nt = tile % p.n_tiles;
    if (KIND == GK_ROUTER) {
        ti.a_row = (tile / p.n_tiles) * GEMM_BM;
        ti.out_row = ti.a_row;
        ti.rows = min(GEMM_BM, p.T - ti.a_row);
        ti.group = 0;
        ti.shared = 0;
    } else {
        const int4 m = p.mtiles[tile / p.n_tiles];
        ti.group = m.x;
        ti.shared = (m.x == p.E);
        ti.rows = m.z;
        if (KIND == GK_GATE_UP) {
            ti.a_row = m.y;                               // X_perm slot, or token for the shared expert
            ti.out_row = ti.shared ? p.kT + m.y : m.y;
        } else {
            ti.a_row = ti.shared ? p.kT + m.y : m.y;      // intermediate rows
            ti.out_row = ti.a_row;
        }
    }
    return ti;
}

template <int KIND>
__device__ __forceinline__ void issue_loads(const GemmParams &p, const TileInfo &ti, int kb, uint32_t sA,
                                            uint32_t sB, uint32_t bar)
{
    using C = GemmCfg<KIND>;
    const int k0 = kb * GEMM_BK;
    if (KIND == GK_ROUTER) {
        tma_load_2d(sA, &p.tmA0, bar, k0, ti.a_row);
#pragma unroll
        for (int s = 0; s < 3; ++s)
            tma_load_2d(sB + s * GemmCfg<GK_ROUTER>::B_PART, &p.tmB0, bar, k0, s * p.E + ti.nt * C::BN);
    } else if (KIND == GK_GATE_UP) {
        const CUtensorMap *ma = ti.shared ? &p.tmA1 : &p.tmA0;
        const CUtensorMap *mb = ti.shared ? &p.tmB1 : &p.tmB0;
        const int wrow = (ti.shared ? 0 : ti.group * 2 * p.I) + ti.nt * 128;
        tma_load_2d(sA, ma, bar, k0, ti.a_row);
        tma_load_2d(sB, mb, bar, k0, wrow);                                      // gate rows
        tma_load_2d(sB + GemmCfg<GK_GATE_UP>::B_HALF, mb, bar, k0, wrow + p.I);  // up rows
    } else {
        const CUtensorMap *mb = ti.shared ? &p.tmB1 : &p.tmB0;
        const int krow = (ti.shared ? 0 : ti.group * p.I) + k0;
        tma_load_2d(sA, &p.tmA0, bar, k0, ti.a_row);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            tma_load_2d(sB + q * GemmCfg<GK_DOWN>::B_ATOM, mb, bar, ti.nt * C::BN + q * 64, krow);
    }
}

template <int KIND>
__device__ __forceinline__ void issue_mmas(uint32_t sA, uint32_t sB, uint32_t d, bool acc_in)
{
    using C = GemmCfg<KIND>;
#pragma unroll
    for (int kk = 0; kk < GEMM_BK / 16; ++kk) {
        const uint64_t ad = sdesc_kmajor_sw128(sA + kk * 32);
        if (KIND == GK_ROUTER) {
#pragma unroll
            for (int s = 0; s < 3; ++s)
                umma_bf16(d, ad, sdesc_kmajor_sw128(sB + s * GemmCfg<GK_ROUTER>::B_PART + kk * 32), C::IDESC,
                          (acc_in || kk > 0 || s > 0) ? 1u : 0u);
        } else if (KIND == GK_GATE_UP) {
            umma_bf16(d, ad, sdesc_kmajor_sw128(sB + kk * 32), C::IDESC, (acc_in || kk > 0) ? 1u : 0u);
        } else {
            // 16 K rows = two 8-row atoms = 2048 B further into each 64-wide N atom
            umma_bf16(d, ad, sdesc_mnmajor_sw128(sB + kk * 2048, GemmCfg<GK_DOWN>::B_ATOM), C::IDESC,
                      (acc_in || kk > 0) ? 1u : 0u);
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float silu_times(float g, float u)
{
    return g / (1.0f + __expf(-g)) * u;
}

// Epilogue of one tile for the thread that owns accumulator row `row`.
template <int KIND>
__device__ __forceinline__ void epilogue_tile(const GemmParams &p, const TileInfo &ti, uint32_t tacc, int row)
{
    const bool valid = row < ti.rows;
    if (KIND == GK_ROUTER) {
        float *dst = static_cast<float *>(p.out) + (size_t)(ti.out_row + row) * p.ld_out + ti.nt * 128;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
            uint32_t r[32];
            tmem_load32(tacc + c, r);
            if (valid) {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    d4[q] = make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
            }
        }
    } else if (KIND == GK_GATE_UP) {
        uint16_t *dst = static_cast<uint16_t *>(p.out) + (size_t)(ti.out_row + row) * p.ld_out + ti.nt * 128;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
            uint32_t g[32], u[32];
            tmem_load32(tacc + c, g);
            tmem_load32(tacc + 128 + c, u);
            if (valid) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(silu_times(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                                        silu_times(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1])));
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        }
    } else {
        uint16_t *dst = static_cast<uint16_t *>(p.out) + (size_t)(ti.out_row + row) * p.ld_out + ti.nt * 256;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
            uint32_t r[32];
            tmem_load32(tacc + c, r);
            if (valid) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        }
    }
}

template <int KIND>
__global__ void __launch_bounds__(GEMM_THREADS, 1) umma_gemm_kernel(const __grid_constant__ GemmParams p)
{
    using C = GemmCfg<KIND>;
    using L = GemmLayout<KIND>;
    extern __shared__ uint8_t dsmem[];

    const uint32_t raw = smem_u32(dsmem);
    const uint32_t base = (raw + 1023u) & ~1023u;                 // swizzle atoms need 1024-B alignment
    uint8_t *base_ptr = dsmem + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base_ptr + C::STAGES * L::STAGE_BYTES);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + L::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    const uint32_t fin_bar = bar0 + 8u * (2 * C::STAGES + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4);
        }
        mbar_init(fin_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&p.tmA0);
        tma_prefetch_map(&p.tmB0);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    const int num_tiles = (KIND == GK_ROUTER) ? p.num_tiles_static : (*p.num_mtiles) * p.n_tiles;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const TileInfo ti = tile_info<KIND>(p, tile);
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = base + stage * L::STAGE_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), L::STAGE_BYTES);
                    issue_loads<KIND>(p, ti, kb, sA, sA + C::A_BYTES, full_bar(stage));
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let the copies in flight land before the CTA's smem goes away
                for (int s = 0; s < C::STAGES; ++s)
                    if ((issued >> s) & 1u)
                        mbar_drain(full_bar(s), (issued_parity >> s) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + acc * C::BN;
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = base + stage * L::STAGE_BYTES;
                    issue_mmas<KIND>(sA, sA + C::A_BYTES, d, kb > 0);
                    umma_commit(empty_bar(stage));   // frees the stage once these MMAs have read it
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok)
                    umma_commit(tfull_bar(acc));     // accumulator ready for the epilogue
            }
            // no MMA may still be writing TMEM when it is freed
            umma_commit(fin_bar);
            mbar_drain(fin_bar, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            __syncwarp();
            tc_fence_after();
            const TileInfo ti = tile_info<KIND>(p, tile);
            const uint32_t tacc = tmem + ((uint32_t)(quad * 32) << 16) + acc * C::BN;
            epilogue_tile<KIND>(p, ti, tacc, row);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(tempty_bar(acc));
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(p.status, ST_TIMEOUT);
}

int gemm_smem_bytes(int kind)
{
    switch (kind) {
    case GK_ROUTER: return GemmLayout<GK_ROUTER>::SMEM;
    case GK_GATE_UP: return GemmLayout<GK_GATE_UP>::SMEM;
    default: return GemmLayout<GK_DOWN>::SMEM;
    }
}

int gemm_tmem_cols(int kind)
{
    switch (kind) {
    case GK_ROUTER: return GemmCfg<GK_ROUTER>::TMEM_COLS;
    case GK_GATE_UP: return GemmCfg<GK_GATE_UP>::TMEM_COLS;
    default: return GemmCfg<GK_DOWN>::TMEM_COLS;
    }
}

template <int KIND>
static cudaError_t launch_kind(const GemmParams &p, int grid, cudaStream_t s)
{
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(umma_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             GemmLayout<KIND>::SMEM);
        if (e != cudaSuccess)
            return e;
        configured_device = dev;
    }
    umma_gemm_kernel<KIND><<<grid, GEMM_THREADS, GemmLayout<KIND>::SMEM, s>>>(p);
    return cudaPeekAtLastError();
}

cudaError_t launch_gemm(int kind, const GemmParams &p, int grid, cudaStream_t s)
{
    switch (kind) {
    case GK_ROUTER: return launch_kind<GK_ROUTER>(p, grid, s);
    case GK_GATE_UP: return launch_kind<GK_GATE_UP>(p, grid, s);
    default: return launch_kind<GK_DOWN>(p, grid, s);
    }
}

}  // namespace glr
