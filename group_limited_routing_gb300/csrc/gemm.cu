// Tensor-core GEMMs of the MoE layer forward on sm_103a (tcgen05 + TMEM + TMA).
//
// One persistent, warp-specialised kernel template serves three products:
//   GK_ROUTER   logits[T, E] = hidden[T, H] . W^T to fp32 accuracy.  (Routing
//               article "InternLumina-U2中256个专家的路由秘密…", section 二 step 1:
//               the router linear layer runs in fp32.)  W (fp32) is pre-split
//               into hi + mid + lo bf16 parts, so every product of a bf16
//               hidden value with a part is exact.  Each 64-wide K block is
//               summed on the tensor core into a fresh TMEM slot (12 MMAs) and
//               the epilogue warps add the K-block partial sums in fp32 with
//               round-to-nearest: the tensor core's own accumulation never
//               runs over more than one K block.
//   GK_GATE_UP  per expert bucket: G = X_e . Wgate^T, U = X_e . Wup^T, written
//               as bf16( silu(G) * U )  (section 四: SwiGLU experts stacked as
//               3D weights; the shared expert of section 五 is the last group).
//   GK_DOWN     per expert bucket: Y = intermediate_e . W_down[e], W_down
//               stacked [E, I, H] as on the page (an MN-major B operand).
//   GK_*_SMALL  the two grouped products for T <= GEMM_SMALL_T (decode): 16 A
//               rows per stage and a 6-deep ring of weight tiles.
//   GK_ROUTER_WIDE  the router with all 256 experts of a token tile in one
//               N = 256 MMA (half the shared-memory operand traffic per flop
//               of the 128-expert tiles), two TMEM K-block slots and eight
//               epilogue warps (two per TMEM lane quadrant, 128 columns each).
//   GK_ROUTER_FUSED  GK_ROUTER_WIDE that also routes and buckets the tokens
//               (section 二 steps 1-3, section 三, section 四's bucketing):
//               after its own tiles a CTA takes finished tiles from a queue,
//               selects their tokens' experts, claims the pairs' rows in the
//               experts' buckets with one integer atomic per expert and tile,
//               and copies the hidden rows there -- so the HBM-bound copies of
//               CTAs with fewer tiles overlap the MMAs of the others.
// The grouped kinds also serve the dense first-layer MLP (one weight group).
//
// Every kernel starts with griddepcontrol.wait (programmatic dependent
// launch): its prologue (barriers, TMEM, descriptor prefetch) overlaps the
// previous kernel's teardown, and nothing global is read before the wait.
//
// Roles (192 threads, 320 for the 256-expert routers; one CTA per SM):
//   warp 0, one lane : TMA producer, fills a STAGES-deep ring of smem stages
//                      (the fused router: then the copy engine of the rows)
//   warp 1           : allocates TMEM; one lane issues tcgen05.mma and commits
//   warps 2..5 (..9) : epilogue, TMEM -> registers -> global; warp w reads TMEM
//                      lanes 32*(w%4) .. +31 (the lane quadrant it may access)
//                      (the fused router: then the routing of queued tiles)
// TMEM holds SLOTS accumulators: two whole-tile accumulators for the grouped
// GEMMs (the epilogue of one tile overlaps the MMAs of the next), four K-block
// slots for the router.  Tiles are 128 rows x BN columns; CTAs walk the tile
// list round-robin.
//
// Every wait is bounded (see ptx.cuh).  When one runs out the CTA sets an
// abort flag, every role leaves its loop, the producer waits (bounded) for its
// TMA copies in flight, the MMA lane drains its MMAs, TMEM is freed and the
// status word gets MOE_STATUS_TIMEOUT.  Nothing traps.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"
#include "route_token.cuh"

namespace glr {

template <int KIND>
struct GemmCfg;

// the product a kind computes (the _SMALL kinds differ only in staging)
__host__ __device__ constexpr int base_kind(int kind)
{
    return (kind == GK_GATE_UP_SMALL || kind == GK_GATE_UP_BWD) ? GK_GATE_UP
           : (kind == GK_DOWN_SMALL || kind == GK_DOWN_COMBINE)  ? GK_DOWN
           : (kind == GK_ROUTER_WIDE || kind == GK_ROUTER_FUSED) ? GK_ROUTER
                                                                : kind;
}

__host__ __device__ constexpr bool wide_router(int kind) { return kind == GK_ROUTER_WIDE || kind == GK_ROUTER_FUSED; }

// K blocks of hidden the wide router prefetches into L2 ahead of its loads
constexpr int ROUTER_PF = 6;

// K blocks (of 64) the router's tensor core sums into one TMEM slot before the
// epilogue adds the slot to its fp32 running sums (48 MMAs per slot: the
// tensor core's own accumulation stays short enough for the logits to stay
// within the fp32-accuracy bound the tests hold them to, and the promotion
// round trip is paid once per 256 K)
constexpr int ROUTER_KPS = 4;

// epilogue warps of a kind (the block is 64 + 32 x this threads)
__host__ __device__ constexpr int epi_warps(int kind)
{
    return (wide_router(kind) || kind == GK_DOWN_COMBINE) ? 8 : 4;
}
__host__ __device__ constexpr int kind_threads(int kind) { return 64 + 32 * epi_warps(kind); }

// the fused router's extra barriers: the epilogue warps' meeting, the logits'
// staging load, the two row tables' full and empty, the copy engine's slots
constexpr int FUSED_ENGINE_SLOTS = 16;                  // rows in flight in the copy engine at most
constexpr int FUSED_BARS = 1 + 1 + 2 + 2 + FUSED_ENGINE_SLOTS;

template <>
struct GemmCfg<GK_ROUTER> {
    static constexpr int BN = 128;                     // experts per tile
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_PART = BN * GEMM_BK * 2;    // 16 KB per W part
    static constexpr int B_BYTES = 3 * B_PART;         // hi, mid, lo
    static constexpr int STAGES = 3;
    static constexpr int SLOTS = 4;                    // one slot per K block in flight
    static constexpr int TMEM_COLS = SLOTS * BN;       // 512
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, false, false);
    static constexpr int A_ROWS = GEMM_BM;
    static constexpr int NBUF = 1;
};

// 128 tokens x all 256 experts per tile: a stage holds 16 KB of hidden and
// 3 x 32 KB of W parts, so only two fit; no staging buffers (the epilogue
// writes each thread's 512 contiguous bytes of logits directly).
template <>
struct GemmCfg<GK_ROUTER_WIDE> {
    static constexpr int BN = 256;
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_PART = BN * GEMM_BK * 2;    // 32 KB per W part
    static constexpr int B_BYTES = 3 * B_PART;
    static constexpr int STAGES = 2;
    static constexpr int SLOTS = 2;
    static constexpr int TMEM_COLS = SLOTS * BN;       // 512
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, false, false);
    static constexpr int A_ROWS = GEMM_BM;
    static constexpr int NBUF = 0;
};

template <>
struct GemmCfg<GK_ROUTER_FUSED> : GemmCfg<GK_ROUTER_WIDE> {};

template <>
struct GemmCfg<GK_GATE_UP> {
    static constexpr int BN = 256;                     // 128 gate + 128 up columns
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_HALF = 128 * GEMM_BK * 2;   // 16 KB
    static constexpr int B_BYTES = BN * GEMM_BK * 2;
    static constexpr int STAGES = 4;
    static constexpr int SLOTS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, false, false);
    static constexpr int A_ROWS = GEMM_BM;             // A rows loaded per stage
    static constexpr int NBUF = 2;                     // staging buffers per epilogue warp
};

template <>
struct GemmCfg<GK_DOWN> {
    static constexpr int BN = 256;                     // hidden columns per tile
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_ATOM = 64 * GEMM_BK * 2;    // 64 N x 64 K box, 8 KB
    static constexpr int B_BYTES = BN * GEMM_BK * 2;
    static constexpr int STAGES = 4;
    static constexpr int SLOTS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, false, true);
    static constexpr int A_ROWS = GEMM_BM;
    static constexpr int NBUF = 2;
};

// The shared expert's down GEMM with the combine in its epilogue: the down
// GEMM's operands, three stages, and 64 KB of staging for the tile's output
// rows in token-major order (128 rows x 512 B).
template <>
struct GemmCfg<GK_DOWN_COMBINE> : GemmCfg<GK_DOWN> {
    static constexpr int STAGES = 3;
    static constexpr int NBUF = 4;
};

// Small-T kinds: only GEMM_SMALL_T A rows per stage (2 KB); the MMA still
// reads 128 rows, the rest alias the stage's B bytes and only feed
// accumulator rows that are never stored.  Six stages of 34 KB keep 192 KB of
// weights in flight per SM instead of 128 KB (decode streams the hit experts'
// weights and nothing else); one staging buffer per epilogue warp, since at
// most one warp has rows to store.
template <int BASE>
struct GemmCfgSmall : GemmCfg<BASE> {
    static constexpr int A_ROWS = GEMM_SMALL_T;
    static constexpr int A_BYTES = A_ROWS * GEMM_BK * 2;
    static constexpr int STAGES = 6;
    static constexpr int NBUF = 1;
};

template <>
struct GemmCfg<GK_GATE_UP_SMALL> : GemmCfgSmall<GK_GATE_UP> {};

// Backward: the gate/up products again, with an epilogue that keeps G and U.
template <>
struct GemmCfg<GK_GATE_UP_BWD> : GemmCfg<GK_GATE_UP> {};

// Backward: d(intermediate) = dOut_perm [rows, H] . W_down[e]^T, W_down[e]
// read as [I, H] rows (K-major, 256 of the I columns per tile).
template <>
struct GemmCfg<GK_DGRAD_DOWN> {
    static constexpr int BN = 256;
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_HALF = 128 * GEMM_BK * 2;
    static constexpr int B_BYTES = BN * GEMM_BK * 2;
    static constexpr int STAGES = 4;
    static constexpr int SLOTS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, false, false);
    static constexpr int A_ROWS = GEMM_BM;
    static constexpr int NBUF = 2;
};

// Backward: weight gradient of one expert, [128 features] x [256 hidden]
// per tile, K = the expert's (64-row padded) bucket rows; A and B MN-major.
template <>
struct GemmCfg<GK_WGRAD> {
    static constexpr int BN = 256;
    static constexpr int ATOM = 64 * GEMM_BK * 2;      // 64 columns x 64 rows, 8 KB
    static constexpr int A_BYTES = 2 * ATOM;
    static constexpr int B_BYTES = 4 * ATOM;
    static constexpr int STAGES = 4;
    static constexpr int SLOTS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(GEMM_BM, BN, true, true);
    static constexpr int A_ROWS = GEMM_BM;
    static constexpr int NBUF = 1;
};

template <>
struct GemmCfg<GK_DOWN_SMALL> : GemmCfgSmall<GK_DOWN> {};

// Run-time tile order: the producer lane claims tiles from a global counter
// and passes each index through a ring of TQ_RING shared-memory entries to the
// MMA lane and the four epilogue warps (TQ_TAKERS arrivals free an entry);
// -1 ends every role's loop.
constexpr int TQ_RING = 8;
constexpr int TQ_TAKERS = 5;

template <int KIND>
struct GemmLayout {
    using C = GemmCfg<KIND>;
    static constexpr int STAGE_BYTES = C::A_BYTES + C::B_BYTES;
    // per epilogue warp, 32 rows x 128 B: one buffer for the router, two for
    // the grouped GEMMs (a TMA store can drain one while the other is filled)
    static constexpr int STAGING = C::NBUF * 4 * 4096;
    // tiles claimed at run time (weight gradients: a tile's K is its expert's
    // bucket, from a few rows to the shared expert's T, so a fixed
    // round-robin leaves some SMs with far more work than others)
    static constexpr bool DYN = (KIND == GK_WGRAD);
    static constexpr int TQ = DYN ? TQ_RING : 0;
    // the fused router's epilogue barrier and per-tile bucket histogram
    static constexpr bool FUSED = (KIND == GK_ROUTER_FUSED);
    static constexpr int HIST = FUSED ? 256 * 4 + 16 + 16 : 0;   // histogram, queue slot, mailbox
    // the router kinds' copy of expert_bias (256 floats at most) for the scored output
    static constexpr int BIAS = (base_kind(KIND) == GK_ROUTER && !FUSED) ? 256 * 4 : 0;
    // full[STAGES], empty[STAGES], tfull[SLOTS], tempty[SLOTS], fin, tq_full[TQ], tq_empty[TQ] (, epi)
    static constexpr int NBARS = 2 * C::STAGES + 2 * C::SLOTS + 1 + 2 * TQ + (FUSED ? FUSED_BARS : 0);
    static constexpr int SMEM = C::STAGES * STAGE_BYTES + STAGING + 1024 /*align*/ + NBARS * 8 + 16 + TQ * 4 + HIST +
                                BIAS;
    static_assert(SMEM <= 232448, "more than 227 KB of shared memory");
    static_assert(C::A_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzle atoms need 1024-B alignment");
};

struct TileInfo {
    int group;    // expert id, E for the shared expert
    int a_row;    // first A row (TMA coordinate)
    int out_row;  // first output row
    int rows;     // valid rows (<= 128)
    int nt;       // n-tile index
    int shared;
    int kblocks;  // K blocks of this tile
    int b_row;    // GK_WGRAD: first B row
    int kp;       // router: K part (its K blocks start at kp * kblocks)
};

template <int KIND>
__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, int tile)
{
    TileInfo ti;
    ti.nt = tile % p.n_tiles;
    ti.kblocks = p.kblocks;
    ti.b_row = 0;
    constexpr int BASE = base_kind(KIND);
    if constexpr (KIND == GK_WGRAD) {
        // tile = (expert, feature block, hidden block); K over the expert's rows
        const int per_e = p.wg_fm * p.wg_fn;
        const int eidx = tile / per_e;
        const int e = (eidx == 0) ? p.E : eidx - 1;      // the shared expert's long tiles first
        const int r = tile % per_e;
        const int2 eo = p.eoff[e];
        ti.group = e;
        ti.shared = (e == p.E);
        ti.nt = r % p.wg_fn;
        ti.rows = 128;
        ti.a_row = eo.x;
        ti.b_row = (ti.shared && p.b_row_shared >= 0) ? p.b_row_shared : eo.x;
        ti.kblocks = eo.y / GEMM_BK;
        ti.out_row = (ti.shared ? 0 : e * p.wg_fm * 128) + (r / p.wg_fn) * 128;   // feature row of the output
        return ti;
    }
    ti.kp = 0;
    if constexpr (KIND == GK_DOWN_COMBINE) {
        // the shared expert's 128-token tiles, n-tiles of one tile adjacent
        const int m = tile / p.n_tiles;
        ti.group = p.E;
        ti.shared = 1;
        ti.rows = min(GEMM_BM, p.T - m * GEMM_BM);
        ti.a_row = p.kT + m * GEMM_BM;                  // the shared rows of the intermediate
        ti.out_row = m * GEMM_BM;                       // the tile's first token
        return ti;
    }
    if (BASE == GK_ROUTER) {
        // tile = (token tile * n_tiles + expert tile) * ksplit + K part
        const int ks = p.ksplit > 1 ? p.ksplit : 1;
        ti.kp = tile % ks;
        const int base = tile / ks;
        ti.nt = base % p.n_tiles;
        ti.a_row = (base / p.n_tiles) * GEMM_BM;
        ti.out_row = ti.a_row;
        ti.rows = min(GEMM_BM, p.T - ti.a_row);
        ti.group = 0;
        ti.shared = 0;
    } else {
        const int4 m = p.mtiles[tile / p.n_tiles];
        ti.group = m.x;
        ti.shared = (m.x == p.E);
        ti.rows = m.z;
        if (BASE == GK_GATE_UP) {
            ti.a_row = (p.cap_rows && !ti.shared) ? m.w : m.y;   // X_perm row, or token for the shared expert
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
    constexpr int BASE = base_kind(KIND);
    const int k0 = kb * GEMM_BK;
    if constexpr (KIND == GK_WGRAD) {
        // A: 128 features x 64 rows (two MN-major boxes), B: 256 hidden x 64 rows (four)
        const int f0 = (ti.out_row % (p.wg_fm * 128));
#pragma unroll
        for (int q = 0; q < 2; ++q)
            tma_load_2d(sA + q * C::ATOM, &p.tmA0, bar, f0 + q * 64, ti.a_row + k0);
        const CUtensorMap *mb = ti.shared ? &p.tmB1 : &p.tmB0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            tma_load_2d(sB + q * C::ATOM, mb, bar, ti.nt * C::BN + q * 64, ti.b_row + k0);
    } else if constexpr (KIND == GK_DGRAD_DOWN) {
        // A: dOut_perm rows (K = H); B: 256 rows of W_down[e] read as [I, H]
        const CUtensorMap *mb = ti.shared ? &p.tmB1 : &p.tmB0;
        const int wrow = (ti.shared ? 0 : ti.group * p.I) + ti.nt * C::BN;
        tma_load_2d(sA, &p.tmA0, bar, k0, ti.a_row);
        tma_load_2d(sB, mb, bar, k0, wrow);
        tma_load_2d(sB + C::B_HALF, mb, bar, k0, wrow + 128);
    } else if constexpr (BASE == GK_ROUTER) {
        const int kr = k0 + ti.kp * p.kblocks * GEMM_BK;   // this K part's columns
        tma_load_2d(sA, &p.tmA0, bar, kr, ti.a_row);
#pragma unroll
        for (int s = 0; s < 3; ++s)
            tma_load_2d(sB + s * C::B_PART, &p.tmB0, bar, kr, s * p.E + ti.nt * C::BN);
    } else if constexpr (BASE == GK_GATE_UP) {
        const CUtensorMap *ma = ti.shared ? &p.tmA1 : &p.tmA0;
        const CUtensorMap *mb = ti.shared ? &p.tmB1 : &p.tmB0;
        const int wrow = (ti.shared ? 0 : ti.group * 2 * p.I) + ti.nt * 128;
        tma_load_2d(sA, ma, bar, k0, ti.a_row);
        tma_load_2d(sB, mb, bar, k0, wrow);                    // gate rows
        tma_load_2d(sB + C::B_HALF, mb, bar, k0, wrow + p.I);  // up rows
    } else {
        const CUtensorMap *mb = ti.shared ? &p.tmB1 : &p.tmB0;
        const int krow = (ti.shared ? 0 : ti.group * p.I) + k0;
        tma_load_2d(sA, &p.tmA0, bar, k0, ti.a_row);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            tma_load_2d(sB + q * C::B_ATOM, mb, bar, ti.nt * C::BN + q * 64, krow);
    }
}

// MMAs of one K block (64) into TMEM column base d; `acc_in` = add to what is there.
template <int KIND>
__device__ __forceinline__ void issue_mmas(uint32_t sA, uint32_t sB, uint32_t d, bool acc_in)
{
    using C = GemmCfg<KIND>;
#pragma unroll
    for (int kk = 0; kk < GEMM_BK / 16; ++kk) {
        const uint64_t ad = sdesc_kmajor_sw128(sA + kk * 32);
        constexpr int BASE = base_kind(KIND);
        if constexpr (BASE == GK_ROUTER) {
#pragma unroll
            for (int s = 0; s < 3; ++s)
                umma_bf16(d, ad, sdesc_kmajor_sw128(sB + s * C::B_PART + kk * 32), C::IDESC,
                          (acc_in || kk > 0 || s > 0) ? 1u : 0u);
        } else if constexpr (BASE == GK_GATE_UP || KIND == GK_DGRAD_DOWN) {
            umma_bf16(d, ad, sdesc_kmajor_sw128(sB + kk * 32), C::IDESC, (acc_in || kk > 0) ? 1u : 0u);
        } else if constexpr (KIND == GK_WGRAD) {
            // both operands MN-major: 16 K rows = 2048 B into every 64-column atom
            umma_bf16(d, sdesc_mnmajor_sw128(sA + kk * 2048, C::ATOM), sdesc_mnmajor_sw128(sB + kk * 2048, C::ATOM),
                      C::IDESC, (acc_in || kk > 0) ? 1u : 0u);
        } else {
            // 16 K rows = two 8-row atoms = 2048 B further into each 64-wide N atom
            umma_bf16(d, ad, sdesc_mnmajor_sw128(sB + kk * 2048, C::B_ATOM), C::IDESC,
                      (acc_in || kk > 0) ? 1u : 0u);
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// sigmoid(g) for the epilogues: one exponential and an approximate
// (branch-free) reciprocal, so that a lane's columns run side by side instead
// of each waiting on a division's special-case branch.  g -> -inf gives
// 1 / inf = 0, g -> +inf gives 1.
__device__ __forceinline__ float sigmoid_fast(float g)
{
    return __fdividef(1.0f, 1.0f + __expf(-g));
}

__device__ __forceinline__ float silu_times(float g, float u)
{
    return g * sigmoid_fast(g) * u;
}

__device__ __forceinline__ float round_bf16(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

// Writes one 128-byte piece of each of the warp's 32 rows (lane = row, eight
// 16-byte chunks in v) to global memory.  The pieces go through the warp's
// 4 KB staging buffer (16-byte chunks XOR-swizzled by row, so both the
// writes and the reads are free of bank conflicts) and come out so that each
// store instruction writes four whole 128-byte lines instead of 32 scattered
// 16-byte pieces.  gbase is the address of the piece of the warp's row 0;
// rows >= valid_rows are not written.
__device__ __forceinline__ void warp_store_rows128(uint8_t *stage, const uint4 (&v)[8], int lane, char *gbase,
                                                   size_t ld_bytes, int valid_rows)
{
#pragma unroll
    for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4 *>(stage + lane * 128 + ((q ^ (lane & 7)) << 4)) = v[q];
    __syncwarp();
    const int q = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = i * 4 + (lane >> 3);
        const uint4 val = *reinterpret_cast<const uint4 *>(stage + r * 128 + ((q ^ (r & 7)) << 4));
        if (r < valid_rows)
            *reinterpret_cast<uint4 *>(gbase + (size_t)r * ld_bytes + q * 16) = val;
    }
    __syncwarp();
}

// One 32-row x 64-column bf16 piece of a grouped-GEMM output (lane = row,
// eight 16-byte chunks in v).  When all 32 rows belong to the tile, the piece
// goes out with a TMA store from a double-buffered, 128B-swizzled staging
// buffer (lane 0 issues it; the buffer is reused only after the store before
// the previous one has read it).  Otherwise -- the last tile of a bucket,
// whose other rows belong to the next expert -- the masked line-wise path.
template <int NBUF>
__device__ __forceinline__ void store_piece(const GemmParams &p, uint8_t *stage2, int &buf, const uint4 (&v)[8],
                                            int lane, int valid_rows, char *gbase, size_t ld_bytes, int col,
                                            int row0)
{
    if (valid_rows >= 32) {
        uint8_t *stage = stage2 + buf * 4096;
        if (lane == 0)
            bulk_wait_group_read<NBUF - 1>();   // this buffer's previous store has left smem
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4 *>(stage + lane * 128 + ((q ^ (lane & 7)) << 4)) = v[q];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(&p.tmOut, smem_u32(stage), col, row0);
            bulk_commit_group();
        }
        buf = (buf + 1) % NBUF;
    } else if (valid_rows > 0) {
        // this path commits no bulk group, so "all but the newest NBUF - 1
        // groups have read smem" no longer means "every other buffer is
        // free": after a masked piece the newest group can be the one that
        // reads this very buffer.  Wait until every store has left smem.
        uint8_t *stage = stage2 + buf * 4096;
        if (lane == 0)
            bulk_wait_group_read<0>();
        __syncwarp();
        warp_store_rows128(stage, v, lane, gbase, ld_bytes, valid_rows);
        buf = (buf + 1) % NBUF;
    }
}

// Epilogue of one grouped-GEMM tile for one epilogue warp (32 rows).
template <int KIND>
__device__ __forceinline__ void epilogue_tile(const GemmParams &p, const TileInfo &ti, uint32_t tacc, int quad,
                                              int lane, uint8_t *stage2, int &buf)
{
    const int valid_rows = ti.rows - quad * 32;
    const size_t ld_bytes = (size_t)p.ld_out * 2;
    const int row0 = ti.out_row + quad * 32;
    if constexpr (base_kind(KIND) == GK_GATE_UP) {
        // TMEM columns [0,128) = gate, [128,256) = up; 64 outputs per pass
        char *gbase = static_cast<char *>(p.out) + (size_t)row0 * ld_bytes + ti.nt * 256;
#pragma unroll 1
        for (int c = 0; c < 128; c += 64) {
            uint32_t g[64], u[64];
            tmem_load64(tacc + c, g);
            tmem_load64(tacc + 128 + c, u);
            uint4 v[8];
            uint32_t *pk = reinterpret_cast<uint32_t *>(v);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                pk[i] = pack_bf16x2(silu_times(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                                    silu_times(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1])));
            store_piece<GemmCfg<KIND>::NBUF>(p, stage2, buf, v, lane, valid_rows, gbase + c * 2, ld_bytes, ti.nt * 128 + c, row0);
        }
    } else {
        char *gbase = static_cast<char *>(p.out) + (size_t)row0 * ld_bytes + ti.nt * 512;
#pragma unroll 1
        for (int c = 0; c < 256; c += 64) {
            uint32_t r[64];
            tmem_load64(tacc + c, r);
            uint4 v[8];
            uint32_t *pk = reinterpret_cast<uint32_t *>(v);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            store_piece<GemmCfg<KIND>::NBUF>(p, stage2, buf, v, lane, valid_rows, gbase + c * 2, ld_bytes, ti.nt * 256 + c, row0);
        }
    }
}

// Named barrier 1 over the eight epilogue warps of GK_DOWN_COMBINE, with the
// AND of `ok` over them (so that all of them leave their tile loop together).
__device__ __forceinline__ bool epi_barrier_and(int ok)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(ok)
        : "memory");
    return r != 0;
}

// A 16-byte load of a routed row, streaming (evict first): each is read once.
__device__ __forceinline__ uint4 ld_row_stream(const uint16_t *ptr)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
    return v;
}

// acc += wgt * (8 bf16 values), in fp32
__device__ __forceinline__ void cmb_add8(float (&acc)[8], const uint4 &v, float wgt)
{
    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(p2[q]);
        acc[2 * q] += wgt * f.x;
        acc[2 * q + 1] += wgt * f.y;
    }
}

// GK_DOWN_COMBINE, one of the eight epilogue warps (two per TMEM lane
// quadrant, each with 128 of the tile's 256 columns).  First the shared
// expert's output rows of the tile, rounded to bf16 as the down GEMM stores
// them, into a token-major tile in shared memory (rows of 512 B; 16-byte
// chunk c of row r at chunk c ^ (r & 31), so that the row-per-lane writes
// and the chunk-per-lane reads below each touch every bank once); the
// accumulator slot then goes back to the MMA.  Then each warp takes 16 of
// the tile's tokens, four at a time, a 16-byte column vector per lane, and
// forms the combine's sum in its order: the eight weighted routed rows (a
// skipped pair, or j >= k, adds weight 0 times a zero row), then the shared
// row, then the residual; one rounding to bf16 into the layer output.
__device__ __forceinline__ void epilogue_down_combine(const GemmParams &p, const TileInfo &ti, uint32_t tslot,
                                                      int warp, int lane, uint8_t *tile_s, uint32_t tempty)
{
    const int ew = warp - 2;
    const int quad = warp & 3, half = ew >> 2;
    {
        const int r = quad * 32 + lane;
        uint8_t *row = tile_s + r * 512;
        const uint32_t tacc = tslot + ((uint32_t)(quad * 32) << 16) + half * 128;
#pragma unroll 1
        for (int c = 0; c < 128; c += 64) {
            uint32_t v[64];
            tmem_load64(tacc + c, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int chunk = (half * 128 + c) / 8 + q;
                const uint4 w4 = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                                            pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                            pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                            pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                *reinterpret_cast<uint4 *>(row + ((chunk ^ (r & 31)) << 4)) = w4;
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0)
        mbar_arrive(tempty);                                    // the slot is in shared memory now
    asm volatile("bar.sync 1, 256;" ::: "memory");              // every row of the tile is
    const size_t H = (size_t)p.H;
    const int K = p.cmb_k;
    const int col = ti.nt * 256 + lane * 8;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
    for (int tb = ew * 16; tb < ew * 16 + 16 && tb < ti.rows; tb += 4) {
        // slots and weights of tokens tb .. tb + 3: lane l holds pair (tb + l / 8, l % 8)
        const int tl = tb + (lane >> 3), j = lane & 7;
        int sl = -1;
        float wl = 0.0f;
        if (tl < ti.rows && j < K) {
            const size_t pi = (size_t)(ti.out_row + tl) * K + j;
            sl = p.cmb_slot[pi];
            wl = p.cmb_w ? p.cmb_w[pi] : 1.0f;
        }
        uint4 yv[4][8];
        float wv[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int sj = __shfl_sync(0xffffffffu, sl, u * 8 + jj);
                const float wj = __shfl_sync(0xffffffffu, wl, u * 8 + jj);
                wv[u][jj] = sj >= 0 ? wj : 0.0f;
                yv[u][jj] = sj >= 0 ? ld_row_stream(p.cmb_y + (size_t)sj * H + col) : zero;
            }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = tb + u;
            if (t < ti.rows) {
                float acc[8], racc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    acc[q] = 0.0f;
                    racc[q] = 0.0f;
                }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    cmb_add8(racc, yv[u][jj], wv[u][jj]);
                const uint4 sv = *reinterpret_cast<const uint4 *>(tile_s + t * 512 + ((lane ^ (t & 31)) << 4));
                cmb_add8(acc, sv, 1.0f);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    acc[q] += racc[q];
                const size_t o = (size_t)(ti.out_row + t) * H + col;
                if (p.cmb_res)
                    cmb_add8(acc, *reinterpret_cast<const uint4 *>(p.cmb_res + o), 1.0f);
                const uint4 ov = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                            pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
                *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + o) = ov;
            }
        }
    }
}

// ---------------------------------------------------------------- backward
// G and U of the backward are kept in bf16 (the activations a bf16 training
// step saves for the SwiGLU backward) in a warp-interleaved layout: for each
// block of 32 rows b and each group j of 8 columns of [G | U] (2I per row),
// the 16-byte pieces of the block's 32 rows lie side by side, at byte
// ((b * 2I / 8 + j) * 32 + row % 32) * 16.  An epilogue warp holds one row
// per lane, so each of its loads and stores moves 512 contiguous bytes.
// Blocks never straddle two buckets: buckets start on 64-row boundaries.
__device__ __forceinline__ uint4 *gu_piece(uint16_t *gu, int I, int row, int col)
{
    const size_t b = (size_t)(row >> 5), j = (size_t)(col >> 3);
    return reinterpret_cast<uint4 *>(gu) + ((b * (size_t)(I >> 2) + j) << 5) + (row & 31);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// GK_GATE_UP_BWD epilogue (one warp, 32 rows): for its 128 gate + 128 up
// columns, G and U (bf16, interleaved as above) into gu_out and
// aw = bf16(w_row * bf16(silu(G) * U)) into aw_out [rows, I] (TMA stores).
__device__ __forceinline__ void epilogue_gu_bwd(const GemmParams &p, const TileInfo &ti, uint32_t tacc, int quad,
                                                int lane, uint8_t *stage2, int &buf)
{
    const int r = quad * 32 + lane;
    const bool valid = r < ti.rows;
    const int row = ti.out_row + r;
    const float w = valid ? p.w_perm[row] : 0.0f;
    const int valid_rows = ti.rows - quad * 32;
    const int row0 = ti.out_row + quad * 32;
    const size_t ld_aw = (size_t)p.I * 2;
    char *aw_base = reinterpret_cast<char *>(p.aw_out) + (size_t)row0 * ld_aw;
#pragma unroll 1
    for (int c = 0; c < 128; c += 64) {
        uint32_t g[64], u[64];
        tmem_load64(tacc + c, g);
        tmem_load64(tacc + 128 + c, u);
        const int col = ti.nt * 128 + c;                 // intermediate column
        if (valid) {
            uint4 *pg = gu_piece(p.gu_out, p.I, row, col);
            uint4 *pu = gu_piece(p.gu_out, p.I, row, p.I + col);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t *gq = g + 8 * q, *uq = u + 8 * q;
                pg[32 * q] = make_uint4(pack_bf16x2(__uint_as_float(gq[0]), __uint_as_float(gq[1])),
                                        pack_bf16x2(__uint_as_float(gq[2]), __uint_as_float(gq[3])),
                                        pack_bf16x2(__uint_as_float(gq[4]), __uint_as_float(gq[5])),
                                        pack_bf16x2(__uint_as_float(gq[6]), __uint_as_float(gq[7])));
                pu[32 * q] = make_uint4(pack_bf16x2(__uint_as_float(uq[0]), __uint_as_float(uq[1])),
                                        pack_bf16x2(__uint_as_float(uq[2]), __uint_as_float(uq[3])),
                                        pack_bf16x2(__uint_as_float(uq[4]), __uint_as_float(uq[5])),
                                        pack_bf16x2(__uint_as_float(uq[6]), __uint_as_float(uq[7])));
            }
        }
        uint4 v[8];
        uint32_t *pk = reinterpret_cast<uint32_t *>(v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            // the forward's intermediate, bit for bit (same silu_times)
            const float a0 = round_bf16(silu_times(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])));
            const float a1 = round_bf16(silu_times(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1])));
            pk[i] = pack_bf16x2(w * a0, w * a1);
        }
        store_piece<GemmCfg<GK_GATE_UP_BWD>::NBUF>(p, stage2, buf, v, lane, valid_rows, aw_base + (size_t)col * 2,
                                                   ld_aw, col, row0);
    }
}

// GK_DGRAD_DOWN epilogue (one warp, 32 rows, 256 intermediate columns): the
// accumulator is dA' = dOut . W_down^T; with a = bf16(silu(G) U) it adds the
// row's partial <a, dA'> (d of the routing weight) to dw_part, then with
// dA = w dA' and s = sigmoid(G):
//   dG = dA U s (1 + G (1 - s)),  dU = dA G s   -> bf16 into dgu_out [rows, 2I]
// (TMA stores, 64 columns of dG and of dU at a time).
__device__ __forceinline__ void epilogue_dgrad(const GemmParams &p, const TileInfo &ti, uint32_t tacc, int quad,
                                               int lane, uint8_t *stage2, int &buf)
{
    const int r = quad * 32 + lane;
    const bool valid = r < ti.rows;
    const int row = ti.out_row + r;
    const float w = valid ? p.w_perm[row] : 0.0f;
    const int valid_rows = ti.rows - quad * 32;
    const int row0 = ti.out_row + quad * 32;
    const int I = p.I;
    const size_t ld = (size_t)2 * I * 2;
    char *dgu_base = reinterpret_cast<char *>(p.dgu_out) + (size_t)row0 * ld;
    float dwp = 0.0f;
#pragma unroll 1
    for (int c = 0; c < 256; c += 64) {
        uint4 dg4[8], du4[8];
        uint32_t *pg = reinterpret_cast<uint32_t *>(dg4);
        uint32_t *pu = reinterpret_cast<uint32_t *>(du4);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t acc[32];
            tmem_load32(tacc + c + half * 32, acc);
            const int col = ti.nt * 256 + c + half * 32;
            float G[32], U[32];
            if (valid) {
                const uint4 *sg = gu_piece(const_cast<uint16_t *>(p.gu_in), I, row, col);
                const uint4 *su = gu_piece(const_cast<uint16_t *>(p.gu_in), I, row, I + col);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 g8 = sg[32 * q], u8 = su[32 * q];
                    const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w}, uw[4] = {u8.x, u8.y, u8.z, u8.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        G[8 * q + 2 * k] = bf16_lo(gw[k]);
                        G[8 * q + 2 * k + 1] = bf16_hi(gw[k]);
                        U[8 * q + 2 * k] = bf16_lo(uw[k]);
                        U[8 * q + 2 * k + 1] = bf16_hi(uw[k]);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    G[i] = U[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float dgv[2], duv[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float g = G[i + h], u = U[i + h], da1 = __uint_as_float(acc[i + h]);
                    const float s = sigmoid_fast(g);
                    const float sg = g * s;                     // silu(G); sg * u == silu_times(g, u)
                    dwp = fmaf(round_bf16(sg * u), da1, dwp);
                    const float da = w * da1;
                    dgv[h] = da * u * s * fmaf(g, 1.0f - s, 1.0f);
                    duv[h] = da * sg;
                }
                pg[half * 16 + i / 2] = pack_bf16x2(dgv[0], dgv[1]);
                pu[half * 16 + i / 2] = pack_bf16x2(duv[0], duv[1]);
            }
        }
        const int col = ti.nt * 256 + c;
        store_piece<GemmCfg<GK_DGRAD_DOWN>::NBUF>(p, stage2, buf, dg4, lane, valid_rows,
                                                  dgu_base + (size_t)col * 2, ld, col, row0);
        store_piece<GemmCfg<GK_DGRAD_DOWN>::NBUF>(p, stage2, buf, du4, lane, valid_rows,
                                                  dgu_base + (size_t)(I + col) * 2, ld, I + col, row0);
    }
    if (valid && !ti.shared)
        p.dw_part[(size_t)row * p.n_tiles + ti.nt] = dwp;
}

// GK_WGRAD epilogue (one warp, 32 feature rows x 256 hidden columns, fp32);
// an expert with no rows gets zeros.
__device__ __forceinline__ void epilogue_wgrad(const GemmParams &p, const TileInfo &ti, uint32_t tacc, int quad,
                                               int lane, uint8_t *stage)
{
    const size_t ld = (size_t)p.H * 4;
    char *base = static_cast<char *>(ti.shared ? p.out_shared : p.out) + (size_t)(ti.out_row + quad * 32) * ld +
                 (size_t)ti.nt * 256 * 4;
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
        uint32_t r[32];
        if (ti.kblocks > 0)
            tmem_load32(tacc + c, r);
        else
#pragma unroll
            for (int i = 0; i < 32; ++i)
                r[i] = 0u;
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            v[q] = make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        warp_store_rows128(stage, v, lane, base + (size_t)c * 4, ld, 32);
    }
}

// ---------------------------------------------------------------------------
// GK_ROUTER_FUSED.  The epilogue warps store each tile's logits like the
// 256-expert router (to p.out, in L2) and mark the tile ready; after the CTA's
// last tile they take tiles from a queue shared by all CTAs (so CTAs that had
// fewer tiles start on the first tiles while the others still multiply) and,
// for each: select every token's experts (route_token, the routing kernel's
// own code: the same bits), count the tile's hits per expert, claim the rows
// in the experts' buckets with one integer atomic per expert, and copy the
// tokens' hidden rows there with bulk copies through the idle stage ring.
struct FusedCtx {
    uint32_t ebar;    // epilogue barrier: 8 warp arrivals per phase
    uint32_t phase;   // phases completed so far
    int *hist;        // smem [256]: a tile's hits per expert, then the bucket bases
    int *unit;        // smem: the tile the CTA took from the queue
    int2 *mail;       // smem [2]: (first token, rows) of the tile in each row table; first < 0: done
    uint32_t stage;   // barrier of the logits' staging load
    uint32_t dfull;   // [2] a row table is filled (epilogue -> copy engine)
    uint32_t dempty;  // [2] a row table is read (copy engine -> epilogue)
    uint32_t eslot;   // [FUSED_ENGINE_SLOTS] the copy engine's row loads
};

// The eight epilogue warps meet; shared-memory writes made before are visible
// to every epilogue thread after.  Bounded like every wait of the kernel.
__device__ __forceinline__ bool epi_sync(FusedCtx &fz, int lane, volatile int *abort_flag, unsigned long long limit)
{
    __syncwarp();
    int ok = 1;
    if (lane == 0) {
        mbar_arrive(fz.ebar);
        ok = mbar_wait(fz.ebar, fz.phase & 1u, abort_flag, limit) ? 1 : 0;
    }
    ++fz.phase;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Bounded wait (lane 0) until all eight epilogue warps of the tile's CTA have
// stored its logits.
__device__ __forceinline__ bool wait_tile_ready(const int *ready, volatile int *abort_flag, unsigned long long limit)
{
    int v = 0;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ready) : "memory");
    if (v >= 8)
        return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ready) : "memory");
        if (v >= 8)
            return true;
        if ((it & 63u) == 0) {
            if (*abort_flag)
                return false;
            if (globaltimer_ns() - t0 > limit) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Post-phase shared memory, carved from the idle stage ring (bytes):
//   [0, 128 K)   the tile's logits, then their scores, [128][256] fp32;
//   group scores [128][8] fp32, the halves' lists [128][2][3 FUSED_MAX_K],
//   two tables of the pairs' bucket rows [2][128][FUSED_MAX_K] (one being
//   filled by the epilogue while the copy engine reads the other), the bias
//   [256]; from FP_SLOTS to the ring's end the copy engine's row slots.
// Their barriers live with the kernel's others (FusedCtx).
constexpr uint32_t FP_LOGITS = 0;
constexpr uint32_t FP_GROUPS = GEMM_BM * 256 * 4;
constexpr uint32_t FP_LISTS = FP_GROUPS + GEMM_BM * 8 * 4;
constexpr uint32_t FP_DEST = FP_LISTS + GEMM_BM * 2 * 3 * FUSED_MAX_K * 4;
constexpr uint32_t FP_BIAS = FP_DEST + 2 * GEMM_BM * FUSED_MAX_K * 4;
constexpr uint32_t FP_END = FP_BIAS + 256 * 4;
constexpr uint32_t FP_SLOTS = (FP_END + 1023u) & ~1023u;

// The post phase of one CTA.  All 256 epilogue threads (ew = 0..255) take
// tiles from the queue; per tile, thread (h = ew / 128,
// r = ew % 128) holds token r's experts 128 h .. 128 h + 127 (groups
// 4 h .. 4 h + 3) and reads them from shared memory starting at column
// r % 32, so the 32 lanes of a warp hit 32 different banks.  The arithmetic
// is the routing kernels' (route.cu): the same score formula, group score
// (the two best biased scores, a repeated best counting twice), group ranking,
// winner order (key desc, expert asc) and sequential normaliser, so the
// results are bit-identical to routing the same logits there.
__device__ __forceinline__ void fused_post(const GemmParams &p, int num_tiles, int lane, int ew, FusedCtx &fz,
                                          uint8_t *ring_ptr, uint32_t ring, volatile int *abort_flag,
                                          unsigned long long limit)
{
    const int K = p.k;
    const int h = ew >> 7, r = ew & 127;
    const int e0 = 128 * h;
    float *sl = reinterpret_cast<float *>(ring_ptr + FP_LOGITS);
    float *sg = reinterpret_cast<float *>(ring_ptr + FP_GROUPS);
    uint32_t *sls = reinterpret_cast<uint32_t *>(ring_ptr + FP_LISTS);
    float *sbias = reinterpret_cast<float *>(ring_ptr + FP_BIAS);
    const uint32_t stage_bar = fz.stage;
    sbias[ew] = p.bias ? __ldg(p.bias + ew) : 0.0f;
    uint32_t stage_par = 0;
    bool nonfinite = false;
    for (int nunit = 0;; ++nunit) {
        const int buf = nunit & 1;
        if (ew == 0) {
            // the row table this tile will fill must have been read by the copy engine
            if (nunit >= 2 && !mbar_wait(fz.dempty + 8u * buf, ((nunit >> 1) - 1) & 1u, abort_flag, limit))
                *fz.unit = -1;
            else
                *fz.unit = atomicAdd(p.unit_ctr, 1);
        }
        if (!epi_sync(fz, lane, abort_flag, limit))
            break;
        const int u = *fz.unit;
        if (u < 0)
            break;
        if (u >= num_tiles) {
            if (ew == 0) {
                fz.mail[buf] = make_int2(-1, 0);   // no more tiles for the copy engine
                mbar_arrive(fz.dfull + 8u * buf);
            }
            break;
        }
        int *sdst = reinterpret_cast<int *>(ring_ptr + FP_DEST) + buf * GEMM_BM * FUSED_MAX_K;
        const int row0 = u * GEMM_BM;
        const int rows = min(GEMM_BM, p.T - row0);
        if (ew == 0) {
            // every thread is done with the previous tile's scores (the meeting
            // above): stage this tile's logits once its CTA has stored them
            bool ok = wait_tile_ready(p.ready + u, abort_flag, limit);
            if (ok) {
                fence_proxy_async_global();       // the logits were stored by generic writes
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(stage_bar, (uint32_t)rows * 1024u);
                bulk_load_g2s(ring + FP_LOGITS, static_cast<const float *>(p.out) + (size_t)row0 * 256,
                              (uint32_t)rows * 1024u, stage_bar);
            }
        }
        if (!mbar_wait(stage_bar, stage_par, abort_flag, limit))
            break;
        stage_par ^= 1u;
        const bool valid = r < rows;
        float *row = sl + r * 256 + e0;

        // scores (section 二 step 1), in place; this half's four group scores
        // on the biased scores (section 三)
        float gs[4];
#pragma unroll 1
        for (int gi = 0; gi < 4; ++gi) {
            uint32_t m1 = 0u, m2 = 0u;
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
                const int c = gi * 32 + ((i + r) & 31);
                const float L = row[c];
                const float b = sbias[e0 + c];
                nonfinite |= valid && (!isfinite(L) || !isfinite(b));
                const float sc = router_sigmoid(L);
                row[c] = sc;
                const uint32_t k = fkey(sc + b);
                m2 = max(m2, min(m1, k));
                m1 = max(m1, k);
            }
            gs[gi] = fkey_value(m1) + fkey_value(m2);
        }
#pragma unroll
        for (int gi = 0; gi < 4; ++gi)
            sg[r * 8 + 4 * h + gi] = gs[gi];
        if (!epi_sync(fz, lane, abort_flag, limit))
            break;
        // keep the topk_group best groups (section 二 step 2), ties to the lower group
        float g[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            g[j] = sg[r * 8 + j];
        uint32_t keep = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int rank = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                rank += (g[q] > g[j] || (g[q] == g[j] && q < j)) ? 1 : 0;
            if (rank < p.topk_group)
                keep |= 1u << j;
        }
        // this half's best FUSED_MAX_K of the kept groups, by (key desc, expert asc)
        uint32_t lk[FUSED_MAX_K];
        int le[FUSED_MAX_K];
        float ls[FUSED_MAX_K];
#pragma unroll
        for (int q = 0; q < FUSED_MAX_K; ++q) {
            lk[q] = 0u;
            le[q] = 0x7fffffff;
            ls[q] = 0.0f;
        }
#pragma unroll 1
        for (int gi = 0; gi < 4; ++gi) {
            if (!((keep >> (4 * h + gi)) & 1u))
                continue;
#pragma unroll 2
            for (int i = 0; i < 32; ++i) {
                const int c = gi * 32 + ((i + r) & 31);
                const float sc = row[c];
                const uint32_t k = fkey(sc + sbias[e0 + c]);
                const int e = e0 + c;
                if (k < lk[FUSED_MAX_K - 1] || (k == lk[FUSED_MAX_K - 1] && e > le[FUSED_MAX_K - 1]))
                    continue;
#pragma unroll
                for (int q = FUSED_MAX_K - 1; q > 0; --q) {
                    const bool up = k > lk[q - 1] || (k == lk[q - 1] && e < le[q - 1]);   // ranks above entry q-1
                    const bool here = k > lk[q] || (k == lk[q] && e < le[q]);
                    lk[q] = up ? lk[q - 1] : (here ? k : lk[q]);
                    le[q] = up ? le[q - 1] : (here ? e : le[q]);
                    ls[q] = up ? ls[q - 1] : (here ? sc : ls[q]);
                }
                if (k > lk[0] || (k == lk[0] && e < le[0])) {
                    lk[0] = k;
                    le[0] = e;
                    ls[0] = sc;
                }
            }
        }
        // the logits area is refilled by bulk copies after the next meeting:
        // order this thread's accesses to it before them
        fence_proxy_async_smem();
        uint32_t *mine = sls + (r * 2 + h) * 3 * FUSED_MAX_K;
#pragma unroll
        for (int q = 0; q < FUSED_MAX_K; ++q) {
            mine[q] = lk[q];
            mine[FUSED_MAX_K + q] = (uint32_t)le[q];
            mine[2 * FUSED_MAX_K + q] = __float_as_uint(ls[q]);
        }
        if (!epi_sync(fz, lane, abort_flag, limit))
            break;

        // the lower half's thread merges the two lists: the token's k experts
        // in output order, their weights (section 二 step 3) and each pair's
        // rank among the tile's hits of its expert
        int oe[FUSED_MAX_K], orank[FUSED_MAX_K];
        if (h == 0) {
            const uint32_t *other = sls + (r * 2 + 1) * 3 * FUSED_MAX_K;
            uint32_t pk[FUSED_MAX_K];
            int pe[FUSED_MAX_K];
            float ps[FUSED_MAX_K];
#pragma unroll
            for (int q = 0; q < FUSED_MAX_K; ++q) {
                pk[q] = other[q];
                pe[q] = (int)other[FUSED_MAX_K + q];
                ps[q] = __uint_as_float(other[2 * FUSED_MAX_K + q]);
            }
            float os[FUSED_MAX_K];
            float den = 0.0f;
#pragma unroll
            for (int j = 0; j < FUSED_MAX_K; ++j) {
                const bool a = lk[0] >= pk[0];      // equal keys: the lower half's expert has the lower id
                oe[j] = a ? le[0] : pe[0];
                os[j] = a ? ls[0] : ps[0];
#pragma unroll
                for (int q = 0; q < FUSED_MAX_K - 1; ++q) {
                    lk[q] = a ? lk[q + 1] : lk[q];
                    le[q] = a ? le[q + 1] : le[q];
                    ls[q] = a ? ls[q + 1] : ls[q];
                    pk[q] = a ? pk[q] : pk[q + 1];
                    pe[q] = a ? pe[q] : pe[q + 1];
                    ps[q] = a ? ps[q] : ps[q + 1];
                }
                lk[FUSED_MAX_K - 1] = a ? 0u : lk[FUSED_MAX_K - 1];
                pk[FUSED_MAX_K - 1] = a ? pk[FUSED_MAX_K - 1] : 0u;
                if (j < K)
                    den += os[j];                   // in output order
            }
            den += p.eps;
#pragma unroll
            for (int j = 0; j < FUSED_MAX_K; ++j) {
                orank[j] = 0;
                if (j < K && valid && oe[j] >= 0 && oe[j] < 256) {
                    const int t = row0 + r;
                    p.idx_out[(size_t)t * K + j] = oe[j];
                    p.w_out[(size_t)t * K + j] = (os[j] / den) * p.rsf;
                    orank[j] = atomicAdd(&fz.hist[oe[j]], 1);
                }
            }
        }
        if (!epi_sync(fz, lane, abort_flag, limit))
            break;
        // one atomic per expert hit in this tile reserves its rows in the
        // bucket; the counters end as the experts' hit counts (section 六)
        {
            const int n = fz.hist[ew];
            if (n > 0)
                fz.hist[ew] = atomicAdd(p.counts + ew, n);
        }
        if (!epi_sync(fz, lane, abort_flag, limit))
            break;
        if (h == 0) {
#pragma unroll
            for (int j = 0; j < FUSED_MAX_K; ++j) {
                int d = -1;
                if (j < K && valid && oe[j] >= 0 && oe[j] < 256) {
                    const int t = row0 + r;
                    const int slot = fz.hist[oe[j]] + orank[j];
                    const bool in = slot < p.T;       // at most T pairs per expert: one per token
                    p.slot_local[(size_t)t * K + j] = in ? slot : -1;
                    d = in ? oe[j] * p.T + slot : -1;
                    if (!in)
                        atomicOr(p.status, ST_COUNT_MISMATCH);
                }
                sdst[r * FUSED_MAX_K + j] = d;
            }
        }
        if (!epi_sync(fz, lane, abort_flag, limit))
            break;
        fz.hist[ew] = 0;                          // every base is read: clear for the next tile

        // hand the row table to the copy engine (the producer warp's lane 0)
        if (ew == 0) {
            fz.mail[buf] = make_int2(row0, rows);
            mbar_arrive(fz.dfull + 8u * buf);
        }
    }
    if (__any_sync(0xffffffffu, nonfinite) && lane == 0)
        atomicOr(p.status, ST_NONFINITE);
}

// The copy engine: the producer warp's lane 0, once its loads are issued.
// For every tile the epilogue warps route (in their order), it loads the
// tokens' hidden rows into its slots at the ring's end and stores each to its
// pairs' bucket rows, so the copies of one tile overlap the routing of the
// next.  Bounded waits; on a failed one it lets its loads in flight land and
// stops.
__device__ __forceinline__ void fused_copy_engine(const GemmParams &p, uint8_t *ring_ptr, uint32_t ring,
                                                 uint32_t ring_bytes, const FusedCtx &fz,
                                                 volatile int *abort_flag, unsigned long long limit)
{
    const uint32_t rowbytes = (uint32_t)p.H * 2;
    const int ns = min((int)((ring_bytes - FP_SLOTS) / rowbytes), FUSED_ENGINE_SLOTS);   // >= 1: H <= 8192
    const int K = p.k;
    uint32_t parity = 0;                      // bit b: parity of slot b's next completion
    for (int n = 0;; ++n) {
        const int buf = n & 1;
        if (!mbar_wait(fz.dfull + 8u * buf, (n >> 1) & 1u, abort_flag, limit))
            break;
        const int2 m = fz.mail[buf];
        if (m.x < 0)
            break;
        const int *sdst = reinterpret_cast<const int *>(ring_ptr + FP_DEST) + buf * GEMM_BM * FUSED_MAX_K;
        bool ok = true;
        for (int i0 = 0; i0 < m.y && ok; i0 += ns) {
            const int nb = min(ns, m.y - i0);
            for (int b = 0; b < nb; ++b) {
                const uint32_t bar = fz.eslot + 8u * b;
                mbar_arrive_expect_tx(bar, rowbytes);
                bulk_load_g2s(ring + FP_SLOTS + (uint32_t)b * rowbytes, p.hidden + (size_t)(m.x + i0 + b) * p.H,
                              rowbytes, bar);
            }
            for (int b = 0; b < nb; ++b) {
                const uint32_t bar = fz.eslot + 8u * b;
                if (ok && !mbar_wait(bar, (parity >> b) & 1u, abort_flag, limit))
                    ok = false;
                if (!ok)
                    mbar_drain(bar, (parity >> b) & 1u);   // let its load land
                parity ^= 1u << b;
                if (!ok)
                    continue;
                const int *dr = sdst + (i0 + b) * FUSED_MAX_K;
                for (int j = 0; j < K; ++j) {
                    const int d = dr[j];
                    if (d >= 0)
                        bulk_store_s2g(p.xperm + (size_t)d * p.H, ring + FP_SLOTS + (uint32_t)b * rowbytes,
                                       rowbytes);
                }
            }
            bulk_commit_group();
            bulk_wait_group_read<0>();            // the slots may be refilled
        }
        if (!ok)
            break;
        mbar_arrive(fz.dempty + 8u * buf);        // this row table is read
    }
    bulk_wait_group_all();
}

// Router epilogue warp: adds the K-block partial sums of its 32 rows in fp32
// (K-block order, round-to-nearest), then writes the 128 logits of each row
// that it owns (columns half * 128 .. of the tile; half = 0 for the 128-expert
// tiles, 0 or 1 for the wide kind's two warps per lane quadrant).
// The fused kind also counts the warp towards the tile's readiness.
template <int KIND>
__device__ __forceinline__ bool router_epilogue_tile(const GemmParams &p, const TileInfo &ti, uint32_t tmem,
                                                     int quad, int half, int lane, uint32_t tfull0,
                                                     uint32_t tempty0, uint32_t &kctr, volatile int *abort_flag,
                                                     uint8_t *stage, unsigned long long limit, int tile,
                                                     const float *sbias, uint32_t tempty_cluster = 0)
{
    using C = GemmCfg<KIND>;
    constexpr int COLS = 128;
    float acc[COLS];
#pragma unroll
    for (int c = 0; c < COLS; ++c)
        acc[c] = 0.0f;
    const int ngroups = (p.kblocks + ROUTER_KPS - 1) / ROUTER_KPS;
    for (int kg = 0; kg < ngroups; ++kg, ++kctr) {
        const uint32_t slot = kctr % C::SLOTS;
        const uint32_t par = (kctr / C::SLOTS) & 1u;
        int ok = 1;
        if (lane == 0)
            ok = mbar_wait(tfull0 + 8u * slot, par, abort_flag, limit) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok)
            return false;
        __syncwarp();
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + slot * C::BN + half * COLS;
        // 64-column loads for the 128-expert tiles; 32-column loads for the
        // wide kind, whose 320-thread block leaves ~200 registers per thread
        constexpr int LD = (C::NBUF == 0) ? 32 : 64;
#pragma unroll
        for (int c = 0; c < COLS; c += LD) {
            uint32_t r[LD];
            if constexpr (LD == 64)
                tmem_load64(taddr + c, r);
            else
                tmem_load32(taddr + c, r);
            if (c + LD == COLS) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // slot free again: the values are in registers (a CTA pair
                    // counts both CTAs' warps on the leader's barrier)
                    if (tempty_cluster)
                        mbar_arrive_cluster(tempty_cluster + 8u * slot);
                    else
                        mbar_arrive(tempty0 + 8u * slot);
                }
            }
#pragma unroll
            for (int i = 0; i < LD; ++i)
                acc[c + i] += __uint_as_float(r[i]);
        }
    }
    const int valid_rows = ti.rows - quad * 32;
    if (p.gscore != nullptr) {
        // scored output (routing page, section 二 step 1 and the group score
        // of step 2, with section 三's bias): the sigmoid of every logit
        // replaces it, and each of the row's four groups of 32 gets its two
        // best biased scores (a tie for the top counts twice; the group score
        // is their sum)
        const int e0 = ti.nt * C::BN + half * COLS;
        bool bad = false;
        float g1[COLS / 32], g2[COLS / 32];
#pragma unroll
        for (int q = 0; q < COLS / 32; ++q) {
            float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float L = acc[32 * q + i];
                bad |= !(fabsf(L) <= 3.402823466e38f);       // NaN or +-inf
                const float sc = router_sigmoid(L);
                acc[32 * q + i] = sc;
                const float b = sc + sbias[e0 + 32 * q + i];   // one address for the warp: a broadcast
                m2 = fmaxf(m2, fminf(m1, b));
                m1 = fmaxf(m1, b);
            }
            g1[q] = m1;
            g2[q] = m2;
        }
        if (lane < valid_rows) {
            float *g = p.gscore + ((size_t)(ti.out_row + quad * 32 + lane) * (p.E / 32) + e0 / 32) * 2;
#pragma unroll
            for (int q = 0; q < COLS / 32; ++q) {
                g[2 * q] = g1[q];
                g[2 * q + 1] = g2[q];
            }
        }
        if (__any_sync(0xffffffffu, bad && lane < valid_rows) && lane == 0)
            atomicOr(p.status, ST_NONFINITE);
    }
    if (valid_rows > 0) {
        const size_t ld_bytes = (size_t)p.ld_out * 4;
        char *gbase = static_cast<char *>(p.out) + (size_t)ti.kp * (size_t)p.part_stride * 4 +
                      (size_t)(ti.out_row + quad * 32) * ld_bytes + (size_t)(ti.nt * C::BN + half * COLS) * 4;
        if constexpr (C::NBUF == 0) {
            // each thread's 512 contiguous bytes, straight from registers
            if (lane < valid_rows) {
                uint4 *dst = reinterpret_cast<uint4 *>(gbase + (size_t)lane * ld_bytes);
#pragma unroll
                for (int q = 0; q < COLS / 4; ++q)
                    dst[q] = make_uint4(__float_as_uint(acc[4 * q]), __float_as_uint(acc[4 * q + 1]),
                                        __float_as_uint(acc[4 * q + 2]), __float_as_uint(acc[4 * q + 3]));
            }
        } else {
#pragma unroll
            for (int c = 0; c < COLS; c += 32) {
                uint4 v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    v[q] = make_uint4(__float_as_uint(acc[c + 4 * q]), __float_as_uint(acc[c + 4 * q + 1]),
                                      __float_as_uint(acc[c + 4 * q + 2]), __float_as_uint(acc[c + 4 * q + 3]));
                warp_store_rows128(stage, v, lane, gbase + c * 4, ld_bytes, valid_rows);
            }
        }
    }
    if constexpr (KIND == GK_ROUTER_FUSED) {
        // this warp's rows of the tile are stored: count it towards the tile's readiness
        __threadfence();
        __syncwarp();
        if (lane == 0)
            atomicAdd(p.ready + tile, 1);
    }
    return true;
}

static_assert(FP_SLOTS + 8192 * 2 <= GemmCfg<GK_ROUTER_FUSED>::STAGES *
                                      (GemmCfg<GK_ROUTER_FUSED>::A_BYTES + GemmCfg<GK_ROUTER_FUSED>::B_BYTES),
              "the fused router's post phase does not fit its stage ring");

template <int KIND>
__global__ void __launch_bounds__(kind_threads(KIND), 1) umma_gemm_kernel(const __grid_constant__ GemmParams p)
{
    using C = GemmCfg<KIND>;
    using L = GemmLayout<KIND>;
    constexpr bool ROUTER = (base_kind(KIND) == GK_ROUTER);
    extern __shared__ uint8_t dsmem[];

    const uint32_t raw = smem_u32(dsmem);
    const uint32_t base = (raw + 1023u) & ~1023u;                 // swizzle atoms need 1024-B alignment
    uint8_t *base_ptr = dsmem + (base - raw);
    uint8_t *staging = base_ptr + C::STAGES * L::STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + L::STAGING);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + L::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *tq = reinterpret_cast<volatile int *>(tmem_holder + 4);   // L::TQ entries
    float *sbias = reinterpret_cast<float *>(const_cast<int *>(tq + L::TQ) + L::HIST / 4);   // L::BIAS bytes

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    const uint32_t tfull0 = bar0 + 8u * (2 * C::STAGES);
    const uint32_t tempty0 = tfull0 + 8u * C::SLOTS;
    const uint32_t fin_bar = tempty0 + 8u * C::SLOTS;
    const uint32_t tqfull0 = fin_bar + 8u;
    const uint32_t tqempty0 = tqfull0 + 8u * L::TQ;
    FusedCtx fz;
    fz.ebar = tqempty0 + 8u * L::TQ;             // (fused router only)
    fz.phase = 0;
    fz.hist = const_cast<int *>(tq + L::TQ);      // (fused router only) L::HIST bytes
    fz.unit = fz.hist + 256;                      // (fused router only)
    fz.mail = reinterpret_cast<int2 *>(fz.hist + 260);
    fz.stage = fz.ebar + 8u;
    fz.dfull = fz.stage + 8u;
    fz.dempty = fz.dfull + 16u;
    fz.eslot = fz.dempty + 16u;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < C::SLOTS; ++a) {
            mbar_init(tfull0 + 8u * a, 1);
            mbar_init(tempty0 + 8u * a, epi_warps(KIND));
        }
        mbar_init(fin_bar, 1);
        for (int i = 0; i < L::TQ; ++i) {
            mbar_init(tqfull0 + 8u * i, 1);
            mbar_init(tqempty0 + 8u * i, TQ_TAKERS);
        }
        if constexpr (L::FUSED) {
            mbar_init(fz.ebar, epi_warps(KIND));
            mbar_init(fz.stage, 1);
            for (int b = 0; b < 2; ++b) {
                mbar_init(fz.dfull + 8u * b, 1);
                mbar_init(fz.dempty + 8u * b, 1);
            }
            for (int b = 0; b < FUSED_ENGINE_SLOTS; ++b)
                mbar_init(fz.eslot + 8u * b, 1);
        }
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
    // the prologue above overlaps the previous kernel's teardown; its outputs
    // (the tile list, A rows) are read only after this
    pdl_wait();

    const int num_tiles =
        (ROUTER || KIND == GK_WGRAD || KIND == GK_DOWN_COMBINE) ? p.num_tiles_static : (*p.num_mtiles) * p.n_tiles;
    const unsigned long long limit = p.wait_limit_ns ? p.wait_limit_ns : WAIT_LIMIT_NS;

    // The CTA's n-th tile for the MMA lane and the epilogue warps' lane 0:
    // blockIdx.x + n gridDim.x, or the producer's n-th claim.  -1: no more
    // tiles; -2: the wait for the claim ran out.
    auto take_tile = [&](int n) -> int {
        if constexpr (!L::DYN) {
            const int t = blockIdx.x + n * gridDim.x;
            return t < num_tiles ? t : -1;
        } else {
            const uint32_t slot = n % TQ_RING, par = (n / TQ_RING) & 1u;
            if (!mbar_wait(tqfull0 + 8u * slot, par, abort_flag, limit))
                return -2;
            const int t = tq[slot];
            mbar_arrive(tqempty0 + 8u * slot);
            return t;
        }
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true;
            for (int n = 0; ok && !p.inject_withhold; ++n) {
                int tile;
                if constexpr (L::DYN) {
                    const uint32_t slot = n % TQ_RING, par = (n / TQ_RING) & 1u;
                    if (!mbar_wait(tqempty0 + 8u * slot, par ^ 1u, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    tile = atomicAdd(p.tile_ctr, 1);
                    if (tile >= num_tiles)
                        tile = -1;
                    tq[slot] = tile;
                    mbar_arrive(tqfull0 + 8u * slot);            // releases the index to the takers
                } else {
                    tile = blockIdx.x + n * gridDim.x;
                    if (tile >= num_tiles)
                        tile = -1;
                }
                if (tile < 0)
                    break;
                const TileInfo ti = tile_info<KIND>(p, tile);
                for (int kb = 0; kb < ti.kblocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = base + stage * L::STAGE_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), L::STAGE_BYTES);
                    issue_loads<KIND>(p, ti, kb, sA, sA + C::A_BYTES, full_bar(stage));
                    if constexpr (wide_router(KIND)) {
                        // two stages cannot hide a DRAM read of the hidden rows:
                        // pull the A box ROUTER_PF K blocks ahead (in this CTA's
                        // tile order) into L2
                        const int q = n * p.kblocks + kb + ROUTER_PF;
                        const int pt = blockIdx.x + (q / p.kblocks) * (int)gridDim.x;
                        if (pt < num_tiles)
                            tma_prefetch_l2_2d(&p.tmA0, (q % p.kblocks) * GEMM_BK, (pt / p.n_tiles) * GEMM_BM);
                    }
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
            if constexpr (L::FUSED) {
                // the fused router's hidden-row copies, tile by tile as the
                // epilogue warps route them
                if (ok)
                    fused_copy_engine(p, base_ptr, base, C::STAGES * L::STAGE_BYTES, fz, abort_flag, limit);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            uint32_t ctr = 0;   // accumulators used so far (tiles, or K blocks for the router)
            for (int n = 0; ok; ++n) {
                const int tile = take_tile(n);
                if (tile < 0)
                    break;
                const int kblocks = (KIND == GK_WGRAD) ? tile_info<KIND>(p, tile).kblocks : p.kblocks;
                if (!ROUTER) {
                    const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
                    if (!mbar_wait(tempty0 + 8u * slot, par ^ 1u, abort_flag, limit))
                        break;
                    tc_fence_after();
                }
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (ROUTER && kb % ROUTER_KPS == 0) {
                        const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
                        if (!mbar_wait(tempty0 + 8u * slot, par ^ 1u, abort_flag, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = base + stage * L::STAGE_BYTES;
                    const uint32_t d = tmem + (ctr % C::SLOTS) * C::BN;
                    issue_mmas<KIND>(sA, sA + C::A_BYTES, d, ROUTER ? (kb % ROUTER_KPS != 0) : kb > 0);
                    umma_commit(empty_bar(stage));               // frees the stage once read
                    if (ROUTER && (kb % ROUTER_KPS == ROUTER_KPS - 1 || kb == kblocks - 1)) {
                        umma_commit(tfull0 + 8u * (ctr % C::SLOTS));  // the slot's partial sum is ready
                        ++ctr;
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ROUTER && ok) {
                    umma_commit(tfull0 + 8u * (ctr % C::SLOTS));      // tile accumulator ready
                    ++ctr;
                }
            }
            // no MMA may still be writing TMEM when it is freed
            umma_commit(fin_bar);
            mbar_drain(fin_bar, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        uint8_t *stage = staging + (warp - 2) * (C::NBUF * 4096);
        int buf = 0;
        uint32_t ctr = 0;
        bool fused_ok = true;
        if constexpr (L::BIAS > 0) {
            // the scored router output adds expert_bias: a copy in shared
            // memory, shared by the epilogue warps (named barrier 1)
            if (p.gscore) {
                const int et = threadIdx.x - 64;
                for (int e = et; e < p.E; e += 32 * epi_warps(KIND))
                    sbias[e] = p.bias ? p.bias[e] : 0.0f;
                asm volatile("bar.sync 1, %0;" ::"r"(32 * epi_warps(KIND)) : "memory");
            }
        }
        if constexpr (L::FUSED)
            fz.hist[(warp - 2) * 32 + lane] = 0;
        for (int n = 0;; ++n) {
            int tile = 0;
            if (lane == 0)
                tile = take_tile(n);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0)
                break;
            const TileInfo ti = tile_info<KIND>(p, tile);
            if constexpr (ROUTER) {
                if (!router_epilogue_tile<KIND>(p, ti, tmem, quad, (warp - 2) >> 2, lane, tfull0, tempty0, ctr,
                                                abort_flag, stage, limit, tile, sbias)) {
                    fused_ok = false;
                    break;
                }
            } else if constexpr (KIND == GK_DOWN_COMBINE) {
                const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
                int ok = 1;
                if (lane == 0)
                    ok = mbar_wait(tfull0 + 8u * slot, par, abort_flag, limit) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                // every epilogue warp is past its reads of the previous tile's
                // rows in shared memory, and all of them agree to go on
                if (!epi_barrier_and(ok))
                    break;
                tc_fence_after();
                epilogue_down_combine(p, ti, tmem + slot * C::BN, warp, lane, staging, tempty0 + 8u * slot);
                ++ctr;
            } else {
                const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
                int ok = 1;
                if (lane == 0)
                    ok = mbar_wait(tfull0 + 8u * slot, par, abort_flag, limit) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
                __syncwarp();
                tc_fence_after();
                const uint32_t tacc = tmem + ((uint32_t)(quad * 32) << 16) + slot * C::BN;
                if constexpr (KIND == GK_GATE_UP_BWD)
                    epilogue_gu_bwd(p, ti, tacc, quad, lane, stage, buf);
                else if constexpr (KIND == GK_DGRAD_DOWN)
                    epilogue_dgrad(p, ti, tacc, quad, lane, stage, buf);
                else if constexpr (KIND == GK_WGRAD)
                    epilogue_wgrad(p, ti, tacc, quad, lane, stage);
                else
                    epilogue_tile<KIND>(p, ti, tacc, quad, lane, stage, buf);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(tempty0 + 8u * slot);
                ++ctr;
            }
        }
        if (!ROUTER && lane == 0)
            bulk_wait_group_all();              // this warp's output stores have completed
        if constexpr (L::FUSED) {
            // the CTA's tiles are multiplied (every MMA done, the ring idle):
            // route and bucket tiles from the shared queue
            if (fused_ok && epi_sync(fz, lane, abort_flag, limit))
                fused_post(p, num_tiles, lane, (warp - 2) * 32 + lane, fz, base_ptr, base, abort_flag, limit);
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

// ---------------------------------------------------------------------------
// GK_ROUTER_PAIR: the 256-expert router on CTA pairs (tcgen05 cta_group::2).
// A pair takes 256 tokens x all 256 experts per tile: each CTA loads its own
// 128 token rows and the hi/mid/lo weight parts of its half of the experts
// (CTA rank r: experts 128 r .. 128 r + 127), so a stage is 16 KB + 48 KB
// instead of the single-CTA wide router's 16 KB + 96 KB; the even CTA issues
// M = 256, N = 256 MMAs that read both CTAs' shared memory and leave each
// CTA's 128 rows of the K-block partial sums in its own TMEM.  Each CTA's
// eight epilogue warps then do exactly what the wide router's do (K-block
// promotion in fp32, scored output), so the logits are bit-identical to it.
// Barriers: the leader's full[stage] counts both CTAs' TMA bytes (the peer's
// loads complete on it across the pair); the MMA commits arrive on empty[] and
// tfull[] of both CTAs; the leader's tempty[] counts both CTAs' epilogue warps.
struct PairRouterCfg {
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;   // this CTA's 128 token rows
    static constexpr int B_PART = 128 * GEMM_BK * 2;        // this CTA's 128 experts of one part
    static constexpr int STAGE_BYTES = A_BYTES + 3 * B_PART; // 64 KB
    static constexpr int STAGES = 3;
    static constexpr int SLOTS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(256, 256, false, false);
    static constexpr int NBARS = 2 * STAGES + 2 * SLOTS + 1;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + NBARS * 8 + 16 + 256 * 4 /*bias*/;
    static_assert(SMEM <= 232448, "more than 227 KB of shared memory");
};
static_assert(GemmCfg<GK_ROUTER_WIDE>::SLOTS == PairRouterCfg::SLOTS && GemmCfg<GK_ROUTER_WIDE>::BN == 256,
              "the pair router reuses the wide router's epilogue");

constexpr int PAIR_THREADS = 64 + 32 * 8;

__global__ void __launch_bounds__(PAIR_THREADS, 1) router_pair_kernel(const __grid_constant__ GemmParams p)
{
    using C = PairRouterCfg;
    extern __shared__ uint8_t dsmem[];
    const uint32_t raw = smem_u32(dsmem);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = dsmem + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base_ptr + C::STAGES * C::STAGE_BYTES);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + C::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    float *sbias = reinterpret_cast<float *>(tmem_holder + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int st) { return bar0 + 8u * st; };
    auto empty_bar = [&](int st) { return bar0 + 8u * (C::STAGES + st); };
    const uint32_t tfull0 = bar0 + 8u * (2 * C::STAGES);
    const uint32_t tempty0 = tfull0 + 8u * C::SLOTS;
    const uint32_t fin_bar = tempty0 + 8u * C::SLOTS;

    if (threadIdx.x == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            mbar_init(full_bar(st), 1);
            mbar_init(empty_bar(st), 1);
        }
        for (int a = 0; a < C::SLOTS; ++a) {
            mbar_init(tfull0 + 8u * a, 1);
            // this CTA's epilogue warps; the leader's also counts the peer's forwarder
            mbar_init(tempty0 + 8u * a, 8 + (leader ? 1 : 0));
        }
        mbar_init(fin_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&p.tmA0);
        tma_prefetch_map(&p.tmB0);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();            // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    pdl_wait();

    const int npairs = (int)gridDim.x / 2;
    const int pair = (int)blockIdx.x / 2;
    const int num_tiles = p.num_tiles_static;           // 256-token tiles
    const unsigned long long limit = p.wait_limit_ns ? p.wait_limit_ns : WAIT_LIMIT_NS;
    bool aborted_peer_loads = false;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            const uint32_t full_leader0 = mapa_shared(full_bar(0), 0);
            // every hidden row is read by one CTA once: its lines go first
            // when L2 needs room, so that the scores this kernel writes stay
            // there for the routing kernel that reads them next
            const uint64_t once = l2_policy_evict_first();
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int tile = pair + n * npairs;
                if (tile >= num_tiles)
                    break;
                const int a_row = tile * 256 + (int)rank * GEMM_BM;
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = base + stage * C::STAGE_BYTES;
                    if (leader)
                        mbar_arrive_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
                    const uint32_t fb = full_leader0 + 8u * stage;
                    tma_load_2d_pair_hint(sA, &p.tmA0, fb, kb * GEMM_BK, a_row, once);
#pragma unroll
                    for (int part = 0; part < 3; ++part)
                        tma_load_2d_pair(sA + C::A_BYTES + part * C::B_PART, &p.tmB0, fb, kb * GEMM_BK,
                                         part * p.E + (int)rank * 128);
                    // pull this CTA's hidden rows ROUTER_PF K blocks ahead into L2
                    const int q = n * p.kblocks + kb + ROUTER_PF;
                    const int pt = pair + (q / p.kblocks) * npairs;
                    const int prow = pt * 256 + (int)rank * GEMM_BM;
                    if (pt < num_tiles && prow < p.T)
                        tma_prefetch_l2_2d_hint(&p.tmA0, (q % p.kblocks) * GEMM_BK, prow, once);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    // the leader's full barriers count both CTAs' copies in flight
                    for (int st = 0; st < C::STAGES; ++st)
                        if ((issued >> st) & 1u)
                            mbar_drain(full_bar(st), (issued_parity >> st) & 1u);
                } else {
                    aborted_peer_loads = issued != 0;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            uint32_t ctr = 0;   // K-block slots used so far
            for (int n = 0; ok; ++n) {
                const int tile = pair + n * npairs;
                if (tile >= num_tiles)
                    break;
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
                    if (kb % ROUTER_KPS == 0) {
                        // (the peer's forwarder arrives here across the pair)
                        if (!mbar_wait_cluster(tempty0 + 8u * slot, par ^ 1u, abort_flag, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = base + stage * C::STAGE_BYTES;
                    const uint32_t d = tmem + slot * 256;
#pragma unroll
                    for (int kk = 0; kk < GEMM_BK / 16; ++kk) {
                        const uint64_t ad = sdesc_kmajor_sw128(sA + kk * 32);
#pragma unroll
                        for (int part = 0; part < 3; ++part)
                            umma_bf16_pair(d, ad, sdesc_kmajor_sw128(sA + C::A_BYTES + part * C::B_PART + kk * 32),
                                           C::IDESC, (kk > 0 || part > 0 || kb % ROUTER_KPS != 0) ? 1u : 0u);
                    }
                    umma_commit_pair(empty_bar(stage), 0x3);          // both CTAs' stage is read
                    if (kb % ROUTER_KPS == ROUTER_KPS - 1 || kb == p.kblocks - 1) {
                        umma_commit_pair(tfull0 + 8u * slot, 0x3);    // the slot's partial sum ready in both TMEMs
                        ++ctr;
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // no MMA may still be writing either CTA's TMEM when it is freed
            umma_commit_pair(fin_bar, 0x1);
            mbar_drain(fin_bar, 0);
        } else if (lane == 0) {
            // ------------------------------------------- the peer's forwarder
            // hands each TMEM slot back to the leader's MMA issuer once this
            // CTA's epilogue warps have read it (their local arrivals need no
            // cluster-scope release)
            const uint32_t tempty_leader = mapa_shared(tempty0, 0);
            const int groups = (p.kblocks + ROUTER_KPS - 1) / ROUTER_KPS;
            uint32_t ctr = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int tile = pair + n * npairs;
                if (tile >= num_tiles)
                    break;
                for (int g = 0; g < groups; ++g, ++ctr) {
                    const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
                    if (!mbar_wait(tempty0 + 8u * slot, par, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_cluster(tempty_leader + 8u * slot);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        uint32_t ctr = 0;
        if (p.gscore) {
            for (int e = threadIdx.x - 64; e < p.E; e += 32 * 8)
                sbias[e] = p.bias ? p.bias[e] : 0.0f;
            asm volatile("bar.sync 1, %0;" ::"r"(32 * 8) : "memory");
        }
        for (int n = 0;; ++n) {
            const int tile = pair + n * npairs;
            if (tile >= num_tiles)
                break;
            TileInfo ti;
            ti.group = 0;
            ti.shared = 0;
            ti.nt = 0;
            ti.kp = 0;
            ti.b_row = 0;
            ti.kblocks = p.kblocks;
            ti.a_row = tile * 256 + (int)rank * GEMM_BM;
            ti.out_row = ti.a_row;
            ti.rows = min(GEMM_BM, p.T - ti.a_row);     // <= 0: the pair's last tile ends in the other CTA
            if (!router_epilogue_tile<GK_ROUTER_WIDE>(p, ti, tmem, quad, (warp - 2) >> 2, lane, tfull0, tempty0,
                                                      ctr, abort_flag, nullptr, limit, tile, sbias))
                break;
        }
    }

    __syncwarp();
    if (aborted_peer_loads) {
        // loads of this CTA complete on the leader's barriers, which this CTA
        // cannot wait on: give copies in flight time to land before the pair
        // leaves (only after a wait has run out)
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 100000ull) {
        }
    }
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(p.status, ST_TIMEOUT);
}

// ---------------------------------------------------------------------------
// GK_DOWN_PAIR: the grouped down GEMM on CTA pairs (tcgen05 cta_group::2).
// A pair tile is 256 consecutive rows of one bucket (the pair-tile list of
// bucket_scatter) x 256 hidden columns: each CTA loads its own 128 rows of the
// intermediate and 128 of the 256 W_down columns (two 64-column MN-major
// atoms), so a stage is 16 + 16 KB instead of 16 + 32 KB and six stages fit
// beside the epilogue's staging buffers; the even CTA issues M = 256, N = 256
// MMAs over both CTAs' shared memory and each CTA's TMEM receives its 128 rows.
// Rows of a pair tile beyond its bucket (the bucket's last tile) belong to the
// next bucket or to nothing; their results are never stored.  The epilogue is
// the single-CTA down GEMM's (bf16 rows, TMA stores), per CTA.
struct PairDownCfg {
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;   // 16 KB
    static constexpr int B_ATOM = 64 * GEMM_BK * 2;         // 64 columns x 64 K, 8 KB
    static constexpr int B_BYTES = 2 * B_ATOM;              // this CTA's 128 columns
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 6;
    static constexpr int SLOTS = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int NBUF = 2;
    static constexpr uint32_t IDESC = idesc_bf16_f32(256, 256, false, true);
    static constexpr int STAGING = NBUF * 4 * 4096;
    static constexpr int NBARS = 2 * STAGES + 2 * SLOTS + 1;
    static constexpr int SMEM = STAGES * STAGE_BYTES + STAGING + 1024 /*align*/ + NBARS * 8 + 16;
    static_assert(SMEM <= 232448, "more than 227 KB of shared memory");
    static_assert(STAGE_BYTES % 1024 == 0, "swizzle atoms need 1024-B alignment");
};
static_assert(GemmCfg<GK_DOWN>::NBUF == PairDownCfg::NBUF, "the pair down GEMM reuses the down GEMM's epilogue");

constexpr int PAIR_DOWN_THREADS = 64 + 32 * 4;

__global__ void __launch_bounds__(PAIR_DOWN_THREADS, 1) down_pair_kernel(const __grid_constant__ GemmParams p)
{
    using C = PairDownCfg;
    extern __shared__ uint8_t dsmem[];
    const uint32_t raw = smem_u32(dsmem);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = dsmem + (base - raw);
    uint8_t *staging = base_ptr + C::STAGES * C::STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + C::STAGING);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + C::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int st) { return bar0 + 8u * st; };
    auto empty_bar = [&](int st) { return bar0 + 8u * (C::STAGES + st); };
    const uint32_t tfull0 = bar0 + 8u * (2 * C::STAGES);
    const uint32_t tempty0 = tfull0 + 8u * C::SLOTS;
    const uint32_t fin_bar = tempty0 + 8u * C::SLOTS;

    if (threadIdx.x == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            mbar_init(full_bar(st), 1);
            mbar_init(empty_bar(st), 1);
        }
        for (int a = 0; a < C::SLOTS; ++a) {
            mbar_init(tfull0 + 8u * a, 1);
            // this CTA's epilogue warps; the leader's also counts the peer's forwarder
            mbar_init(tempty0 + 8u * a, 4 + (leader ? 1 : 0));
        }
        mbar_init(fin_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&p.tmA0);
        tma_prefetch_map(&p.tmB0);
        tma_prefetch_map(&p.tmB1);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();            // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    pdl_wait();                // the pair-tile list and the A rows come from earlier kernels

    const int npairs = (int)gridDim.x / 2;
    const int pair = (int)blockIdx.x / 2;
    const int num_tiles = (*p.num_mtiles) * p.n_tiles;
    const unsigned long long limit = p.wait_limit_ns ? p.wait_limit_ns : WAIT_LIMIT_NS;
    bool aborted_peer_loads = false;

    // this CTA's half of pair tile `tile`
    auto half_tile = [&](int tile) {
        const int4 m = p.mtiles[tile / p.n_tiles];
        TileInfo ti;
        ti.group = m.x;
        ti.shared = (m.x == p.E);
        ti.nt = tile % p.n_tiles;
        ti.kblocks = p.kblocks;
        ti.kp = 0;
        ti.b_row = 0;
        ti.a_row = (ti.shared ? p.kT + m.y : m.y) + (int)rank * GEMM_BM;   // intermediate rows
        ti.out_row = ti.a_row;
        ti.rows = min(GEMM_BM, m.z - (int)rank * GEMM_BM);                 // <= 0: nothing to store
        return ti;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            const uint32_t full_leader0 = mapa_shared(full_bar(0), 0);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int tile = pair + n * npairs;
                if (tile >= num_tiles)
                    break;
                const TileInfo ti = half_tile(tile);
                const CUtensorMap *mb = ti.shared ? &p.tmB1 : &p.tmB0;
                const int col0 = ti.nt * 256 + (int)rank * 128;
                // a half with no rows of the bucket (its last pair tile ends in
                // the even CTA) loads rows past the end of the intermediate:
                // TMA fills them with zeros without reading memory
                const int a_row = ti.rows > 0 ? ti.a_row : p.kT + p.T;
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = base + stage * C::STAGE_BYTES;
                    if (leader)
                        mbar_arrive_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
                    const uint32_t fb = full_leader0 + 8u * stage;
                    const int k0 = kb * GEMM_BK;
                    const int krow = (ti.shared ? 0 : ti.group * p.I) + k0;
                    tma_load_2d_pair(sA, &p.tmA0, fb, k0, a_row);
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        tma_load_2d_pair(sA + C::A_BYTES + q * C::B_ATOM, mb, fb, col0 + q * 64, krow);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    for (int st = 0; st < C::STAGES; ++st)
                        if ((issued >> st) & 1u)
                            mbar_drain(full_bar(st), (issued_parity >> st) & 1u);
                } else {
                    aborted_peer_loads = issued != 0;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            uint32_t ctr = 0;   // tile accumulators used so far
            for (int n = 0; ok; ++n) {
                const int tile = pair + n * npairs;
                if (tile >= num_tiles)
                    break;
                const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
                // (the peer's forwarder arrives here across the pair)
                if (!mbar_wait_cluster(tempty0 + 8u * slot, par ^ 1u, abort_flag, limit))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + slot * 256;
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sA = base + stage * C::STAGE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < GEMM_BK / 16; ++kk)
                        // 16 K rows = two 8-row atoms = 2048 B further into each 64-wide N atom
                        umma_bf16_pair(d, sdesc_kmajor_sw128(sA + kk * 32),
                                       sdesc_mnmajor_sw128(sA + C::A_BYTES + kk * 2048, C::B_ATOM), C::IDESC,
                                       (kb > 0 || kk > 0) ? 1u : 0u);
                    umma_commit_pair(empty_bar(stage), 0x3);          // both CTAs' stage is read
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) {
                    umma_commit_pair(tfull0 + 8u * slot, 0x3);        // tile accumulator ready in both TMEMs
                    ++ctr;
                }
            }
            umma_commit_pair(fin_bar, 0x1);
            mbar_drain(fin_bar, 0);
        } else if (lane == 0) {
            // ------------------------------------------- the peer's forwarder
            const uint32_t tempty_leader = mapa_shared(tempty0, 0);
            uint32_t ctr = 0;
            for (int n = 0;; ++n, ++ctr) {
                const int tile = pair + n * npairs;
                if (tile >= num_tiles)
                    break;
                const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
                if (!mbar_wait(tempty0 + 8u * slot, par, abort_flag, limit))
                    break;
                mbar_arrive_cluster(tempty_leader + 8u * slot);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        uint8_t *stage = staging + (warp - 2) * (C::NBUF * 4096);
        int buf = 0;
        uint32_t ctr = 0;
        for (int n = 0;; ++n) {
            const int tile = pair + n * npairs;
            if (tile >= num_tiles)
                break;
            const TileInfo ti = half_tile(tile);
            const uint32_t slot = ctr % C::SLOTS, par = (ctr / C::SLOTS) & 1u;
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait(tfull0 + 8u * slot, par, abort_flag, limit) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            __syncwarp();
            tc_fence_after();
            const uint32_t tacc = tmem + ((uint32_t)(quad * 32) << 16) + slot * 256;
            epilogue_tile<GK_DOWN>(p, ti, tacc, quad, lane, stage, buf);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(tempty0 + 8u * slot);   // (the peer's forwarder passes it on to the leader)
            ++ctr;
        }
        if (lane == 0)
            bulk_wait_group_all();              // this warp's output stores have completed
    }

    __syncwarp();
    if (aborted_peer_loads) {
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 100000ull) {
        }
    }
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(p.status, ST_TIMEOUT);
}

int gemm_smem_bytes(int kind)
{
    switch (kind) {
    case GK_ROUTER_PAIR: return PairRouterCfg::SMEM;
    case GK_DOWN_PAIR: return PairDownCfg::SMEM;
    case GK_ROUTER: return GemmLayout<GK_ROUTER>::SMEM;
    case GK_ROUTER_WIDE: return GemmLayout<GK_ROUTER_WIDE>::SMEM;
    case GK_ROUTER_FUSED: return GemmLayout<GK_ROUTER_FUSED>::SMEM;
    case GK_GATE_UP: return GemmLayout<GK_GATE_UP>::SMEM;
    case GK_GATE_UP_SMALL: return GemmLayout<GK_GATE_UP_SMALL>::SMEM;
    case GK_DOWN_SMALL: return GemmLayout<GK_DOWN_SMALL>::SMEM;
    case GK_DOWN_COMBINE: return GemmLayout<GK_DOWN_COMBINE>::SMEM;
    case GK_GATE_UP_BWD: return GemmLayout<GK_GATE_UP_BWD>::SMEM;
    case GK_DGRAD_DOWN: return GemmLayout<GK_DGRAD_DOWN>::SMEM;
    case GK_WGRAD: return GemmLayout<GK_WGRAD>::SMEM;
    default: return GemmLayout<GK_DOWN>::SMEM;
    }
}

int gemm_tmem_cols(int kind)
{
    if (kind == GK_ROUTER_PAIR)
        return PairRouterCfg::TMEM_COLS;
    if (kind == GK_DOWN_PAIR)
        return PairDownCfg::TMEM_COLS;
    switch (kind) {
    case GK_ROUTER: return GemmCfg<GK_ROUTER>::TMEM_COLS;
    case GK_ROUTER_WIDE: case GK_ROUTER_FUSED: return GemmCfg<GK_ROUTER_WIDE>::TMEM_COLS;
    case GK_GATE_UP: case GK_GATE_UP_SMALL: return GemmCfg<GK_GATE_UP>::TMEM_COLS;
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
    const cudaError_t le = launch_pdl(umma_gemm_kernel<KIND>, dim3(grid), dim3(kind_threads(KIND)),
                                      (size_t)GemmLayout<KIND>::SMEM, s, p);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// A CTA-pair kernel: grid = 2 x clusters (at most what fits at once), each
// cluster two CTAs on one TPC, with programmatic stream serialisation.
template <int KIND>
static cudaError_t launch_pair(const GemmParams &p, int grid, cudaStream_t s)
{
    constexpr bool ROUTER = (KIND == GK_ROUTER_PAIR);
    auto kernel = ROUTER ? router_pair_kernel : down_pair_kernel;
    constexpr int SMEM = ROUTER ? PairRouterCfg::SMEM : PairDownCfg::SMEM;
    constexpr int THREADS = ROUTER ? PAIR_THREADS : PAIR_DOWN_THREADS;
    static int configured_device = -1;
    static int max_clusters = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess)
            return e;
        cfg.gridDim = dim3(2);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        if (e != cudaSuccess)
            return e;
        if (n < 1)
            return cudaErrorInvalidConfiguration;
        max_clusters = n;
        configured_device = dev;
    }
    const int clusters = std::max(1, std::min(grid / 2, max_clusters));
    cfg.gridDim = dim3(2 * clusters);
    const cudaError_t le = cudaLaunchKernelEx(&cfg, kernel, p);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

cudaError_t launch_gemm(int kind, const GemmParams &p, int grid, cudaStream_t s)
{
    switch (kind) {
    case GK_ROUTER_PAIR: return launch_pair<GK_ROUTER_PAIR>(p, grid, s);
    case GK_DOWN_PAIR: return launch_pair<GK_DOWN_PAIR>(p, grid, s);
    case GK_ROUTER: return launch_kind<GK_ROUTER>(p, grid, s);
    case GK_ROUTER_WIDE: return launch_kind<GK_ROUTER_WIDE>(p, grid, s);
    case GK_ROUTER_FUSED: return launch_kind<GK_ROUTER_FUSED>(p, grid, s);
    case GK_GATE_UP: return launch_kind<GK_GATE_UP>(p, grid, s);
    case GK_GATE_UP_SMALL: return launch_kind<GK_GATE_UP_SMALL>(p, grid, s);
    case GK_DOWN_SMALL: return launch_kind<GK_DOWN_SMALL>(p, grid, s);
    case GK_DOWN_COMBINE: return launch_kind<GK_DOWN_COMBINE>(p, grid, s);
    case GK_GATE_UP_BWD: return launch_kind<GK_GATE_UP_BWD>(p, grid, s);
    case GK_DGRAD_DOWN: return launch_kind<GK_DGRAD_DOWN>(p, grid, s);
    case GK_WGRAD: return launch_kind<GK_WGRAD>(p, grid, s);
    default: return launch_kind<GK_DOWN>(p, grid, s);
    }
}

}  // namespace glr
