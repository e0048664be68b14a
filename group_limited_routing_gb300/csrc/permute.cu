// Bucketing (permute) and combine kernels of the MoE layer forward (SIMT, sm_103a).
//
// The routing page ("InternLumina-U2中256个专家的路由秘密：分组受限Top-K、Expert
// Bias与Fused MoE详解", section 四, the eager inference path) sorts tokens into
// one bucket per expert, runs each bucket through its expert and sums the
// weighted results.  Here:
//   bucket_hist    per PERM_CHUNK-token chunk, hits per expert  (reads topk_idx)
//   bucket_scan    each chunk's start inside every bucket (relative) and the
//                  bucket sizes
//   bucket_scatter bucket offsets (exclusive scan of the sizes) and, block 0,
//                  the m-tile list of the grouped GEMMs (the shared expert is
//                  group E, all T tokens); then, per chunk:
//                  stable slot of every (token, j) pair -- slots in a bucket in
//                  ascending (token, j) order -- and the gather of hidden rows
//                  into the bucketed activation matrix X_perm
//   bucket_tiles   after the fused router (which bucketed the pairs itself):
//                  bucket offsets and the m-tile list only
//   combine        out[t] = bf16( sum_j w[t,j] * Y[slot(t,j)] + Y_shared[t]
//                  (+ residual[t]) ) in fp32 (section 五: the shared expert is
//                  added directly)
// Everything is deterministic: no float atomics, fixed summation order.
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"

namespace glr {

// ---------------------------------------------------------------------------
// Per-chunk expert histograms hist[e][c] (chunks of PERM_CHUNK tokens).  A
// block counts HIST_CHUNKS consecutive chunks in shared memory and writes each
// expert's HIST_CHUNKS counts side by side (fewer, fuller stores than one
// block per chunk).
constexpr int HIST_CHUNKS = 4;

__global__ void __launch_bounds__(256) bucket_hist_kernel(const int32_t *__restrict__ idx, int T, int E, int K,
                                                          int nchunk, int32_t *__restrict__ hist,
                                                          int *__restrict__ status)
{
    pdl_wait();
    extern __shared__ int sh[];                     // [HIST_CHUNKS][E]
    for (int i = threadIdx.x; i < HIST_CHUNKS * E; i += blockDim.x)
        sh[i] = 0;
    __syncthreads();
    const int c0 = blockIdx.x * HIST_CHUNKS;
    const long long n0 = (long long)c0 * PERM_CHUNK * K;
    const long long n1 = min((long long)T * K, n0 + (long long)HIST_CHUNKS * PERM_CHUNK * K);
    bool bad = false;
    for (long long i = n0 + threadIdx.x; i < n1; i += blockDim.x) {
        const int e = idx[i];
        const int q = (int)((i - n0) / (PERM_CHUNK * K));
        if (e >= 0 && e < E)
            atomicAdd(&sh[q * E + e], 1);
        else
            bad = true;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0)
        atomicOr(status, ST_BAD_INDEX);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
#pragma unroll
        for (int q = 0; q < HIST_CHUNKS; ++q)
            if (c0 + q < nchunk)
                hist[(size_t)e * nchunk + c0 + q] = sh[q * E + e];   // [expert][chunk]
}

cudaError_t launch_bucket_hist(const int32_t *idx, int T, int E, int k, int32_t *hist, int *status, cudaStream_t s)
{
    const int nchunk = (T + PERM_CHUNK - 1) / PERM_CHUNK;
    const int blocks = (nchunk + HIST_CHUNKS - 1) / HIST_CHUNKS;
    const cudaError_t le = launch_pdl(bucket_hist_kernel, dim3(blocks), dim3(256), HIST_CHUNKS * E * sizeof(int), s,
                                      idx, T, E, k, nchunk, hist, status);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// Per-bucket scan: one block per expert.  hist is [expert][chunk]; in place,
// hist[e][c] becomes the number of bucket-e rows of the chunks before c, and
// sizes[e] the bucket's size.  Thread i takes a run of consecutive chunks:
// its run's sum, a block-wide exclusive scan of the 256 sums (warp shuffles,
// then the 8 warp totals in warp order), then the run is rewritten in place.
// The bucket offsets follow in bucket_scatter.
__global__ void __launch_bounds__(256) bucket_scan_kernel(int32_t *__restrict__ hist, int nchunk, int E,
                                                          int32_t *__restrict__ sizes, int32_t *__restrict__ sizes2)
{
    pdl_wait();
    __shared__ int wtot[8];
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int32_t *row = hist + (size_t)e * nchunk;
    const int per = (nchunk + blockDim.x - 1) / blockDim.x;
    const int c0 = threadIdx.x * per;
    const int c1 = min(nchunk, c0 + per);
    // runs of up to SCAN_REG chunks stay in registers between the two passes
    // (16-byte loads and stores when the rows and runs allow it)
    constexpr int SCAN_REG = 16;
    int v[SCAN_REG];
    const bool in_regs = per <= SCAN_REG;
    const bool vec = in_regs && (per % 4 == 0) && (nchunk % 4 == 0);
    int sum = 0;
    if (vec) {
#pragma unroll
        for (int q = 0; q < SCAN_REG / 4; ++q) {
            if (4 * q < per && c0 + 4 * q < nchunk) {
                const int4 x = *reinterpret_cast<const int4 *>(row + c0 + 4 * q);
                v[4 * q] = x.x;
                v[4 * q + 1] = x.y;
                v[4 * q + 2] = x.z;
                v[4 * q + 3] = x.w;
            } else {
                v[4 * q] = v[4 * q + 1] = v[4 * q + 2] = v[4 * q + 3] = 0;
            }
        }
#pragma unroll
        for (int i = 0; i < SCAN_REG; ++i)
            sum += v[i];
    } else if (in_regs) {
#pragma unroll
        for (int i = 0; i < SCAN_REG; ++i) {
            v[i] = (i < per && c0 + i < c1) ? row[c0 + i] : 0;
            sum += v[i];
        }
    } else {
        for (int c = c0; c < c1; ++c)
            sum += row[c];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off)
            incl += y;
    }
    if (lane == 31)
        wtot[w] = incl;
    __syncthreads();
    int run = incl - sum;                         // exclusive within the warp
    for (int q = 0; q < w; ++q)
        run += wtot[q];
    if (vec) {
#pragma unroll
        for (int q = 0; q < SCAN_REG / 4; ++q) {
            int4 x;
            x.x = run;
            run += v[4 * q];
            x.y = run;
            run += v[4 * q + 1];
            x.z = run;
            run += v[4 * q + 2];
            x.w = run;
            run += v[4 * q + 3];
            if (4 * q < per && c0 + 4 * q < nchunk)
                *reinterpret_cast<int4 *>(row + c0 + 4 * q) = x;
        }
    } else if (in_regs) {
#pragma unroll
        for (int i = 0; i < SCAN_REG; ++i) {
            if (i < per && c0 + i < c1)
                row[c0 + i] = run;
            run += v[i];
        }
    } else {
        for (int c = c0; c < c1; ++c) {
            const int h = row[c];
            row[c] = run;
            run += h;
        }
    }
    if (threadIdx.x == blockDim.x - 1) {
        sizes[e] = run;                           // the last run ends at the bucket's size
        if (sizes2)
            sizes2[e] = run;                      // (moe_layer's expert_counts output)
    }
}

cudaError_t launch_bucket_scan(int32_t *hist, int nchunk, int E, int32_t *sizes, cudaStream_t s, int32_t *sizes2)
{
    const cudaError_t le = launch_pdl(bucket_scan_kernel, dim3(E), dim3(256), 0, s, hist, nchunk, E, sizes, sizes2);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// Bucket offsets (exclusive scan of the E sizes, each rounded up to `pad`
// rows: 1 for the forward, BWD_ROW_ALIGN for the backward) and first m-tile of
// every group, by a 256-thread block into shared memory; thread 0 also checks
// that every pair was bucketed.  With `write_tiles`, the block writes the
// m-tile list of the grouped GEMMs (the shared expert is group E, all T
// tokens) and, when eoff is given, every bucket's (first row, padded rows),
// the shared expert's rows starting at shared_base.  With cap > 0 the routed
// rows were bucketed at e * cap + r (the fused router's layout): the fourth
// field of every m-tile is then its first A row (the token for the shared
// expert's m-tiles).
//
// With ptiles (the forward's CTA-pair GEMMs), the block also writes the list
// of pair tiles: every bucket (and the shared expert's T rows) cut into
// 256-row tiles {group, first row, rows <= 256, 0}, their count in
// hdr->num_ptiles.
__device__ void bucket_offsets(const int32_t *__restrict__ sizes, int T, int E, int K, int *offset, int *tstart,
                               int *wsum_rows, int *wsum_tiles, bool write_tiles, int4 *__restrict__ mtiles,
                               WsHeader *__restrict__ hdr, int pad = 1, int2 *__restrict__ eoff = nullptr,
                               int shared_base = 0, int cap = 0, int4 *__restrict__ ptiles = nullptr,
                               bool with_shared = true)
{
    __shared__ int true_rows;
    __shared__ int wsum_pt[8];
    __shared__ int pt_total;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int e = threadIdx.x;   // blockDim.x == 256 >= E
    const int n0 = (e < E) ? sizes[e] : 0;
    const int n = (n0 + pad - 1) / pad * pad;    // rows the bucket occupies
    const int nt = (n0 + GEMM_BM - 1) / GEMM_BM;
    const int np = (n0 + 2 * GEMM_BM - 1) / (2 * GEMM_BM);
    if (threadIdx.x == 0)
        true_rows = 0;
    __syncthreads();
    if (n0)
        atomicAdd(&true_rows, n0);               // integer: exact in any order
    int a = n, b = nt, c = np;   // inclusive warp scans
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, a, off);
        const int yb = __shfl_up_sync(0xffffffffu, b, off);
        const int yc = __shfl_up_sync(0xffffffffu, c, off);
        if (lane >= off) {
            a += ya;
            b += yb;
            c += yc;
        }
    }
    if (lane == 31) {
        wsum_rows[w] = a;
        wsum_tiles[w] = b;
        wsum_pt[w] = c;
    }
    __syncthreads();
    int ra = 0, rb = 0, rc = 0;
    for (int q = 0; q < w; ++q) {
        ra += wsum_rows[q];
        rb += wsum_tiles[q];
        rc += wsum_pt[q];
    }
    offset[e] = ra + a - n;
    tstart[e] = rb + b - nt;
    const int pstart = rc + c - np;
    __syncthreads();
    if (threadIdx.x == 0) {
        int off = 0, tiles = 0, pts = 0;
        for (int q = 0; q < 8; ++q) {
            off += wsum_rows[q];
            tiles += wsum_tiles[q];
            pts += wsum_pt[q];
        }
        offset[E] = off;             // padded rows of all buckets (== K*T for pad 1 and valid indices)
        tstart[E] = tiles;
        pt_total = pts;
        if (write_tiles && ptiles) {
            hdr->num_ptiles = pts + (with_shared ? (T + 2 * GEMM_BM - 1) / (2 * GEMM_BM) : 0);
            hdr->num_ptiles_routed = pts;
        }
        if (write_tiles) {
            hdr->num_mtiles = tiles + (with_shared ? (T + GEMM_BM - 1) / GEMM_BM : 0);
            if (true_rows != K * T)
                atomicOr(&hdr->status, ST_COUNT_MISMATCH);
            if (eoff)
                eoff[E] = make_int2(shared_base, (T + pad - 1) / pad * pad);
        }
    }
    __syncthreads();
    if (write_tiles) {
        if (e < E && eoff)
            eoff[e] = make_int2(offset[e], n);
        if (e < E)
            for (int i = 0, r = 0; r < n0; ++i, r += GEMM_BM)
                mtiles[tstart[e] + i] = make_int4(e, offset[e] + r, min(GEMM_BM, n0 - r), cap > 0 ? e * cap + r : 0);
        const int ntile_sh = with_shared ? (T + GEMM_BM - 1) / GEMM_BM : 0;
        for (int i = threadIdx.x; i < ntile_sh; i += blockDim.x)
            mtiles[tstart[E] + i] = make_int4(E, i * GEMM_BM, min(GEMM_BM, T - i * GEMM_BM), cap > 0 ? i * GEMM_BM : 0);
        if (ptiles) {
            constexpr int PM = 2 * GEMM_BM;
            if (e < E)
                for (int i = 0, r = 0; r < n0; ++i, r += PM)
                    ptiles[pstart + i] = make_int4(e, offset[e] + r, min(PM, n0 - r), 0);
            const int np_sh = with_shared ? (T + PM - 1) / PM : 0;
            for (int i = threadIdx.x; i < np_sh; i += blockDim.x)
                ptiles[pt_total + i] = make_int4(E, i * PM, min(PM, T - i * PM), 0);
        }
    }
}

// A 16-byte store marked as streaming (evict first): the bucketed copy of the
// rows is written once and read once by the next kernel, and should not push
// other lines out of L2 on the way.
__device__ __forceinline__ void st_global_streaming(uint4 *p, const uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Stable slots for one chunk, then the row gather.  Warp 0 assigns slots in
// (token, j) order, 32 pairs at a time: lanes holding the same expert find
// each other with __match_any_sync and take consecutive slots by lane rank.
// With `bw` (the backward), buckets start on BWD_ROW_ALIGN-row boundaries,
// every bucket row also receives the token's output gradient row (unweighted)
// and its routing weight, and the shared expert's rows (after the padded
// routed rows) receive every token's gradient row with weight 1.
struct ScatterBwd {
    const uint16_t *dout;   // [T, H]
    const float *w;         // [T, K]
    uint16_t *do_perm;      // [rows, H]
    float *w_perm;          // [rows]
    int2 *eoff;             // [E + 1]
    int shared_base;        // first shared-expert row (past every routed row for any routing)
};

template <bool EARLY>
__global__ void __launch_bounds__(256) bucket_scatter_kernel(const int32_t *__restrict__ idx,
                                                             const uint16_t *__restrict__ x,
                                                             const int32_t *__restrict__ chunk_base,
                                                             const int32_t *__restrict__ sizes, int T, int H,
                                                             int E, int K, int32_t *__restrict__ slot_of,
                                                             uint16_t *__restrict__ x_perm, int4 *__restrict__ mtiles,
                                                             WsHeader *__restrict__ hdr, ScatterBwd bw,
                                                             int4 *__restrict__ ptiles, int with_shared)
{
    pdl_wait();
    __shared__ int offset[258];
    __shared__ int tstart[258];
    __shared__ int wsum_rows[8];
    __shared__ int wsum_tiles[8];
    extern __shared__ int sm[];
    int *next = sm;            // [E]   next free slot of each bucket for this chunk
    int *slots = sm + E;       // [PERM_CHUNK * K]
    const int t0 = blockIdx.x * PERM_CHUNK;
    const int nt = min(PERM_CHUNK, T - t0);
    const bool backward = bw.do_perm != nullptr;
    // forward, with a whole number of rows per pass (H / 8 divides the block):
    // every thread loads its 16-byte column of the chunk's rows now, so that
    // the loads are in flight while the offsets and slots are worked out
    const int vec_per_row = H / 8;                    // 16-byte vectors
    const bool early = EARLY && !backward && vec_per_row <= (int)blockDim.x && blockDim.x % vec_per_row == 0;
    const int rpp = early ? (int)blockDim.x / vec_per_row : 1;
    uint4 val_e[EARLY ? PERM_CHUNK : 1];
    if (early) {
        const int sub = threadIdx.x / vec_per_row, v = threadIdx.x % vec_per_row;
#pragma unroll
        for (int u = 0; u < PERM_CHUNK; ++u) {
            const int tt = sub + u * rpp;
            if (u * rpp < PERM_CHUNK && tt < nt)
                val_e[u] = reinterpret_cast<const uint4 *>(x + (size_t)(t0 + tt) * H)[v];
        }
    }
    bucket_offsets(sizes, T, E, K, offset, tstart, wsum_rows, wsum_tiles, blockIdx.x == 0, mtiles, hdr,
                   backward ? BWD_ROW_ALIGN : 1, bw.eoff, bw.shared_base, 0, ptiles, with_shared != 0);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        next[e] = offset[e] + chunk_base[(size_t)e * gridDim.x + blockIdx.x];   // [expert][chunk]
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int n = nt * K;
        const int32_t *src = idx + (size_t)t0 * K;
        for (int base = 0; base < n; base += 32) {
            const int i = base + lane;
            const bool in = i < n;
            const int e = in ? src[i] : -1;
            const bool ok = in && e >= 0 && e < E;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
            int slot = -1;
            if (ok)
                slot = next[e] + __popc(peers & ((1u << lane) - 1u));
            __syncwarp();
            if (ok && (__ffs(peers) - 1) == lane)   // lowest lane of the peer group
                next[e] += __popc(peers);
            __syncwarp();
            if (in) {
                slots[i] = slot;
                slot_of[(size_t)t0 * K + i] = slot;
                if (backward && slot >= 0)
                    bw.w_perm[slot] = bw.w[(size_t)t0 * K + i];
            }
        }
    }
    if (backward)
        for (int tt = threadIdx.x; tt < nt; tt += blockDim.x)
            bw.w_perm[bw.shared_base + t0 + tt] = 1.0f;   // shared-expert rows
    __syncthreads();
    if (early) {
        // each token row read once (above) and written to its K slots
        const int sub = threadIdx.x / vec_per_row, v = threadIdx.x % vec_per_row;
#pragma unroll
        for (int u = 0; u < PERM_CHUNK; ++u) {
            const int tt = sub + u * rpp;
            if (u * rpp < PERM_CHUNK && tt < nt)
                for (int j = 0; j < K; ++j) {
                    const int slot = slots[tt * K + j];
                    if (slot >= 0)
                        st_global_streaming(reinterpret_cast<uint4 *>(x_perm + (size_t)slot * H) + v, val_e[u]);
                }
        }
        return;
    }
    // gather: each token row is read once and written to its K slots
    const int rows_per_pass = blockDim.x / vec_per_row > 0 ? blockDim.x / vec_per_row : 1;
    const int sub = threadIdx.x / vec_per_row;
    const int v = threadIdx.x % vec_per_row;
    if (sub < rows_per_pass) {
        for (int vv = v; vv < vec_per_row; vv += blockDim.x) {
            // four tokens per step so that four loads are in flight per thread
            for (int tl = sub; tl < nt; tl += 4 * rows_per_pass) {
                uint4 val[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int tt = tl + u * rows_per_pass;
                    if (tt < nt)
                        val[u] = reinterpret_cast<const uint4 *>(x + (size_t)(t0 + tt) * H)[vv];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int tt = tl + u * rows_per_pass;
                    if (tt < nt)
                        for (int j = 0; j < K; ++j) {
                            const int slot = slots[tt * K + j];
                            if (slot >= 0)
                                reinterpret_cast<uint4 *>(x_perm + (size_t)slot * H)[vv] = val[u];
                        }
                }
                if (backward) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int tt = tl + u * rows_per_pass;
                        if (tt < nt) {
                            const uint4 g = reinterpret_cast<const uint4 *>(bw.dout + (size_t)(t0 + tt) * H)[vv];
                            reinterpret_cast<uint4 *>(bw.do_perm + (size_t)(bw.shared_base + t0 + tt) * H)[vv] = g;
                            for (int j = 0; j < K; ++j) {
                                const int slot = slots[tt * K + j];
                                if (slot >= 0)
                                    reinterpret_cast<uint4 *>(bw.do_perm + (size_t)slot * H)[vv] = g;
                            }
                        }
                    }
                }
            }
        }
    }
}

cudaError_t launch_bucket_scatter(const int32_t *idx, const uint16_t *x, const int32_t *chunk_base,
                                  const int32_t *sizes, int T, int H, int E, int k, int32_t *slot_of,
                                  uint16_t *x_perm, int4 *mtiles, WsHeader *hdr, cudaStream_t s, int4 *ptiles,
                                  bool with_shared)
{
    const int blocks = (T + PERM_CHUNK - 1) / PERM_CHUNK;
    const size_t smem = (size_t)(E + PERM_CHUNK * k) * sizeof(int);
    const ScatterBwd none = {nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    // (the row loads go out before the slots are known when whole rows fit a
    // pass of the block: H / 8 divides 256)
    const int vpr = H / 8;
    const bool early = vpr <= 256 && 256 % vpr == 0;
    const cudaError_t le = early ? launch_pdl(bucket_scatter_kernel<true>, dim3(blocks), dim3(256), smem, s, idx, x,
                                              chunk_base, sizes, T, H, E, k, slot_of, x_perm, mtiles, hdr, none, ptiles,
                                              with_shared ? 1 : 0)
                                 : launch_pdl(bucket_scatter_kernel<false>, dim3(blocks), dim3(256), smem, s, idx, x,
                                              chunk_base, sizes, T, H, E, k, slot_of, x_perm, mtiles, hdr, none, ptiles,
                                              with_shared ? 1 : 0);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

cudaError_t launch_bucket_scatter_bwd(const int32_t *idx, const uint16_t *x, const int32_t *chunk_base,
                                      const int32_t *sizes, int T, int H, int E, int k, int32_t *slot_of,
                                      uint16_t *x_perm, int4 *mtiles, WsHeader *hdr, const uint16_t *dout,
                                      const float *w, uint16_t *do_perm, float *w_perm, int2 *eoff, int shared_base,
                                      cudaStream_t s)
{
    const int blocks = (T + PERM_CHUNK - 1) / PERM_CHUNK;
    const size_t smem = (size_t)(E + PERM_CHUNK * k) * sizeof(int);
    const ScatterBwd bw = {dout, w, do_perm, w_perm, eoff, shared_base};
    const cudaError_t le = launch_pdl(bucket_scatter_kernel<false>, dim3(blocks), dim3(256), smem, s, idx, x,
                                      chunk_base, sizes, T, H, E, k, slot_of, x_perm, mtiles, hdr, bw, (int4 *)nullptr, 1);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// Zeroes the padding rows of every backward bucket (the weight-gradient GEMMs
// run their K loop over whole 64-row blocks): rows [first + n, first + padded)
// of the routed buckets in x_perm and all three of do_perm, aw, dgu; of the
// shared rows in do_perm, aw, dgu.  Block b takes bucket b (b == E: shared).
__global__ void zero_pad_kernel(const int2 *__restrict__ eoff, const int32_t *__restrict__ sizes, int T, int E,
                                int H, int I, uint16_t *__restrict__ x_perm, uint16_t *__restrict__ do_perm,
                                uint16_t *__restrict__ aw, uint16_t *__restrict__ dgu, int *__restrict__ tile_ctr)
{
    pdl_wait();
    const int e = blockIdx.x;
    if (e == 0 && threadIdx.x < 2)
        tile_ctr[threadIdx.x] = 0;
    const int2 eo = eoff[e];
    const int n = (e < E) ? sizes[e] : T;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int r = eo.x + n; r < eo.x + eo.y; ++r) {
        for (int v = threadIdx.x; v < H / 8; v += blockDim.x) {
            if (e < E)
                reinterpret_cast<uint4 *>(x_perm + (size_t)r * H)[v] = z;
            reinterpret_cast<uint4 *>(do_perm + (size_t)r * H)[v] = z;
        }
        for (int v = threadIdx.x; v < I / 8; v += blockDim.x)
            reinterpret_cast<uint4 *>(aw + (size_t)r * I)[v] = z;
        for (int v = threadIdx.x; v < 2 * I / 8; v += blockDim.x)
            reinterpret_cast<uint4 *>(dgu + (size_t)r * 2 * I)[v] = z;
    }
}

cudaError_t launch_zero_pad(const int2 *eoff, const int32_t *sizes, int T, int E, int H, int I, uint16_t *x_perm,
                            uint16_t *do_perm, uint16_t *aw, uint16_t *dgu, int *tile_ctr, cudaStream_t s)
{
    const cudaError_t le = launch_pdl(zero_pad_kernel, dim3(E + 1), dim3(256), 0, s, eoff, sizes, T, E, H, I, x_perm,
                                      do_perm, aw, dgu, tile_ctr);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// d topk_w[t, j] = sum over the n-tiles of the partial dot products of the
// pair's bucket row (fixed order); a skipped pair gets 0.
__global__ void dw_reduce_kernel(const int32_t *__restrict__ slot_of, const float *__restrict__ dw_part, int n,
                                 int ntiles, float *__restrict__ dw)
{
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    const int slot = slot_of[i];
    float v = 0.0f;
    if (slot >= 0)
        for (int q = 0; q < ntiles; ++q)
            v += dw_part[(size_t)slot * ntiles + q];
    dw[i] = v;
}

cudaError_t launch_dw_reduce(const int32_t *slot_of, const float *dw_part, int n, int ntiles, float *dw,
                             cudaStream_t s)
{
    const cudaError_t le = launch_pdl(dw_reduce_kernel, dim3((n + 255) / 256), dim3(256), 0, s, slot_of, dw_part, n,
                                      ntiles, dw);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// After the fused router (which bucketed every pair at e * T + its slot and
// counted the buckets' sizes): the bucket offsets of the compact layout the
// grouped GEMMs write (offs[e], offs[E] = k T) and the m-tile list, one block.
__global__ void __launch_bounds__(256) bucket_tiles_kernel(const int32_t *__restrict__ sizes, int T, int E, int K,
                                                           int4 *__restrict__ mtiles, WsHeader *__restrict__ hdr,
                                                           int32_t *__restrict__ offs)
{
    pdl_wait();
    __shared__ int offset[257], tstart[257], wr[8], wt[8];
    bucket_offsets(sizes, T, E, K, offset, tstart, wr, wt, true, mtiles, hdr, 1, nullptr, 0, T);
    for (int e = threadIdx.x; e <= E; e += blockDim.x)
        offs[e] = offset[e];
}

cudaError_t launch_bucket_tiles(const int32_t *sizes, int T, int E, int k, int4 *mtiles, WsHeader *hdr,
                                int32_t *offs, cudaStream_t s)
{
    if (E > 256)
        return cudaErrorInvalidValue;
    const cudaError_t le = launch_pdl(bucket_tiles_kernel, dim3(1), dim3(256), 0, s, sizes, T, E, k, mtiles, hdr,
                                      offs);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// Small batches (T <= BUCKET_SMALL_MAX_T): the three bucketing steps in one
// launch.  Every block recomputes the (tiny) bucketing from topk_idx in shared
// memory -- per-expert counts with shared-memory atomics (exact, order-free),
// a block scan gives the bucket offsets, then one warp walks the pairs in
// (token, j) order, 32 at a time, and hands out slots with __match_any_sync,
// so slots are stable exactly as in the general path -- and copies its share
// of the hidden rows into X_perm; block 0 also writes the bucket sizes,
// slot_of and the m-tile list, in tiles of at most `mt` rows (16 for the
// small-T GEMM kinds, else 128; a bucket can exceed T rows when a token lists
// an expert twice), then the shared group (all T tokens).
__global__ void __launch_bounds__(256) bucket_small_kernel(const int32_t *__restrict__ idx,
                                                           const uint16_t *__restrict__ x, int T, int H, int E,
                                                           int K, int mt, int32_t *__restrict__ sizes,
                                                           int32_t *__restrict__ slot_of,
                                                           uint16_t *__restrict__ x_perm, int4 *__restrict__ mtiles,
                                                           WsHeader *__restrict__ hdr)
{
    pdl_wait();
    __shared__ int s_idx[BUCKET_SMALL_MAX_T * 32];
    __shared__ int s_slot[BUCKET_SMALL_MAX_T * 32];
    __shared__ int s_wsum[8][2];
    __shared__ int s_cnt[256];
    __shared__ int s_next[256];
    const int n = T * K;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    s_cnt[tid] = 0;                          // blockDim.x == 256 >= E
    __syncthreads();
    bool bad = false;
    for (int i = tid; i < n; i += blockDim.x) {
        const int e = idx[i];
        const bool ok = e >= 0 && e < E;
        bad |= !ok;
        s_idx[i] = ok ? e : -1;
        s_slot[i] = -1;
        if (ok)
            atomicAdd(&s_cnt[e], 1);
    }
    __syncthreads();
    const int e = tid;
    const int cnt = (e < E) ? s_cnt[e] : 0;
    const int ntile = (cnt + mt - 1) / mt;   // m-tiles of bucket e
    int a = cnt, b = ntile;                  // inclusive warp scans: rows, m-tiles
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, a, off);
        const int yb = __shfl_up_sync(0xffffffffu, b, off);
        if (lane >= off) {
            a += ya;
            b += yb;
        }
    }
    if (lane == 31) {
        s_wsum[w][0] = a;
        s_wsum[w][1] = b;
    }
    __syncthreads();
    int ra = 0, rb = 0, ta = 0, tb = 0;
    for (int q = 0; q < 8; ++q) {
        if (q < w) {
            ra += s_wsum[q][0];
            rb += s_wsum[q][1];
        }
        ta += s_wsum[q][0];
        tb += s_wsum[q][1];
    }
    const int offset = ra + a - cnt;         // first slot of bucket e
    const int tile = rb + b - ntile;         // its first m-tile
    s_next[e] = offset;
    __syncthreads();
    if (w == 0) {
        // stable slots: pairs in (token, j) order, a bucket's rows in that order
        for (int base = 0; base < n; base += 32) {
            const int i = base + lane;
            const int ei = (i < n) ? s_idx[i] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, ei);
            int slot = -1;
            if (ei >= 0)
                slot = s_next[ei] + __popc(peers & ((1u << lane) - 1u));
            __syncwarp();
            if (ei >= 0 && (__ffs(peers) - 1) == lane)   // lowest lane of the peer group
                s_next[ei] += __popc(peers);
            __syncwarp();
            if (i < n)
                s_slot[i] = slot;
        }
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        if (e < E) {
            sizes[e] = cnt;
            for (int q = 0; q < ntile; ++q)
                mtiles[tile + q] = make_int4(e, offset + q * mt, min(mt, cnt - q * mt), 0);
        }
        for (int i = tid; i < n; i += blockDim.x)
            slot_of[i] = s_slot[i];
        const int nsh = (T + mt - 1) / mt;
        for (int q = tid; q < nsh; q += blockDim.x)
            mtiles[tb + q] = make_int4(E, q * mt, min(mt, T - q * mt), 0);
        if (tid == 0) {
            hdr->num_mtiles = tb + nsh;
            if (ta != n)
                atomicOr(&hdr->status, ST_COUNT_MISMATCH);
        }
        if (__syncthreads_or(bad) && tid == 0)
            atomicOr(&hdr->status, ST_BAD_INDEX);
    }
    const int vpr = H / 8;                   // 16-byte vectors per row
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int slot = s_slot[i];
        if (slot < 0)
            continue;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(i / K) * H);
        uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)slot * H);
        for (int v = tid; v < vpr; v += blockDim.x)
            dst[v] = src[v];
    }
}

cudaError_t launch_bucket_small(const int32_t *idx, const uint16_t *x, int T, int H, int E, int k, int mt,
                                int32_t *sizes, int32_t *slot_of, uint16_t *x_perm, int4 *mtiles, WsHeader *hdr,
                                cudaStream_t s)
{
    if (T > BUCKET_SMALL_MAX_T || k > 32 || E > 256 || mt <= 0)
        return cudaErrorInvalidValue;
    const int blocks = T * k;                // one row copy per block
    const cudaError_t le = launch_pdl(bucket_small_kernel, dim3(blocks), dim3(256), 0, s, idx, x, T, H, E, k, mt,
                                      sizes, slot_of, x_perm, mtiles, hdr);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// Dense MLP: every token runs through the one weight set, so the m-tile list
// is just the T tokens in tiles of `mt` rows (the GEMMs' "shared" group).
__global__ void dense_tiles_kernel(int T, int mt, int4 *__restrict__ mtiles, WsHeader *__restrict__ hdr)
{
    pdl_wait();
    const int n = (T + mt - 1) / mt;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        mtiles[i] = make_int4(0, i * mt, min(mt, T - i * mt), 0);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        hdr->num_mtiles = n;
}

cudaError_t launch_dense_tiles(int T, int mt, int4 *mtiles, WsHeader *hdr, cudaStream_t s)
{
    const int n = (T + mt - 1) / mt;
    const cudaError_t le = launch_pdl(dense_tiles_kernel, dim3((n + 255) / 256), dim3(256), 0, s, T, mt, mtiles, hdr);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// out[t] = bf16( Y[K*T + t] + sum_j w[t,j] * Y[slot_of[t,j]] (+ residual[t]) ),
// fp32 accumulation in j order.  A block owns one contiguous slice of the
// tokens (all slices within a token of the same length) and takes it ctok <=
// COMBINE_TOK tokens at a time: their slots and weights are loaded once into
// shared memory, then a thread owns one 16-byte column vector (8 values) of a
// token and issues all of its row loads before the first use.
constexpr int COMBINE_TOK = 32;

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 &v, float wgt)
{
    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(p2[q]);
        acc[2 * q] += wgt * f.x;
        acc[2 * q + 1] += wgt * f.y;
    }
}

// A 16-byte load marked as streaming (evict first): every row of Y is read
// once, by one token.
__device__ __forceinline__ uint4 ld_stream(const uint16_t *p)
{
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// One token's 16-byte column vector: the K expert rows (in batches of eight,
// every load of a batch issued before any use) and the shared row.
__device__ __forceinline__ void combine_one(const uint16_t *__restrict__ Y, const int *s_slot, const float *s_w,
                                            const uint16_t *__restrict__ residual, size_t srow0, int H, int K, int t,
                                            int tl, int vv, uint16_t *__restrict__ out)
{
    float acc[8], racc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        acc[q] = 0.0f;
        racc[q] = 0.0f;
    }
    const uint4 sv = ld_stream(Y + (srow0 + t) * H + (size_t)vv * 8);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int j0 = 0; j0 < K; j0 += 8) {
        uint4 yv[8];
        float wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = j0 + u;
            const int slot = (j < K) ? s_slot[tl * K + j] : -1;
            wv[u] = (slot >= 0) ? s_w[tl * K + j] : 0.0f;
            yv[u] = (slot >= 0) ? ld_stream(Y + (size_t)slot * H + (size_t)vv * 8) : zero;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            add_bf16x8(racc, yv[u], wv[u]);      // skipped pairs hold weight 0 and a zero row
    }
    add_bf16x8(acc, sv, 1.0f);
#pragma unroll
    for (int q = 0; q < 8; ++q)
        acc[q] += racc[q];
    if (residual)
        add_bf16x8(acc, reinterpret_cast<const uint4 *>(residual + (size_t)t * H)[vv], 1.0f);
    uint4 o;
    uint32_t *op = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
        op[q] = *reinterpret_cast<uint32_t *>(&b);
    }
    reinterpret_cast<uint4 *>(out + (size_t)t * H)[vv] = o;
}

// Two tokens at once: both tokens' row loads are issued before any is used
// (same arithmetic, in the same order, as combine_one for each token).
__device__ __forceinline__ void combine_two(const uint16_t *__restrict__ Y, const int *s_slot, const float *s_w,
                                            const uint16_t *__restrict__ residual, size_t srow0, int H, int K,
                                            int ta, int tla, int tb, int tlb, int vv, uint16_t *__restrict__ out)
{
    if (K > 8) {
        combine_one(Y, s_slot, s_w, residual, srow0, H, K, ta, tla, vv, out);
        combine_one(Y, s_slot, s_w, residual, srow0, H, K, tb, tlb, vv, out);
        return;
    }
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint4 ya[8], yb[8];
    float wa[8], wb[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int sa = (u < K) ? s_slot[tla * K + u] : -1;
        const int sb = (u < K) ? s_slot[tlb * K + u] : -1;
        wa[u] = (sa >= 0) ? s_w[tla * K + u] : 0.0f;
        wb[u] = (sb >= 0) ? s_w[tlb * K + u] : 0.0f;
        ya[u] = (sa >= 0) ? ld_stream(Y + (size_t)sa * H + (size_t)vv * 8) : zero;
        yb[u] = (sb >= 0) ? ld_stream(Y + (size_t)sb * H + (size_t)vv * 8) : zero;
    }
    const uint4 sva = ld_stream(Y + (srow0 + ta) * H + (size_t)vv * 8);
    const uint4 svb = ld_stream(Y + (srow0 + tb) * H + (size_t)vv * 8);
    uint4 rva = zero, rvb = zero;
    if (residual) {
        rva = reinterpret_cast<const uint4 *>(residual + (size_t)ta * H)[vv];
        rvb = reinterpret_cast<const uint4 *>(residual + (size_t)tb * H)[vv];
    }
    float acc[8], racc[8];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            acc[q] = 0.0f;
            racc[q] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            add_bf16x8(racc, half ? yb[u] : ya[u], half ? wb[u] : wa[u]);
        add_bf16x8(acc, half ? svb : sva, 1.0f);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            acc[q] += racc[q];
        if (residual)
            add_bf16x8(acc, half ? rvb : rva, 1.0f);
        uint4 o;
        uint32_t *op = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
            op[q] = *reinterpret_cast<uint32_t *>(&b);
        }
        reinterpret_cast<uint4 *>(out + (size_t)(half ? tb : ta) * H)[vv] = o;
    }
}

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t *__restrict__ Y,
                                                      const int32_t *__restrict__ slot_of,
                                                      const float *__restrict__ w,
                                                      const uint16_t *__restrict__ residual, int T, int H, int K,
                                                      int ctok, long long shared_row0, uint16_t *__restrict__ out,
                                                      const int32_t *__restrict__ idx,
                                                      const int32_t *__restrict__ offs, int E, long long y_rows)
{
    pdl_wait();
    __shared__ int s_slot[COMBINE_TOK * 32];
    __shared__ float s_w[COMBINE_TOK * 32];
    const int vpr = H / 8;                                   // 16-byte vectors per row
    const int rpp = max(1, (int)blockDim.x / vpr);           // tokens per pass
    const int sub = threadIdx.x / vpr, v = threadIdx.x % vpr;
    // this block's tokens: one contiguous slice, the same length (to a token)
    // for every block, so that all blocks end together
    const int t_begin = (int)((long long)T * blockIdx.x / gridDim.x);
    const int t_end = (int)((long long)T * (blockIdx.x + 1) / gridDim.x);
    for (int t0 = t_begin; t0 < t_end; t0 += ctok) {
        const int nt = min(ctok, t_end - t0);
        __syncthreads();
        for (int i = threadIdx.x; i < nt * K; i += blockDim.x) {
            int slot = slot_of[(size_t)t0 * K + i];
            if (offs && slot >= 0) {
                const int e = idx[(size_t)t0 * K + i];      // bucket row -> row of the compact layout
                slot = (e >= 0 && e < E) ? slot + offs[e] : -1;
            }
            s_slot[i] = (slot < y_rows) ? slot : -1;        // a caller's row index past Y is skipped
            s_w[i] = w ? w[(size_t)t0 * K + i] : 1.0f;
        }
        __syncthreads();
        if (sub >= rpp)
            continue;
        for (int vv = v; vv < vpr; vv += blockDim.x) {
            for (int tl = sub; tl < nt; tl += 2 * rpp) {
                if (tl + rpp < nt)
                    combine_two(Y, s_slot, s_w, residual, (size_t)shared_row0, H, K, t0 + tl, tl, t0 + tl + rpp,
                                tl + rpp, vv, out);
                else
                    combine_one(Y, s_slot, s_w, residual, (size_t)shared_row0, H, K, t0 + tl, tl, vv, out);
            }
        }
    }
}

cudaError_t launch_combine(const uint16_t *Y, const int32_t *slot_of, const float *w, const uint16_t *residual,
                           int T, int H, int k, uint16_t *out, cudaStream_t s, long long shared_row0,
                           const int32_t *idx, const int32_t *offs, int E, long long y_rows)
{
    if (y_rows < 0)
        y_rows = 1ll << 62;
    if (shared_row0 < 0)
        shared_row0 = (long long)k * T;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // tokens per chunk: COMBINE_TOK, halved (down to 2) until there is at
    // least one chunk per SM (longer-lived blocks keep more row loads in
    // flight: at T=8192 this measured 0.073 -> 0.069 ms against four chunks
    // per SM), so that small batches still spread over the GPU
    int ctok = COMBINE_TOK;
    while (ctok > 2 && (T + ctok - 1) / ctok < sms)
        ctok >>= 1;
    // one slice of tokens per block, two blocks per SM (the kernel's
    // registers allow two): every block streams its slice to the end instead
    // of a last partial round of 32-token blocks
    const int blocks = (int)std::min<long long>(((long long)T + ctok - 1) / ctok, 2ll * sms);
    const cudaError_t le = launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, s, Y, slot_of, w, residual, T, H, k,
                                      ctok, shared_row0, out, idx, offs, offs ? E : 0, y_rows);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

// ---------------------------------------------------------------------------
// Expert parallelism (the training-pitfalls article's section "专家并行（EP）
// 怎么切": the expert stacks sharded along their first dimension over R
// ranks, rank r holding experts [r E/R, (r + 1) E/R)).

// dest[i] = idx[i] / per_rank (the rank that holds the pair's expert); an id
// outside [0, E) gets -1 (skipped by the bucketing, flagged there)
__global__ void ep_dest_kernel(const int32_t *__restrict__ idx, long long n, int E, int per_rank,
                               int32_t *__restrict__ dest)
{
    pdl_wait();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int e = idx[i];
        dest[i] = (e >= 0 && e < E) ? e / per_rank : -1;
    }
}

// e_send[slot_of[i]] = idx[i] - dest * per_rank: every sent row's expert, as
// an id local to the rank that receives it
__global__ void ep_local_ids_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ slot_of,
                                    long long n, int per_rank, int32_t *__restrict__ e_send)
{
    pdl_wait();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int slot = slot_of[i];
        if (slot >= 0)
            e_send[slot] = idx[i] % per_rank;
    }
}

// out[i] = rows[slot_of[i]] (bf16 rows of H, 16-byte pieces); a row whose
// slot is -1 gets zeros
__global__ void rows_gather_kernel(const uint16_t *__restrict__ rows, const int32_t *__restrict__ slot_of, int n,
                                   int H, uint16_t *__restrict__ out)
{
    pdl_wait();
    const int vpr = H / 8;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < (long long)n * vpr;
         q += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(q / vpr), v = (int)(q % vpr);
        const int slot = slot_of[i];
        reinterpret_cast<uint4 *>(out + (size_t)i * H)[v] =
            slot >= 0 ? reinterpret_cast<const uint4 *>(rows + (size_t)slot * H)[v] : make_uint4(0u, 0u, 0u, 0u);
    }
}

static int grid_for(long long n)
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return (int)std::max<long long>(1, std::min<long long>((n + 255) / 256, (long long)sms * 8));
}

cudaError_t launch_ep_dest(const int32_t *idx, long long n, int E, int per_rank, int32_t *dest, cudaStream_t s)
{
    const cudaError_t le = launch_pdl(ep_dest_kernel, dim3(grid_for(n)), dim3(256), 0, s, idx, n, E, per_rank, dest);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

cudaError_t launch_ep_local_ids(const int32_t *idx, const int32_t *slot_of, long long n, int per_rank,
                                int32_t *e_send, cudaStream_t s)
{
    const cudaError_t le = launch_pdl(ep_local_ids_kernel, dim3(grid_for(n)), dim3(256), 0, s, idx, slot_of, n,
                                      per_rank, e_send);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

cudaError_t launch_rows_gather(const uint16_t *rows, const int32_t *slot_of, int n, int H, uint16_t *out,
                               cudaStream_t s)
{
    const cudaError_t le = launch_pdl(rows_gather_kernel, dim3(grid_for((long long)n * (H / 8))), dim3(256), 0, s,
                                      rows, slot_of, n, H, out);
    if (le != cudaSuccess)
        return le;
    return cudaPeekAtLastError();
}

}  // namespace glr
