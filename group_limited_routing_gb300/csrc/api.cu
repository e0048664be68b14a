// C-ABI entry points (include/moe.h): argument checks, workspace layout,
// TMA tensor maps and the launch sequence of the MoE layer forward.
//
// Every check runs on the host before any CUDA call, so a wrong argument
// returns an error code without touching the device.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "moe.h"

using namespace glr;

namespace {

thread_local int g_last_launches = 0;

// ------------------------------------------------------------- profiling
enum KernelId {
    KID_SPLIT = 0, KID_ROUTER_GEMM, KID_SELECT, KID_FINALIZE, KID_HIST, KID_SCAN, KID_SCATTER,
    KID_GEMM_GATE_UP, KID_GEMM_DOWN, KID_COMBINE, KID_DENSE_TILES, KID_BWD_RECOMPUTE, KID_BWD_DGRAD,
    KID_BWD_DX, KID_BWD_WGRAD, KID_BWD_MISC, KID_ROUTE_FUSED, KID_TILES,
    KID_STAGE_ROUTE_PERMUTE   // (per-stage timing) the routing and bucketing kernels as one interval
};
const char *const kKernelNames[MOE_KERNEL_COUNT] = {
    "split_router", "router_gemm", "route_select", "route_finalize", "bucket_hist",
    "bucket_scan", "bucket_scatter", "gemm_gate_up_swiglu", "gemm_down", "combine", "dense_tiles",
    "bwd_gate_up_recompute", "bwd_dgrad_down_swiglu", "bwd_dgrad_x", "bwd_weight_grads", "bwd_pad_and_dw",
    "router_route_bucket", "bucket_tiles", "router_plus_permute"};

struct ProfRecord {
    cudaEvent_t start, stop;
    int kid;
};

std::atomic<int> g_prof_on{0};
std::atomic<int> g_inject_timeouts{0};   // test-only: gate/up GEMM launches left to sabotage
std::mutex g_prof_mu;
std::vector<ProfRecord> g_prof_pending;
std::vector<cudaEvent_t> g_event_pool;
double g_prof_ms[MOE_KERNEL_COUNT];
long long g_prof_n[MOE_KERNEL_COUNT];

cudaEvent_t pool_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Per-stage timing (moe_profile_enable(2)): the kernels of the routing and
// bucketing stage form one interval and every other kernel its own, and
// events are recorded only where the stage changes, so that the kernels of
// one stage still overlap each other's launch and tail (programmatic stream
// serialisation) as they do unprofiled.  The open stage of this thread:
thread_local int t_stage = -1;
thread_local cudaEvent_t t_stage_start = nullptr;
thread_local cudaStream_t t_stage_stream = nullptr;

int prof_stage(int kid)
{
    switch (kid) {
    case KID_SPLIT: case KID_ROUTER_GEMM: case KID_SELECT: case KID_FINALIZE: case KID_HIST: case KID_SCAN:
    case KID_SCATTER: case KID_ROUTE_FUSED: case KID_TILES:
        return KID_STAGE_ROUTE_PERMUTE;
    default:
        return kid;
    }
}

// ends the open stage with an event on its stream (g_prof_mu held)
void prof_close_stage_locked()
{
    if (t_stage < 0)
        return;
    cudaEvent_t stop = pool_event();
    cudaEventRecord(stop, t_stage_stream);
    g_prof_pending.push_back(ProfRecord{t_stage_start, stop, t_stage});
    t_stage = -1;
}

struct ProfScope {
    bool on;
    ProfRecord r;
    cudaStream_t s;
    ProfScope(int kid, cudaStream_t st) : on(g_prof_on.load(std::memory_order_relaxed) != 0), s(st)
    {
        if (!on)
            return;
        std::lock_guard<std::mutex> g(g_prof_mu);
        if (g_prof_on.load(std::memory_order_relaxed) == 2) {
            const int stage = prof_stage(kid);
            if (stage != t_stage || st != t_stage_stream) {
                prof_close_stage_locked();
                t_stage = stage;
                t_stage_stream = st;
                t_stage_start = pool_event();
                cudaEventRecord(t_stage_start, st);
            }
            on = false;
            return;
        }
        r.start = pool_event();
        r.stop = pool_event();
        r.kid = kid;
        cudaEventRecord(r.start, s);
    }
    void done()
    {
        if (!on)
            return;
        cudaEventRecord(r.stop, s);
        std::lock_guard<std::mutex> g(g_prof_mu);
        g_prof_pending.push_back(r);
        on = false;
    }
};

// At the end of every public call that launches kernels: closes the stage
// left open by its last launch.
struct ProfCall {
    ~ProfCall()
    {
        if (g_prof_on.load(std::memory_order_relaxed) != 2)
            return;
        std::lock_guard<std::mutex> g(g_prof_mu);
        prof_close_stage_locked();
    }
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------- validation
int check_route_cfg(const moe_cfg *c)
{
    if (!c)
        return MOE_ERR_INVALID_ARG;
    if (c->T < 1 || c->H < 1 || c->E < 1 || c->n_group < 1 || c->topk_group < 1 || c->k < 1)
        return MOE_ERR_INVALID_ARG;
    if (c->E % c->n_group != 0 || c->E / c->n_group < 2 || c->topk_group > c->n_group ||
        c->k > c->topk_group * (c->E / c->n_group))
        return MOE_ERR_INVALID_ARG;
    if (!isfinite(c->rsf) || !isfinite(c->eps) || c->eps < 0.0f)
        return MOE_ERR_INVALID_ARG;
    if (c->E != 32 * c->n_group || c->n_group > MAX_GROUPS || c->E % 128 != 0 || c->k > 32)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->H % GEMM_BK != 0 || c->T > (1 << 24))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

int check_forward_cfg(const moe_cfg *c)
{
    if (!c)
        return MOE_ERR_INVALID_ARG;
    if (c->T < 1 || c->H < 1 || c->E < 1 || c->k < 1 || c->I < 1 || c->Is < 1 || c->k > c->E)
        return MOE_ERR_INVALID_ARG;
    if (c->E > 256 || c->k > 32 || c->T > (1 << 24))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->H % 256 != 0 || c->I % 128 != 0 || c->Is != c->I)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

// ---------------------------------------------------------------- layouts
struct RouteLayout {
    size_t w3, logits, gscore, ppart, pfin, total;
    int nchunk;
    int ksplit;   // K parts of the router GEMM's logits region
};

// K parts of the router GEMM: when the 128-expert tiles are few, each tile's
// K range is split into parts that run on different SMs (partial logits, added
// in part order by the routing kernel), up to ROUTER_MAX_KSPLIT parts and
// ~ROUTER_SPLIT_UNITS work units.  The decode-size CUDA-core router and the
// wide tiles never split.
constexpr int ROUTER_SPLIT_UNITS = 152;

// tokens from which the grouped down GEMM runs on CTA pairs
constexpr int PAIR_DOWN_MIN_T = 24576;

int router_ksplit(const moe_cfg &c)
{
    if (c.T <= ROUTER_SIMT_MAX_T)
        return 1;
    const int tiles = ((c.T + GEMM_BM - 1) / GEMM_BM) * (c.E / 128);
    const int kb = c.H / GEMM_BK;
    int ks = 1;
    while (ks < ROUTER_MAX_KSPLIT && tiles * ks * 2 <= ROUTER_SPLIT_UNITS && kb % (ks * 2) == 0)
        ks *= 2;
    return ks;
}

RouteLayout route_layout(const moe_cfg &c)
{
    RouteLayout L;
    L.nchunk = (c.T + route_chunk(c.T) - 1) / route_chunk(c.T);
    L.ksplit = router_ksplit(c);
    size_t off = sizeof(WsHeader);
    L.w3 = off;
    off = align_up(off + 3ull * c.E * c.H * 2, 256);
    L.logits = off;
    off = align_up(off + (size_t)L.ksplit * c.T * c.E * 4, 256);
    L.gscore = off;                     // each group's two best scores, scored router output [T, E / 32, 2]
    off = align_up(off + (size_t)c.T * (c.E / 32) * 2 * 4, 256);
    L.ppart = off;
    off = align_up(off + (size_t)L.nchunk * c.E * 4, 256);
    L.pfin = off;
    off = align_up(off + (size_t)ROUTE_FIN_BLOCKS * c.E * 4, 256);
    L.total = off;
    return L;
}

struct FwdLayout {
    size_t hist, sizes, mtiles, ptiles, slot_of, xperm, aint, y, total;
    int nchunk, max_mtiles, max_ptiles;
};

// xperm_rows: rows of the bucketed activations (0: k T, the compact layout;
// the fused router's buckets take E T)
FwdLayout fwd_layout(const moe_cfg &c, size_t xperm_rows = 0)
{
    FwdLayout L;
    const size_t T = c.T, K = c.k, H = c.H, I = c.I;
    L.nchunk = (c.T + PERM_CHUNK - 1) / PERM_CHUNK;
    // sum over buckets of ceil(n_e / mt) <= K T / mt + E, plus the shared group;
    // mt = rows per m-tile (GEMM_SMALL_T for the small-T GEMM kinds)
    const size_t mt = (c.T <= GEMM_SMALL_T) ? GEMM_SMALL_T : GEMM_BM;
    L.max_mtiles = (int)((K * T) / mt + c.E + (T + mt - 1) / mt + 1);
    // 256-row pair tiles of the CTA-pair down GEMM: the same bound for 256 rows
    L.max_ptiles = (int)((K * T) / (2 * GEMM_BM) + c.E + (T + 2 * GEMM_BM - 1) / (2 * GEMM_BM) + 1);
    size_t off = sizeof(WsHeader);
    L.hist = off;
    off = align_up(off + (size_t)L.nchunk * c.E * 4, 256);
    L.sizes = off;
    off = align_up(off + (size_t)c.E * 4, 256);
    L.mtiles = off;
    off = align_up(off + (size_t)L.max_mtiles * 16, 256);
    L.ptiles = off;
    off = align_up(off + (size_t)L.max_ptiles * 16, 256);
    L.slot_of = off;
    off = align_up(off + T * K * 4, 256);
    L.xperm = off;
    off = align_up(off + (xperm_rows ? xperm_rows : K * T) * H * 2, 256);
    L.aint = off;
    off = align_up(off + (K + 1) * T * I * 2, 256);
    L.y = off;
    off = align_up(off + (K + 1) * T * H * 2, 256);
    L.total = off;
    return L;
}

struct BwdLayout {
    size_t hist, sizes, mtiles, slot_of, eoff, xperm, dop, wperm, gu, aw, dgu, dx, dwp, total;
    int nchunk, max_mtiles, kTp, rows;
};

// Backward workspace.  Buckets start on BWD_ROW_ALIGN-row boundaries, so the
// routed rows take at most k T + E (BWD_ROW_ALIGN - 1), rounded up to kTp;
// the shared expert's rows follow at kTp whatever the routing, padded to a
// whole block.  G and U (gu) are kept warp-interleaved (32-row blocks).
BwdLayout bwd_layout(const moe_cfg &c)
{
    BwdLayout L;
    const size_t T = c.T, K = c.k, H = c.H, I = c.I;
    L.nchunk = (c.T + PERM_CHUNK - 1) / PERM_CHUNK;
    L.max_mtiles = (int)((K * T) / GEMM_BM + c.E + (T + GEMM_BM - 1) / GEMM_BM + 1);
    L.kTp = (int)align_up(K * T + (size_t)c.E * (BWD_ROW_ALIGN - 1), BWD_ROW_ALIGN);
    L.rows = L.kTp + (c.T + BWD_ROW_ALIGN - 1) / BWD_ROW_ALIGN * BWD_ROW_ALIGN;
    const size_t R = (size_t)L.rows;
    size_t off = sizeof(WsHeader);
    L.hist = off;
    off = align_up(off + (size_t)L.nchunk * c.E * 4, 256);
    L.sizes = off;
    off = align_up(off + (size_t)c.E * 4, 256);
    L.mtiles = off;
    off = align_up(off + (size_t)L.max_mtiles * 16, 256);
    L.slot_of = off;
    off = align_up(off + T * K * 4, 256);
    L.eoff = off;
    off = align_up(off + (size_t)(c.E + 1) * 8, 256);
    L.xperm = off;
    off = align_up(off + (size_t)L.kTp * H * 2, 256);
    L.dop = off;
    off = align_up(off + R * H * 2, 256);
    L.wperm = off;
    off = align_up(off + R * 4, 256);
    L.gu = off;
    off = align_up(off + R * 2 * I * 2, 256);
    L.aw = off;
    off = align_up(off + R * I * 2, 256);
    L.dgu = off;
    off = align_up(off + R * 2 * I * 2, 256);
    L.dx = off;
    off = align_up(off + R * H * 2, 256);
    L.dwp = off;
    off = align_up(off + (size_t)L.kTp * (I / 256) * 4, 256);
    L.total = off;
    return L;
}

int check_backward_cfg(const moe_cfg *c)
{
    int rc = check_forward_cfg(c);
    if (rc != MOE_OK)
        return rc;
    if (c->I % 256 != 0)
        return MOE_ERR_UNSUPPORTED_SHAPE;     // the d(intermediate) tiles are 256 columns wide
    return MOE_OK;
}

// --------------------------------------------------------------- device
int device_check(int *sms)
{
    static int cached_sms[64];
    static int cached_ok[64];   // 0 unknown, 1 ok, -1 unsupported
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64)
        return MOE_ERR_UNSUPPORTED_DEVICE;
    if (cached_ok[dev] == 0) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        cached_sms[dev] = n;
        cached_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (cached_ok[dev] < 0)
        return MOE_ERR_UNSUPPORTED_DEVICE;
    *sms = cached_sms[dev];
    return MOE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 2D bf16 tensor [rows, cols] (row-major), box [box_rows, box_cols], 128-byte
// swizzle (box_cols * 2 == 128), zero fill outside the tensor.
bool make_map_bf16(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                   uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

WsHeader *header(void *ws) { return static_cast<WsHeader *>(ws); }

template <typename T>
T *at(void *ws, size_t off)
{
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

#define GLR_LAUNCH(kid, expr)                  \
    do {                                       \
        ProfScope prof_scope_((kid), s);       \
        if ((expr) != cudaSuccess)             \
            return MOE_ERR_CUDA;               \
        prof_scope_.done();                    \
        ++launches;                            \
    } while (0)

// counts (nullable) is cleared by the split kernel, for the routing kernel after it.
// W_split: the bf16 x 3 split of W made by moe_prepare_router, or NULL to
// split W into the workspace here (that launch also clears counts).
// ksplit_max: K parts the logits buffer has room for (L.ksplit, or 1 for a
// caller's [T, E] buffer); nparts receives the parts actually written.
// Whether router_gemm gives the scored output when asked: the tensor-core
// router without a K split, for the routing page's 256 experts in 8 groups of
// which 4 are kept.
bool router_scores(const moe_cfg &c, const RouteLayout &L, const float *W, int sms)
{
    if (c.T <= ROUTER_SIMT_MAX_T && c.H % 8 == 0 && aligned(W, 16))
        return false;                     // the CUDA-core router
    const bool wide = c.E % 256 == 0 && (c.T + GEMM_BM - 1) / GEMM_BM >= sms;
    const int ks = wide ? 1 : L.ksplit;
    return ks == 1 && c.E == 256 && c.n_group == 8 && c.topk_group == 4;
}

// gscore (nullable): ask for the scored output (sigmoid scores in `logits`,
// each group's two best scores in gscore, bias = `bias`); `scored` tells
// whether it was produced (router_scores).  counts (nullable) is cleared.
int router_gemm(const moe_cfg &c, const moe_bf16 *hidden, const float *W, const moe_bf16 *W_split, float *logits,
                int32_t *counts, void *ws, const RouteLayout &L, int sms, cudaStream_t s, int &launches,
                int ksplit_max, int &nparts, const float *bias = nullptr, float *gscore = nullptr,
                bool *scored = nullptr)
{
    nparts = 1;
    if (scored)
        *scored = false;
    if (c.T <= ROUTER_SIMT_MAX_T && c.H % 8 == 0 && aligned(W, 16)) {
        // a few token tiles cannot fill the tensor-core kernel: CUDA cores, fp32 W as is
        // (16-byte loads of W; a W that is only 4-byte aligned takes the tensor-core path)
        GLR_LAUNCH(KID_ROUTER_GEMM, launch_router_simt(hidden, W, c.T, c.E, c.H, logits, counts, s));
        return MOE_OK;
    }
    const uint16_t *W3 = reinterpret_cast<const uint16_t *>(W_split);
    if (!W3) {
        uint16_t *W3ws = at<uint16_t>(ws, L.w3);
        GLR_LAUNCH(KID_SPLIT, launch_split_router(W, W3ws, c.E, c.H, counts, s));
        W3 = W3ws;
    } else if (counts && cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, s) != cudaSuccess) {
        return MOE_ERR_CUDA;
    }
    // all experts of a token tile in one N = 256 MMA when E is a multiple of 256
    // and there are enough token tiles to give every SM one (below that the
    // 128-expert tiles spread the work over twice as many SMs)
    // (on CTA pairs, each CTA loading the weight parts of 128 experts, when E
    // is exactly 256)
    const bool wide = c.E % 256 == 0 && (c.T + GEMM_BM - 1) / GEMM_BM >= sms;
    const bool pair = wide && c.E == 256;
    const int bn = (wide && !pair) ? 256 : 128;
    GemmParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map_bf16(&p.tmA0, hidden, c.T, c.H, GEMM_BK, GEMM_BM) ||
        !make_map_bf16(&p.tmB0, W3, 3ull * c.E, c.H, GEMM_BK, bn))
        return MOE_ERR_CUDA;
    const int ks = wide ? 1 : std::max(1, std::min(ksplit_max, L.ksplit));
    p.out = logits;
    p.n_tiles = c.E / bn;
    p.ksplit = ks;
    p.part_stride = (long long)c.T * c.E;
    p.num_tiles_static = ((c.T + GEMM_BM - 1) / GEMM_BM) * p.n_tiles * ks;
    p.kblocks = c.H / GEMM_BK / ks;
    p.T = c.T;
    p.E = c.E;
    p.H = c.H;
    p.ld_out = c.E;
    p.status = &header(ws)->status;
    const bool sc = gscore && ks == 1 && c.E == 256 && c.n_group == 8 && c.topk_group == 4;
    if (sc) {
        p.gscore = gscore;
        p.bias = bias;
    }
    if (pair) {
        p.n_tiles = 1;
        p.num_tiles_static = (c.T + 255) / 256;
        GLR_LAUNCH(KID_ROUTER_GEMM, launch_gemm(GK_ROUTER_PAIR, p, 2 * std::min(sms / 2, p.num_tiles_static), s));
    } else {
        GLR_LAUNCH(KID_ROUTER_GEMM,
                   launch_gemm(wide ? GK_ROUTER_WIDE : GK_ROUTER, p, std::min(sms, p.num_tiles_static), s));
    }
    nparts = ks;
    if (scored)
        *scored = sc;
    return MOE_OK;
}

// counts must be zero on the stream when this runs.
// logits: nparts K-part buffers of [T, E] (see router_gemm).
// scored: `logits` holds the router's scored output (router_gemm); then
// chunk_hist (nullable) receives the bucketing histogram [E][ceil(T / 16)]
// from the same launch.
int route_select(const moe_cfg &c, const float *logits, int nparts, const float *bias, int32_t *idx, float *w,
                 int32_t *counts, float *aux_P, float *aux_loss, void *ws, const RouteLayout &L, cudaStream_t s,
                 int &launches, bool scored = false, int32_t *chunk_hist = nullptr)
{
    float *ppart = (aux_P || aux_loss) ? at<float>(ws, L.ppart) : nullptr;
    int *ticket = ppart ? &header(ws)->fin_ticket : nullptr;
    int nchunk = L.nchunk;
    if (scored) {
        GLR_LAUNCH(KID_SELECT, launch_route_select_scored(logits, at<float>(ws, L.gscore), bias, c.T, c.E, c.k, c.rsf,
                                                          c.eps, idx, w, counts, ppart, &header(ws)->status, ticket,
                                                          chunk_hist, s));
        nchunk = (c.T + route_chunk_hist(c.T) - 1) / route_chunk_hist(c.T);
    } else {
        GLR_LAUNCH(KID_SELECT, launch_route_select(logits, nparts, (long long)c.T * c.E, bias, c.T, c.E, c.n_group,
                                                   c.topk_group, c.k, c.rsf, c.eps, idx, w, counts, ppart,
                                                   &header(ws)->status, ticket, s));
    }
    if (ppart)
        GLR_LAUNCH(KID_FINALIZE, launch_route_finalize(counts, ppart, nchunk, c.T, c.E, c.k, at<float>(ws, L.pfin),
                                                       &header(ws)->fin_ticket, aux_P, aux_loss, s));
    return MOE_OK;
}

// Router GEMM and selection (moe_route's kernels): the scored router output
// when the shape allows it.  With chunk_hist, hist_done tells whether the
// selection wrote the bucketing histogram there, and counts_left whether it
// left `counts` to the scan of that histogram (no balance loss asked for:
// the loss needs the counts before the scan runs).
int route_all(const moe_cfg &c, const moe_bf16 *hidden, const float *W, const moe_bf16 *W_split, const float *bias,
              int32_t *idx, float *w, int32_t *counts, float *aux_P, float *aux_loss, void *ws, const RouteLayout &L,
              int sms, cudaStream_t s, int &launches, int32_t *chunk_hist = nullptr, bool *hist_done = nullptr,
              bool *counts_left = nullptr)
{
    float *logits = at<float>(ws, L.logits);
    int nparts = 1;
    bool scored = false;
    // with the histogram asked for, the expert stage's scan of it forms the
    // counts: the routing kernel then leaves them alone (no atomics, no clear)
    const bool by_scan = chunk_hist && !aux_P && !aux_loss && router_scores(c, L, W, sms);
    int rc = router_gemm(c, hidden, W, W_split, logits, by_scan ? nullptr : counts, ws, L, sms, s, launches,
                         L.ksplit, nparts, bias, at<float>(ws, L.gscore), &scored);
    if (rc == MOE_OK && by_scan && !scored)
        rc = MOE_ERR_CUDA;               // (router_scores disagrees with the router: never expected)
    if (rc == MOE_OK)
        rc = route_select(c, logits, nparts, bias, idx, w, by_scan ? nullptr : counts, aux_P, aux_loss, ws, L, s,
                          launches, scored, scored ? chunk_hist : nullptr);
    if (hist_done)
        *hist_done = scored && chunk_hist;
    if (counts_left)
        *counts_left = by_scan;
    return rc;
}

int check_ws(void *ws, size_t ws_bytes, size_t need)
{
    if (!ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(ws, 256))
        return MOE_ERR_MISALIGNED;
    if (ws_bytes < need)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    return MOE_OK;
}

// ------------------------------------------------------------ moe_layer
// One workspace for routing and the expert stage: the routing region, then
// the expert stage's (its X_perm sized for the fused router's buckets when
// that path is taken), then the fused router's scratch.  One header (status).
struct LayerLayout {
    RouteLayout r;
    FwdLayout f;
    size_t sync, offs, total;   // sync: the fused router's tile queue counter, then one ready count per tile
    bool fused;
};

// the fused router's shape: 256 experts in 8 groups, at most FUSED_MAX_K per
// token, every bucket row index e T + slot within int32, a hidden row within
// one warp's share (16 KB) of the 256-expert router's ring
bool fusable(const moe_cfg &c)
{
    return c.E == 256 && c.n_group == 8 && c.k <= FUSED_MAX_K && (long long)c.E * c.T < (1ll << 31) &&
           c.H <= 8192;   // a hidden row fits one copy slot of the router's shared-memory ring
}

bool layer_fused(const moe_cfg &c, int flags)
{
    return (flags & MOE_LAYER_FUSED_ROUTER) && fusable(c);
}

LayerLayout layer_layout(const moe_cfg &c, int flags)
{
    LayerLayout L;
    L.fused = layer_fused(c, flags);
    L.r = route_layout(c);
    L.f = fwd_layout(c, L.fused ? (size_t)c.E * c.T : 0);
    const size_t b = L.r.total - sizeof(WsHeader);   // the expert stage's region follows the routing region
    L.f.hist += b;
    L.f.sizes += b;
    L.f.mtiles += b;
    L.f.ptiles += b;
    L.f.slot_of += b;
    L.f.xperm += b;
    L.f.aint += b;
    L.f.y += b;
    L.f.total += b;
    const size_t tiles = (size_t)(c.T + GEMM_BM - 1) / GEMM_BM;
    size_t off = L.f.total;
    L.sync = off;
    off = align_up(off + (tiles + 1) * 4, 256);
    L.offs = off;
    off = align_up(off + (size_t)(c.E + 1) * 4, 256);
    L.total = off;
    return L;
}

// Routing and bucketing in one launch of the fused router, then the m-tile
// list.  counts is cleared first (the split launch does it when W_split is
// NULL); the caller checked every argument.
int fused_route(const moe_cfg &c, const moe_bf16 *hidden, const float *W, const moe_bf16 *W_split,
                const float *bias, int32_t *idx, float *w, int32_t *counts, void *ws, const LayerLayout &L, int sms,
                cudaStream_t s, int &launches)
{
    const uint16_t *W3 = reinterpret_cast<const uint16_t *>(W_split);
    if (!W3) {
        uint16_t *W3ws = at<uint16_t>(ws, L.r.w3);
        GLR_LAUNCH(KID_SPLIT, launch_split_router(W, W3ws, c.E, c.H, counts, s));
        W3 = W3ws;
    } else if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, s) != cudaSuccess) {
        return MOE_ERR_CUDA;
    }
    const int tiles = (c.T + GEMM_BM - 1) / GEMM_BM;
    int *sync = at<int>(ws, L.sync);
    if (cudaMemsetAsync(sync, 0, sizeof(int) * (tiles + 1), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    GemmParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map_bf16(&p.tmA0, hidden, c.T, c.H, GEMM_BK, GEMM_BM) ||
        !make_map_bf16(&p.tmB0, W3, 3ull * c.E, c.H, GEMM_BK, 256))
        return MOE_ERR_CUDA;
    p.n_tiles = 1;
    p.ksplit = 1;
    p.num_tiles_static = tiles;
    p.kblocks = c.H / GEMM_BK;
    p.T = c.T;
    p.E = c.E;
    p.H = c.H;
    p.status = &header(ws)->status;
    p.bias = bias;
    p.idx_out = idx;
    p.w_out = w;
    p.counts = counts;
    p.slot_local = at<int32_t>(ws, L.f.slot_of);
    p.unit_ctr = sync;
    p.ready = sync + 1;
    p.out = at<float>(ws, L.r.logits);
    p.ld_out = c.E;
    p.hidden = hidden;
    p.xperm = at<uint16_t>(ws, L.f.xperm);
    p.topk_group = c.topk_group;
    p.k = c.k;
    p.rsf = c.rsf;
    p.eps = c.eps;
    GLR_LAUNCH(KID_ROUTE_FUSED, launch_gemm(GK_ROUTER_FUSED, p, std::min(sms, tiles), s));
    WsHeader *hdr = header(ws);
    GLR_LAUNCH(KID_TILES, launch_bucket_tiles(counts, c.T, c.E, c.k, at<int4>(ws, L.f.mtiles), hdr,
                                              at<int32_t>(ws, L.offs), s));
    return MOE_OK;
}

// The expert stage of the forward: bucketing (unless offs is given: the fused
// router then bucketed the pairs itself, bucket e at rows e T .. of X_perm,
// slot_of holding rows inside the buckets and offs the compact offsets), the
// two grouped GEMMs and the combine.  Arguments are checked by the caller.
int forward_impl(const moe_cfg &c, const moe_bf16 *hidden, const moe_bf16 *W_gate_up, const moe_bf16 *W_down,
                 const moe_bf16 *shared_gate_up, const moe_bf16 *shared_down, const int32_t *topk_idx,
                 const float *topk_w, const moe_bf16 *residual, moe_bf16 *out, void *ws, const FwdLayout &L,
                 const int32_t *offs, int sms, cudaStream_t s, int &launches, bool hist_ready = false,
                 bool with_shared = true, int32_t *counts_out = nullptr, bool fused_combine = false)
{
    // with_shared = false (moe_expert_rows): no shared-expert group, k = 1, and
    // out receives every pair's unweighted expert row in pair order instead
    // of the combine
    WsHeader *hdr = header(ws);
    int32_t *hist = at<int32_t>(ws, L.hist);
    int4 *mtiles = at<int4>(ws, L.mtiles);
    int32_t *slot_of = at<int32_t>(ws, L.slot_of);
    uint16_t *xperm = at<uint16_t>(ws, L.xperm);
    uint16_t *aint = at<uint16_t>(ws, L.aint);
    uint16_t *y = at<uint16_t>(ws, L.y);
    const uint64_t kT = (uint64_t)c.k * c.T;

    // bucket the (token, expert) pairs by expert (stable), gather rows --
    // unless the fused router has done it (bucket e at rows e T .., offsets in offs)
    int32_t *sizes = at<int32_t>(ws, L.sizes);
    if (!offs && c.T <= BUCKET_SMALL_MAX_T && with_shared) {
        // a handful of tokens: the three bucketing steps in one launch
        const int mt = c.T <= GEMM_SMALL_T ? GEMM_SMALL_T : GEMM_BM;
        GLR_LAUNCH(KID_SCATTER, launch_bucket_small(topk_idx, hidden, c.T, c.H, c.E, c.k, mt, sizes, slot_of,
                                                    xperm, mtiles, hdr, s));
    } else if (!offs) {
        // (the routing kernel of moe_layer may have written the histogram already)
        if (!hist_ready)
            GLR_LAUNCH(KID_HIST, launch_bucket_hist(topk_idx, c.T, c.E, c.k, hist, &hdr->status, s));
        GLR_LAUNCH(KID_SCAN, launch_bucket_scan(hist, L.nchunk, c.E, sizes, s, counts_out));
        GLR_LAUNCH(KID_SCATTER, launch_bucket_scatter(topk_idx, hidden, hist, sizes, c.T, c.H, c.E, c.k, slot_of,
                                                      xperm, mtiles, hdr, s, at<int4>(ws, L.ptiles), with_shared));
    }
    if (!with_shared) {
        // (placeholders for the shared group's operands, which no tile reads)
        shared_gate_up = W_gate_up;
        shared_down = W_down;
    }
    // the down GEMM runs on CTA pairs over 256-row tiles at large T (the
    // bucketing above writes their list); below that the 128-row tiles waste
    // fewer rows in buckets' part-filled last tiles (measured, workload-4
    // recipe: T = 4096 / 8192 / 16384 / 32768 took 0.119 / 0.169 / 0.280 /
    // 0.510 ms on single CTAs and 0.133 / 0.181 / 0.283 / 0.492 ms on pairs)
    const bool pair_down = !offs && c.T >= PAIR_DOWN_MIN_T;

    // grouped gate/up GEMM with the SwiGLU epilogue (shared expert = group E);
    // for T <= GEMM_SMALL_T no bucket has more than T rows: the small kinds
    // load only that many A rows per stage and keep more weights in flight
    const bool small = c.T <= GEMM_SMALL_T && with_shared;
    const int a_rows = small ? GEMM_SMALL_T : GEMM_BM;
    GemmParams p1;
    memset(&p1, 0, sizeof(p1));
    if (!make_map_bf16(&p1.tmA0, xperm, offs ? (uint64_t)c.E * c.T : kT, c.H, GEMM_BK, a_rows) ||
        !make_map_bf16(&p1.tmA1, hidden, c.T, c.H, GEMM_BK, a_rows) ||
        !make_map_bf16(&p1.tmB0, W_gate_up, 2ull * c.I * c.E, c.H, GEMM_BK, 128) ||
        !make_map_bf16(&p1.tmB1, shared_gate_up, 2ull * c.I, c.H, GEMM_BK, 128))
        return MOE_ERR_CUDA;
    if (!make_map_bf16(&p1.tmOut, aint, kT + c.T, c.I, 64, 32))
        return MOE_ERR_CUDA;
    p1.out = aint;
    p1.mtiles = mtiles;
    p1.num_mtiles = &hdr->num_mtiles;
    p1.n_tiles = c.I / 128;
    p1.kblocks = c.H / GEMM_BK;
    p1.T = c.T;
    p1.E = c.E;
    p1.I = c.I;
    p1.H = c.H;
    p1.kT = (int)kT;
    p1.ld_out = c.I;
    p1.status = &hdr->status;
    p1.cap_rows = offs ? 1 : 0;
    if (g_inject_timeouts.load() > 0 && g_inject_timeouts.fetch_sub(1) > 0) {
        p1.inject_withhold = 1;
        p1.wait_limit_ns = 50000000ull;
    }
    GLR_LAUNCH(KID_GEMM_GATE_UP, launch_gemm(small ? GK_GATE_UP_SMALL : GK_GATE_UP, p1,
                                             std::min(sms, L.max_mtiles * p1.n_tiles), s));

    // grouped down GEMM (W_down stacked [E, I, H]: an MN-major B operand)
    GemmParams p2;
    memset(&p2, 0, sizeof(p2));
    if (!make_map_bf16(&p2.tmA0, aint, kT + c.T, c.I, GEMM_BK, a_rows) ||
        !make_map_bf16(&p2.tmB0, W_down, (uint64_t)c.I * c.E, c.H, 64, GEMM_BK) ||
        !make_map_bf16(&p2.tmB1, shared_down, (uint64_t)c.I, c.H, 64, GEMM_BK))
        return MOE_ERR_CUDA;
    if (!make_map_bf16(&p2.tmOut, y, kT + c.T, c.H, 64, 32))
        return MOE_ERR_CUDA;
    p2.out = y;
    p2.mtiles = mtiles;
    p2.num_mtiles = &hdr->num_mtiles;
    p2.n_tiles = c.H / 256;
    p2.kblocks = c.I / GEMM_BK;
    p2.T = c.T;
    p2.E = c.E;
    p2.I = c.I;
    p2.H = c.H;
    p2.kT = (int)kT;
    p2.ld_out = c.H;
    p2.status = &hdr->status;
    // with fused_combine (moe_layer's MOE_LAYER_FUSED_COMBINE): the shared
    // expert's down GEMM with the combine in its epilogue, after the routed
    // pair tiles, whose rows it reads; no shared rows in Y and no separate
    // combine launch.  Bit-identical to the default, and slower on a GB300
    // (its eight epilogue warps keep fewer row loads in flight than the
    // combine kernel), so not the default.
    const bool down_combine = fused_combine && pair_down && with_shared && c.k <= 8;
    if (pair_down) {
        p2.mtiles = at<int4>(ws, L.ptiles);
        p2.num_mtiles = down_combine ? &hdr->num_ptiles_routed : &hdr->num_ptiles;
        GLR_LAUNCH(KID_GEMM_DOWN, launch_gemm(GK_DOWN_PAIR, p2, 2 * std::min(sms / 2, L.max_ptiles * p2.n_tiles), s));
        if (down_combine) {
            GemmParams p3 = p2;
            p3.mtiles = nullptr;
            p3.num_mtiles = nullptr;
            p3.num_tiles_static = ((c.T + GEMM_BM - 1) / GEMM_BM) * p3.n_tiles;
            p3.out = out;
            p3.cmb_y = y;
            p3.cmb_slot = slot_of;
            p3.cmb_w = topk_w;
            p3.cmb_res = residual;
            p3.cmb_k = c.k;
            GLR_LAUNCH(KID_COMBINE, launch_gemm(GK_DOWN_COMBINE, p3, std::min(sms, p3.num_tiles_static), s));
            return MOE_OK;
        }
    } else {
        GLR_LAUNCH(KID_GEMM_DOWN, launch_gemm(small ? GK_DOWN_SMALL : GK_DOWN, p2,
                                              std::min(sms, L.max_mtiles * p2.n_tiles), s));
    }

    if (!with_shared) {
        // every row's expert output, back in the rows' own order
        GLR_LAUNCH(KID_COMBINE, launch_rows_gather(y, slot_of, c.T, c.H, out, s));
        return MOE_OK;
    }
    // weighted combine + shared expert (+ residual), one rounding to bf16
    GLR_LAUNCH(KID_COMBINE, launch_combine(y, slot_of, topk_w, residual, c.T, c.H, c.k, out, s, -1, topk_idx, offs,
                                           c.E));
    return MOE_OK;
}

// ------------------------------------------------------ expert parallelism
struct EpLayout {
    size_t dest, hist, mtiles, total;
    int nchunk;
};

EpLayout ep_layout(const moe_cfg &c, int ranks)
{
    EpLayout L;
    const size_t n = (size_t)c.T * c.k;
    L.nchunk = (c.T + PERM_CHUNK - 1) / PERM_CHUNK;
    size_t off = sizeof(WsHeader);
    L.dest = off;
    off = align_up(off + n * 4, 256);
    L.hist = off;
    off = align_up(off + (size_t)L.nchunk * ranks * 4, 256);
    L.mtiles = off;
    off = align_up(off + (n / GEMM_BM + ranks + 2) * 16, 256);
    L.total = off;
    return L;
}

int check_ep(const moe_cfg *c, int ranks)
{
    if (!c || ranks < 1 || c->T < 1 || c->k < 1 || c->E < 1 || c->H < 8)
        return MOE_ERR_INVALID_ARG;
    if (c->E % ranks != 0 || ranks > 256 || c->k > 32 || c->H % 8 != 0 || c->T > (1 << 24))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}


}  // namespace

// ===================================================================== ABI
extern "C" {

size_t moe_workspace_bytes(const moe_cfg *cfg, int which)
{
    if (which == MOE_WS_ROUTE)
        return check_route_cfg(cfg) == MOE_OK ? route_layout(*cfg).total : 0;
    if (which == MOE_WS_FORWARD)
        return check_forward_cfg(cfg) == MOE_OK ? fwd_layout(*cfg).total : 0;
    if (which == MOE_WS_BACKWARD)
        return check_backward_cfg(cfg) == MOE_OK ? bwd_layout(*cfg).total : 0;
    return 0;
}

int moe_workspace_init(void *ws, size_t ws_bytes, void *stream)
{
    int rc = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (rc != MOE_OK)
        return rc;
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_router_logits(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router, float *logits, void *ws,
                      size_t ws_bytes, void *stream)
{
    ProfCall prof_call_;
    int rc = check_route_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (!hidden || !W_router || !logits)
        return MOE_ERR_INVALID_ARG;
    const RouteLayout L = route_layout(*cfg);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(hidden, 16) || !aligned(W_router, 4) || !aligned(logits, 16))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    int launches = 0;
    int nparts = 1;
    rc = router_gemm(*cfg, hidden, W_router, nullptr, logits, nullptr, ws, L, sms,
                     static_cast<cudaStream_t>(stream), launches, 1, nparts);
    g_last_launches = launches;
    return rc;
}

int moe_route_from_logits(const moe_cfg *cfg, const float *logits, const float *expert_bias, int32_t *topk_idx,
                          float *topk_w, int32_t *expert_counts, float *aux_P, float *aux_loss, void *ws,
                          size_t ws_bytes, void *stream)
{
    ProfCall prof_call_;
    int rc = check_route_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (!logits || !topk_idx || !topk_w || !expert_counts)
        return MOE_ERR_INVALID_ARG;
    const RouteLayout L = route_layout(*cfg);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(logits, 4) || !aligned(expert_bias, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
        !aligned(expert_counts, 4) || !aligned(aux_P, 4) || !aligned(aux_loss, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    int launches = 0;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * cfg->E, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    rc = route_select(*cfg, logits, 1, expert_bias, topk_idx, topk_w, expert_counts, aux_P, aux_loss, ws, L, s,
                      launches);
    g_last_launches = launches;
    return rc;
}

int moe_router_scores(const float *logits, float *scores, int64_t n, void *stream)
{
    ProfCall prof_call_;
    if (!logits || !scores || n < 1)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(scores, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0, rc = MOE_OK;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    if (launch_router_scores(logits, scores, (long long)n, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    g_last_launches = 1;
    return MOE_OK;
}

int moe_route(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router, const float *expert_bias,
              int32_t *topk_idx, float *topk_w, int32_t *expert_counts, float *aux_P, float *aux_loss, void *ws,
              size_t ws_bytes, void *stream)
{
    ProfCall prof_call_;
    int rc = check_route_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (!hidden || !W_router || !topk_idx || !topk_w || !expert_counts)
        return MOE_ERR_INVALID_ARG;
    const RouteLayout L = route_layout(*cfg);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(hidden, 16) || !aligned(W_router, 4) || !aligned(expert_bias, 4) || !aligned(topk_idx, 4) ||
        !aligned(topk_w, 4) || !aligned(expert_counts, 4) || !aligned(aux_P, 4) || !aligned(aux_loss, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    rc = route_all(*cfg, hidden, W_router, nullptr, expert_bias, topk_idx, topk_w, expert_counts, aux_P, aux_loss, ws,
                   L, sms, s, launches);
    g_last_launches = launches;
    return rc;
}

int moe_prepare_router(const moe_cfg *cfg, const float *W_router, moe_bf16 *W_split, void *stream)
{
    ProfCall prof_call_;
    int rc = check_route_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (!W_router || !W_split)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(W_router, 4) || !aligned(W_split, 16))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    GLR_LAUNCH(KID_SPLIT, launch_split_router(W_router, reinterpret_cast<uint16_t *>(W_split), cfg->E, cfg->H,
                                              nullptr, s));
    g_last_launches = launches;
    return MOE_OK;
}

int moe_route_prepared(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router, const moe_bf16 *W_split,
                       const float *expert_bias, int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                       float *aux_P, float *aux_loss, void *ws, size_t ws_bytes, void *stream)
{
    ProfCall prof_call_;
    int rc = check_route_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (!hidden || !W_router || !W_split || !topk_idx || !topk_w || !expert_counts)
        return MOE_ERR_INVALID_ARG;
    const RouteLayout L = route_layout(*cfg);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(hidden, 16) || !aligned(W_router, 4) || !aligned(W_split, 16) || !aligned(expert_bias, 4) ||
        !aligned(topk_idx, 4) || !aligned(topk_w, 4) || !aligned(expert_counts, 4) || !aligned(aux_P, 4) ||
        !aligned(aux_loss, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    rc = route_all(*cfg, hidden, W_router, W_split, expert_bias, topk_idx, topk_w, expert_counts, aux_P, aux_loss, ws,
                   L, sms, s, launches);
    g_last_launches = launches;
    return rc;
}

int check_dense(int32_t T, int32_t H, int32_t I)
{
    if (T < 1 || H < 1 || I < 1)
        return MOE_ERR_INVALID_ARG;
    if (T > (1 << 24) || H % 256 != 0 || I % 128 != 0)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

struct DenseLayout {
    size_t mtiles, aint, y, total;
    int mt;
};

DenseLayout dense_layout(int32_t T, int32_t H, int32_t I)
{
    DenseLayout L;
    L.mt = (T <= GEMM_SMALL_T) ? GEMM_SMALL_T : GEMM_BM;
    size_t off = sizeof(WsHeader);
    L.mtiles = off;
    off = align_up(off + (size_t)((T + L.mt - 1) / L.mt + 1) * 16, 256);
    L.aint = off;
    off = align_up(off + (size_t)T * I * 2, 256);
    L.y = off;
    off = align_up(off + (size_t)T * H * 2, 256);
    L.total = off;
    return L;
}

size_t moe_dense_workspace_bytes(int32_t T, int32_t H, int32_t I)
{
    return check_dense(T, H, I) == MOE_OK ? dense_layout(T, H, I).total : 0;
}

int moe_dense_ffn(int32_t T, int32_t H, int32_t I, const moe_bf16 *hidden, const moe_bf16 *W_gate_up,
                  const moe_bf16 *W_down, const moe_bf16 *residual, moe_bf16 *out, void *ws, size_t ws_bytes,
                  void *stream)
{
    ProfCall prof_call_;
    int rc = check_dense(T, H, I);
    if (rc != MOE_OK)
        return rc;
    if (!hidden || !W_gate_up || !W_down || !out)
        return MOE_ERR_INVALID_ARG;
    const DenseLayout L = dense_layout(T, H, I);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(hidden, 16) || !aligned(W_gate_up, 16) || !aligned(W_down, 16) || !aligned(residual, 16) ||
        !aligned(out, 16))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    WsHeader *hdr = header(ws);
    int4 *mtiles = at<int4>(ws, L.mtiles);
    uint16_t *aint = at<uint16_t>(ws, L.aint);
    uint16_t *y = at<uint16_t>(ws, L.y);
    const bool small = T <= GEMM_SMALL_T;
    const int a_rows = small ? GEMM_SMALL_T : GEMM_BM;
    const int ntile = (T + L.mt - 1) / L.mt;
    GLR_LAUNCH(KID_DENSE_TILES, launch_dense_tiles(T, L.mt, mtiles, hdr, s));

    // the grouped GEMMs with one group: group 0 == E = 0 takes the "shared"
    // operands (tmA1 / tmB1), rows 0 .. T-1 of the intermediate and of Y
    GemmParams p1;
    memset(&p1, 0, sizeof(p1));
    if (!make_map_bf16(&p1.tmA1, hidden, T, H, GEMM_BK, a_rows) ||
        !make_map_bf16(&p1.tmB1, W_gate_up, 2ull * I, H, GEMM_BK, 128) ||
        !make_map_bf16(&p1.tmOut, aint, T, I, 64, 32))
        return MOE_ERR_CUDA;
    p1.tmA0 = p1.tmA1;
    p1.tmB0 = p1.tmB1;
    p1.out = aint;
    p1.mtiles = mtiles;
    p1.num_mtiles = &hdr->num_mtiles;
    p1.n_tiles = I / 128;
    p1.kblocks = H / GEMM_BK;
    p1.T = T;
    p1.E = 0;
    p1.I = I;
    p1.H = H;
    p1.kT = 0;
    p1.ld_out = I;
    p1.status = &hdr->status;
    GLR_LAUNCH(KID_GEMM_GATE_UP, launch_gemm(small ? GK_GATE_UP_SMALL : GK_GATE_UP, p1,
                                             std::min(sms, ntile * p1.n_tiles), s));
    GemmParams p2;
    memset(&p2, 0, sizeof(p2));
    if (!make_map_bf16(&p2.tmA0, aint, T, I, GEMM_BK, a_rows) ||
        !make_map_bf16(&p2.tmB1, W_down, (uint64_t)I, H, 64, GEMM_BK) ||
        !make_map_bf16(&p2.tmOut, y, T, H, 64, 32))
        return MOE_ERR_CUDA;
    p2.tmB0 = p2.tmB1;
    p2.out = y;
    p2.mtiles = mtiles;
    p2.num_mtiles = &hdr->num_mtiles;
    p2.n_tiles = H / 256;
    p2.kblocks = I / GEMM_BK;
    p2.T = T;
    p2.E = 0;
    p2.I = I;
    p2.H = H;
    p2.kT = 0;
    p2.ld_out = H;
    p2.status = &hdr->status;
    GLR_LAUNCH(KID_GEMM_DOWN, launch_gemm(small ? GK_DOWN_SMALL : GK_DOWN, p2, std::min(sms, ntile * p2.n_tiles),
                                          s));
    // k = 0 combine: out = bf16(Y (+ residual))
    GLR_LAUNCH(KID_COMBINE, launch_combine(y, nullptr, nullptr, residual, T, H, 0, out, s));
    g_last_launches = launches;
    return MOE_OK;
}

int moe_backward(const moe_cfg *cfg, const moe_bf16 *hidden, const moe_bf16 *W_gate_up, const moe_bf16 *W_down,
                 const moe_bf16 *shared_gate_up, const moe_bf16 *shared_down, const int32_t *topk_idx,
                 const float *topk_w, const moe_bf16 *d_out, moe_bf16 *d_hidden, float *dW_gate_up, float *dW_down,
                 float *d_shared_gate_up, float *d_shared_down, float *d_topk_w, void *ws, size_t ws_bytes,
                 void *stream)
{
    ProfCall prof_call_;
    int rc = check_backward_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (!hidden || !W_gate_up || !W_down || !shared_gate_up || !shared_down || !topk_idx || !topk_w || !d_out ||
        !d_hidden || !dW_gate_up || !dW_down || !d_shared_gate_up || !d_shared_down || !d_topk_w)
        return MOE_ERR_INVALID_ARG;
    const BwdLayout L = bwd_layout(*cfg);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(hidden, 16) || !aligned(W_gate_up, 16) || !aligned(W_down, 16) || !aligned(shared_gate_up, 16) ||
        !aligned(shared_down, 16) || !aligned(d_out, 16) || !aligned(d_hidden, 16) || !aligned(dW_gate_up, 16) ||
        !aligned(dW_down, 16) || !aligned(d_shared_gate_up, 16) || !aligned(d_shared_down, 16) ||
        !aligned(topk_idx, 4) || !aligned(topk_w, 4) || !aligned(d_topk_w, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    const moe_cfg &c = *cfg;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    WsHeader *hdr = header(ws);
    int32_t *hist = at<int32_t>(ws, L.hist);
    int32_t *sizes = at<int32_t>(ws, L.sizes);
    int4 *mtiles = at<int4>(ws, L.mtiles);
    int32_t *slot_of = at<int32_t>(ws, L.slot_of);
    int2 *eoff = at<int2>(ws, L.eoff);
    uint16_t *xperm = at<uint16_t>(ws, L.xperm);
    uint16_t *dop = at<uint16_t>(ws, L.dop);
    float *wperm = at<float>(ws, L.wperm);
    uint16_t *gu = at<uint16_t>(ws, L.gu);
    uint16_t *aw = at<uint16_t>(ws, L.aw);
    uint16_t *dgu = at<uint16_t>(ws, L.dgu);
    uint16_t *dx = at<uint16_t>(ws, L.dx);
    float *dwp = at<float>(ws, L.dwp);
    const uint64_t R = (uint64_t)L.rows;

    // 1. buckets on 64-row boundaries: X rows, dOut rows, weights per bucket row
    GLR_LAUNCH(KID_HIST, launch_bucket_hist(topk_idx, c.T, c.E, c.k, hist, &hdr->status, s));
    GLR_LAUNCH(KID_SCAN, launch_bucket_scan(hist, L.nchunk, c.E, sizes, s));
    GLR_LAUNCH(KID_SCATTER, launch_bucket_scatter_bwd(topk_idx, hidden, hist, sizes, c.T, c.H, c.E, c.k, slot_of,
                                                      xperm, mtiles, hdr, d_out, topk_w, dop, wperm, eoff, L.kTp,
                                                      s));
    GLR_LAUNCH(KID_BWD_MISC, launch_zero_pad(eoff, sizes, c.T, c.E, c.H, c.I, xperm, dop, aw, dgu, hdr->tile_ctr, s));

    // 2. the gate/up products again: G, U (bf16) and w * a (bf16)
    GemmParams p1;
    memset(&p1, 0, sizeof(p1));
    if (!make_map_bf16(&p1.tmA0, xperm, (uint64_t)L.kTp, c.H, GEMM_BK, GEMM_BM) ||
        !make_map_bf16(&p1.tmA1, hidden, c.T, c.H, GEMM_BK, GEMM_BM) ||
        !make_map_bf16(&p1.tmB0, W_gate_up, 2ull * c.I * c.E, c.H, GEMM_BK, 128) ||
        !make_map_bf16(&p1.tmB1, shared_gate_up, 2ull * c.I, c.H, GEMM_BK, 128))
        return MOE_ERR_CUDA;
    p1.mtiles = mtiles;
    p1.num_mtiles = &hdr->num_mtiles;
    p1.n_tiles = c.I / 128;
    p1.kblocks = c.H / GEMM_BK;
    p1.T = c.T;
    p1.E = c.E;
    p1.I = c.I;
    p1.H = c.H;
    p1.kT = L.kTp;
    p1.status = &hdr->status;
    if (!make_map_bf16(&p1.tmOut, aw, R, c.I, 64, 32))
        return MOE_ERR_CUDA;
    p1.w_perm = wperm;
    p1.gu_out = gu;
    p1.aw_out = aw;
    GLR_LAUNCH(KID_BWD_RECOMPUTE, launch_gemm(GK_GATE_UP_BWD, p1, std::min(sms, L.max_mtiles * p1.n_tiles), s));

    // 3. dA' = dOut_perm . W_down^T, then dw partials and the SwiGLU backward
    GemmParams p2;
    memset(&p2, 0, sizeof(p2));
    if (!make_map_bf16(&p2.tmA0, dop, R, c.H, GEMM_BK, GEMM_BM) ||
        !make_map_bf16(&p2.tmB0, W_down, (uint64_t)c.I * c.E, c.H, GEMM_BK, 128) ||
        !make_map_bf16(&p2.tmB1, shared_down, (uint64_t)c.I, c.H, GEMM_BK, 128) ||
        !make_map_bf16(&p2.tmOut, dgu, R, 2ull * c.I, 64, 32))
        return MOE_ERR_CUDA;
    p2.mtiles = mtiles;
    p2.num_mtiles = &hdr->num_mtiles;
    p2.n_tiles = c.I / 256;
    p2.kblocks = c.H / GEMM_BK;
    p2.T = c.T;
    p2.E = c.E;
    p2.I = c.I;
    p2.H = c.H;
    p2.kT = L.kTp;
    p2.status = &hdr->status;
    p2.w_perm = wperm;
    p2.gu_in = gu;
    p2.dgu_out = dgu;
    p2.dw_part = dwp;
    GLR_LAUNCH(KID_BWD_DGRAD, launch_gemm(GK_DGRAD_DOWN, p2, std::min(sms, L.max_mtiles * p2.n_tiles), s));

    // 4. dX_perm = [dG dU] . W_gate_up[e]: the down GEMM with K = 2I
    GemmParams p3;
    memset(&p3, 0, sizeof(p3));
    if (!make_map_bf16(&p3.tmA0, dgu, R, 2ull * c.I, GEMM_BK, GEMM_BM) ||
        !make_map_bf16(&p3.tmB0, W_gate_up, 2ull * c.I * c.E, c.H, 64, GEMM_BK) ||
        !make_map_bf16(&p3.tmB1, shared_gate_up, 2ull * c.I, c.H, 64, GEMM_BK) ||
        !make_map_bf16(&p3.tmOut, dx, R, c.H, 64, 32))
        return MOE_ERR_CUDA;
    p3.out = dx;
    p3.mtiles = mtiles;
    p3.num_mtiles = &hdr->num_mtiles;
    p3.n_tiles = c.H / 256;
    p3.kblocks = 2 * c.I / GEMM_BK;
    p3.T = c.T;
    p3.E = c.E;
    p3.I = 2 * c.I;
    p3.H = c.H;
    p3.kT = L.kTp;
    p3.ld_out = c.H;
    p3.status = &hdr->status;
    GLR_LAUNCH(KID_BWD_DX, launch_gemm(GK_DOWN, p3, std::min(sms, L.max_mtiles * p3.n_tiles), s));

    // 5. d_hidden = sum over the token's rows (weights already applied), d topk_w
    GLR_LAUNCH(KID_COMBINE, launch_combine(dx, slot_of, nullptr, nullptr, c.T, c.H, c.k, d_hidden, s, L.kTp));
    GLR_LAUNCH(KID_BWD_MISC, launch_dw_reduce(slot_of, dwp, c.T * c.k, c.I / 256, d_topk_w, s));

    // 6. weight gradients per expert, K over its rows: dW_down = (w a)^T dOut,
    //    dW_gate_up = [dG dU]^T X
    for (int which = 0; which < 2; ++which) {
        GemmParams p4;
        memset(&p4, 0, sizeof(p4));
        const uint64_t F = which == 0 ? (uint64_t)c.I : 2ull * c.I;
        bool ok = make_map_bf16(&p4.tmA0, which == 0 ? aw : dgu, R, F, 64, GEMM_BK);
        if (which == 0) {
            ok = ok && make_map_bf16(&p4.tmB0, dop, R, c.H, 64, GEMM_BK);
            p4.tmB1 = p4.tmB0;
            p4.b_row_shared = -1;
        } else {
            ok = ok && make_map_bf16(&p4.tmB0, xperm, (uint64_t)L.kTp, c.H, 64, GEMM_BK) &&
                 make_map_bf16(&p4.tmB1, hidden, c.T, c.H, 64, GEMM_BK);
            p4.b_row_shared = 0;
        }
        if (!ok)
            return MOE_ERR_CUDA;
        p4.out = which == 0 ? (void *)dW_down : (void *)dW_gate_up;
        p4.out_shared = which == 0 ? (void *)d_shared_down : (void *)d_shared_gate_up;
        p4.eoff = eoff;
        p4.wg_fm = (int)(F / 128);
        p4.wg_fn = c.H / 256;
        p4.n_tiles = 1;
        p4.num_tiles_static = (c.E + 1) * p4.wg_fm * p4.wg_fn;
        p4.T = c.T;
        p4.E = c.E;
        p4.I = c.I;
        p4.H = c.H;
        p4.status = &hdr->status;
        p4.tile_ctr = &hdr->tile_ctr[which];
        GLR_LAUNCH(KID_BWD_WGRAD, launch_gemm(GK_WGRAD, p4, std::min(sms, p4.num_tiles_static), s));
    }
    g_last_launches = launches;
    return MOE_OK;
}

int moe_forward(const moe_cfg *cfg, const moe_bf16 *hidden, const moe_bf16 *W_gate_up, const moe_bf16 *W_down,
                const moe_bf16 *shared_gate_up, const moe_bf16 *shared_down, const int32_t *topk_idx,
                const float *topk_w, const moe_bf16 *residual, moe_bf16 *out, void *ws, size_t ws_bytes,
                void *stream)
{
    ProfCall prof_call_;
    int rc = check_forward_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (!hidden || !W_gate_up || !W_down || !shared_gate_up || !shared_down || !topk_idx || !topk_w || !out)
        return MOE_ERR_INVALID_ARG;
    const FwdLayout L = fwd_layout(*cfg);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(hidden, 16) || !aligned(W_gate_up, 16) || !aligned(W_down, 16) || !aligned(shared_gate_up, 16) ||
        !aligned(shared_down, 16) || !aligned(residual, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) ||
        !aligned(topk_w, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    int launches = 0;
    rc = forward_impl(*cfg, hidden, W_gate_up, W_down, shared_gate_up, shared_down, topk_idx, topk_w, residual, out,
                      ws, L, nullptr, sms, static_cast<cudaStream_t>(stream), launches);
    g_last_launches = launches;
    return rc;
}

size_t moe_layer_workspace_bytes(const moe_cfg *cfg, int flags)
{
    if (check_route_cfg(cfg) != MOE_OK || check_forward_cfg(cfg) != MOE_OK)
        return 0;
    return layer_layout(*cfg, flags).total;
}

int moe_layer(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router, const moe_bf16 *W_split,
              const float *expert_bias, const moe_bf16 *W_gate_up, const moe_bf16 *W_down,
              const moe_bf16 *shared_gate_up, const moe_bf16 *shared_down, const moe_bf16 *residual,
              int32_t *topk_idx, float *topk_w, int32_t *expert_counts, float *aux_P, float *aux_loss,
              moe_bf16 *out, int flags, void *ws, size_t ws_bytes, void *stream)
{
    ProfCall prof_call_;
    int rc = check_route_cfg(cfg);
    if (rc == MOE_OK)
        rc = check_forward_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (flags & ~(MOE_LAYER_FUSED_ROUTER | MOE_LAYER_FUSED_COMBINE))
        return MOE_ERR_INVALID_ARG;
    if ((aux_P || aux_loss) && layer_fused(*cfg, flags))
        return MOE_ERR_INVALID_ARG;          // the fused router forms no balance-loss sums
    if (!hidden || !W_router || !W_gate_up || !W_down || !shared_gate_up || !shared_down || !topk_idx || !topk_w ||
        !expert_counts || !out)
        return MOE_ERR_INVALID_ARG;
    const LayerLayout L = layer_layout(*cfg, flags);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(hidden, 16) || !aligned(W_router, 4) || !aligned(W_split, 16) || !aligned(expert_bias, 4) ||
        !aligned(W_gate_up, 16) || !aligned(W_down, 16) || !aligned(shared_gate_up, 16) ||
        !aligned(shared_down, 16) || !aligned(residual, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) ||
        !aligned(topk_w, 4) || !aligned(expert_counts, 4) || !aligned(aux_P, 4) || !aligned(aux_loss, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    const moe_cfg &c = *cfg;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    if (L.fused) {
        rc = fused_route(c, hidden, W_router, W_split, expert_bias, topk_idx, topk_w, expert_counts, ws, L, sms, s,
                         launches);
        if (rc == MOE_OK)
            rc = forward_impl(c, hidden, W_gate_up, W_down, shared_gate_up, shared_down, topk_idx, topk_w, residual,
                              out, ws, L.f, at<int32_t>(ws, L.offs), sms, s, launches);
    } else {
        // the routing kernel also writes the bucketing histogram where the
        // expert stage reads it (when the router's scored output is taken)
        bool hist_done = false, counts_left = false;
        rc = route_all(c, hidden, W_router, W_split, expert_bias, topk_idx, topk_w, expert_counts, aux_P, aux_loss, ws,
                       L.r, sms, s, launches, at<int32_t>(ws, L.f.hist), &hist_done, &counts_left);
        if (rc == MOE_OK)
            rc = forward_impl(c, hidden, W_gate_up, W_down, shared_gate_up, shared_down, topk_idx, topk_w, residual,
                              out, ws, L.f, nullptr, sms, s, launches, hist_done, true,
                              counts_left ? expert_counts : nullptr, (flags & MOE_LAYER_FUSED_COMBINE) != 0);
    }
    g_last_launches = launches;
    return rc;
}

int moe_expert_feedback(const moe_cfg *cfg, const int32_t *expert_counts, float gamma, float *expert_bias,
                        int64_t *totals, void *stream)
{
    ProfCall prof_call_;
    if (!cfg || cfg->E < 1 || cfg->T < 1 || cfg->k < 1 || !expert_counts || !isfinite(gamma))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(expert_counts, 4) || !aligned(expert_bias, 4) || !aligned(totals, 8))
        return MOE_ERR_MISALIGNED;
    int sms = 0, rc = device_check(&sms);
    if (rc != MOE_OK)
        return rc;
    if (launch_expert_feedback(expert_counts, cfg->E, cfg->T, cfg->k, gamma, expert_bias,
                               reinterpret_cast<long long *>(totals), static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    g_last_launches = 1;
    return MOE_OK;
}

int moe_rmsnorm(int32_t T, int32_t H, const moe_bf16 *x, moe_bf16 *out, float eps, void *stream)
{
    ProfCall prof_call_;
    if (T < 1 || H < 8 || H % 8 != 0 || !x || !out || !isfinite(eps) || eps < 0.0f)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(out, 16))
        return MOE_ERR_MISALIGNED;
    int sms = 0, rc = device_check(&sms);
    if (rc != MOE_OK)
        return rc;
    if (launch_rmsnorm(x, out, T, H, eps, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    g_last_launches = 1;
    return MOE_OK;
}

int moe_get_status(void *ws, size_t ws_bytes, void *stream, int32_t *status, int reset)
{
    int rc = check_ws(ws, ws_bytes, sizeof(WsHeader));
    if (rc != MOE_OK)
        return rc;
    if (!status)
        return MOE_ERR_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, &header(ws)->status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (reset && cudaMemsetAsync(&header(ws)->status, 0, sizeof(int32_t), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    *status = v;
    return MOE_OK;
}

int moe_last_launch_count(void) { return g_last_launches; }

int moe_debug_inject_timeout(int launches)
{
    if (launches < 0)
        return MOE_ERR_INVALID_ARG;
    g_inject_timeouts.store(launches);
    return MOE_OK;
}

int moe_profile_enable(int on)
{
    if (on < 0 || on > 2)
        return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(g_prof_mu);
    prof_close_stage_locked();
    g_prof_on.store(on);
    return MOE_OK;
}

int moe_profile_read(int kernel_id, double *total_ms, int32_t *launches, int reset)
{
    if (kernel_id < 0 || kernel_id >= MOE_KERNEL_COUNT || !total_ms || !launches)
        return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(g_prof_mu);
    int rc = MOE_OK;
    for (const ProfRecord &r : g_prof_pending) {
        float ms = 0.0f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
            rc = MOE_ERR_CUDA;
        g_prof_ms[r.kid] += ms;
        g_prof_n[r.kid] += 1;
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_prof_pending.clear();
    *total_ms = g_prof_ms[kernel_id];
    *launches = (int32_t)g_prof_n[kernel_id];
    if (reset) {
        g_prof_ms[kernel_id] = 0.0;
        g_prof_n[kernel_id] = 0;
    }
    return rc;
}

const char *moe_kernel_name(int kernel_id)
{
    if (kernel_id < 0 || kernel_id >= MOE_KERNEL_COUNT)
        return "";
    return kKernelNames[kernel_id];
}

const char *moe_strerror(int code)
{
    switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive size or inconsistent config)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "shape not supported by this implementation";
    case MOE_ERR_MISALIGNED: return "pointer not aligned (16 bytes for tensor-core operands, 256 for workspaces)";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than moe_workspace_bytes()";
    case MOE_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case MOE_ERR_DEVICE_STATUS: return "the device reported a fault in the status word";
    case MOE_ERR_TIMEOUT: return "a bounded device wait ran out";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300)";
    default: return "unknown error code";
    }
}

size_t moe_ep_dispatch_workspace_bytes(const moe_cfg *cfg, int32_t ranks)
{
    return check_ep(cfg, ranks) == MOE_OK ? ep_layout(*cfg, ranks).total : 0;
}

int moe_ep_dispatch(const moe_cfg *cfg, int32_t ranks, const moe_bf16 *hidden, const int32_t *topk_idx,
                    int32_t *send_counts, moe_bf16 *x_send, int32_t *e_send, int32_t *slot_of, void *ws,
                    size_t ws_bytes, void *stream)
{
    ProfCall prof_call_;
    int rc = check_ep(cfg, ranks);
    if (rc != MOE_OK)
        return rc;
    if (!hidden || !topk_idx || !send_counts || !x_send || !e_send || !slot_of)
        return MOE_ERR_INVALID_ARG;
    const EpLayout L = ep_layout(*cfg, ranks);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(hidden, 16) || !aligned(x_send, 16) || !aligned(topk_idx, 4) || !aligned(send_counts, 4) ||
        !aligned(e_send, 4) || !aligned(slot_of, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    const moe_cfg &c = *cfg;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader *hdr = header(ws);
    int32_t *dest = at<int32_t>(ws, L.dest);
    int32_t *hist = at<int32_t>(ws, L.hist);
    const long long n = (long long)c.T * c.k;
    int launches = 0;
    // the pairs bucketed by destination rank, stably (rows to one rank in
    // ascending (token, j) order), with the same kernels that bucket them by
    // expert; the bucketed copy of the rows is the send buffer
    GLR_LAUNCH(KID_HIST, launch_ep_dest(topk_idx, n, c.E, c.E / ranks, dest, s));
    GLR_LAUNCH(KID_HIST, launch_bucket_hist(dest, c.T, ranks, c.k, hist, &hdr->status, s));
    GLR_LAUNCH(KID_SCAN, launch_bucket_scan(hist, L.nchunk, ranks, send_counts, s));
    GLR_LAUNCH(KID_SCATTER, launch_bucket_scatter(dest, reinterpret_cast<const uint16_t *>(hidden), hist, send_counts,
                                                  c.T, c.H, ranks, c.k, slot_of, reinterpret_cast<uint16_t *>(x_send),
                                                  at<int4>(ws, L.mtiles), hdr, s, nullptr, false));
    GLR_LAUNCH(KID_SCATTER, launch_ep_local_ids(topk_idx, slot_of, n, c.E / ranks, e_send, s));
    g_last_launches = launches;
    return MOE_OK;
}

size_t moe_expert_rows_workspace_bytes(const moe_cfg *cfg, int32_t rows)
{
    if (!cfg || rows < 1)
        return 0;
    moe_cfg c = *cfg;
    c.T = rows;
    c.k = 1;
    c.Is = c.I;
    return check_forward_cfg(&c) == MOE_OK ? fwd_layout(c).total : 0;
}

int moe_expert_rows(const moe_cfg *cfg, int32_t rows, const moe_bf16 *x, const int32_t *expert,
                    const moe_bf16 *W_gate_up, const moe_bf16 *W_down, moe_bf16 *y, void *ws, size_t ws_bytes,
                    void *stream)
{
    ProfCall prof_call_;
    if (!cfg || rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (rows == 0) {
        g_last_launches = 0;
        return MOE_OK;                        // nothing received
    }
    moe_cfg c = *cfg;
    c.T = rows;
    c.k = 1;
    c.Is = c.I;
    int rc = check_forward_cfg(&c);
    if (rc != MOE_OK)
        return rc;
    if (!x || !expert || !W_gate_up || !W_down || !y)
        return MOE_ERR_INVALID_ARG;
    const FwdLayout L = fwd_layout(c);
    if ((rc = check_ws(ws, ws_bytes, L.total)) != MOE_OK)
        return rc;
    if (!aligned(x, 16) || !aligned(W_gate_up, 16) || !aligned(W_down, 16) || !aligned(y, 16) ||
        !aligned(expert, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    int launches = 0;
    rc = forward_impl(c, x, W_gate_up, W_down, nullptr, nullptr, expert, nullptr, nullptr, y, ws, L, nullptr, sms,
                      static_cast<cudaStream_t>(stream), launches, false, false);
    g_last_launches = launches;
    return rc;
}

int moe_combine(const moe_cfg *cfg, const moe_bf16 *Y, int64_t y_rows, int64_t shared_row0, const int32_t *slot_of,
                const float *topk_w, const moe_bf16 *residual, moe_bf16 *out, void *stream)
{
    ProfCall prof_call_;
    if (!cfg || cfg->T < 1 || cfg->k < 1 || cfg->k > 32 || cfg->H < 8 || !Y || !slot_of || !out)
        return MOE_ERR_INVALID_ARG;
    if (cfg->H % 8 != 0)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (shared_row0 < 0 || shared_row0 + cfg->T > y_rows)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(Y, 16) || !aligned(residual, 16) || !aligned(out, 16) || !aligned(slot_of, 4) ||
        !aligned(topk_w, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0, rc = MOE_OK;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    GLR_LAUNCH(KID_COMBINE, launch_combine(reinterpret_cast<const uint16_t *>(Y), slot_of, topk_w,
                                           reinterpret_cast<const uint16_t *>(residual), cfg->T, cfg->H, cfg->k,
                                           reinterpret_cast<uint16_t *>(out), s, shared_row0, nullptr, nullptr, 0,
                                           y_rows));
    g_last_launches = launches;
    return MOE_OK;
}

// ------------------------------------------------------ moe_route_static
// The scratch of moe_route_static: one array per device, zero at module load.
static __device__ __align__(256) unsigned char g_route_static_scratch[MOE_ROUTE_STATIC_SCRATCH_BYTES];

static std::mutex g_static_mu;

// A __device__ array has one address per CUDA context, not per device: a host
// that makes its own driver context current, or a process that resets the
// device, sees a new address.  So the looked-up address is cached per context,
// keyed by the driver's unique context id (never reused within a process).
struct StaticAddr {
    unsigned long long ctx_id;
    void *addr;
};
static StaticAddr g_static_addr[64];
static int g_static_n = 0, g_static_next = 0;

typedef CUresult (*PFN_ctx_get_current)(CUcontext *);
typedef CUresult (*PFN_ctx_get_id)(CUcontext, unsigned long long *);

// id of the context current on this thread; false when there is none yet
static bool current_ctx_id(unsigned long long *id)
{
    static PFN_ctx_get_current get_cur = nullptr;
    static PFN_ctx_get_id get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) == cudaSuccess &&
            r1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) == cudaSuccess &&
            r2 == cudaDriverEntryPointSuccess) {
            get_cur = reinterpret_cast<PFN_ctx_get_current>(p);
            get_id = reinterpret_cast<PFN_ctx_get_id>(q);
        }
        looked_up = true;
    }
    if (!get_cur || !get_id)
        return false;
    CUcontext c = nullptr;
    if (get_cur(&c) != CUDA_SUCCESS || !c)
        return false;
    return get_id(c, id) == CUDA_SUCCESS;
}

// Device address of the array in the current context.  The first call in a
// context looks it up with cudaGetSymbolAddress (host code only ever sees a
// stand-in for the symbol, so it must never hand `g_route_static_scratch` to a
// kernel); later calls in the same context reuse it.
static int static_scratch(void **addr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_static_mu);
    unsigned long long id = 0;
    if (current_ctx_id(&id)) {
        for (int i = 0; i < g_static_n; ++i)
            if (g_static_addr[i].ctx_id == id) {
                *addr = g_static_addr[i].addr;
                return MOE_OK;
            }
    }
    // set-up in this context (the lookup also makes the runtime's context
    // current when none was)
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_static_scratch) != cudaSuccess || !p)
        return MOE_ERR_CUDA;
    if (!current_ctx_id(&id))
        return MOE_ERR_CUDA;
    const int slot = g_static_n < 64 ? g_static_n++ : (g_static_next++ & 63);
    g_static_addr[slot] = StaticAddr{id, p};
    *addr = p;
    return MOE_OK;
}

int moe_route_static(const moe_cfg *cfg, const moe_bf16 *hidden, const float *W_router, const float *expert_bias,
                     int32_t *topk_idx, float *topk_w, int32_t *expert_counts, float *aux_P, float *aux_loss,
                     int32_t *status_out, void *stream)
{
    ProfCall prof_call_;
    int rc = check_route_cfg(cfg);
    if (rc != MOE_OK)
        return rc;
    if (!hidden || !W_router || !topk_idx || !topk_w || !expert_counts)
        return MOE_ERR_INVALID_ARG;
    const RouteLayout L = route_layout(*cfg);
    if (L.total > (size_t)MOE_ROUTE_STATIC_SCRATCH_BYTES)
        return MOE_ERR_UNSUPPORTED_SHAPE;   // needs more scratch than the fixed array holds
    if (!aligned(hidden, 16) || !aligned(W_router, 4) || !aligned(expert_bias, 4) || !aligned(topk_idx, 4) ||
        !aligned(topk_w, 4) || !aligned(expert_counts, 4) || !aligned(aux_P, 4) || !aligned(aux_loss, 4) ||
        !aligned(status_out, 4))
        return MOE_ERR_MISALIGNED;
    int sms = 0;
    if ((rc = device_check(&sms)) != MOE_OK)
        return rc;
    void *ws = nullptr;
    if ((rc = static_scratch(&ws)) != MOE_OK)
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the status word must start at zero
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    int launches = 0;
    rc = route_all(*cfg, hidden, W_router, nullptr, expert_bias, topk_idx, topk_w, expert_counts, aux_P, aux_loss, ws,
                   L, sms, s, launches);
    if (rc == MOE_OK && status_out &&
        cudaMemcpyAsync(status_out, &header(ws)->status, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        rc = MOE_ERR_CUDA;
    g_last_launches = launches;
    return rc;
}

}  // extern "C"
