// tdg_moe.cu -- expert-parallel AllToAll dispatch / combine as a permutation
// of token rows between W logical ranks (paper summary, 实验: AllToAll dispatch
// and combine; "Triton-distributed 正把通信纳入编译器的职责范围", "DITRON 加入三级
// 分块": per-expert row counts are only known at run time, so the receive
// layout is computed on the device).
//
// Routing (integer, bit-exact):
//   1. moe_hist_kernel    one CTA per (source rank, 64-token chunk): shared-
//                         memory histogram of the chunk's expert ids.
//   2. moe_scan_kernel    one CTA: per-(src, e) counts, the expert-major
//                         exclusive scan base[e], and every chunk's first row
//                         per expert, base[e] + rows of e from earlier ranks +
//                         rows of e from earlier chunks of the same rank.
//   3. moe_slot_kernel    one warp per chunk walks its tokens in order; lanes
//                         are the k routing slots; equal expert ids inside a
//                         token are ranked by lane (match.any), so rows of an
//                         expert follow (src, t, kk) order exactly.
// Dispatch (HBM bound): copy warps bulk-load a row chunk (<= 16 KB) into
//   shared memory once and bulk-store it to its k receive rows.
// Combine (HBM bound): one CTA per token; 16-byte loads of the k rows, fp32
//   gate-weighted sum in kk order, bf16 (round to nearest even) store.
#include "tdg_internal.h"

namespace tdg {

namespace moe {
constexpr int TC = 64;            // tokens per routing chunk
constexpr int DW = 6;             // copy warps per dispatch CTA
constexpr int DCHUNK = 16384;     // max bytes of one row chunk
constexpr int D_SMEM = DW * 2 * DCHUNK + DW * 2 * 8 + 1024;
constexpr int MAX_E = 4096;
} // namespace moe

struct MoeParams {
    DevStatus *status;
    uint32_t epoch;
    int W, E, k, n_chunks;
    int64_t T, H;
    uint8_t *regions;
    uint64_t region_bytes;
    uint64_t x_off, topk_off, gate_off, out_off;
    uint8_t *recv;
    const uint8_t *y;
    int64_t *counts, *base, *slot;
    int32_t *row_src, *row_tok, *row_k;
    int32_t *chunk_hist; // [W][n_chunks][E]
    int32_t *chunk_base; // [W][n_chunks][E]
    uint64_t timeout_ns;
};

__device__ __forceinline__ const int32_t *moe_topk(const MoeParams &p, int src)
{
    return reinterpret_cast<const int32_t *>(p.regions + (uint64_t)src * p.region_bytes + p.topk_off);
}

__global__ void moe_hist_kernel(const __grid_constant__ MoeParams p)
{
    extern __shared__ int32_t hist[];
    const int chunk = blockIdx.x, src = blockIdx.y;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x)
        hist[e] = 0;
    __syncthreads();
    const int32_t *tk = moe_topk(p, src);
    const int64_t t0 = (int64_t)chunk * moe::TC;
    const int64_t t1 = min(p.T, t0 + moe::TC);
    const int64_t n = (t1 - t0) * p.k;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        const int64_t q = t0 * p.k + i;
        const int e = tk[q];
        if (e >= 0 && e < p.E)
            atomicAdd(&hist[e], 1);
        else
            report_fault(p.status, TDG_ERR_DEVICE, TDG_WHERE_MOE_EXPERT,
                         (uint32_t)((uint64_t)src * p.T * p.k + q), p.epoch);
    }
    __syncthreads();
    int32_t *out = p.chunk_hist + ((int64_t)src * p.n_chunks + chunk) * p.E;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x)
        out[e] = hist[e];
}

__global__ void __launch_bounds__(1024) moe_scan_kernel(const __grid_constant__ MoeParams p)
{
    extern __shared__ int64_t tot[]; // [E] then [1024] segment sums
    int64_t *seg = tot + p.E;
    const int W = p.W, E = p.E, nc = p.n_chunks;
    // counts[src][e] and the per-chunk exclusive prefix (in place)
    for (int idx = threadIdx.x; idx < W * E; idx += blockDim.x) {
        const int src = idx / E, e = idx % E;
        int32_t *h = p.chunk_hist + (int64_t)src * nc * E + e;
        int64_t run = 0;
        for (int c = 0; c < nc; ++c) {
            const int32_t v = h[(int64_t)c * E];
            h[(int64_t)c * E] = (int32_t)run;
            run += v;
        }
        p.counts[idx] = run;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int64_t s = 0;
        for (int src = 0; src < W; ++src)
            s += p.counts[(int64_t)src * E + e];
        tot[e] = s;
    }
    __syncthreads();
    // exclusive scan of tot over experts: contiguous segments per thread
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int lo = min(E, (int)threadIdx.x * per), hi = min(E, lo + per);
    int64_t s = 0;
    for (int e = lo; e < hi; ++e)
        s += tot[e];
    seg[threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t run = 0;
        for (int i = 0; i < (int)blockDim.x; ++i) {
            const int64_t v = seg[i];
            seg[i] = run;
            run += v;
        }
        p.base[E] = run;
    }
    __syncthreads();
    s = seg[threadIdx.x];
    for (int e = lo; e < hi; ++e) {
        const int64_t v = tot[e];
        p.base[e] = s;
        tot[e] = s; // tot now holds base
        s += v;
    }
    __syncthreads();
    // first receive row of every (src, chunk, e)
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int64_t run = tot[e];
        for (int src = 0; src < W; ++src) {
            for (int c = 0; c < nc; ++c) {
                const int64_t at = ((int64_t)src * nc + c) * E + e;
                p.chunk_base[at] = (int32_t)(run + p.chunk_hist[at]);
            }
            run += p.counts[(int64_t)src * E + e];
        }
    }
}

__global__ void __launch_bounds__(32) moe_slot_kernel(const __grid_constant__ MoeParams p)
{
    extern __shared__ int32_t sm[]; // cursor[E], then topk of the chunk
    int32_t *cursor = sm;
    int32_t *tks = sm + p.E;
    const int chunk = blockIdx.x, src = blockIdx.y, lane = threadIdx.x;
    const int32_t *cb = p.chunk_base + ((int64_t)src * p.n_chunks + chunk) * p.E;
    for (int e = lane; e < p.E; e += 32)
        cursor[e] = cb[e];
    const int64_t t0 = (int64_t)chunk * moe::TC;
    const int64_t t1 = min(p.T, t0 + moe::TC);
    const int k = p.k;
    const int32_t *tk = moe_topk(p, src) + t0 * k;
    for (int64_t i = lane; i < (t1 - t0) * k; i += 32)
        tks[i] = tk[i];
    __syncwarp();
    const unsigned active = (k >= 32) ? 0xffffffffu : ((1u << k) - 1u);
    for (int64_t t = t0; t < t1; ++t) {
        if (lane < k) {
            const int e = tks[(t - t0) * k + lane];
            const bool valid = e >= 0 && e < p.E;
            const int key = valid ? e : -1 - lane; // invalid ids never match
            const unsigned peers = __match_any_sync(active, key);
            const int64_t q = ((int64_t)src * p.T + t) * k + lane;
            if (valid) {
                const int rank = __popc(peers & ((1u << lane) - 1u));
                const int32_t s = cursor[e] + rank;
                p.slot[q] = s;
                if (p.row_src) {
                    p.row_src[s] = src;
                    p.row_tok[s] = (int32_t)t;
                    p.row_k[s] = lane;
                }
                __syncwarp(active);
                if (rank == 0)
                    cursor[e] += __popc(peers);
            } else {
                p.slot[q] = -1;
                __syncwarp(active);
            }
            __syncwarp(active);
        }
        __syncwarp();
    }
}

// Dispatch: recv[slot(src,t,kk)] = x_src[t].
__global__ void __launch_bounds__(moe::DW * 32) moe_dispatch_kernel(const __grid_constant__ MoeParams p,
                                                                    int64_t units, int chunks_per_row,
                                                                    uint32_t chunk_bytes)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *buf = smem + warp * 2 * moe::DCHUNK;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + moe::DW * 2 * moe::DCHUNK) + warp * 2;
    if (lane == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncwarp();
    const uint64_t row_bytes = (uint64_t)p.H * 2;
    const int64_t wid = (int64_t)blockIdx.x * moe::DW + warp;
    const int64_t nw = (int64_t)gridDim.x * moe::DW;
    auto unit_src = [&](int64_t u, uint32_t &bytes) -> const uint8_t * {
        const int64_t tok = u / chunks_per_row; // global token id src*T + t
        const int c = (int)(u % chunks_per_row);
        const int src = (int)(tok / p.T);
        const int64_t t = tok % p.T;
        const uint64_t off = (uint64_t)c * chunk_bytes;
        bytes = (uint32_t)min((uint64_t)chunk_bytes, row_bytes - off);
        return p.regions + (uint64_t)src * p.region_bytes + p.x_off + (uint64_t)t * row_bytes + off;
    };
    uint32_t phase = 0;
    uint32_t pending = 0; // buffers with a load in flight (lane 0)
    int64_t u = wid;
    if (u < units && lane == 0) {
        uint32_t b;
        const uint8_t *s = unit_src(u, b);
        mbar_arrive_expect_tx(&bar[0], b);
        bulk_load(buf, s, b, &bar[0]);
        pending |= 1u;
    }
    for (int i = 0; u < units; ++i, u += nw) {
        const int cur = i & 1;
        const int64_t tok = u / chunks_per_row;
        const int c = (int)(u % chunks_per_row);
        int64_t sl = -1;
        if (lane < p.k)
            sl = p.slot[tok * p.k + lane];
        bool ok = true;
        if (lane == 0) {
            const int64_t un = u + nw;
            if (un < units) {
                bulk_wait_read<0>(); // the other buffer's stores have read it
                uint32_t b;
                const uint8_t *s = unit_src(un, b);
                mbar_arrive_expect_tx(&bar[cur ^ 1], b);
                bulk_load(buf + (cur ^ 1) * moe::DCHUNK, s, b, &bar[cur ^ 1]);
                pending |= 1u << (cur ^ 1);
            }
            ok = mbar_wait(&bar[cur], (phase >> cur) & 1u, p.timeout_ns);
            if (ok) {
                phase ^= 1u << cur;
                pending &= ~(1u << cur);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) {
            if (lane == 0) {
                report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_PIPE, (uint32_t)u, p.epoch);
                // drain this warp's other load in flight (bounded) before leaving
                if ((pending >> (cur ^ 1)) & 1u)
                    (void)mbar_wait(&bar[cur ^ 1], (phase >> (cur ^ 1)) & 1u, p.timeout_ns);
            }
            break;
        }
        uint32_t bytes = 0;
        (void)unit_src(u, bytes);
        for (int kk = 0; kk < p.k; ++kk) {
            const int64_t s = __shfl_sync(0xffffffffu, sl, kk);
            if (lane == 0 && s >= 0)
                bulk_store(p.recv + (uint64_t)s * row_bytes + (uint64_t)c * chunk_bytes,
                           buf + cur * moe::DCHUNK, bytes);
        }
        if (lane == 0)
            bulk_commit();
        __syncwarp();
    }
    if (lane == 0)
        bulk_wait<0>();
}

// Combine: out_src[t] = bf16(sum_kk gate[t][kk] * y[slot(src,t,kk)]).
__global__ void __launch_bounds__(128) moe_combine_kernel(const __grid_constant__ MoeParams p)
{
    __shared__ float g[32];
    __shared__ int64_t sl[32];
    const int64_t tok = blockIdx.x; // src*T + t
    const int src = (int)(tok / p.T);
    const int64_t t = tok % p.T;
    const int k = p.k;
    if ((int)threadIdx.x < k) {
        const float *gate = reinterpret_cast<const float *>(p.regions + (uint64_t)src * p.region_bytes + p.gate_off);
        g[threadIdx.x] = gate[t * k + threadIdx.x];
        sl[threadIdx.x] = p.slot[tok * k + threadIdx.x];
    }
    __syncthreads();
    const int64_t nvec = p.H / 8;
    const uint64_t row_bytes = (uint64_t)p.H * 2;
    uint8_t *out = p.regions + (uint64_t)src * p.region_bytes + p.out_off + (uint64_t)t * row_bytes;
    for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            acc[j] = 0.f;
        for (int k0 = 0; k0 < k; k0 += 8) {
            uint4 val[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (k0 + j < k && sl[k0 + j] >= 0)
                    val[j] = __ldg(reinterpret_cast<const uint4 *>(p.y + (uint64_t)sl[k0 + j] * row_bytes) + v);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (k0 + j < k && sl[k0 + j] >= 0) {
                    const float w = g[k0 + j];
                    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&val[j]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h[e]);
                        acc[2 * e] = fmaf(w, f.x, acc[2 * e]);
                        acc[2 * e + 1] = fmaf(w, f.y, acc[2 * e + 1]);
                    }
                }
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4 *>(out)[v] = o;
    }
}

} // namespace tdg

using namespace tdg;
using namespace tdg_host;

extern "C" size_t tdg_moe_workspace_bytes(int world, int64_t T, int E)
{
    if (world <= 0 || T < 0 || E <= 0)
        return 0;
    const int64_t nc = (T + moe::TC - 1) / moe::TC;
    return (size_t)2 * world * (nc > 0 ? nc : 1) * E * sizeof(int32_t);
}

namespace {

// Every argument check of tdg_moe_dispatch_combine except the workspace's:
// TDG_OK when the call may go ahead (T == 0 included).
int moe_validate(const tdg_symm *h, const tdg_moe_args *a)
{
    const int W = a->world, E = a->E, k = a->k;
    const int64_t T = a->T, H = a->H;
    if (W != h->world || T < 0 || H < 0 || E <= 0 || E > moe::MAX_E || E % W || k < 1 || k > 32 || k > E)
        return TDG_ERR_INVALID;
    if ((a->phases & ~TDG_MOE_ALL) || a->phases == 0)
        return TDG_ERR_INVALID;
    if (T == 0)
        return TDG_OK;
    const int64_t total = (int64_t)W * T * k;
    if (total >= INT32_MAX || H % 8 || !aligned16(a->x_off) || !aligned16(a->out_off) ||
        (a->topk_off & 3) || (a->gate_off & 3))
        return TDG_ERR_INVALID;
    const uint64_t R = h->region_bytes;
    const bool route = a->phases & TDG_MOE_ROUTE, disp = a->phases & TDG_MOE_DISPATCH,
               comb = a->phases & TDG_MOE_COMBINE;
    if (a->topk_off + (uint64_t)T * k * 4 > R || a->gate_off + (uint64_t)T * k * 4 > R ||
        a->x_off + (uint64_t)T * H * 2 > R || a->out_off + (uint64_t)T * H * 2 > R)
        return TDG_ERR_NOMEM;
    if (!a->slot || (route && (!a->counts || !a->base)))
        return TDG_ERR_INVALID;
    // combine writes out while it reads the gates
    if (comb && a->out_off < a->gate_off + (uint64_t)T * k * 4 && a->gate_off < a->out_off + (uint64_t)T * H * 2)
        return TDG_ERR_INVALID;
    if ((disp || (comb && !a->y)) && (!a->recv || !aligned16(a->recv)))
        return TDG_ERR_INVALID;
    if (a->y && !aligned16(a->y))
        return TDG_ERR_INVALID;
    if ((a->row_src || a->row_tok || a->row_k) && !(a->row_src && a->row_tok && a->row_k))
        return TDG_ERR_INVALID;
    return TDG_OK;
}

} // namespace

extern "C" int tdg_moe_dispatch_combine(tdg_symm *h, const tdg_moe_args *a, void *stream)
{
    if (!h || !a)
        return TDG_ERR_INVALID;
    if (const int drc = check_device(h))
        return drc;
    if (const int vrc = moe_validate(h, a))
        return vrc;
    const int W = a->world, E = a->E, k = a->k;
    const int64_t T = a->T, H = a->H;
    if (T == 0)
        return TDG_OK;
    const uint64_t R = h->region_bytes;
    const bool route = a->phases & TDG_MOE_ROUTE, disp = a->phases & TDG_MOE_DISPATCH,
               comb = a->phases & TDG_MOE_COMBINE;
    const int nc = (int)((T + moe::TC - 1) / moe::TC);
    if (route && (!a->workspace || a->workspace_bytes < tdg_moe_workspace_bytes(W, T, E)))
        return TDG_ERR_NOMEM;

    MoeParams p;
    memset(&p, 0, sizeof p);
    p.status = h->status;
    p.epoch = next_epoch(h);
    p.W = W;
    p.E = E;
    p.k = k;
    p.n_chunks = nc;
    p.T = T;
    p.H = H;
    p.regions = h->base;
    p.region_bytes = R;
    p.x_off = a->x_off;
    p.topk_off = a->topk_off;
    p.gate_off = a->gate_off;
    p.out_off = a->out_off;
    p.recv = static_cast<uint8_t *>(a->recv);
    p.y = a->y ? static_cast<const uint8_t *>(a->y) : static_cast<const uint8_t *>(a->recv);
    p.counts = a->counts;
    p.base = a->base;
    p.slot = a->slot;
    p.row_src = a->row_src;
    p.row_tok = a->row_tok;
    p.row_k = a->row_k;
    p.chunk_hist = static_cast<int32_t *>(a->workspace);
    p.chunk_base = p.chunk_hist ? p.chunk_hist + (size_t)W * nc * E : nullptr;
    p.timeout_ns = timeout_or_default(0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *args[] = {&p};
    cudaError_t e;
    if (route) {
        e = launch(reinterpret_cast<const void *>(&moe_hist_kernel), dim3(nc, W), dim3(256),
                   (size_t)E * 4, s, args, false);
        if (e != cudaSuccess)
            return cuda_err(e, "moe hist");
        e = launch(reinterpret_cast<const void *>(&moe_scan_kernel), dim3(1), dim3(1024),
                   (size_t)(E + 1024) * 8, s, args, false);
        if (e != cudaSuccess)
            return cuda_err(e, "moe scan");
        const size_t slot_smem = (size_t)E * 4 + (size_t)moe::TC * k * 4;
        e = launch(reinterpret_cast<const void *>(&moe_slot_kernel), dim3(nc, W), dim3(32), slot_smem,
                   s, args, false);
        if (e != cudaSuccess)
            return cuda_err(e, "moe slot");
    }
    if (disp) {
        e = set_smem(reinterpret_cast<const void *>(&moe_dispatch_kernel), moe::D_SMEM);
        if (e != cudaSuccess)
            return cuda_err(e, "moe dispatch smem");
        const uint64_t row_bytes = (uint64_t)H * 2;
        const int cpr = (int)((row_bytes + moe::DCHUNK - 1) / moe::DCHUNK);
        // equal chunks, 16-byte multiples
        uint32_t cb = (uint32_t)((row_bytes + cpr - 1) / cpr);
        cb = (cb + 15) & ~15u;
        int64_t units = (int64_t)W * T * cpr;
        int64_t ucopy = units;
        uint32_t cbc = cb;
        int cprc = cpr;
        void *dargs[] = {&p, &ucopy, &cprc, &cbc};
        int grid = h->sm_count;
        e = launch(reinterpret_cast<const void *>(&moe_dispatch_kernel), dim3(grid), dim3(moe::DW * 32),
                   moe::D_SMEM, s, dargs, false);
        if (e != cudaSuccess)
            return cuda_err(e, "moe dispatch");
    }
    if (comb) {
        e = launch(reinterpret_cast<const void *>(&moe_combine_kernel), dim3((unsigned)(W * T)), dim3(128),
                   0, s, args, false);
        if (e != cudaSuccess)
            return cuda_err(e, "moe combine");
    }
    return TDG_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the routing scratch lives in a fixed device array
// of this file instead of a caller-provided workspace, for callers that cannot
// allocate device memory when they call.  Host code cannot pass the array's
// name to a kernel (on the host it is only a stand-in symbol); its device
// address is looked up with cudaGetSymbolAddress, with the device current,
// the first time a context uses it, and kept per (device, context): a context
// built again after a device reset looks it up afresh.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

static __device__ __align__(256) int32_t g_moe_static_ws[TDG_MOE_STATIC_WORKSPACE_BYTES / sizeof(int32_t)];

struct StaticWs {
    int dev;
    void *ctx;
    void *ptr;
};
std::mutex g_static_ws_mu;
StaticWs g_static_ws[64] = {};
int g_static_ws_n = 0;

} // namespace

extern "C" int tdg_moe_dispatch_combine_noalloc(tdg_symm *h, const tdg_moe_args *a, void *stream)
{
    if (!h || !a)
        return TDG_ERR_INVALID;
    if (const int drc = check_device(h))
        return drc;
    // the arguments first, so that a bad argument gives the regular entry
    // point's code whatever workspace it would need
    if (const int vrc = moe_validate(h, a))
        return vrc;
    if (a->T == 0)
        return TDG_OK;
    if ((a->phases & TDG_MOE_ROUTE) &&
        tdg_moe_workspace_bytes(a->world, a->T, a->E) > (size_t)TDG_MOE_STATIC_WORKSPACE_BYTES) {
        if (getenv("TDG_LOG"))
            fprintf(stderr, "[tdg] moe noalloc: routing needs %zu bytes of scratch, the fixed array holds %u\n",
                    tdg_moe_workspace_bytes(a->world, a->T, a->E), TDG_MOE_STATIC_WORKSPACE_BYTES);
        return TDG_ERR_NOMEM;
    }
    void *ctx = current_context();
    if (!ctx)
        return TDG_ERR_CUDA;
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_ws_mu);
        for (int i = 0; i < g_static_ws_n; ++i)
            if (g_static_ws[i].dev == h->device && g_static_ws[i].ctx == ctx)
                ws = g_static_ws[i].ptr;
        if (!ws) {
            void *p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_moe_static_ws);
            if (e != cudaSuccess || !p)
                return cuda_err(e != cudaSuccess ? e : cudaErrorInvalidSymbol, "moe noalloc symbol");
            // one entry per (device, context); a full table reuses its oldest slot
            StaticWs &slot = g_static_ws[g_static_ws_n < 64 ? g_static_ws_n++ : 0];
            slot = StaticWs{h->device, ctx, p};
            ws = p;
        }
    }
    tdg_moe_args b = *a;
    b.workspace = ws;
    b.workspace_bytes = TDG_MOE_STATIC_WORKSPACE_BYTES;
    return tdg_moe_dispatch_combine(h, &b, stream);
}
