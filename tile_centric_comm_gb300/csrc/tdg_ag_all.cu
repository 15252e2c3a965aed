// tdg_ag_all.cu -- AllGather + GEMM for every logical rank in one call
// ("Triton-distributed 语义", 内核设计模式 "AllGather + GEMM 重叠", run by every
// PE at once; paper summary, 方法: the intra-node AllGather on the copy engine).
//
// Rank r holds the shard A_r and its own weight shard B_r (the columns of the
// tensor-parallel weight it owns).  Every rank gathers all W shards and
// computes C_r = concat(A_0, ..., A_{W-1}) @ B_r: W times the work of one
// rank's call, with W x (W-1) shard copies.
//
// CE mode: the shard copies run on the copy engine (side stream), rank by
// rank -- rank r's remote shards in the order r+1, r+2, ... -- each followed
// by a stream-ordered write of rank r's flag for that signal group.  One
// persistent tcgen05 GEMM launch on the main stream runs every rank's tiles,
// rank by rank (each rank's B_r stays in L2 while its tiles run), each rank's
// m tiles in Triton-distributed's swizzled order (its own shard first, read in place);
// a tile's loader waits on the groups of its A rows with a bounded
// ld.acquire spin before its TMA loads.
// Push mode (CE): the senders order the copies step by step -- at step j
// every sender s copies its shard to destination (s + j) mod W -- so each
// destination receives one shard per step from a different sender, and the
// GEMM follows the steps: each rank's own shard first (step 0), then at step
// j the shard (r - j) mod W of every rank r.  Pull goes rank by rank.
// SERIAL mode: the same copies on the main stream, then the GEMM launch,
// which does not wait.
#include "tdg_gemm.cuh"
#include "tdg_internal.h"

namespace tdg {

struct AgAllParams {
    CUtensorMap tmA_g; // gathered A of every rank: {K, M, W}, plane stride = region bytes
    CUtensorMap tmA_l; // the shards, read in place: {K, Ms, W}
    CUtensorMap tmB;   // B_r: KN {N, K, W} box {64, 64, 1}; NK {K, N, W} box {64, rows, 1}
    CUtensorMap tmC;   // C_r: bf16 {N, M, W} box {64, 32, 1}, or fp32 box {32, 32, 1}
    DevStatus *status;
    uint32_t epoch;
    uint64_t timeout_ns;      // bound of a flag wait
    uint64_t pipe_timeout_ns; // bound of an intra-CTA pipeline wait (longer)
    int k_blocks;
    int W;
    int64_t M, K, N, Ms;
    int m_tiles, n_tiles; // per rank, tiles of 128 * cl rows
    int pair;             // 1: CTA pairs (cta_group::2)
    int cl;               // CTAs per cluster (1, 2 or 4)
    int group_m;          // 0: m-major per rank; > 0: groups of group_m m tiles, n outer
    int inplace;          // 1: Ms is a whole number of tiles, each rank's own shard is read in place
    int tiles_per_shard;  // Ms / (128 * cl) when inplace
    const uint32_t *flags; // rank 0's flag words
    uint64_t nsig;         // flag words per rank
    int wait_flags;
    int64_t sig_rows;
    int c_f32; // 1: C_r is fp32
    int stages; // GEMM ring stages in use
    int full_n; // N is a multiple of BN: every tile is full width
    int edge_n;   // > 0: only the last n-tile column is narrow, an MMA of edge_n columns
    int steps;  // 1: push order (items step by step, see tile()); 0: rank by rank
};

template <int BMN, bool F32 = false> struct AgAllPolicy {
    using Params = AgAllParams;
    static constexpr int B_MN = BMN;
    // C_r is bf16, or with F32 the fp32 accumulator itself (32-column chunks)
    static constexpr bool F32_OUT = F32;
    __device__ static bool out_f32(const Params &) { return true; }
    struct EpiState {};

    __device__ static int64_t num_items(const Params &p) { return (int64_t)p.W * p.m_tiles * p.n_tiles; }

    // item -> (rank r, m tile, n tile): ranks one after another; inside a rank
    // the single-rank AG-GEMM's order, its m tiles rotated by the rank swizzle
    __device__ static void tile(const Params &p, int64_t item, TileInfo &t, int sub)
    {
        const int tm = p.cl * gm::BM;
        const int64_t per_rank = (int64_t)p.m_tiles * p.n_tiles;
        if (p.steps) {
            // push order (whole tiles per shard): step j, then rank r, then the
            // m tiles of shard (r - j) mod W, n inner
            const int64_t per_shard = (int64_t)p.tiles_per_shard * p.n_tiles;
            const int64_t per_step = (int64_t)p.W * per_shard;
            int64_t rem, in, pn;
            const int j = (int)divmod(item, per_step, rem);
            const int r = (int)divmod(rem, per_shard, in);
            const int shard = ((r - j) % p.W + p.W) % p.W;
            const int pm = shard * p.tiles_per_shard + (int)divmod(in, p.n_tiles, pn);
            t.pn = (int)pn;
            set_tile(p, t, r, pm, sub, tm);
            return;
        }
        int64_t tid, r64;
        const int r = (int)divmod(item, per_rank, tid);
        int pm0;
        const int GM = p.group_m;
        if (GM <= 0) {
            pm0 = (int)divmod(tid, p.n_tiles, r64);
            t.pn = (int)r64;
        } else {
            const int64_t per_group = (int64_t)GM * p.n_tiles;
            int64_t in;
            const int grp = (int)divmod(tid, per_group, in);
            const int rows = min(GM, p.m_tiles - grp * GM);
            t.pn = (int)divmod(in, rows, r64);
            pm0 = grp * GM + (int)r64;
        }
        // Triton-distributed's swizzle: pid_m = (pid_m + rank * tiles_per_pe) % total
        const int pm = (pm0 + (int)(((int64_t)r * p.Ms / tm) % p.m_tiles)) % p.m_tiles;
        set_tile(p, t, r, pm, sub, tm);
    }

    // the rest of tile (r, pm, t.pn): rows, columns, A source
    __device__ static void set_tile(const Params &p, TileInfo &t, int r, int pm, int sub, int tm)
    {
        t.m0 = pm * tm + sub * gm::BM;
        t.n0 = t.pn * gm::BN;
        t.n_valid = (int)min((int64_t)gm::BN, p.N - t.n0);
        const int q = p.pair ? 32 : 16;
        t.n_mma = (t.n_valid + q - 1) / q * q;
        t.owner = r;
        t.m_loc = pm;
        if (p.inplace && pm >= r * p.tiles_per_shard && pm < (r + 1) * p.tiles_per_shard) {
            t.a_sel = 1;
            t.a_row = t.m0 - (int)(r * p.Ms);
        } else {
            t.a_sel = 0;
            t.a_row = t.m0;
        }
    }

    // wait(ptr, n) on rank r's groups that this CTA's rows fall into, then the
    // consume_token fence before the TMA reads of those rows
    __device__ static void before_a(const Params &p, const TileInfo &t, bool &gave_up)
    {
        if (t.a_sel == 1 || !p.wait_flags || t.m0 >= p.M)
            return;
        const int64_t r0 = t.m0;
        const int64_t r1 = min(p.M, (int64_t)t.m0 + gm::BM) - 1;
        const uint32_t *fl = p.flags + (uint64_t)t.owner * p.nsig;
        for (int64_t g = r0 / p.sig_rows; g <= r1 / p.sig_rows && !gave_up; ++g) {
            if (!wait_flag(fl + g, p.epoch, p.timeout_ns)) {
                report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_AG_FLAG,
                             (uint32_t)((uint64_t)t.owner * p.nsig + g), p.epoch);
                gave_up = true;
            }
        }
        fence_proxy_async_global();
    }

    // The TMA form is chosen at compile time: a kernel holds either only
    // cta_group::1 or only cta_group::2 instructions, never both.
    template <int CL>
    __device__ static void load(void *dst, const CUtensorMap *m, uint32_t bar, int x, int y, int z)
    {
        if constexpr (CL >= 2)
            tma_load_3d_pair(dst, m, bar, x, y, z);
        else
            tma_load_3d_addr(dst, m, bar, x, y, z);
    }

    template <int CL>
    __device__ static void load_a(const Params &p, const TileInfo &t, void *dst, uint32_t bar, int kb)
    {
        load<CL>(dst, t.a_sel ? &p.tmA_l : &p.tmA_g, bar, kb * gm::BK, t.a_row, t.owner);
    }

    // B_r slices of 64 columns (8 KB); with CL = 4 pair `pidx` fetches slices
    // pidx, pidx + 2, ... and multicasts each to CTA `half` of both pairs
    template <int CL>
    __device__ static void load_b(const Params &p, const TileInfo &t, void *dst, uint32_t bar, int kb,
                                  int col0, int cols, int pidx, int half)
    {
        uint8_t *d = static_cast<uint8_t *>(dst);
        if constexpr (CL == 4) {
            const uint16_t mask = (uint16_t)((1u << half) | (1u << (2 + half)));
            const int nch = BMN ? (cols + 63) >> 6 : 2;
            for (int j = pidx; j < nch; j += 2) {
                if (BMN)
                    tma_load_3d_pair_mc(d + j * 8192, &p.tmB, bar, col0 + 64 * j, kb * gm::BK, t.owner, mask);
                else
                    tma_load_3d_pair_mc(d + j * 8192, &p.tmB, bar, kb * gm::BK, col0 + 64 * j, t.owner, mask);
            }
        } else if (BMN) {
            const int nch = (cols + 63) >> 6;
            for (int j = 0; j < nch; ++j)
                load<CL>(d + j * 8192, &p.tmB, bar, col0 + 64 * j, kb * gm::BK, t.owner);
        } else {
            load<CL>(dst, &p.tmB, bar, kb * gm::BK, col0, t.owner);
        }
    }

    __device__ static uint32_t b_bytes(const Params &p, const TileInfo &, int cols)
    {
        return BMN ? (uint32_t)(((cols + 63) >> 6) * 8192) : (uint32_t)((p.pair ? gm::BN / 2 : gm::BN) * gm::BK * 2);
    }

    __device__ static void store_chunk(const Params &p, const TileInfo &t, const void *buf, int ch, int q)
    {
        const int row = t.m0 + 32 * q;
        if (row < p.M)
            tma_store_3d(&p.tmC, buf, t.n0 + 64 * ch, row, t.owner);
    }

    // (the second 32-column half of a 64-column chunk may start past N: skipped)
    __device__ static void store_chunk_f32(const Params &p, const TileInfo &t, const void *buf, int sub, int q)
    {
        const int row = t.m0 + 32 * q;
        const int col = t.n0 + 32 * sub;
        if (row < p.M && col < p.N)
            tma_store_3d(&p.tmC, buf, col, row, t.owner);
    }

    __device__ static void after_tile(const Params &, const TileInfo &, int, int, EpiState &, bool) {}
};

template <int BMN, int CL, bool F32>
__global__ void __launch_bounds__(gm::NUM_THREADS, 1) ag_all_gemm_kernel(const __grid_constant__ AgAllParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    gemm_consumer<AgAllPolicy<BMN, F32>, CL>(p, smem, (int)blockIdx.x / CL, (int)gridDim.x / CL);
}

} // namespace tdg

using namespace tdg;
using namespace tdg_host;

namespace {

template <int BMN, bool F32> const void *ag_all_kernel_cl(int cl)
{
    return cl == 4   ? reinterpret_cast<const void *>(&ag_all_gemm_kernel<BMN, 4, F32>)
           : cl == 2 ? reinterpret_cast<const void *>(&ag_all_gemm_kernel<BMN, 2, F32>)
                     : reinterpret_cast<const void *>(&ag_all_gemm_kernel<BMN, 1, F32>);
}

const void *ag_all_kernel_fn(int b_layout, int cl, bool f32)
{
    if (b_layout == TDG_B_KN)
        return f32 ? ag_all_kernel_cl<1, true>(cl) : ag_all_kernel_cl<1, false>(cl);
    return f32 ? ag_all_kernel_cl<0, true>(cl) : ag_all_kernel_cl<0, false>(cl);
}

bool meet(uint64_t x0, uint64_t x1, uint64_t y0, uint64_t y1) { return x0 < y1 && y0 < x1; }

} // namespace

extern "C" int tdg_ag_gemm_all_ranks(tdg_symm *h, const tdg_ag_gemm_all_args *a, void *stream,
                                     void *side_stream)
{
    if (!h || !a)
        return TDG_ERR_INVALID;
    if (const int drc = check_device(h))
        return drc;
    const int W = a->world;
    if (W != h->world || a->Ms < 0 || a->K < 0 || a->N < 0)
        return TDG_ERR_INVALID;
    if (a->mode != TDG_MODE_CE && a->mode != TDG_MODE_SERIAL)
        return TDG_ERR_INVALID;
    if (a->b_layout != TDG_B_KN && a->b_layout != TDG_B_NK)
        return TDG_ERR_INVALID;
    if (a->c_f32 != 0 && a->c_f32 != 1)
        return TDG_ERR_INVALID;
    const int64_t Ms = a->Ms, K = a->K, N = a->N, M = (int64_t)W * Ms;
    const uint64_t c_elem = a->c_f32 ? 4 : 2;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0)
        return TDG_OK;
    if (!aligned16(a->a_off) || !aligned16(a->g_off) || !aligned16(a->b_off) || !aligned16(a->c_off) ||
        K % 8 || N % 8 || M > INT32_MAX || K > INT32_MAX || N > INT32_MAX)
        return TDG_ERR_INVALID;
    const uint64_t R = h->region_bytes;
    const uint64_t a_end = a->a_off + (uint64_t)Ms * K * 2, g_end = a->g_off + (uint64_t)M * K * 2;
    const uint64_t b_end = a->b_off + (uint64_t)K * N * 2, c_end = a->c_off + (uint64_t)M * N * c_elem;
    if (a_end > R || g_end > R || b_end > R || c_end > R)
        return TDG_ERR_NOMEM;
    // the buffers written (gathered, C) overlap nothing else
    if (K > 0 && (meet(a->g_off, g_end, a->a_off, a_end) || meet(a->g_off, g_end, a->b_off, b_end) ||
                  meet(a->g_off, g_end, a->c_off, c_end)))
        return TDG_ERR_INVALID;
    if (meet(a->c_off, c_end, a->a_off, a_end) || meet(a->c_off, c_end, a->b_off, b_end))
        return TDG_ERR_INVALID;
    if (K == 0) {
        for (int r = 0; r < W; ++r) {
            cudaError_t e = cudaMemsetAsync(h->base + (size_t)r * R + a->c_off, 0, (size_t)(M * N * c_elem), s);
            if (e != cudaSuccess)
                return cuda_err(e, "ag all K==0");
        }
        return TDG_OK;
    }

    const int BM = gm::BM;
    const int cl = pick_cluster(a->cluster, M > BM, Ms % (4 * BM) == 0);
    const int stages = cl ? pick_stages(a->stages, cl) : 0;
    if (!cl || !stages || (a->push & ~1))
        return TDG_ERR_INVALID;
    const int pair = cl >= 2 ? 1 : 0;
    const int TM = cl * BM;
    const bool inplace = (Ms % TM) == 0;
    int64_t sig_rows = a->signal_rows > 0 ? a->signal_rows : Ms;
    if (sig_rows > Ms || Ms % sig_rows)
        return TDG_ERR_INVALID;
    if ((uint64_t)(M / sig_rows) > h->nsig)
        return TDG_ERR_NOMEM;

    AgAllParams p;
    memset(&p, 0, sizeof p);
    bool ok = map_bf16_3d(&p.tmA_g, h->base + a->g_off, K, M, W, K * 2, R, 64, BM, 1);
    ok = ok && map_bf16_3d(&p.tmA_l, h->base + a->a_off, K, Ms, W, K * 2, R, 64, BM, 1);
    if (a->b_layout == TDG_B_KN)
        ok = ok && map_bf16_3d(&p.tmB, h->base + a->b_off, N, K, W, N * 2, R, 64, 64, 1);
    else
        ok = ok && map_bf16_3d(&p.tmB, h->base + a->b_off, K, N, W, K * 2, R, 64,
                               cl == 4 ? 64 : (pair ? 128 : 256), 1);
    ok = ok && (a->c_f32 ? map_f32_3d(&p.tmC, h->base + a->c_off, N, M, W, N * 4, R, 32, 32, 1)
                         : map_bf16_3d(&p.tmC, h->base + a->c_off, N, M, W, N * 2, R, 64, 32, 1));
    if (!ok)
        return TDG_ERR_CUDA;
    const uint32_t epoch = next_epoch(h);
    p.status = h->status;
    p.epoch = epoch;
    p.timeout_ns = timeout_or_default(a->timeout_ns);
    p.pipe_timeout_ns = pipe_timeout(p.timeout_ns);
    p.k_blocks = (int)((K + gm::BK - 1) / gm::BK);
    p.W = W;
    p.M = M;
    p.K = K;
    p.N = N;
    p.Ms = Ms;
    p.m_tiles = (int)((M + TM - 1) / TM);
    p.n_tiles = (int)((N + gm::BN - 1) / gm::BN);
    p.pair = pair;
    p.cl = cl;
    // B_r larger than about half of L2: groups of 8 m tiles, n outer
    p.group_m = ((uint64_t)K * N * 2 > (64ull << 20)) ? 8 : 0;
    p.inplace = inplace ? 1 : 0;
    p.tiles_per_shard = inplace ? (int)(Ms / TM) : 0;
    p.flags = h->flags;
    p.nsig = h->nsig;
    p.sig_rows = sig_rows;
    p.c_f32 = a->c_f32;
    p.stages = stages;
    p.full_n = (N % gm::BN) == 0 ? 1 : 0;
    // the GEMM follows the push steps when every shard is whole tiles (else it
    // keeps the rank-by-rank order: the same result, only the waits differ)
    p.steps = (a->push && a->mode == TDG_MODE_CE && inplace) ? 1 : 0;
    // both orders without groups put item i in n-tile column i mod n_tiles
    // (every block of the order is whole rows of n_tiles items)
    p.edge_n = 0;
    if (!p.full_n && p.group_m <= 0) {
        const int q16 = p.pair ? 32 : 16;
        const int nv = (int)(N - (int64_t)(p.n_tiles - 1) * gm::BN);
        p.edge_n = (nv + q16 - 1) / q16 * q16;
    }

    const void *fn = ag_all_kernel_fn(a->b_layout, cl, a->c_f32 != 0);
    if (cudaError_t e = set_smem(fn, gm::SMEM_BYTES); e != cudaSuccess)
        return cuda_err(e, "ag all set smem");
    int grid = h->sm_count;
    if (cl > 1) {
        const int mc = max_clusters(fn, gm::NUM_THREADS, gm::SMEM_BYTES, cl);
        const int n = mc < h->sm_count / cl ? mc : h->sm_count / cl;
        if (n <= 0)
            return TDG_ERR_UNSUPPORTED;
        grid = cl * n;
    }
    const int64_t items = (int64_t)W * p.m_tiles * p.n_tiles;
    if (grid / cl > items)
        grid = (int)(cl * items);

    // One shard copy: shard `shard` into rank r's gathered buffer, one signal
    // group per copy, each followed by rank r's flag for it.
    auto copy_shard = [&](cudaStream_t cs, bool signal, int r, int shard) -> int {
        const int64_t ups = Ms / sig_rows;
        uint8_t *gathered = h->base + (size_t)r * R + a->g_off;
        uint32_t *fl = h->flags + (size_t)r * h->nsig;
        for (int64_t part = 0; part < ups; ++part) {
            const int64_t row0 = part * sig_rows, grow = (int64_t)shard * Ms + row0;
            const uint8_t *src = h->base + (size_t)shard * R + a->a_off + (size_t)row0 * K * 2;
            cudaError_t e = cudaMemcpyAsync(gathered + (size_t)grow * K * 2, src, (size_t)sig_rows * K * 2,
                                            cudaMemcpyDeviceToDevice, cs);
            if (e != cudaSuccess)
                return cuda_err(e, "ag all memcpy");
            const int64_t g = grow / sig_rows;
            const bool skip = r == 0 && ((a->test_skip_notify >> (g & 63)) & 1ull);
            if (signal && !skip && !stream_write_u32(cs, fl + g, epoch))
                return TDG_ERR_UNSUPPORTED;
        }
        return TDG_OK;
    };
    // Pull: rank by rank, rank r's remote shards r+1, r+2, ... (its own shard
    // last when it is read in place, else first).  Push: step by step, sender
    // s to destination (s + j) mod W at step j (the own shards as step 0: last
    // when read in place, else first).
    auto copies = [&](cudaStream_t cs, bool signal) -> int {
        int rc = TDG_OK;
        if (!a->push) {
            for (int r = 0; r < W && rc == TDG_OK; ++r)
                for (int j = 0; j < W && rc == TDG_OK; ++j)
                    rc = copy_shard(cs, signal, r, inplace ? (r + 1 + j) % W : (r + j) % W);
            return rc;
        }
        for (int jj = 0; jj < W && rc == TDG_OK; ++jj) {
            const int j = inplace ? (jj + 1) % W : jj;
            for (int snd = 0; snd < W && rc == TDG_OK; ++snd)
                rc = copy_shard(cs, signal, (snd + j) % W, snd);
        }
        return rc;
    };
    void *args[] = {&p};
    if (a->mode == TDG_MODE_SERIAL) {
        int rc = copies(s, false);
        if (rc != TDG_OK)
            return rc;
        p.wait_flags = 0;
        return cuda_err(launch(fn, dim3(grid), dim3(gm::NUM_THREADS), gm::SMEM_BYTES, s, args, false, cl),
                        "ag all gemm launch");
    }
    // CE mode: the copies on the side stream, the GEMM on the main stream
    cudaStream_t side = static_cast<cudaStream_t>(side_stream);
    if (!side || side == s)
        return TDG_ERR_INVALID;
    cudaEvent_t ev0, ev1;
    if (!ce_events(h, ev0, ev1))
        return TDG_ERR_CUDA;
    int rc = TDG_OK;
    cudaError_t e = cudaEventRecord(ev0, s);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(side, ev0, 0);
    if (e != cudaSuccess)
        rc = cuda_err(e, "ag all events");
    // The copies and their flag writes are queued before the GEMM that waits
    // on them (the producer transfers, then signals; the consumer waits), so
    // the call completes whatever order the two streams run in -- one after
    // the other included.  The side stream starts only after ev0, so the GEMM
    // is not behind the copies: the tiles of each rank's own shard start at once.
    if (rc == TDG_OK)
        rc = copies(side, true);
    if (rc == TDG_OK) {
        p.wait_flags = 1;
        rc = cuda_err(launch(fn, dim3(grid), dim3(gm::NUM_THREADS), gm::SMEM_BYTES, s, args, false, cl),
                      "ag all gemm launch");
    }
    // the call completes on the main stream only when the side stream has too
    e = cudaEventRecord(ev1, side);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(s, ev1, 0);
    if (e != cudaSuccess && rc == TDG_OK)
        rc = cuda_err(e, "ag all join");
    return rc;
}
