// tdg_ag.cu -- tile-centric overlapped AllGather + GEMM ("Triton-distributed
// 语义", 内核设计模式 "AllGather + GEMM 重叠"; paper summary, 方法: AllGather
// on SMs or on the copy engine, resource partitioning, NVSwitch swizzle).
//
// SM mode: one cooperative persistent launch.  CTAs [0, P) are producers:
// their copy workers (one thread per warp, 1-D TMA bulk copies through a
// shared-memory ring) pull shard tiles from the peer regions into the
// gathered buffer, one signal group at a time, in source order
// (rank+1, rank+2, ..., rank) -- one source at a time, the NVSwitch order the
// pages describe -- and publish each finished group with st.release of the
// call's epoch.  CTAs [P, grid) are the persistent tcgen05 GEMM; its loader
// waits on the groups of each A tile with a bounded ld.acquire spin, then
// fences the async proxy and issues TMA.  The local shard is read in place.
// CE mode: cudaMemcpyAsync per group on the side stream, each followed by a
// stream-ordered cuStreamWriteValue32 of the flag; the GEMM-only launch on
// the main stream waits on the flags.
// SERIAL mode: a copy-only launch (all SMs), then a GEMM-only launch that does
// not wait; the two are ordered by the stream.
#include "tdg_gemm.cuh"
#include "tdg_internal.h"

namespace tdg {

namespace ag {
constexpr int PW = 4;          // copy workers (warps) per producer CTA
constexpr int PSLOTS = 3;      // ring slots per worker
constexpr int PCHUNK = 16384;  // bytes per bulk copy
constexpr int OFF_PBAR = PW * PSLOTS * PCHUNK;
static_assert(OFF_PBAR + PW * PSLOTS * 8 <= gm::SMEM_BYTES - 1024, "producer smem");
} // namespace ag

struct AgParams {
    CUtensorMap tmA_g; // gathered A: M x K
    CUtensorMap tmA_l; // local shard in place: Ms x K
    CUtensorMap tmB;   // KN: {N, K} box {64, 64}; NK: {K, N} box {64, 256}
    CUtensorMap tmC;   // C: {N, M} box {64, 32}
    DevStatus *status;
    uint32_t epoch;
    uint64_t timeout_ns;      // bound of a cross-CTA signal wait
    uint64_t pipe_timeout_ns; // bound of an intra-CTA pipeline wait (longer)
    int k_blocks;
    int64_t M, K, N, Ms;
    int m_tiles, n_tiles;
    int swz; // m-tile offset of the rank swizzle
    int local_inplace, local_lo, local_hi;
    const uint32_t *flags;
    int wait_flags;
    int64_t sig_rows;
    // producer side
    int n_prod;
    const uint8_t *regions;
    uint64_t region_bytes;
    uint64_t a_off;
    uint8_t *gathered;
    int rank, W;
    int64_t unit_rows;
    int64_t units_per_shard;
    int64_t n_units;
    int signal;
    int local_last;
    uint32_t *flags_w;
    uint64_t skip_mask;
};

template <int BMN> struct AgPolicy {
    using Params = AgParams;
    static constexpr int B_MN = BMN;

    __device__ static int64_t num_items(const Params &p) { return (int64_t)p.m_tiles * p.n_tiles; }

    __device__ static void tile(const Params &p, int64_t item, TileInfo &t)
    {
        const int pm0 = (int)(item / p.n_tiles);
        t.pn = (int)(item % p.n_tiles);
        // the pages' swizzle: pid_m = (pid_m + rank * tiles_per_pe) % total
        const int pm = (pm0 + p.swz) % p.m_tiles;
        t.m0 = pm * gm::BM;
        t.n0 = t.pn * gm::BN;
        t.n_valid = (int)min((int64_t)gm::BN, p.N - t.n0);
        if (p.local_inplace && pm >= p.local_lo && pm < p.local_hi) {
            t.a_sel = 1;
            t.a_row = t.m0 - p.local_lo * gm::BM;
        } else {
            t.a_sel = 0;
            t.a_row = t.m0;
        }
        t.owner = 0;
        t.m_loc = pm;
    }

    __device__ static void before_a(const Params &p, const TileInfo &t, bool &gave_up)
    {
        if (t.a_sel == 1 || !p.wait_flags)
            return;
        const int64_t r0 = t.m0;
        const int64_t r1 = min(p.M, (int64_t)t.m0 + gm::BM) - 1;
        // wait(ptr, n): every signal group the tile's rows fall into
        for (int64_t g = r0 / p.sig_rows; g <= r1 / p.sig_rows && !gave_up; ++g) {
            if (!wait_flag(p.flags + g, p.epoch, p.timeout_ns)) {
                report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_AG_FLAG, (uint32_t)g, p.epoch);
                gave_up = true;
            }
        }
        // consume_token: the data read below goes through the async proxy
        fence_proxy_async_global();
    }

    __device__ static void load_a(const Params &p, const TileInfo &t, void *dst, uint64_t *bar, int kb)
    {
        tma_load_2d(dst, t.a_sel ? &p.tmA_l : &p.tmA_g, bar, kb * gm::BK, t.a_row);
    }

    __device__ static void load_b(const Params &p, const TileInfo &t, void *dst, uint64_t *bar, int kb)
    {
        if (BMN) {
            const int nch = (t.n_valid + 63) >> 6;
            for (int j = 0; j < nch; ++j)
                tma_load_2d(static_cast<uint8_t *>(dst) + j * 8192, &p.tmB, bar, t.n0 + 64 * j,
                            kb * gm::BK);
        } else {
            tma_load_2d(dst, &p.tmB, bar, kb * gm::BK, t.n0);
        }
    }

    __device__ static uint32_t b_bytes(const TileInfo &t)
    {
        return BMN ? (uint32_t)(((t.n_valid + 63) >> 6) * 8192) : (uint32_t)gm::B_BYTES;
    }

    __device__ static void store_chunk(const Params &p, const TileInfo &t, const void *buf, int ch, int q)
    {
        const int row = t.m0 + 32 * q;
        if (row < p.M)
            tma_store_2d(&p.tmC, buf, t.n0 + 64 * ch, row);
    }

    __device__ static void after_tile(const Params &, const TileInfo &, int, int) {}
};

// One copy worker: copy `bytes` from src to dst through its ring.  Returns
// false if a wait ran out of time (after draining its own loads in flight).
__device__ bool ring_copy(uint8_t *dst, const uint8_t *src, uint64_t bytes, uint8_t *ring,
                          uint64_t *bar, uint32_t &phases, uint64_t tmo)
{
    using namespace ag;
    const int64_t nch = (int64_t)((bytes + PCHUNK - 1) / PCHUNK);
    uint32_t pending = 0;
    auto csize = [&](int64_t i) -> uint32_t {
        const uint64_t off = (uint64_t)i * PCHUNK;
        return (uint32_t)min((uint64_t)PCHUNK, bytes - off);
    };
    for (int64_t i = 0; i < nch && i < PSLOTS; ++i) {
        mbar_arrive_expect_tx(&bar[i], csize(i));
        bulk_load(ring + i * PCHUNK, src + (uint64_t)i * PCHUNK, csize(i), &bar[i]);
        pending |= 1u << i;
    }
    for (int64_t i = 0; i < nch; ++i) {
        const int s = (int)(i % PSLOTS);
        if (!mbar_wait(&bar[s], (phases >> s) & 1u, tmo)) {
            for (int t = 0; t < PSLOTS; ++t)
                if ((pending >> t) & 1u) {
                    if (t != s && mbar_wait(&bar[t], (phases >> t) & 1u, tmo))
                        phases ^= 1u << t;
                }
            bulk_wait<0>();
            return false;
        }
        phases ^= 1u << s;
        pending &= ~(1u << s);
        bulk_store(dst + (uint64_t)i * PCHUNK, ring + s * PCHUNK, csize(i));
        bulk_commit();
        const int64_t j = i - 1 + PSLOTS;
        if (i >= 1 && j < nch) {
            bulk_wait_read<1>(); // the store of chunk i-1 has read its slot
            const int s2 = (int)(j % PSLOTS);
            mbar_arrive_expect_tx(&bar[s2], csize(j));
            bulk_load(ring + s2 * PCHUNK, src + (uint64_t)j * PCHUNK, csize(j), &bar[s2]);
            pending |= 1u << s2;
        }
    }
    return true;
}

// Producer CTA: PW copy workers (lane 0 of warps 0..PW-1).
__device__ void ag_producer(const AgParams &p, uint8_t *smem)
{
    using namespace ag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= PW || lane != 0)
        return;
    uint8_t *ring = smem + warp * PSLOTS * PCHUNK;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_PBAR) + warp * PSLOTS;
    for (int i = 0; i < PSLOTS; ++i)
        mbar_init(&bar[i], 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    uint32_t phases = 0;
    const int64_t worker = (int64_t)blockIdx.x * PW + warp;
    const int64_t nworkers = (int64_t)p.n_prod * PW;
    const uint64_t row_bytes = (uint64_t)p.K * 2;
    for (int64_t u = worker; u < p.n_units; u += nworkers) {
        const int seq = (int)(u / p.units_per_shard);
        const int64_t part = u % p.units_per_shard;
        const int shard = p.local_last ? (p.rank + 1 + seq) % p.W : (p.rank + seq) % p.W;
        const int64_t row0 = part * p.unit_rows;
        const int64_t rows = min(p.unit_rows, p.Ms - row0);
        const uint8_t *src = p.regions + (uint64_t)shard * p.region_bytes + p.a_off + (uint64_t)row0 * row_bytes;
        const int64_t grow = (int64_t)shard * p.Ms + row0;
        uint8_t *dst = p.gathered + (uint64_t)grow * row_bytes;
        if (!ring_copy(dst, src, (uint64_t)rows * row_bytes, ring, bar, phases, p.timeout_ns)) {
            report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_PIPE, (uint32_t)u, p.epoch);
            return;
        }
        bulk_wait<0>();             // the group's writes are complete ...
        fence_proxy_async_global(); // ... and ordered before the generic release
        if (p.signal) {
            const int64_t g = grow / p.sig_rows;
            if (!((p.skip_mask >> (g & 63)) & 1ull))
                st_release_gpu(p.flags_w + g, p.epoch); // notify
        }
    }
}

template <int BMN>
__global__ void __launch_bounds__(gm::NUM_THREADS, 1) ag_gemm_kernel(const __grid_constant__ AgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    if ((int)blockIdx.x < p.n_prod) {
        ag_producer(p, smem);
        return;
    }
    gemm_consumer<AgPolicy<BMN>>(p, smem, (int)blockIdx.x - p.n_prod, (int)gridDim.x - p.n_prod);
}

} // namespace tdg

using namespace tdg;
using namespace tdg_host;

namespace {

const void *ag_kernel_fn(int b_layout)
{
    return b_layout == TDG_B_KN ? reinterpret_cast<const void *>(&ag_gemm_kernel<1>)
                                : reinterpret_cast<const void *>(&ag_gemm_kernel<0>);
}

int launch_ag(const AgParams &p, int b_layout, int grid, bool coop, cudaStream_t s)
{
    const void *fn = ag_kernel_fn(b_layout);
    static bool smem_set[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    bool &done = smem_set[b_layout & 1][dev & 63];
    if (!done) {
        cudaError_t e = set_smem(fn, gm::SMEM_BYTES);
        if (e != cudaSuccess)
            return cuda_err(e, "ag set smem");
        done = true;
    }
    void *args[] = {const_cast<AgParams *>(&p)};
    return cuda_err(launch(fn, dim3(grid), dim3(gm::NUM_THREADS), gm::SMEM_BYTES, s, args, coop),
                    "ag launch");
}

} // namespace

extern "C" int tdg_ag_gemm(tdg_symm *h, const tdg_ag_gemm_args *a, void *stream, void *side_stream)
{
    if (!h || !a)
        return TDG_ERR_INVALID;
    const int W = a->world, rank = a->rank;
    if (W != h->world || rank < 0 || rank >= W || a->Ms < 0 || a->K < 0 || a->N < 0)
        return TDG_ERR_INVALID;
    if (a->mode != TDG_MODE_SM && a->mode != TDG_MODE_CE && a->mode != TDG_MODE_SERIAL &&
        a->mode != TDG_MODE_LL)
        return TDG_ERR_INVALID;
    if (a->b_layout != TDG_B_KN && a->b_layout != TDG_B_NK)
        return TDG_ERR_INVALID;
    const int64_t Ms = a->Ms, K = a->K, N = a->N, M = (int64_t)W * Ms;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0)
        return TDG_OK;
    if (!a->C || !a->B || !aligned16(a->C) || !aligned16(a->B) || !aligned16(a->a_off) ||
        !aligned16(a->g_off) || (K % 8) != 0 || (N % 8) != 0)
        return TDG_ERR_INVALID;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return TDG_ERR_INVALID;
    const uint64_t shard_bytes = (uint64_t)Ms * K * 2, gath_bytes = (uint64_t)M * K * 2;
    if (a->a_off + shard_bytes > h->region_bytes || a->g_off + gath_bytes > h->region_bytes)
        return TDG_ERR_NOMEM;
    if (a->g_off < a->a_off + shard_bytes && a->a_off < a->g_off + gath_bytes && K > 0)
        return TDG_ERR_INVALID; // the gathered buffer overlaps the shard
    if (K == 0)
        return cuda_err(cudaMemsetAsync(a->C, 0, (size_t)M * N * 2, s), "ag K==0");
    if (a->mode == TDG_MODE_LL)
        return TDG_ERR_UNSUPPORTED;

    const int BM = gm::BM;
    const bool inplace = (Ms % BM) == 0;
    int64_t sig_rows = a->signal_rows;
    if (sig_rows <= 0)
        sig_rows = (a->mode == TDG_MODE_CE) ? Ms : (inplace ? (Ms % 32 == 0 ? 32 : Ms) : Ms);
    if (sig_rows > Ms || (Ms % sig_rows) != 0)
        return TDG_ERR_INVALID;
    const int64_t n_groups = M / sig_rows;
    if ((size_t)n_groups > h->nsig)
        return TDG_ERR_NOMEM;

    uint8_t *region_r = static_cast<uint8_t *>(tdg_symm_region(h, rank));
    uint8_t *gathered = region_r + a->g_off;
    uint32_t *flags = tdg_symm_flags(h, rank);

    AgParams p;
    memset(&p, 0, sizeof p);
    bool ok = map_bf16_2d(&p.tmA_g, gathered, K, M, K * 2, 64, BM);
    ok = ok && map_bf16_2d(&p.tmA_l, region_r + a->a_off, K, Ms, K * 2, 64, BM);
    if (a->b_layout == TDG_B_KN)
        ok = ok && map_bf16_2d(&p.tmB, a->B, N, K, N * 2, 64, 64);
    else
        ok = ok && map_bf16_2d(&p.tmB, a->B, K, N, K * 2, 64, 256);
    ok = ok && map_bf16_2d(&p.tmC, a->C, N, M, N * 2, 64, 32);
    if (!ok)
        return TDG_ERR_CUDA;

    const uint32_t epoch = next_epoch(h);
    p.status = h->status;
    p.epoch = epoch;
    p.timeout_ns = timeout_or_default(a->timeout_ns);
    p.pipe_timeout_ns = pipe_timeout(p.timeout_ns);
    p.k_blocks = (int)((K + gm::BK - 1) / gm::BK);
    p.M = M;
    p.K = K;
    p.N = N;
    p.Ms = Ms;
    p.m_tiles = (int)((M + BM - 1) / BM);
    p.n_tiles = (int)((N + gm::BN - 1) / gm::BN);
    p.swz = a->swizzle ? (int)(((int64_t)rank * Ms / BM) % p.m_tiles) : 0;
    p.local_inplace = inplace ? 1 : 0;
    p.local_lo = inplace ? (int)(rank * Ms / BM) : 0;
    p.local_hi = inplace ? (int)((rank + 1) * Ms / BM) : 0;
    p.flags = flags;
    p.sig_rows = sig_rows;
    p.regions = h->base;
    p.region_bytes = h->region_bytes;
    p.a_off = a->a_off;
    p.gathered = gathered;
    p.rank = rank;
    p.W = W;
    p.local_last = inplace ? 1 : 0;
    p.flags_w = flags;
    p.skip_mask = a->test_skip_notify;

    const int sms = h->sm_count;
    if (a->mode == TDG_MODE_SM) {
        int nprod = a->producers > 0 ? a->producers : 16;
        if (nprod >= sms)
            return TDG_ERR_INVALID;
        p.n_prod = nprod;
        p.wait_flags = 1;
        p.signal = 1;
        p.unit_rows = sig_rows;
        p.units_per_shard = Ms / sig_rows;
        p.n_units = (int64_t)W * p.units_per_shard;
        return launch_ag(p, a->b_layout, sms, true, s);
    }
    if (a->mode == TDG_MODE_SERIAL) {
        // copy phase: every SM copies, fine-grained units, no signals
        AgParams c = p;
        c.n_prod = sms;
        c.signal = 0;
        c.wait_flags = 0;
        c.unit_rows = Ms >= 8 ? 8 : Ms;
        while (Ms % c.unit_rows)
            c.unit_rows--;
        c.units_per_shard = Ms / c.unit_rows;
        c.n_units = (int64_t)W * c.units_per_shard;
        c.local_last = 0;
        int rc = launch_ag(c, a->b_layout, sms, false, s);
        if (rc != TDG_OK)
            return rc;
        // GEMM phase: stream-ordered after the copy, no waits
        AgParams g = p;
        g.n_prod = 0;
        g.wait_flags = 0;
        g.n_units = 0;
        return launch_ag(g, a->b_layout, sms, false, s);
    }
    // CE mode
    cudaStream_t side = static_cast<cudaStream_t>(side_stream);
    if (!side || side == s)
        return TDG_ERR_INVALID;
    cudaEvent_t ev0, ev1;
    if (cudaEventCreateWithFlags(&ev0, cudaEventDisableTiming) != cudaSuccess)
        return TDG_ERR_CUDA;
    if (cudaEventCreateWithFlags(&ev1, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(ev0);
        return TDG_ERR_CUDA;
    }
    int rc = TDG_OK;
    cudaError_t e = cudaEventRecord(ev0, s);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(side, ev0, 0);
    if (e != cudaSuccess)
        rc = cuda_err(e, "ce events");
    const int64_t ups = Ms / sig_rows;
    for (int seq = 0; seq < W && rc == TDG_OK; ++seq) {
        const int shard = inplace ? (rank + 1 + seq) % W : (rank + seq) % W;
        for (int64_t part = 0; part < ups && rc == TDG_OK; ++part) {
            const int64_t row0 = part * sig_rows;
            const int64_t grow = (int64_t)shard * Ms + row0;
            const uint8_t *src = h->base + (size_t)shard * h->region_bytes + a->a_off + (size_t)row0 * K * 2;
            e = cudaMemcpyAsync(gathered + (size_t)grow * K * 2, src, (size_t)sig_rows * K * 2,
                                cudaMemcpyDeviceToDevice, side);
            if (e != cudaSuccess) {
                rc = cuda_err(e, "ce memcpy");
                break;
            }
            const int64_t g = grow / sig_rows;
            if (!((a->test_skip_notify >> (g & 63)) & 1ull) && !stream_write_u32(side, flags + g, epoch))
                rc = TDG_ERR_UNSUPPORTED;
        }
    }
    if (rc == TDG_OK) {
        AgParams g = p;
        g.n_prod = 0;
        g.wait_flags = 1;
        g.n_units = 0;
        rc = launch_ag(g, a->b_layout, sms, false, s);
    }
    // the call completes on the main stream only when the side stream has too
    e = cudaEventRecord(ev1, side);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(s, ev1, 0);
    if (e != cudaSuccess && rc == TDG_OK)
        rc = cuda_err(e, "ce join");
    cudaEventDestroy(ev0);
    cudaEventDestroy(ev1);
    return rc;
}
