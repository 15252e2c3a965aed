// tdg_rs.cu -- tile-centric overlapped GEMM + ReduceScatter ("Triton-distributed
// 语义", 内核设计模式 "GEMM + ReduceScatter 重叠"; paper summary, 方法: push-mode
// intra-node ReduceScatter, the reduction running in parallel and synchronised
// by signals).
//
// One persistent tcgen05 GEMM runs every rank's partial product.  Work items
// are (owner block, rank r, owner o in the block, m tile inside o, n tile):
// all ranks' items of one block run back to back, so each B_r is streamed
// once per block (by default one block of all owners: once per call), and
// with smaller blocks every output tile gathers its W partials closer
// together in time.  The epilogue pushes each partial tile (bf16,
// or fp32 when asked; tile-contiguous, 128 x 256) into owner o's staging area
// (region o) with TMA, waits for the write to complete, fences the async
// proxy, and increments the owner's per-(tile, row-quarter) arrival counter
// with acq_rel semantics (Triton-distributed's "increment" signal; the counter word is
// tagged with the call's epoch).  The epilogue warp whose increment completes
// the count of W acquires the other W-1 pushes and owes the reduction of its
// 32 rows: summing the W partials in fixed rank order (fp32, 16-byte
// coalesced loads) and writing the bf16 rows of out_o, all at once or a few
// rows after each of its next tiles.  No CTA ever spins on another: the last
// arriver does the work.
// SERIAL mode: the GEMM stores every partial, then a separate reduction
// launch (all SMs) sums them -- same arithmetic, no overlap.
#include "tdg_gemm.cuh"
#include "tdg_internal.h"

namespace tdg {

struct RsParams {
    CUtensorMap tmA; // {K, M, W}, plane stride = region bytes, box {64, 128, 1}
    CUtensorMap tmB; // KN: {N, K, W} box {64, 64, 1}; NK: {K, N, W} box {64, 256, 1}
    CUtensorMap tmS; // staging {256, rows per owner, W}: bf16 box {64, 32, 1}, fp32 box {32, 32, 1}
    DevStatus *status;
    uint32_t epoch;
    uint64_t timeout_ns;      // bound of a cross-CTA signal wait
    uint64_t pipe_timeout_ns; // bound of an intra-CTA pipeline wait (longer)
    int k_blocks;
    int W;
    int64_t M, K, N, Mo;
    int mt;      // 128-row tiles per owner (Mo / 128): the staging layout
    int mtp;     // scheduled tiles per owner (Mo / (128 * cl))
    int pair;    // 1: CTA pairs (cta_group::2)
    int cl;      // CTAs per cluster (1, 2 or 4): tiles of 128 * cl rows
    int n_tiles;
    int order;   // 0: owner blocks of `ob` owners, then rank, owner, m, n; 1: rank fastest
    int ob;      // owners per block in order 0 (1 = owner by owner, W = rank-major)
    int fused_reduce;
    uint8_t *regions;
    uint64_t region_bytes;
    uint64_t stage_off, out_off;
    uint32_t *counters;
    uint64_t nsig;
    int f32; // 1: partials are pushed as fp32, 0: as bf16
    int red_rows; // rows of owed reductions an epilogue warp works off per tile
    int stages;   // GEMM ring stages in use
    int full_n;   // N is a multiple of BN: every tile is full width
    int edge_n;   // 0: the narrow-last-column fast path is not used here
    int64_t item_lo, item_hi; // this launch's items (item_hi < 0: all)
    int evict_partials; // bf16 partials pushed with an L2 evict-first policy
    int dep;      // 1: a second launch on the spare SMs follows this one;
                  // 2: this is that launch (it ends after the first)
};

__device__ __forceinline__ uint8_t *rs_stage_row(const RsParams &p, int o, int r, int m_loc, int pn, int row)
{
    const uint64_t idx = ((uint64_t)r * p.mt + m_loc) * p.n_tiles + pn;
    return p.regions + (uint64_t)o * p.region_bytes + p.stage_off + ((idx * 128 + row) << (p.f32 ? 10 : 9));
}

// Sum the W partial rows [row0, row1) of tile (o, m_loc, pn) in rank order
// (row1 - row0 a multiple of 4) and write the bf16 result into out_o.  One
// warp; lane l owns columns
// [8l, 8l + 8) of the tile, which are one 16-byte unit of each bf16 partial
// row or two units of each fp32 one (p.f32); the units are loaded one after
// the other, so both forms keep the same 4 rows x 8 ranks in flight.  Each
// partial is read here once, after the counter's acquire: bf16 partials with
// streaming loads (evict-first), so that they do not push the GEMM's operands
// out of L2 (+0.8 % at the Qwen-32B down-projection shape); fp32 partials,
// reduced a few rows per tile from L2-warm blocks, with L2-only loads (the
// streaming form measured 20 % slower there).
__device__ void rs_reduce_rows(const RsParams &p, int o, int m_loc, int pn, int n_valid, int row0, int row1,
                               int lane)
{
    const int col = lane * 8;
    if (col >= n_valid)
        return;
    uint8_t *out_base = p.regions + (uint64_t)o * p.region_bytes + p.out_off;
    const int64_t n0 = (int64_t)pn * gm::BN;
    const bool f32 = p.f32 != 0;
    const int units = f32 ? 2 : 1;
    const int lane_off = col * (f32 ? 4 : 2);
    constexpr int RR = 4; // rows in flight per lane: RR x 8 ranks x 16 B
    for (int rr = row0; rr < row1; rr += RR) {
        float acc[RR][8];
#pragma unroll
        for (int a = 0; a < RR; ++a)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                acc[a][j] = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (u >= units)
                break;
            for (int r0 = 0; r0 < p.W; r0 += 8) {
                uint4 v[RR][8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (r0 + j < p.W) {
#pragma unroll
                        for (int a = 0; a < RR; ++a) {
                            const uint4 *src = reinterpret_cast<const uint4 *>(
                                rs_stage_row(p, o, r0 + j, m_loc, pn, rr + a) + lane_off + 16 * u);
                            v[a][j] = f32 ? __ldcg(src) : __ldcs(src);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (r0 + j < p.W) {
#pragma unroll
                        for (int a = 0; a < RR; ++a) {
                            if (f32) {
                                const float *f = reinterpret_cast<const float *>(&v[a][j]);
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    acc[a][4 * u + e] += f[e];
                            } else {
                                const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v[a][j]);
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f = __bfloat1622float2(h[e]);
                                    acc[a][2 * e] += f.x;
                                    acc[a][2 * e + 1] += f.y;
                                }
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int a = 0; a < RR; ++a) {
            const int64_t orow = (int64_t)m_loc * gm::BM + rr + a;
            uint4 w;
            w.x = pack_bf16x2(acc[a][0], acc[a][1]);
            w.y = pack_bf16x2(acc[a][2], acc[a][3]);
            w.z = pack_bf16x2(acc[a][4], acc[a][5]);
            w.w = pack_bf16x2(acc[a][6], acc[a][7]);
            __stcs(reinterpret_cast<uint4 *>(out_base + ((uint64_t)orow * p.N + n0 + col) * 2), w); // not read here again
        }
    }
}

// The push signal of a tile quarter: increment its arrival counter and return
// the count before this push.  The word holds the call's epoch in bits 31..7
// (its low 25 bits) and the count in bits 6..0 (W <= 64), so a word left by
// an earlier call -- one that ended early on a fault, say -- counts as 0
// instead of corrupting this call.  A CAS that keeps losing (it cannot: each
// loss is another push landing) is bounded and reported.
__device__ __forceinline__ uint32_t rs_arrive(const RsParams &p, uint32_t *ctr)
{
    const uint32_t tag = (p.epoch & 0x01FFFFFFu) << 7;
    uint32_t v = *reinterpret_cast<volatile uint32_t *>(ctr);
    for (int i = 0; i < 4096; ++i) {
        const bool same = (v & ~0x7Fu) == tag;
        const uint32_t seen = atom_cas_acq_rel_gpu(ctr, v, same ? v + 1 : (tag | 1u));
        if (seen == v)
            return same ? (v & 0x7Fu) : 0u;
        v = seen;
    }
    report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_RS_SIGNAL, 0, p.epoch);
    return 0xFFFFFFFFu; // never the last arriver
}

template <int BMN> struct RsPolicy {
    using Params = RsParams;
    static constexpr int B_MN = BMN;

    __device__ static int64_t num_items(const Params &p)
    {
        return (int64_t)p.W * p.W * p.mtp * p.n_tiles;
    }

    __device__ static void tile(const Params &p, int64_t item, TileInfo &t, int sub)
    {
        const int64_t per_rank = (int64_t)p.mtp * p.n_tiles;
        int o, r;
        int64_t rem, x;
        if (p.order == 1) {
            const int64_t rest = divmod(item, p.W, x);
            r = (int)x;
            o = (int)divmod(rest, per_rank, rem);
        } else {
            // blocks of ob owners; inside a block every rank's tiles run back
            // to back, so B_r is streamed once per block and every output tile
            // of the block gathers its W partials within the block
            const int64_t per_block = (int64_t)p.W * p.ob * per_rank;
            const int blk = (int)divmod(item, per_block, x);
            r = (int)divmod(x, (int64_t)p.ob * per_rank, x);
            o = blk * p.ob + (int)divmod(x, per_rank, rem);
        }
        t.owner = o;
        t.a_sel = r;
        int64_t pn;
        t.m_loc = (int)divmod(rem, p.n_tiles, pn) * p.cl + sub; // 128-row tile in the owner
        t.pn = (int)pn;
        t.m0 = (o * p.mt + t.m_loc) * gm::BM;
        t.a_row = t.m0;
        t.n0 = t.pn * gm::BN;
        t.n_valid = (int)min((int64_t)gm::BN, p.N - t.n0);
        const int q = p.pair ? 32 : 16;
        t.n_mma = (t.n_valid + q - 1) / q * q;
    }

    __device__ static void before_a(const Params &, const TileInfo &, bool &) {}

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
        load<CL>(dst, &p.tmA, bar, kb * gm::BK, t.a_row, t.a_sel);
    }

    // B slices of 64 columns (8 KB): MN-major boxes {64 cols, 64 K}; K-major
    // boxes {64 K, 64 rows} with CL = 4, else one box of all the columns.
    // With CL = 4 pair `pidx` fetches slices pidx, pidx + 2, ... and
    // multicasts each to CTA `half` of both pairs.
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
                    tma_load_3d_pair_mc(d + j * 8192, &p.tmB, bar, col0 + 64 * j, kb * gm::BK, t.a_sel, mask);
                else
                    tma_load_3d_pair_mc(d + j * 8192, &p.tmB, bar, kb * gm::BK, col0 + 64 * j, t.a_sel, mask);
            }
        } else if (BMN) {
            const int nch = (cols + 63) >> 6;
            for (int j = 0; j < nch; ++j)
                load<CL>(d + j * 8192, &p.tmB, bar, col0 + 64 * j, kb * gm::BK, t.a_sel);
        } else {
            load<CL>(dst, &p.tmB, bar, kb * gm::BK, col0, t.a_sel);
        }
    }

    __device__ static uint32_t b_bytes(const Params &p, const TileInfo &, int cols)
    {
        return BMN ? (uint32_t)(((cols + 63) >> 6) * 8192) : (uint32_t)((p.pair ? gm::BN / 2 : gm::BN) * gm::BK * 2);
    }

    // push: the partial tile goes to the owner's staging area, as bf16 chunks
    // of 64 columns or (F32_OUT, when p.f32) fp32 chunks of 32 columns
    static constexpr bool F32_OUT = true;
    __device__ static bool out_f32(const Params &p) { return p.f32 != 0; }

    __device__ static void store_chunk(const Params &p, const TileInfo &t, const void *buf, int ch, int q)
    {
        const uint64_t idx = ((uint64_t)t.a_sel * p.mt + t.m_loc) * p.n_tiles + t.pn;
        if (p.evict_partials)
            tma_store_3d_evict_first(&p.tmS, buf, 64 * ch, (int)(idx * 128 + 32 * q), t.owner);
        else
            tma_store_3d(&p.tmS, buf, 64 * ch, (int)(idx * 128 + 32 * q), t.owner);
    }

    __device__ static void store_chunk_f32(const Params &p, const TileInfo &t, const void *buf, int sub, int q)
    {
        const uint64_t idx = ((uint64_t)t.a_sel * p.mt + t.m_loc) * p.n_tiles + t.pn;
        tma_store_3d(&p.tmS, buf, 32 * sub, (int)(idx * 128 + 32 * q), t.owner);
    }

    // The reductions an epilogue warp owes, oldest first: rows [row0, 32) of
    // its quarter of tile (o0, m0, pn0), then all of tiles 1 and 2.  At most
    // three wait; a fourth finishes the oldest at once.  (With fp32 partials
    // in blocks of 2 owners a block's last-rank pass can leave a warp three
    // quarters to work off; finishing one of them at once stalled the next
    // accumulator drain and made the call bimodal, 1440-1538 TFLOP/s at the
    // Qwen-32B down-projection shape against a steady 1553-1562 now.)
    struct EpiState {
        int n;
        int o0, m0, pn0, nv0, row0;
        int o1, m1, pn1, nv1;
        int o2, m2, pn2, nv2;
        int o3, m3, pn3, nv3;
    };

    // After each tile: signal the push (increment the tile quarter's arrival
    // counter); the warp whose increment completes the count of W owes the
    // reduction of that quarter.  Each warp then works off at most red_rows
    // rows of what it owes, so that no single tile's drain waits behind a
    // whole 32-row reduction; the tail pass after the last tile finishes all.
    __device__ static void after_tile(const Params &p, const TileInfo &t, int q, int lane, EpiState &st,
                                      bool tail)
    {
        if (!p.fused_reduce)
            return;
        int budget = tail ? 128 : p.red_rows;
        if (!tail) {
            uint32_t *ctr = p.counters + (uint64_t)t.owner * p.nsig +
                            ((uint64_t)t.m_loc * p.n_tiles + t.pn) * 4 + q;
            uint32_t old = 0;
            if (lane == 0) {
                bulk_wait<0>();             // this warp's pushed rows are written ...
                fence_proxy_async_global(); // ... and ordered before the signal
                old = rs_arrive(p, ctr);
            }
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == (uint32_t)(p.W - 1)) {
                __threadfence();
                if (st.n == 0) {
                    st.o0 = t.owner, st.m0 = t.m_loc, st.pn0 = t.pn, st.nv0 = t.n_valid, st.row0 = 0;
                } else if (st.n == 1) {
                    st.o1 = t.owner, st.m1 = t.m_loc, st.pn1 = t.pn, st.nv1 = t.n_valid;
                } else if (st.n == 2) {
                    st.o2 = t.owner, st.m2 = t.m_loc, st.pn2 = t.pn, st.nv2 = t.n_valid;
                } else {
                    st.o3 = t.owner, st.m3 = t.m_loc, st.pn3 = t.pn, st.nv3 = t.n_valid;
                    budget += 32 - st.row0; // the oldest is finished now
                }
                ++st.n;
            }
        }
        while (st.n > 0 && budget > 0) {
            const int rows = min(budget, 32 - st.row0);
            rs_reduce_rows(p, st.o0, st.m0, st.pn0, st.nv0, 32 * q + st.row0, 32 * q + st.row0 + rows, lane);
            st.row0 += rows;
            budget -= rows;
            if (st.row0 == 32) {
                __syncwarp();
                if (lane == 0) // tidy; any value from an earlier call counts as 0
                    st_relaxed_gpu(p.counters + (uint64_t)st.o0 * p.nsig +
                                       ((uint64_t)st.m0 * p.n_tiles + st.pn0) * 4 + q,
                                   0u);
                st.o0 = st.o1, st.m0 = st.m1, st.pn0 = st.pn1, st.nv0 = st.nv1, st.row0 = 0;
                st.o1 = st.o2, st.m1 = st.m2, st.pn1 = st.pn2, st.nv1 = st.nv2;
                st.o2 = st.o3, st.m2 = st.m3, st.pn2 = st.pn3, st.nv2 = st.nv3;
                --st.n;
            }
        }
    }
};

template <int BMN, int CL>
__global__ void __launch_bounds__(gm::NUM_THREADS, 1) rs_gemm_kernel(const __grid_constant__ RsParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    if (p.dep == 1)
        griddep_launch_dependents(); // every CTA is resident: the spare-SM launch may start
    gemm_consumer<RsPolicy<BMN>, CL>(p, smem, (int)blockIdx.x / CL, (int)gridDim.x / CL, p.item_lo, p.item_hi);
    if (p.dep == 2)
        griddep_wait(); // what follows in the stream then also follows the first launch
}

// SERIAL reduction: one 4-warp CTA per output tile.
__global__ void __launch_bounds__(128) rs_reduce_kernel(const __grid_constant__ RsParams p)
{
    const int64_t tile = blockIdx.x;
    const int per_owner = p.mt * p.n_tiles;
    const int o = (int)(tile / per_owner);
    const int rem = (int)(tile % per_owner);
    const int m_loc = rem / p.n_tiles, pn = rem % p.n_tiles;
    const int n_valid = (int)min((int64_t)gm::BN, p.N - (int64_t)pn * gm::BN);
    const int row0 = 32 * (int)(threadIdx.x >> 5);
    rs_reduce_rows(p, o, m_loc, pn, n_valid, row0, row0 + 32, threadIdx.x & 31);
}

} // namespace tdg

using namespace tdg;
using namespace tdg_host;

extern "C" size_t tdg_gemm_rs_stage_bytes(int world, int64_t M, int64_t N)
{
    if (world <= 0 || M <= 0 || N <= 0 || M % world)
        return 0;
    const int64_t Mo = M / world;
    const int64_t mt = (Mo + gm::BM - 1) / gm::BM;
    const int64_t nt = (N + gm::BN - 1) / gm::BN;
    return (size_t)world * mt * nt * gm::BM * gm::BN * 2;
}

extern "C" int tdg_gemm_rs(tdg_symm *h, const tdg_gemm_rs_args *a, void *stream)
{
    if (!h || !a)
        return TDG_ERR_INVALID;
    if (const int drc = check_device(h))
        return drc;
    const int W = a->world;
    if (W != h->world || a->M < 0 || a->K < 0 || a->N < 0)
        return TDG_ERR_INVALID;
    if (a->mode != TDG_MODE_SM && a->mode != TDG_MODE_SERIAL)
        return TDG_ERR_INVALID;
    if (a->b_layout != TDG_B_KN && a->b_layout != TDG_B_NK)
        return TDG_ERR_INVALID;
    if (a->partial_f32 != 0 && a->partial_f32 != 1)
        return TDG_ERR_INVALID;
    const int f32 = a->partial_f32;
    const int64_t M = a->M, K = a->K, N = a->N;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 0 || N == 0)
        return TDG_OK;
    if (M % W)
        return TDG_ERR_INVALID;
    const int64_t Mo = M / W;
    if (Mo % gm::BM || K % 8 || N % 8 || !aligned16(a->a_off) || !aligned16(a->b_off) ||
        !aligned16(a->stage_off) || !aligned16(a->out_off) || M > INT32_MAX || K > INT32_MAX ||
        N > INT32_MAX)
        return TDG_ERR_INVALID;
    const size_t stage_bytes = tdg_gemm_rs_stage_bytes(W, M, N) * (f32 ? 2 : 1);
    const uint64_t R = h->region_bytes;
    const uint64_t a_end = a->a_off + (uint64_t)M * K * 2, b_end = a->b_off + (uint64_t)K * N * 2;
    const uint64_t s_end = a->stage_off + stage_bytes, o_end = a->out_off + (uint64_t)Mo * N * 2;
    if (a_end > R || b_end > R || s_end > R || o_end > R)
        return TDG_ERR_NOMEM;
    // the buffers written (staging, out) overlap nothing else
    auto meet = [](uint64_t x0, uint64_t x1, uint64_t y0, uint64_t y1) { return x0 < y1 && y0 < x1; };
    if (meet(a->stage_off, s_end, a->a_off, a_end) || meet(a->stage_off, s_end, a->b_off, b_end) ||
        meet(a->stage_off, s_end, a->out_off, o_end) || meet(a->out_off, o_end, a->a_off, a_end) ||
        meet(a->out_off, o_end, a->b_off, b_end))
        return TDG_ERR_INVALID;
    const int mt = (int)(Mo / gm::BM);
    const int n_tiles = (int)((N + gm::BN - 1) / gm::BN);
    if ((size_t)mt * n_tiles * 4 > h->nsig)
        return TDG_ERR_NOMEM;
    if (K == 0) {
        for (int o = 0; o < W; ++o) {
            cudaError_t e = cudaMemsetAsync(h->base + (size_t)o * R + a->out_off, 0, (size_t)Mo * N * 2, s);
            if (e != cudaSuccess)
                return cuda_err(e, "rs K==0");
        }
        return TDG_OK;
    }

    // CTA pairs when every owner holds whole 256-row tiles; two pairs sharing
    // B when it holds whole 512-row tiles
    const int cl = pick_cluster(a->cluster, Mo % (2 * gm::BM) == 0, Mo % (4 * gm::BM) == 0);
    const int stages = cl ? pick_stages(a->stages, cl) : 0;
    if (!cl || !stages || (a->order & ~1) ||
        (a->red_rows != 0 && (a->red_rows < 4 || a->red_rows > 32 || 32 % a->red_rows)) ||
        a->spare < 0 || a->spare >= W * W)
        return TDG_ERR_INVALID;
    const int pair = cl >= 2 ? 1 : 0;
    RsParams p;
    memset(&p, 0, sizeof p);
    bool ok = map_bf16_3d(&p.tmA, h->base + a->a_off, K, M, W, K * 2, R, 64, gm::BM, 1);
    if (a->b_layout == TDG_B_KN)
        ok = ok && map_bf16_3d(&p.tmB, h->base + a->b_off, N, K, W, N * 2, R, 64, 64, 1);
    else
        ok = ok && map_bf16_3d(&p.tmB, h->base + a->b_off, K, N, W, K * 2, R, 64,
                               cl == 4 ? 64 : (pair ? 128 : 256), 1);
    const uint64_t rows_per_owner = (uint64_t)W * mt * n_tiles * gm::BM;
    if (f32)
        ok = ok && map_f32_3d(&p.tmS, h->base + a->stage_off, gm::BN, rows_per_owner, W, gm::BN * 4, R, 32, 32, 1);
    else
        ok = ok && map_bf16_3d(&p.tmS, h->base + a->stage_off, gm::BN, rows_per_owner, W, gm::BN * 2, R, 64, 32, 1);
    if (!ok)
        return TDG_ERR_CUDA;
    p.status = h->status;
    p.epoch = next_epoch(h);
    p.timeout_ns = timeout_or_default(a->timeout_ns);
    p.pipe_timeout_ns = pipe_timeout(p.timeout_ns);
    p.k_blocks = (int)((K + gm::BK - 1) / gm::BK);
    p.W = W;
    p.M = M;
    p.K = K;
    p.N = N;
    p.Mo = Mo;
    p.mt = mt;
    p.pair = pair;
    p.cl = cl;
    p.mtp = mt / cl;
    p.n_tiles = n_tiles;
    p.order = a->order;
    p.stages = stages;
    p.full_n = (N % gm::BN) == 0 ? 1 : 0;
    // Default block, measured at the Qwen-32B down-projection shape: with bf16
    // partials all owners in one block (each B_r streamed once; 1.7-2.9 %
    // over blocks of 2), with fp32 partials (twice the bytes to keep warm)
    // blocks of 2 owners (1 for odd W), whose reductions come every few
    // tiles instead of in one late stretch (+4 % over blocks of 4)
    if (a->owner_block < 0 || (a->owner_block > 0 && W % a->owner_block))
        return TDG_ERR_INVALID;
    const int ob_default = f32 ? (W % 2 ? 1 : 2) : W;
    p.ob = a->owner_block > 0 ? a->owner_block : ob_default;
    // with one block of all owners a partial is reduced only after every
    // rank's GEMM reached its tile, long after it left L2: let the pushes
    // go first (measured +0.45 % at the Qwen-32B down-projection shape)
    p.evict_partials = (p.ob == W && !f32 && a->order == 0) ? 1 : 0;
    p.fused_reduce = a->mode == TDG_MODE_SM ? 1 : 0;
    p.regions = h->base;
    p.region_bytes = R;
    p.stage_off = a->stage_off;
    p.out_off = a->out_off;
    p.counters = h->counters;
    p.nsig = h->nsig;
    p.f32 = f32;
    // measured at the Qwen-32B down-projection shape: a bf16 quarter's
    // reduction fits in the slack of one tile, so it is done at once; an fp32
    // one (twice the bytes) goes fastest in slices of 4 rows per tile with
    // blocks of 2 owners (1530-1550 TFLOP/s against 1080 at once and
    // 1470 for blocks of 4 in slices of 8; the serial twin 1495-1500)
    p.red_rows = a->red_rows ? a->red_rows : (f32 ? 4 : 32);

    const void *fn;
    if (a->b_layout == TDG_B_KN)
        fn = cl == 4   ? reinterpret_cast<const void *>(&rs_gemm_kernel<1, 4>)
             : cl == 2 ? reinterpret_cast<const void *>(&rs_gemm_kernel<1, 2>)
                       : reinterpret_cast<const void *>(&rs_gemm_kernel<1, 1>);
    else
        fn = cl == 4   ? reinterpret_cast<const void *>(&rs_gemm_kernel<0, 4>)
             : cl == 2 ? reinterpret_cast<const void *>(&rs_gemm_kernel<0, 2>)
                       : reinterpret_cast<const void *>(&rs_gemm_kernel<0, 1>);
    if (cudaError_t e = set_smem(fn, gm::SMEM_BYTES); e != cudaSuccess)
        return cuda_err(e, "rs set smem");
    int grid = h->sm_count;
    if (cl > 1) {
        const int mc = max_clusters(fn, gm::NUM_THREADS, gm::SMEM_BYTES, cl);
        const int n = mc < h->sm_count / cl ? mc : h->sm_count / cl;
        if (n <= 0)
            return TDG_ERR_UNSUPPORTED;
        grid = cl * n;
    }
    // no more clusters than work items (a small problem launches few CTAs)
    const int64_t items = (int64_t)W * W * p.mtp * n_tiles;
    if (grid / cl > items)
        grid = (int)(cl * items);
    p.item_lo = 0;
    p.item_hi = -1;
    // The SMs that the 4-CTA clusters leave idle (152 - 144 on a GB300) take
    // a share of the tiles as CTA pairs.  The tile order of order 0 is a
    // sequence of (owner block, rank, owner) groups of Mo/512 x n_tiles
    // cluster tiles, each of which is twice as many pair tiles in the same
    // place of the pairs' order, so the pairs take the last groups and the
    // clusters the rest.  The pairs launch after the clusters (programmatic
    // serialisation: once every cluster CTA is resident, so they cannot take
    // a cluster's place) and end after them.
    // Measured at the Qwen-32B down-projection shape: as fast as the clusters
    // alone in short bursts, up to a few percent faster on some boxes; under
    // sustained load the GPU sits at its power cap and the extra SMs only
    // lower the clock, so it is off by default.
    const int spare_pairs = cl == 4 ? (h->sm_count - grid) / 2 : 0;
    const int groups = (spare_pairs > 0 && a->order == 0 && a->b_layout == TDG_B_KN) ? a->spare : 0;
    RsParams q = p;
    const void *fn2 = nullptr;
    if (groups > 0) {
        fn2 = reinterpret_cast<const void *>(&rs_gemm_kernel<1, 2>);
        if (cudaError_t e = set_smem(fn2, gm::SMEM_BYTES); e != cudaSuccess)
            return cuda_err(e, "rs set smem");
        const int64_t per_group = (int64_t)p.mtp * n_tiles; // cluster tiles
        p.item_hi = items - groups * per_group;
        p.dep = 1;
        q.cl = 2;
        q.pair = 1;
        q.mtp = mt / 2;
        q.item_lo = 2 * p.item_hi;
        q.item_hi = 2 * items;
        q.dep = 2;
    }
    // no more pairs than the pairs' tiles
    const int64_t pair_items = groups > 0 ? 2 * (items - p.item_hi) : 0;
    const int n_pairs = pair_items < spare_pairs ? (int)pair_items : spare_pairs;
    void *args[] = {&p};
    int rc = cuda_err(launch(fn, dim3(grid), dim3(gm::NUM_THREADS), gm::SMEM_BYTES, s, args, false, cl),
                      "rs gemm launch");
    if (rc == TDG_OK && fn2) {
        void *args2[] = {&q};
        rc = cuda_err(launch(fn2, dim3(2 * n_pairs), dim3(gm::NUM_THREADS), gm::SMEM_BYTES, s, args2, false,
                             2, true),
                      "rs spare launch");
    }
    if (rc != TDG_OK || a->mode == TDG_MODE_SM)
        return rc;
    const unsigned tiles = (unsigned)(W * mt * n_tiles);
    return cuda_err(launch(reinterpret_cast<const void *>(&rs_reduce_kernel), dim3(tiles), dim3(128), 0, s,
                           args, false),
                    "rs reduce launch");
}
