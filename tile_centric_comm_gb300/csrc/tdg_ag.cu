// tdg_ag.cu -- tile-centric overlapped AllGather + GEMM ("Triton-distributed
// 语义", 内核设计模式 "AllGather + GEMM 重叠"; paper summary, 方法: AllGather
// on SMs or on the copy engine, push or pull, resource partitioning, NVSwitch
// swizzle).
//
// SM mode: one cooperative persistent launch.  CTAs [0, P) are producers:
// each has a few copy workers (one thread per warp) that stream their signal
// groups of shard rows from the peer regions into the gathered buffer through
// a ring in shared memory (1-D TMA bulk copies, global -> shared -> global),
// keeping all but one ring slot loading at all times, across group
// boundaries.  A group's flag is released (st.release of the call's epoch)
// once its stores are complete, while the stores of later groups are still
// in flight.  Sources go one at a time (the NVSwitch order: rank+1, rank+2,
// ..., the local shard last) or all at once (round robin over sources).
// CTAs [P, grid) are the persistent tcgen05 GEMM; its loader waits on the
// groups of each A tile with a bounded ld.acquire spin, then fences the async
// proxy and issues TMA.  The local shard is read in place.  Once its copies
// are done, a producer cluster takes GEMM items from the end of the order.
// Push mode: the senders choose the order -- sender s reaches destination
// (s + j) mod W at step j -- so rank r receives rank-1, rank-2, ..., and the
// GEMM visits the m tiles in that order; pull: rank+1, rank+2, ...
// CE mode: cudaMemcpyAsync per group on the side stream, each followed by a
// stream-ordered cuStreamWriteValue32 of the flag, all queued before the
// GEMM-only launch on the main stream that waits on the flags.
// LL mode: one cooperative launch of sender CTAs (8-byte {payload, epoch}
// words into the rank's LL buffer), receiver CTAs (poll every word, unpack it
// into the gathered buffer, release the group's flag) and the GEMM, which
// waits on those flags as in SM mode.
// SERIAL mode: a copy-only launch (all SMs), then a GEMM-only launch that does
// not wait; the two are ordered by the stream.
// Tile order: Triton-distributed's rank swizzle over m tiles (mirrored in push
// mode); m-major while B fits in about half of L2, else groups of 8 m tiles
// with n outer inside a group.
#include "tdg_gemm.cuh"
#include "tdg_internal.h"

namespace tdg {

namespace ag {
// The producer's ring is the GEMM's operand ring (a producer CTA is not a
// GEMM CTA until its copies are done); its slot barriers sit after it, in
// the GEMM's epilogue staging area.
constexpr int PRING = gm::RING_BYTES;
constexpr int PMAX_SLOTS = 32;      // per worker (one phase bit each)
constexpr int PMAX_WARPS = 4;
constexpr int OFF_PBAR = PRING;
constexpr int LAG_DONE = 4;         // a group's flag waits until all but its 4 latest stores are complete
constexpr int PFIFO = 8;            // groups whose stores are issued but whose flag is not yet released
constexpr int DEF_WARPS = 2;
constexpr uint32_t DEF_CHUNK = 32768;
static_assert(OFF_PBAR + PMAX_WARPS * PMAX_SLOTS * 8 <= gm::SMEM_BYTES - 1024, "producer smem");
} // namespace ag

struct AgParams {
    CUtensorMap tmA_g; // gathered A: M x K
    CUtensorMap tmA_l; // local shard in place: Ms x K
    CUtensorMap tmB;   // KN: {N, K} box {64, 64}; NK: {K, N} box {64, 256}
    CUtensorMap tmC;   // C: bf16 {N, M} box {64, 32}, or fp32 {N, M} box {32, 32}
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
    int pair; // 1: CTA pairs (cta_group::2)
    int cl;   // CTAs per cluster (1, 2 or 4): tiles of 128 * cl rows
    int split; // tiles of the last, partial wave split in two 128-column halves
    int mesh;  // 1: producers take all sources at once (round robin over sources)
    int group_m; // m rows per raster group
    int64_t tail_lo; // SM mode: items [tail_lo, T) go to the producer clusters once their copies are done
    // LL mode: producer CTAs [0, n_send) send, [n_send, n_prod) receive
    int ll;
    int n_send;
    uint64_t *ll_buf; // M * K / 2 words in region(rank)
    int c_f32;        // 1: C is fp32
    int stages;       // GEMM ring stages in use
    int push;         // 1: sources in push order (rank-1, rank-2, ...)
    int mirror;       // 1: the m tiles in push order (push with the swizzle on)
    int t_end;        // the m tile of the local shard's last row (the mirror's start)
    int pw;           // copy workers per producer CTA
    uint32_t pchunk;  // bytes per bulk copy
    int pslots;       // ring slots per worker
    int full_n;       // N is a multiple of BN and no tile is split: every tile is full width
    int edge_n;       // m-major order, no split, N not a multiple of BN: the last column's MMA width
};

template <int BMN, bool F32 = false> struct AgPolicy {
    using Params = AgParams;
    static constexpr int B_MN = BMN;

    // With a persistent grid of U scheduling units (CTAs or clusters) and T tiles,
    // the last wave holds only T mod U tiles.  Optionally, when twice that still
    // fits in a wave, those `split` tiles are cut into two 128-column halves.
    __device__ static int64_t num_items(const Params &p) { return (int64_t)p.m_tiles * p.n_tiles + p.split; }

    // tiles are 128 * cl rows (one CTA, a CTA pair, or two pairs); `sub`
    // picks this CTA's 128-row slice
    __device__ static void tile(const Params &p, int64_t item, TileInfo &t, int sub)
    {
        const int tm = p.cl * gm::BM;
        const int64_t full = (int64_t)p.m_tiles * p.n_tiles - p.split;
        int64_t tid = item;
        int nhalf = -1; // -1: whole tile; 0 / 1: a half of a split tail tile
        if (item >= full) {
            tid = full + (item - full) / 2;
            nhalf = (int)((item - full) & 1);
        }
        int64_t r64;
        // Two rasters.  group_m == 0: m-major (all n tiles of one m row, then
        // the next row), so the tiles of a wave follow the shards in arrival
        // order and wait on as few signals as possible (B stays in L2).
        // group_m > 0: groups of group_m m rows, n outer inside a group, so a
        // wave reuses those rows of A and a few columns of B from L2 instead
        // of streaming all of B (chosen when B does not fit in L2).
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
        // (local shard first, then rank+1, rank+2, ...).  Push mode mirrors it,
        // pid_m = (t_end - pid_m) mod total: the local shard first, then
        // rank-1, rank-2, ..., the order in which the senders deliver.
        const int pm = p.mirror ? ((p.t_end - pm0) % p.m_tiles + p.m_tiles) % p.m_tiles
                              : (pm0 + p.swz) % p.m_tiles;
        t.m0 = pm * tm + sub * gm::BM;
        t.n0 = t.pn * gm::BN;
        t.n_valid = (int)min((int64_t)gm::BN, p.N - t.n0);
        if (nhalf >= 0) {
            t.n0 += nhalf * (gm::BN / 2);
            t.n_valid = (int)min((int64_t)gm::BN / 2, p.N - t.n0); // <= 0: null item
        }
        const int q = p.pair ? 32 : 16;
        t.n_mma = (t.n_valid + q - 1) / q * q;
        if (p.local_inplace && pm >= p.local_lo && pm < p.local_hi) {
            t.a_sel = 1;
            t.a_row = t.m0 - p.local_lo * tm;
        } else {
            t.a_sel = 0;
            t.a_row = t.m0;
        }
        t.owner = 0;
        t.m_loc = pm;
    }

    __device__ static void before_a(const Params &p, const TileInfo &t, bool &gave_up)
    {
        if (t.a_sel == 1 || !p.wait_flags || t.m0 >= p.M)
            return;
        const int64_t r0 = t.m0;
        const int64_t r1 = min(p.M, (int64_t)t.m0 + gm::BM) - 1;
        // wait(ptr, n): every signal group this CTA's rows fall into.  In LL
        // mode a receiver that gives up still releases its group, so the GEMM
        // waits twice as long and the receiver's report comes first.
        const uint64_t tmo = p.ll ? 2 * p.timeout_ns : p.timeout_ns;
        for (int64_t g = r0 / p.sig_rows; g <= r1 / p.sig_rows && !gave_up; ++g) {
            if (!wait_flag(p.flags + g, p.epoch, tmo)) {
                report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_AG_FLAG, (uint32_t)g, p.epoch);
                gave_up = true;
            }
        }
        // consume_token: the data read below goes through the async proxy
        fence_proxy_async_global();
    }

    // The TMA form is chosen at compile time: a kernel holds either only
    // cta_group::1 or only cta_group::2 instructions, never both.
    template <int CL>
    __device__ static void load(void *dst, const CUtensorMap *m, uint32_t bar, int x, int y)
    {
        if constexpr (CL >= 2)
            tma_load_2d_pair(dst, m, bar, x, y);
        else
            tma_load_2d_addr(dst, m, bar, x, y);
    }

    template <int CL>
    __device__ static void load_a(const Params &p, const TileInfo &t, void *dst, uint32_t bar, int kb)
    {
        load<CL>(dst, t.a_sel ? &p.tmA_l : &p.tmA_g, bar, kb * gm::BK, t.a_row);
    }

    // B slices of 64 columns (8 KB): MN-major boxes {64 cols, 64 K}; K-major
    // boxes {64 K, 64 rows} with CL = 4, else one box of all the columns
    template <int CL>
    __device__ static void load_b(const Params &p, const TileInfo &, void *dst, uint32_t bar, int kb,
                                  int col0, int cols, int pidx, int half)
    {
        uint8_t *d = static_cast<uint8_t *>(dst);
        if constexpr (CL == 4) {
            // B (K x N) stays in L2 for every m row of tiles and C leaves it
            // first (+0.8 % at the Qwen-32B up-projection with the copy
            // engine's traffic beside the GEMM)
            const uint16_t mask = (uint16_t)((1u << half) | (1u << (2 + half)));
            const int nch = BMN ? (cols + 63) >> 6 : 2;
            for (int j = pidx; j < nch; j += 2) {
                if (BMN)
                    tma_load_2d_pair_mc_evict_last(d + j * 8192, &p.tmB, bar, col0 + 64 * j, kb * gm::BK, mask);
                else
                    tma_load_2d_pair_mc(d + j * 8192, &p.tmB, bar, kb * gm::BK, col0 + 64 * j, mask);
            }
        } else if (BMN) {
            const int nch = (cols + 63) >> 6;
            for (int j = 0; j < nch; ++j)
                load<CL>(d + j * 8192, &p.tmB, bar, col0 + 64 * j, kb * gm::BK);
        } else {
            load<CL>(dst, &p.tmB, bar, kb * gm::BK, col0);
        }
    }

    __device__ static uint32_t b_bytes(const Params &p, const TileInfo &, int cols)
    {
        return BMN ? (uint32_t)(((cols + 63) >> 6) * 8192) : (uint32_t)((p.pair ? gm::BN / 2 : gm::BN) * gm::BK * 2);
    }

    // C is bf16 (RNE of the fp32 accumulator), or with F32 the accumulator
    // itself, stored as fp32 chunks of 32 columns
    static constexpr bool F32_OUT = F32;
    __device__ static bool out_f32(const Params &) { return true; }

    __device__ static void store_chunk(const Params &p, const TileInfo &t, const void *buf, int ch, int q)
    {
        const int row = t.m0 + 32 * q;
        if (row < p.M)
            tma_store_2d_evict_first(&p.tmC, buf, t.n0 + 64 * ch, row);
    }

    // (the second 32-column half of a 64-column chunk may start past N: skipped)
    __device__ static void store_chunk_f32(const Params &p, const TileInfo &t, const void *buf, int sub, int q)
    {
        const int row = t.m0 + 32 * q;
        const int col = t.n0 + 32 * sub;
        if (row < p.M && col < p.N)
            tma_store_2d(&p.tmC, buf, col, row);
    }

    struct EpiState {};
    __device__ static void after_tile(const Params &, const TileInfo &, int, int, EpiState &, bool) {}
};

// Unit u of the producers (one signal group of one shard): the source and
// destination rows.  Sources one at a time: every part of the first source,
// then the next; all at once: part 0 of every source, then part 1, ...  Pull
// visits rank+1, rank+2, ... (the local shard last when it is read in place,
// first otherwise); push visits rank-1, rank-2, ..., and the parts of a shard
// from its last rows to its first, the order in which the GEMM takes them.
struct CopyUnit {
    const uint8_t *src;
    uint8_t *dst;
    uint64_t bytes;
    int64_t g; // flag word of the group
};

__device__ CopyUnit copy_unit(const AgParams &p, int64_t u)
{
    const int seq = p.mesh ? (int)(u % p.W) : (int)(u / p.units_per_shard);
    int64_t part = p.mesh ? u / p.W : u % p.units_per_shard;
    int shard;
    if (p.push) {
        const int back = p.local_last ? 1 + seq : seq;
        shard = ((p.rank - back) % p.W + p.W) % p.W;
        part = p.units_per_shard - 1 - part;
    } else {
        shard = p.local_last ? (p.rank + 1 + seq) % p.W : (p.rank + seq) % p.W;
    }
    const uint64_t row_bytes = (uint64_t)p.K * 2;
    const int64_t row0 = part * p.unit_rows;
    const int64_t rows = min(p.unit_rows, p.Ms - row0);
    const int64_t grow = (int64_t)shard * p.Ms + row0;
    CopyUnit c;
    c.src = p.regions + (uint64_t)shard * p.region_bytes + p.a_off + (uint64_t)row0 * row_bytes;
    c.dst = p.gathered + (uint64_t)grow * row_bytes;
    c.bytes = (uint64_t)rows * row_bytes;
    c.g = grow / p.sig_rows;
    return c;
}

// notify: the group's stores are complete (the caller waited on their bulk
// groups); order them before the generic release of the flag
__device__ __forceinline__ void producer_notify(const AgParams &p, int64_t g)
{
    fence_proxy_async_global();
    if (p.signal && !((p.skip_mask >> (g & 63)) & 1ull))
        st_release_gpu(p.flags_w + g, p.epoch);
}

// One copy worker (one thread): it copies its units u = worker, worker +
// nworkers, ... chunk by chunk through a ring of S slots of `chunk` bytes
// (1-D TMA bulk copies global -> shared -> global).  Loads run S - 1 chunks
// ahead of the stores, across unit boundaries; a slot is refilled as soon as
// the store of its previous chunk has read it.  A unit's flag is released
// once all but the LAG_DONE latest stores are complete, so the pipeline never
// drains between units.  Returns false when a wait ran out of time (after
// waiting, bounded, for its own loads in flight).
__device__ bool copy_worker(const AgParams &p, int64_t worker, int64_t nworkers, uint8_t *ring,
                            uint64_t *bar, int S, uint32_t chunk)
{
    using namespace ag;
    if (worker >= p.n_units)
        return true;
    // load cursor (unit lu, byte lo) and store cursor (unit su, byte so)
    int64_t lu = worker, su = worker;
    uint64_t lo = 0, so = 0;
    CopyUnit lc = copy_unit(p, lu), sc = lc;
    uint32_t ql = 0, q = 0; // chunks loaded (issued) and stored so far
    uint32_t phases = 0, pending = 0;
    int64_t fg[PFIFO];
    uint32_t flast[PFIFO];
    int fh = 0, fn = 0;
    auto load_next = [&]() {
        if (lu >= p.n_units)
            return;
        const int s = (int)(ql % (uint32_t)S);
        const uint32_t b = (uint32_t)min((uint64_t)chunk, lc.bytes - lo);
        mbar_arrive_expect_tx(&bar[s], b);
        bulk_load(ring + (size_t)s * chunk, lc.src + lo, b, &bar[s]);
        pending |= 1u << s;
        ++ql;
        lo += b;
        if (lo >= lc.bytes) {
            lu += nworkers;
            lo = 0;
            if (lu < p.n_units)
                lc = copy_unit(p, lu);
        }
    };
    for (int i = 0; i < S - 1; ++i)
        load_next();
    while (q < ql) {
        const int s = (int)(q % (uint32_t)S);
        if (!mbar_wait(&bar[s], (phases >> s) & 1u, p.timeout_ns)) {
            report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_PIPE, (uint32_t)su, p.epoch);
            for (int t = 0; t < S; ++t) // every load in flight, this one included (bounded)
                if ((pending >> t) & 1u)
                    (void)mbar_wait(&bar[t], (phases >> t) & 1u, p.timeout_ns);
            bulk_wait<0>();
            return false;
        }
        phases ^= 1u << s;
        pending &= ~(1u << s);
        const uint32_t b = (uint32_t)min((uint64_t)chunk, sc.bytes - so);
        bulk_store(sc.dst + so, ring + (size_t)s * chunk, b);
        bulk_commit();
        so += b;
        if (so >= sc.bytes) { // the unit's last store is issued
            if (fn == PFIFO) { // (units of one chunk each): release the oldest at once
                bulk_wait<0>();
                while (fn > 0) {
                    producer_notify(p, fg[fh]);
                    fh = (fh + 1) % PFIFO;
                    --fn;
                }
            }
            fg[(fh + fn) % PFIFO] = sc.g;
            flast[(fh + fn) % PFIFO] = q;
            ++fn;
            su += nworkers;
            so = 0;
            if (su < p.n_units)
                sc = copy_unit(p, su);
        }
        ++q;
        // the slot to refill held the chunk before the one just stored: wait
        // until that store has read it (all but the latest store group)
        bulk_wait_read<1>();
        load_next();
        // stores 0 .. q-1 are issued; all but the LAG_DONE latest complete
        // means every unit whose last store is at most q-1-LAG_DONE is done
        if (fn > 0 && flast[fh] + LAG_DONE < q) {
            bulk_wait<LAG_DONE>();
            while (fn > 0 && flast[fh] + LAG_DONE < q) {
                producer_notify(p, fg[fh]);
                fh = (fh + 1) % PFIFO;
                --fn;
            }
        }
    }
    bulk_wait<0>();
    while (fn > 0) {
        producer_notify(p, fg[fh]);
        fh = (fh + 1) % PFIFO;
        --fn;
    }
    return true;
}

// Producer CTA: p.pw copy workers (lane 0 of warps 0 .. pw-1), each with
// p.pslots slots of p.pchunk bytes.
__device__ void ag_producer(const AgParams &p, uint8_t *smem)
{
    using namespace ag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= p.pw || lane != 0)
        return;
    const int S = p.pslots;
    uint8_t *ring = smem + (size_t)warp * S * p.pchunk;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_PBAR) + warp * PMAX_SLOTS;
    for (int i = 0; i < S; ++i)
        mbar_init(&bar[i], 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    const int64_t worker = (int64_t)blockIdx.x * p.pw + warp;
    const int64_t nworkers = (int64_t)p.n_prod * p.pw;
    (void)copy_worker(p, worker, nworkers, ring, bar, S, p.pchunk);
    // the ring's shared memory may serve another role next
    for (int i = 0; i < S; ++i)
        mbar_inval(&bar[i]);
}

// LL sender (paper summary, 方法: the low-latency protocol stores data and
// flag together in 8-byte blocks, so no separate signal follows a transfer).
// Each thread packs two bf16 of a shard (4 bytes) with the call's epoch into
// one word and writes it into rank `rank`'s LL buffer, at the word's position
// in the gathered matrix.  Sources in the same order as the bulk producers.
__device__ void ll_sender(const AgParams &p, int cta, int ncta)
{
    constexpr int LB = 8;               // words per thread per pass: independent loads in flight
    const int64_t wps = p.Ms * p.K / 2; // words per shard
    // in the all-sources order every source's words are visited in runs of 64
    // (the last run of a source padded), so the loop covers ceil(wps/64)*64*W
    const int64_t total = p.mesh ? (wps + 63) / 64 * 64 * p.W : wps * p.W;
    const uint64_t hi = (uint64_t)p.epoch << 32;
    for (int64_t w0 = ((int64_t)cta * blockDim.x + threadIdx.x) * LB; w0 < total;
         w0 += (int64_t)ncta * blockDim.x * LB) {
        int64_t gw[LB];
        uint32_t payload[LB];
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            const int64_t w = w0 + j;
            gw[j] = -1;
            if (w >= total)
                continue;
            // source order as for the bulk producers, in units of 64-word runs
            int seq;
            int64_t off;
            if (p.mesh) {
                const int64_t run = w / 64, in = w % 64;
                seq = (int)(run % p.W);
                off = (run / p.W) * 64 + in;
                if (off >= wps)
                    continue;
            } else {
                seq = (int)(w / wps);
                off = w % wps;
            }
            const int shard = p.push ? ((p.rank - 1 - seq) % p.W + p.W) % p.W : (p.rank + 1 + seq) % p.W;
            const int64_t word = (int64_t)shard * wps + off;
            const int64_t g = (word * 2 / p.K) / p.sig_rows;
            if ((p.skip_mask >> (g & 63)) & 1ull)
                continue;
            gw[j] = word;
            payload[j] = *reinterpret_cast<const uint32_t *>(
                p.regions + (uint64_t)shard * p.region_bytes + p.a_off + (uint64_t)off * 4);
        }
#pragma unroll
        for (int j = 0; j < LB; ++j)
            if (gw[j] >= 0)
                st_relaxed_gpu_u64(p.ll_buf + gw[j], hi | payload[j]);
    }
}

// LL receiver: spin (bounded) on every word of a signal group until its flag
// is this call's epoch, unpack the payload into the gathered buffer, then hand
// the group to the GEMM with one release of the group's flag.  Each thread
// loads LB consecutive words before it looks at any, so LB loads are in flight.
__device__ void ll_receiver(const AgParams &p, int cta, int ncta)
{
    constexpr int LB = 8;
    const int64_t wpg = p.sig_rows * p.K / 2; // words per group
    const int64_t n_groups = p.M / p.sig_rows;
    uint32_t *g32 = reinterpret_cast<uint32_t *>(p.gathered);
    bool gave_up = false;
    for (int64_t g = cta; g < n_groups; g += ncta) {
        for (int64_t i0 = (int64_t)threadIdx.x * LB; i0 < wpg; i0 += (int64_t)blockDim.x * LB) {
            const int64_t w0 = g * wpg + i0;
            const int n = (int)min((int64_t)LB, wpg - i0);
            uint64_t v[LB];
#pragma unroll
            for (int j = 0; j < LB; ++j)
                if (j < n)
                    v[j] = ld_relaxed_gpu_u64(p.ll_buf + w0 + j);
            // words not yet delivered are polled together: one round trip
            // per poll for the whole batch
            uint32_t pending = 0;
#pragma unroll
            for (int j = 0; j < LB; ++j)
                if (j < n && (uint32_t)(v[j] >> 32) != p.epoch)
                    pending |= 1u << j;
            if (pending && !gave_up) {
                const uint64_t t0 = globaltimer();
                for (int spin = 0; pending; ++spin) {
                    if (spin >= 16)
                        __nanosleep(64);
#pragma unroll
                    for (int j = 0; j < LB; ++j)
                        if ((pending >> j) & 1u)
                            v[j] = ld_relaxed_gpu_u64(p.ll_buf + w0 + j);
#pragma unroll
                    for (int j = 0; j < LB; ++j)
                        if (((pending >> j) & 1u) && (uint32_t)(v[j] >> 32) == p.epoch)
                            pending &= ~(1u << j);
                    if (pending && globaltimer() - t0 > p.timeout_ns) {
                        report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_LL, (uint32_t)g, p.epoch);
                        gave_up = true;
                        break;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < LB; ++j)
                if (j < n)
                    g32[w0 + j] = (uint32_t)v[j];
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            st_release_gpu(p.flags_w + g, p.epoch);
        }
    }
}

template <int BMN, int CL, bool F32>
__global__ void __launch_bounds__(gm::NUM_THREADS, 1) ag_gemm_kernel(const __grid_constant__ AgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const int64_t T = (int64_t)p.m_tiles * p.n_tiles + p.split;
    if ((int)blockIdx.x < p.n_prod) {
        // producer CTAs fill whole clusters; in SM mode, once a cluster's copies
        // are done, it takes the last items of the GEMM (whose shards arrive last)
        if (!p.ll) {
            ag_producer(p, smem);
            if (p.tail_lo < T) {
                __syncthreads(); // every copy worker of this CTA is done with the ring
                gemm_consumer<AgPolicy<BMN, F32>, CL>(p, smem, (int)blockIdx.x / CL, p.n_prod / CL, p.tail_lo, T);
            }
        } else if ((int)blockIdx.x < p.n_send) {
            ll_sender(p, blockIdx.x, p.n_send);
        } else {
            ll_receiver(p, blockIdx.x - p.n_send, p.n_prod - p.n_send);
        }
        return;
    }
    const int c = (int)blockIdx.x - p.n_prod, nc = (int)gridDim.x - p.n_prod;
    gemm_consumer<AgPolicy<BMN, F32>, CL>(p, smem, c / CL, nc / CL, 0, p.tail_lo < T ? p.tail_lo : T);
}

} // namespace tdg

using namespace tdg;
using namespace tdg_host;

namespace {

template <int BMN, bool F32> const void *ag_kernel_cl(int cl)
{
    return cl == 4   ? reinterpret_cast<const void *>(&ag_gemm_kernel<BMN, 4, F32>)
           : cl == 2 ? reinterpret_cast<const void *>(&ag_gemm_kernel<BMN, 2, F32>)
                     : reinterpret_cast<const void *>(&ag_gemm_kernel<BMN, 1, F32>);
}

const void *ag_kernel_fn(int b_layout, int cl, bool f32)
{
    if (b_layout == TDG_B_KN)
        return f32 ? ag_kernel_cl<1, true>(cl) : ag_kernel_cl<1, false>(cl);
    return f32 ? ag_kernel_cl<0, true>(cl) : ag_kernel_cl<0, false>(cl);
}

int prepare(const void *fn)
{
    const cudaError_t e = set_smem(fn, gm::SMEM_BYTES);
    return e == cudaSuccess ? TDG_OK : cuda_err(e, "ag set smem");
}

// grid for a launch with n_prod producer CTAs plus consumers on every other SM
int ag_grid(const AgParams &p, int b_layout, int sms)
{
    if (p.cl == 1)
        return sms;
    if (prepare(ag_kernel_fn(b_layout, p.cl, p.c_f32 != 0)) != TDG_OK)
        return 0;
    const int mc = max_clusters(ag_kernel_fn(b_layout, p.cl, p.c_f32 != 0), gm::NUM_THREADS, gm::SMEM_BYTES, p.cl);
    const int n = mc > 0 ? (mc < sms / p.cl ? mc : sms / p.cl) : 0;
    return p.cl * n;
}

// SM mode: once a producer cluster has copied its share of the shards it
// takes GEMM items from the end of the order (rows that arrive last).
// `req` > 0 gives them the last req items, -1 none; 0 balances the rounds of
// tiles: GEMM clusters run ceil(T_c / n_cc) rounds, producer clusters c
// rounds' worth of copying and then ceil((T - T_c) / n_pc) rounds, with c
// estimated from the bytes each producer CTA moves (PROD_BPS) against the
// time of one tile (TILE_FLOPS per SM).  Returns the first item of the
// producers' share.
//
// PROD_BPS: an SM writes to memory at most about 63 GB/s (TMA bulk stores and
// plain stores alike, measured on one GB300), so a global -> global copy runs
// at about 50 GB/s per producer CTA with the default ring; a GEMM CTA
// computes about 12 TFLOP/s.
constexpr double PROD_BPS = 48e9;
constexpr double TILE_FLOPS = 12e12;

// Default producer CTAs in SM mode: enough to copy the shards within the
// time of the GEMM on every SM (so that the copies stay ahead of the tiles
// that need them), in whole clusters, 4 .. 32; 32 when there is no GEMM
// (N == 0: the AllGather alone).
int default_producers(const AgParams &p, int grid, int TM)
{
    const int lo = (4 + p.cl - 1) / p.cl * p.cl, hi = 32 / p.cl * p.cl;
    const double tiles = (double)p.m_tiles * p.n_tiles;
    const double tile_s = 2.0 * TM * gm::BN * p.K / (p.cl * TILE_FLOPS);
    const double gemm_s = tiles * tile_s / ((double)grid / p.cl);
    if (!(gemm_s > 0.0))
        return hi;
    const double want = (double)p.W * p.Ms * p.K * 2.0 / (gemm_s * PROD_BPS);
    if (want >= hi)
        return hi;
    const int n = ((int)ceil(want) + p.cl - 1) / p.cl * p.cl;
    return n < lo ? lo : (n > hi ? hi : n);
}
int64_t producer_tail_lo(const AgParams &p, int grid, int TM, int req)
{
    const int64_t T = (int64_t)p.m_tiles * p.n_tiles;
    const int n_pc = p.n_prod / p.cl, n_cc = (grid - p.n_prod) / p.cl;
    if (n_pc <= 0 || n_cc <= 0 || req < 0)
        return T;
    if (req > 0)
        return req >= T ? 0 : T - req;
    const double copy_s = (double)p.W * p.Ms * p.K * 2.0 / p.n_prod / PROD_BPS;
    const double tile_s = 2.0 * TM * gm::BN * p.K / (p.cl * TILE_FLOPS);
    const int64_t c = (int64_t)ceil(copy_s / tile_s);
    int64_t best_t = 0, best_r = (T + n_cc - 1) / n_cc;
    for (int64_t t = 1; t <= T; ++t) {
        const int64_t rc = (T - t + n_cc - 1) / n_cc;
        const int64_t rp = c + (t + n_pc - 1) / n_pc;
        const int64_t r = rc > rp ? rc : rp;
        if (r < best_r) {
            best_r = r;
            best_t = t;
        }
    }
    return T - best_t;
}

int launch_ag(const AgParams &p, int b_layout, int grid, bool coop, cudaStream_t s, int split_tail = 0)
{
    const void *fn = ag_kernel_fn(b_layout, p.cl, p.c_f32 != 0);
    int rc = prepare(fn);
    if (rc != TDG_OK)
        return rc;
    if (grid < 1 || grid < p.n_prod) // a copy-only launch has no consumers
        return TDG_ERR_UNSUPPORTED;
    AgParams q = p;
    int64_t units = (grid - p.n_prod) / p.cl;
    const int64_t T = (int64_t)p.m_tiles * p.n_tiles;
    // no more GEMM clusters than tiles (a small problem launches few CTAs)
    if (units > T && units > 0) {
        units = T;
        grid = p.n_prod + (int)(p.cl * units);
    }
    q.split = 0;
    // opt-in (split_tail): measured slower at the Qwen-32B up-projection
    // shape, where the half-width tiles move more operand bytes per FLOP and the
    // tail tiles wait on the shard that arrives last anyway.  Not combined with
    // producer clusters that take the last items.
    if (split_tail && p.tail_lo >= T && units > 0 && T > units && (T % units) > 0 &&
        2 * (T % units) <= units)
        q.split = (int)(T % units);
    if (q.tail_lo >= T)
        q.tail_lo = T + q.split; // every item goes to the GEMM CTAs
    q.full_n = (p.N % gm::BN) == 0 && q.split == 0 ? 1 : 0;
    q.edge_n = 0;
    if (!q.full_n && q.split == 0 && q.group_m <= 0) {
        // m-major order (item = pm0 * n_tiles + pn): only the last column is narrow
        const int q16 = p.pair ? 32 : 16;
        const int nv = (int)(p.N - (int64_t)(p.n_tiles - 1) * gm::BN);
        q.edge_n = (nv + q16 - 1) / q16 * q16;
    }
    void *args[] = {&q};
    cudaError_t e = launch(fn, dim3(grid), dim3(gm::NUM_THREADS), gm::SMEM_BYTES, s, args, coop, p.cl);
    if (e != cudaSuccess && coop && p.cl > 1) {
        // co-residency then rests on the grid being no larger than the number
        // of clusters that fit at once (the bounded waits cover the rest)
        (void)cudaGetLastError();
        e = launch(fn, dim3(grid), dim3(gm::NUM_THREADS), gm::SMEM_BYTES, s, args, false, p.cl);
    }
    return cuda_err(e, "ag launch");
}

} // namespace

extern "C" int tdg_ag_gemm(tdg_symm *h, const tdg_ag_gemm_args *a, void *stream, void *side_stream)
{
    if (!h || !a)
        return TDG_ERR_INVALID;
    if (const int drc = check_device(h))
        return drc;
    const int W = a->world, rank = a->rank;
    if (W != h->world || rank < 0 || rank >= W || a->Ms < 0 || a->K < 0 || a->N < 0)
        return TDG_ERR_INVALID;
    if (a->mode != TDG_MODE_SM && a->mode != TDG_MODE_CE && a->mode != TDG_MODE_SERIAL &&
        a->mode != TDG_MODE_LL)
        return TDG_ERR_INVALID;
    if (a->b_layout != TDG_B_KN && a->b_layout != TDG_B_NK)
        return TDG_ERR_INVALID;
    if (a->c_f32 != 0 && a->c_f32 != 1)
        return TDG_ERR_INVALID;
    const int64_t Ms = a->Ms, K = a->K, N = a->N, M = (int64_t)W * Ms;
    const size_t c_elem = a->c_f32 ? 4 : 2;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 0)
        return TDG_OK;
    // N == 0: the AllGather alone (gathered buffer and flags), no GEMM
    const bool gemm = N > 0;
    if ((gemm && (!a->C || !a->B || !aligned16(a->C) || !aligned16(a->B))) || !aligned16(a->a_off) ||
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
        return gemm ? cuda_err(cudaMemsetAsync(a->C, 0, (size_t)M * N * c_elem, s), "ag K==0") : TDG_OK;
    const bool ll = a->mode == TDG_MODE_LL;
    const uint64_t ll_bytes = (uint64_t)M * K * 4;
    if (ll) {
        if (!aligned16(a->ll_off) || a->ll_off + ll_bytes > h->region_bytes)
            return a->ll_off + ll_bytes > h->region_bytes ? TDG_ERR_NOMEM : TDG_ERR_INVALID;
        if ((a->ll_off < a->a_off + shard_bytes && a->a_off < a->ll_off + ll_bytes) ||
            (a->ll_off < a->g_off + gath_bytes && a->g_off < a->ll_off + ll_bytes))
            return TDG_ERR_INVALID; // the LL buffer overlaps the shard or the gathered buffer
    }

    const int BM = gm::BM;
    // CTA pairs (256-row tiles) once there is more than one 128-row tile; two
    // pairs sharing B (512-row tiles) when every shard is a whole number of them
    const int cl = pick_cluster(a->cluster, M > BM, Ms % (4 * BM) == 0);
    const int stages = cl ? pick_stages(a->stages, cl) : 0;
    if (!cl || !stages || (a->split_tail & ~1) || (a->push & ~1) || a->producer_items < -1 ||
        a->producer_warps < 0 || a->producer_warps > ag::PMAX_WARPS || a->producer_chunk < 0)
        return TDG_ERR_INVALID;
    const int pair = cl >= 2 ? 1 : 0;
    const int pw = a->producer_warps ? a->producer_warps : ag::DEF_WARPS;
    const uint32_t pchunk = a->producer_chunk ? (uint32_t)a->producer_chunk : ag::DEF_CHUNK;
    if (pchunk % 1024 || pchunk < 4096 || pchunk > 65536)
        return TDG_ERR_INVALID;
    const int pslots = (int)min((uint32_t)ag::PMAX_SLOTS, (uint32_t)ag::PRING / (uint32_t)pw / pchunk);
    if (pslots < 3) // at least two loads in flight per worker
        return TDG_ERR_INVALID;
    const int TM = cl * BM;
    const bool inplace = (Ms % TM) == 0;
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
    bool ok = true;
    if (gemm) {
        ok = map_bf16_2d(&p.tmA_g, gathered, K, M, K * 2, 64, BM);
        ok = ok && map_bf16_2d(&p.tmA_l, region_r + a->a_off, K, Ms, K * 2, 64, BM);
        if (a->b_layout == TDG_B_KN)
            ok = ok && map_bf16_2d(&p.tmB, a->B, N, K, N * 2, 64, 64);
        else
            ok = ok && map_bf16_2d(&p.tmB, a->B, K, N, K * 2, 64, cl == 4 ? 64 : (pair ? 128 : 256));
        ok = ok && (a->c_f32 ? map_f32_2d(&p.tmC, a->C, N, M, N * 4, 32, 32)
                             : map_bf16_2d(&p.tmC, a->C, N, M, N * 2, 64, 32));
    }
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
    p.pair = pair;
    p.cl = cl;
    p.m_tiles = (int)((M + TM - 1) / TM);
    // B larger than about half of L2: group 8 m rows per raster group;
    // otherwise m-major
    p.group_m = ((uint64_t)K * N * 2 > (64ull << 20)) ? 8 : 0;
    p.n_tiles = (int)((N + gm::BN - 1) / gm::BN);
    p.tail_lo = (int64_t)p.m_tiles * p.n_tiles; // no items for the producer CTAs
    p.c_f32 = a->c_f32;
    p.swz = a->swizzle ? (int)(((int64_t)rank * Ms / TM) % p.m_tiles) : 0;
    p.local_inplace = inplace ? 1 : 0;
    p.local_lo = inplace ? (int)(rank * Ms / TM) : 0;
    p.local_hi = inplace ? (int)((rank + 1) * Ms / TM) : 0;
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
    if (a->source_order != 0 && a->source_order != 1)
        return TDG_ERR_INVALID;
    p.mesh = a->source_order;
    p.stages = stages;
    p.push = a->push;
    p.mirror = a->push && a->swizzle;
    p.t_end = (int)((((int64_t)rank + 1) * Ms - 1) / TM);
    p.pw = pw;
    p.pchunk = pchunk;
    p.pslots = pslots;

    const int sms = h->sm_count;
    const int ggrid = ag_grid(p, a->b_layout, sms); // GEMM-only grid
    if (ggrid <= 0)
        return TDG_ERR_UNSUPPORTED;
    if (ll) {
        // sender and receiver CTAs beside the GEMM, all in one cooperative launch
        const int n_send = a->producers > 0 ? a->producers : 8;
        const int64_t groups = M / sig_rows;
        // as many receivers as senders (8 by default), at most one per group
        int n_recv = (int)(groups < n_send ? groups : n_send);
        // senders and receivers fill whole clusters (spare receivers find no group)
        n_recv = (n_send + n_recv + cl - 1) / cl * cl - n_send;
        if (n_send + n_recv >= ggrid)
            return TDG_ERR_INVALID;
        p.ll = 1;
        p.ll_buf = reinterpret_cast<uint64_t *>(region_r + a->ll_off);
        p.n_send = n_send;
        p.n_prod = n_send + n_recv;
        p.wait_flags = 1;
        p.n_units = 0;
        return launch_ag(p, a->b_layout, gemm ? ggrid : p.n_prod, true, s, a->split_tail);
    }
    if (a->mode == TDG_MODE_SM) {
        int nprod = a->producers > 0 ? a->producers : default_producers(p, ggrid, TM);
        nprod = (nprod + cl - 1) / cl * cl; // producer CTAs fill whole clusters
        if (nprod >= ggrid)
            return TDG_ERR_INVALID;
        p.n_prod = nprod;
        p.wait_flags = 1;
        p.signal = 1;
        p.unit_rows = sig_rows;
        p.units_per_shard = Ms / sig_rows;
        p.n_units = (int64_t)W * p.units_per_shard;
        p.tail_lo = producer_tail_lo(p, ggrid, TM, a->producer_items);
        return launch_ag(p, a->b_layout, gemm ? ggrid : nprod, true, s, a->split_tail);
    }
    if (a->mode == TDG_MODE_SERIAL) {
        // copy phase: every SM (or `producers` CTAs) copies, fine-grained
        // units, no signals
        AgParams c = p;
        c.n_prod = a->producers > 0 ? (a->producers < sms ? a->producers : sms) : sms;
        c.signal = 0;
        c.wait_flags = 0;
        // units of a few rows, about 4 per copy worker (the workers stream
        // their units back to back, so small units cost nothing but balance
        // the load)
        const int64_t workers = (int64_t)c.n_prod * c.pw;
        c.unit_rows = M / (4 * workers);
        c.unit_rows = c.unit_rows < 1 ? 1 : (c.unit_rows > 64 ? 64 : c.unit_rows);
        if (c.unit_rows > Ms)
            c.unit_rows = Ms;
        while (Ms % c.unit_rows)
            c.unit_rows--;
        c.units_per_shard = Ms / c.unit_rows;
        c.n_units = (int64_t)W * c.units_per_shard;
        c.local_last = 0;
        c.pair = 0;
        c.cl = 1;
        c.stages = pick_stages(0, 1);
        int rc = launch_ag(c, a->b_layout, c.n_prod, false, s);
        if (rc != TDG_OK || !gemm)
            return rc;
        // GEMM phase: stream-ordered after the copy, no waits
        AgParams g = p;
        g.n_prod = 0;
        g.wait_flags = 0;
        g.n_units = 0;
        return launch_ag(g, a->b_layout, ggrid, false, s, a->split_tail);
    }
    // CE mode
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
        rc = cuda_err(e, "ce events");
    const int64_t ups = Ms / sig_rows;
    for (int64_t u = 0; u < (int64_t)W * ups && rc == TDG_OK; ++u) {
        // the producers' order (see copy_unit): pull rank+1, rank+2, ...;
        // push rank-1, rank-2, ..., each shard's groups from its last rows
        const int seq = p.mesh ? (int)(u % W) : (int)(u / ups);
        int64_t part = p.mesh ? u / W : u % ups;
        int shard;
        if (a->push) {
            shard = ((rank - (inplace ? 1 + seq : seq)) % W + W) % W;
            part = ups - 1 - part;
        } else {
            shard = inplace ? (rank + 1 + seq) % W : (rank + seq) % W;
        }
        {
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
    if (rc == TDG_OK && gemm) {
        AgParams g = p;
        g.n_prod = 0;
        g.wait_flags = 1;
        g.n_units = 0;
        rc = launch_ag(g, a->b_layout, ggrid, false, s, a->split_tail);
    }
    // the call completes on the main stream only when the side stream has too
    e = cudaEventRecord(ev1, side);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(s, ev1, 0);
    if (e != cudaSuccess && rc == TDG_OK)
        rc = cuda_err(e, "ce join");
    return rc;
}
