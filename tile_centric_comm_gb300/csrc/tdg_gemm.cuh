// tdg_gemm.cuh -- persistent, warp-specialised bf16 GEMM on the 5th-generation
// tensor cores (tcgen05 + TMEM), the consumer of the AllGather and the producer
// of the ReduceScatter ("Triton-distributed 语义", 内核设计模式: the consumer
// waits for each tile and computes on it at once; the GEMM producer signals
// each finished output tile).
//
// Each CTA runs 6 warps:
//   warp 0      TMA loader: per tile it first runs the policy's signal wait
//               (Triton-distributed's wait / consume_token), then streams
//               BK-wide slices of A and B into a shared-memory ring.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (K=16 per
//               instruction) into one of two TMEM accumulators (2 x 256 fp32
//               columns) and frees ring slots with tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld -> bf16 (round to nearest even) ->
//               128B-swizzled staging -> TMA store (or fp32 as it is, when the
//               policy asks); then the policy's
//               after-tile hook (the GEMM+RS signal and reduction).
//
// Three shapes of the same pipeline (template parameter CL, CTAs per cluster):
//   CL = 1  one CTA per SM owns a 128 x 256 tile; 4 stages of 48 KB.
//   CL = 2  a cluster of two CTAs (an SM pair) owns a 256 x 256 tile:
//           each CTA loads its 128 rows of A and half of the tile's columns
//           of B; the leader CTA issues tcgen05.mma.cta_group::2, which
//           reads both CTAs' shared memory and writes each CTA's TMEM
//           (its own 128 rows).  Both CTAs' loads complete on the leader's
//           barrier; the leader's commits arrive on both CTAs' barriers.
//           Stages are 32 KB, so 6 are in flight, and each SM moves a third
//           less operand data per FLOP than with CL = 1.
//   CL = 4  two such pairs stacked in M own a 512 x 256 tile and share B:
//           each B slice (64 columns x 64 K) is fetched once from L2 by one
//           pair and multicast into the same slot of the other pair, so
//           every CTA requests 24 KB instead of 32 KB per stage.  A slot is
//           refilled only after both pairs' MMAs have released it (each
//           leader's commit arrives on the empty barrier of all four CTAs).
// A tile at the right edge of N issues a narrower MMA and stores only its
// valid columns; rows past M come from TMA zero fill and are not stored.
// Operands: A is K-major (rows of K); B is either MN-major (K x N row-major,
// the transpose bit of the instruction descriptor) or K-major (N x K).
#pragma once

#include <type_traits>

#include "tdg.h"
#include "tdg_ptx.cuh"

namespace tdg {
namespace gm {
constexpr int BM = 128; // rows per CTA
constexpr int BN = 256; // columns per tile
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2; // 16 KB
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 4;
constexpr int EPI_BUF = 32 * 128;     // 32 rows x 64 bf16 (128 B)
constexpr int RING_BYTES = 196608;    // 4 x 48 KB or 6 x 32 KB
constexpr int OFF_EPI = RING_BYTES;
constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * 2 * EPI_BUF; // 229376
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;     // + alignment slack
constexpr uint32_t TMEM_COLS = 512;

template <int PAIR> struct Shape {
    static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;  // B columns held per CTA
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = RING_BYTES / STAGE_BYTES;        // 4 or 6
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;              // rows per tile
};
static_assert(Shape<0>::STAGES == 4 && Shape<1>::STAGES == 6, "ring layout");
} // namespace gm

struct TileInfo {
    int m0;      // first output row handled by THIS CTA (tile row + 128 * sub)
    int n0;      // first output column of the tile
    int n_valid; // columns of this tile inside N (1..BN)
    int n_mma;   // MMA N: n_valid rounded up (16 for one CTA, 32 for a pair)
    int a_row;   // row coordinate of this CTA's A slice in the selected map
    int a_sel;   // policy-defined: which A map / which rank
    int owner;   // policy-defined (RS: owner rank)
    int m_loc;   // policy-defined (RS: 128-row tile inside the owner)
    int pn;      // n tile index
};

struct PipeSmem {
    uint64_t full[6];
    uint64_t empty[6];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;     // used only after an abort, to drain issued MMAs
    uint32_t tmem_base;
    volatile int abort;
    int is_last;
    uint32_t issued;    // ring fills issued by this CTA's loader
    uint32_t consumed;  // ring fills consumed by the leader's MMA issuer
};
static_assert(sizeof(PipeSmem) <= gm::BAR_BYTES, "barrier block");

// q = a / b and r = a % b for a >= 0, b > 0, in 32-bit arithmetic whenever
// both fit (an unsigned 32-bit division is a short instruction sequence, a
// 64-bit one a long software routine); the tile decoders of the policies run
// once per tile in the loader and in every epilogue warp.
__device__ __forceinline__ int64_t divmod(int64_t a, int64_t b, int64_t &r)
{
    if ((static_cast<uint64_t>(a) | static_cast<uint64_t>(b)) < 0x100000000ull) {
        const uint32_t q = static_cast<uint32_t>(a) / static_cast<uint32_t>(b);
        r = static_cast<int64_t>(static_cast<uint32_t>(a) - q * static_cast<uint32_t>(b));
        return q;
    }
    const int64_t q = a / b;
    r = a - q * b;
    return q;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Policy P provides:
//   struct Params { ... DevStatus *status; uint32_t epoch; uint64_t timeout_ns, pipe_timeout_ns;
//                   int k_blocks; int stages; int full_n; int edge_n; int n_tiles; };
//       (stages: ring stages in use, 2 .. Shape::STAGES; full_n: every item is
//        a tile of the full BN columns -- N a multiple of BN, no null items --
//        so the MMA issuer needs no per-tile arithmetic; edge_n > 0: no null
//        items, item i is in n-tile column i mod n_tiles, and only the last
//        column is narrower, with an MMA of edge_n columns)
//   static constexpr int B_MN;                                   // 1: B is K x N
//   __device__ static int64_t num_items(const Params&);
//   __device__ static void tile(const Params&, int64_t item, TileInfo&, int sub);
//       (sub: this CTA's 128-row slice of the cluster's tile; an item with
//        n_valid <= 0 is a null item: every role skips it)
//   __device__ static void before_a(const Params&, const TileInfo&, bool &gave_up);  // loader thread
//   template <int CL> __device__ static void load_a(const Params&, const TileInfo&, void *dst,
//                                                   uint32_t bar, int kb);
//   template <int CL> __device__ static void load_b(const Params&, const TileInfo&, void *dst,
//                                                   uint32_t bar, int kb, int col0, int cols,
//                                                   int pidx, int half);
//       (CL = 4: pair pidx fetches the 64-column slices j with j % 2 == pidx
//        and multicasts each to CTA `half` of both pairs)
//   __device__ static uint32_t b_bytes(const Params&, const TileInfo&, int cols);
//   __device__ static void store_chunk(const Params&, const TileInfo&, const void *buf, int ch, int q);
//       (stores the bf16 rows [32q, 32q + 32) x columns [64ch, 64ch + 64) staged in buf)
//   static constexpr bool F32_OUT;  // true: the policy may ask for fp32 output, then
//   __device__ static bool out_f32(const Params&);
//   __device__ static void store_chunk_f32(const Params&, const TileInfo&, const void *buf, int sub, int q);
//       (fp32 rows [32q, 32q + 32) x columns [32sub, 32sub + 32))
//   struct EpiState;  // per epilogue warp, zero-initialised, kept across its tiles
//   __device__ static void after_tile(const Params&, const TileInfo&, int q, int lane, EpiState&,
//                                     bool tail);  // per epilogue warp after each tile; once
//       more with tail = true (and no tile) after the last one
// The load hooks receive the mbarrier as a shared::cluster address (the pair
// leader's barrier when CL >= 2) and issue pair TMA when CL >= 2.  All
// tcgen05 and TMA instructions of one kernel use a single cta_group.
// Items [item_lo, item_hi) (item_hi < 0: all of P::num_items) are dealt to
// `nunits` scheduling units round robin; this CTA's unit is `unit`.
template <class P, int CL>
__device__ void gemm_consumer(const typename P::Params &p, uint8_t *smem, int unit, int nunits,
                              int64_t item_lo = 0, int64_t item_hi = -1)
{
    using namespace gm;
    constexpr int PAIR = CL >= 2 ? 1 : 0;
    constexpr bool QUAD = CL == 4;
    using S = Shape<PAIR>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int crank = PAIR ? (int)cluster_ctarank() : 0; // this CTA's 128-row slice of the tile
    const int half = crank & 1;                           // CTA in its pair
    const int pidx = crank >> 1;                          // pair in the cluster
    const bool leader = half == 0;
    const uint32_t lead_rank = (uint32_t)(crank & ~1);
    const uint16_t pair_mask = (uint16_t)(3u << (2 * pidx));
    const uint16_t empty_mask = QUAD ? (uint16_t)0xF : pair_mask;
    PipeSmem *ps = reinterpret_cast<PipeSmem *>(smem + OFF_BAR);
    // ring stages in use (the host checks the range; the ring holds S::STAGES)
    const int NST = (p.stages >= 2 && p.stages < S::STAGES) ? p.stages : S::STAGES;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S::STAGES; ++i) {
            mbar_init(&ps->full[i], 1);
            mbar_init(&ps->empty[i], QUAD ? 2 : 1); // one commit per pair sharing the slot
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ps->tfull[i], 1);
            mbar_init(&ps->tempty[i], EPI_WARPS * (PAIR ? 2 : 1));
        }
        mbar_init(&ps->drain, 1);
        ps->issued = 0;
        ps->consumed = 0;
        ps->abort = 0;
        ps->is_last = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(&ps->tmem_base, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&ps->tmem_base, TMEM_COLS);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    __syncthreads();
    if (PAIR)
        cluster_sync(); // the peer's barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = ps->tmem_base;
    // this launch's share of the items: [item_lo, items), unit by unit
    const int64_t items = item_hi >= 0 ? item_hi : P::num_items(p);
    const uint64_t tmo = p.pipe_timeout_ns;
    // the barrier a load completes on / an epilogue releases: the pair leader's
    const uint32_t full0 = PAIR ? mapa_shared(smem_u32(&ps->full[0]), lead_rank) : smem_u32(&ps->full[0]);
    const uint32_t tempty0 =
        PAIR ? mapa_shared(smem_u32(&ps->tempty[0]), lead_rank) : smem_u32(&ps->tempty[0]);

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool gave_up = false;
            uint32_t issued = 0; // kept in a register; published once for the abort drain
            for (int64_t it = item_lo + unit; it < items && !ps->abort; it += nunits) {
                TileInfo ti;
                P::tile(p, it, ti, crank);
                if (ti.n_valid <= 0)
                    continue; // a null item (an empty half of a split tail tile)
                P::before_a(p, ti, gave_up);
                const int cols = PAIR ? ti.n_mma / 2 : ti.n_mma;
                const int col0 = ti.n0 + (PAIR ? half * cols : 0);
                const uint32_t my_bytes = A_BYTES + P::b_bytes(p, ti, cols);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait_sleep(&ps->empty[stage], phase ^ 1u, tmo, 64)) {
                        report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_PIPE, 0, p.epoch);
                        ps->abort = 1;
                        break;
                    }
                    uint8_t *sa = smem + stage * S::STAGE_BYTES;
                    // the leader arms its barrier for both CTAs' bytes
                    if (leader)
                        mbar_arrive_expect_tx(&ps->full[stage], PAIR ? 2 * my_bytes : my_bytes);
                    const uint32_t bar = full0 + stage * 8;
                    P::template load_a<CL>(p, ti, sa, bar, kb);
                    P::template load_b<CL>(p, ti, sa + A_BYTES, bar, kb, col0, cols, pidx, half);
                    ++issued;
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            ps->issued = issued;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            uint32_t consumed = 0; // kept in a register; published once for the abort drain
            const uint32_t sbase = smem_u32(smem);
            // The issuing thread spends 60-85 cycles on each MMA (256 x 256 x
            // 16, 128 cycles of tensor-pipe work), so what it does between a
            // stage's MMAs and the next stage's decides whether the pipe's
            // queue stays full: with full-width tiles only (the common case)
            // it skips the tile's index arithmetic (64-bit divisions) and
            // issues with a compile-time instruction descriptor, which
            // measured 1.5 % of the GEMM at 50 k-blocks per tile.  Where only
            // the last n-tile column is narrow (edge_n), the column is tracked
            // without division and only that column's tiles take the general
            // copy of the loop (+2 % at the Qwen-32B up-projection shape,
            // N = 3200).  With every ring slot in use, the full-width loop
            // runs whole rounds of the ring unrolled, so that each slot's
            // barriers and descriptors are fixed offsets from hoisted bases
            // (no stage arithmetic or wrap test between the stages' MMAs).
            // The descriptors' start-address field counts 16-byte units, and
            // the ring (under 256 KB of shared memory) never carries into the
            // next field, so adding a slot's offset to the base descriptor
            // equals building the descriptor at the slot.
            // MN-major B: 64-column chunks 8 KB apart (LBO), 8 K-rows 1 KB
            // apart (SBO); a K step of 16 rows is 2 KB.  K-major B: same form
            // as A (a K step of 16 elements is 32 bytes).
            const uint64_t a_desc0 = sdesc_sw128(sbase, 16, 1024);
            const uint64_t b_desc0 =
                P::B_MN ? sdesc_sw128(sbase + A_BYTES, 8192, 1024) : sdesc_sw128(sbase + A_BYTES, 16, 1024);
            // one ring stage in slot st: wait for its data, issue its MMAs, free it
            auto stage_mma = [&](int kb, int st, uint32_t ph, uint32_t idesc, uint32_t d_tmem) -> bool {
                const uint64_t ad0 = a_desc0 + (uint64_t)(st * (S::STAGE_BYTES >> 4));
                const uint64_t bd0 = b_desc0 + (uint64_t)(st * (S::STAGE_BYTES >> 4));
                if (!mbar_wait(&ps->full[st], ph, tmo))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint64_t ad = ad0 + (uint64_t)(k * 2);
                    const uint64_t bd = bd0 + (uint64_t)(P::B_MN ? k * 128 : k * 2);
                    if (PAIR)
                        umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                    else
                        umma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                }
                if (PAIR)
                    umma_commit_pair_mask(&ps->empty[st], empty_mask);
                else
                    umma_commit(&ps->empty[st]);
                return true;
            };
            // Returns the k-blocks consumed: all of them, or fewer when a wait
            // ran out.
            auto k_loop = [&](auto full_width, uint32_t idesc_rt, uint32_t d_tmem) -> int {
                constexpr bool FULL = decltype(full_width)::value;
                const uint32_t idesc = FULL ? idesc_bf16(S::TILE_M, BN, P::B_MN) : idesc_rt;
                int kb = 0;
                if (FULL && NST == S::STAGES) {
                    // up to slot 0, then whole rounds of the ring unrolled
                    for (; kb < p.k_blocks && stage != 0; ++kb) {
                        if (!stage_mma(kb, stage, phase, idesc, d_tmem))
                            goto timed_out;
                        if (++stage == NST) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    for (; kb + S::STAGES <= p.k_blocks; kb += S::STAGES) {
#pragma unroll
                        for (int st = 0; st < S::STAGES; ++st)
                            if (!stage_mma(kb + st, st, phase, idesc, d_tmem)) {
                                kb += st;
                                goto timed_out;
                            }
                        phase ^= 1u;
                    }
                }
                for (; kb < p.k_blocks; ++kb) {
                    if (!stage_mma(kb, stage, phase, idesc, d_tmem))
                        goto timed_out;
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                return p.k_blocks;
            timed_out:
                report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_PIPE, 2, p.epoch);
                ps->abort = 1;
                return kb;
            };
            // with edge_n, the column of this unit's items walks on by nunits
            // mod n_tiles per item (no division in the loop)
            int col = 0, col_step = 0;
            if (!p.full_n && p.edge_n > 0) {
                col = (int)((item_lo + unit) % p.n_tiles);
                col_step = (int)(nunits % p.n_tiles);
            }
            for (int64_t it = item_lo + unit; it < items && !ps->abort; it += nunits) {
                uint32_t idesc_rt = 0;
                bool full = p.full_n != 0;
                if (!full && p.edge_n > 0) {
                    full = col != p.n_tiles - 1;
                    idesc_rt = idesc_bf16(S::TILE_M, p.edge_n, P::B_MN);
                    col += col_step;
                    if (col >= p.n_tiles)
                        col -= p.n_tiles;
                } else if (!full) {
                    TileInfo ti;
                    P::tile(p, it, ti, crank);
                    if (ti.n_valid <= 0)
                        continue;
                    idesc_rt = idesc_bf16(S::TILE_M, ti.n_mma, P::B_MN);
                }
                if (!mbar_wait(&ps->tempty[acc], acc_phase ^ 1u, tmo)) {
                    report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_PIPE, 1, p.epoch);
                    ps->abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const int done = full ? k_loop(std::true_type{}, 0u, d_tmem)
                                      : k_loop(std::false_type{}, idesc_rt, d_tmem);
                consumed += (uint32_t)done;
                if (done < p.k_blocks)
                    break;
                if (PAIR)
                    umma_commit_pair_mask(&ps->tfull[acc], pair_mask);
                else
                    umma_commit(&ps->tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            ps->consumed = consumed;
            if (ps->abort) {
                // let every MMA this thread issued finish before TMEM is freed
                if (PAIR)
                    umma_commit_pair_mask(&ps->drain, pair_mask);
                else
                    umma_commit(&ps->drain);
                (void)mbar_wait(&ps->drain, 0, tmo);
            }
        }
        __syncwarp();
    } else {
        // epilogue warps: TMEM lane quarter q = warp % 4 (hardware rule)
        const int q = warp & 3;
        uint8_t *bufs = smem + OFF_EPI + (warp - EPI_WARP0) * 2 * EPI_BUF;
        int acc = 0;
        uint32_t acc_phase = 0;
        int buf = 0;
        typename P::EpiState est{};
        // after the last tile, one more pass with no tile (tail = true) lets
        // the policy finish work it deferred
        for (int64_t it = item_lo + unit;; it += nunits) {
            TileInfo ti;
            if (it >= items) {
                if (!ps->abort)
                    P::after_tile(p, ti, q, lane, est, true);
                break;
            }
            P::tile(p, it, ti, crank);
            if (ti.n_valid <= 0)
                continue;
            // one lane polls the barrier; the warp follows it (fewer shared
            // memory probes while the mainloop runs)
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait_sleep(&ps->tfull[acc], acc_phase, tmo, 256);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok || ps->abort) {
                if (lane == 0 && !ok)
                    report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_PIPE, 3, p.epoch);
                ps->abort = 1;
                break;
            }
            tc_fence_after();
            const int nch = (ti.n_valid + 63) >> 6;
            for (int ch = 0; ch < nch; ++ch) {
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(acc * BN + ch * 64);
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(taddr, r0);
                tmem_ld_32x32b_x32(taddr + 32, r1);
                tmem_ld_wait();
                if constexpr (P::F32_OUT) {
                    if (P::out_f32(p)) {
                        // fp32 output: two 32-column chunks, stored as they are
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const uint32_t *src = hf ? r1 : r0;
                            if (lane == 0)
                                bulk_wait_read<1>();
                            __syncwarp();
                            uint8_t *frow = bufs + buf * EPI_BUF + lane * 128;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                *reinterpret_cast<uint4 *>(frow + ((j ^ (lane & 7)) << 4)) =
                                    make_uint4(src[4 * j], src[4 * j + 1], src[4 * j + 2], src[4 * j + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                P::store_chunk_f32(p, ti, bufs + buf * EPI_BUF, 2 * ch + hf, q);
                                bulk_commit();
                            }
                            buf ^= 1;
                        }
                        continue;
                    }
                }
                if (lane == 0)
                    bulk_wait_read<1>();
                __syncwarp();
                uint8_t *row = bufs + buf * EPI_BUF + lane * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t *src = (j < 4) ? &r0[j * 8] : &r1[(j - 4) * 8];
                    const uint32_t w0 = pack_bf16x2(__uint_as_float(src[0]), __uint_as_float(src[1]));
                    const uint32_t w1 = pack_bf16x2(__uint_as_float(src[2]), __uint_as_float(src[3]));
                    const uint32_t w2 = pack_bf16x2(__uint_as_float(src[4]), __uint_as_float(src[5]));
                    const uint32_t w3 = pack_bf16x2(__uint_as_float(src[6]), __uint_as_float(src[7]));
                    *reinterpret_cast<uint4 *>(row + ((j ^ (lane & 7)) << 4)) = make_uint4(w0, w1, w2, w3);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    P::store_chunk(p, ti, bufs + buf * EPI_BUF, ch, q);
                    bulk_commit();
                }
                buf ^= 1;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    mbar_arrive_remote(tempty0 + acc * 8);
                else
                    mbar_arrive(&ps->tempty[acc]);
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            P::after_tile(p, ti, q, lane, est, false);
        }
        if (lane == 0)
            bulk_wait<0>();
    }
    __syncthreads();
    if (ps->abort && threadIdx.x == 0) {
        // wait (bounded) until no TMA write of this CTA is still in flight.
        if (!PAIR || leader) {
            for (uint32_t f = ps->consumed; f < ps->issued; ++f)
                (void)mbar_wait(&ps->full[f % NST], (f / NST) & 1u, tmo);
        } else {
            // a peer's fill is known done once the leader has freed its slot
            for (uint32_t f = ps->issued > (uint32_t)NST ? ps->issued - NST : 0u;
                 f < ps->issued; ++f)
                (void)mbar_wait(&ps->empty[f % NST], (f / NST) & 1u, tmo);
        }
    }
    __syncthreads();
    if (PAIR)
        cluster_sync(); // no CTA leaves while another may still touch it
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

} // namespace tdg
