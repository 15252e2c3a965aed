/*
 * tdg.h -- C ABI of libtdg: tile-centric overlapped AllGather+GEMM,
 * GEMM+ReduceScatter and MoE dispatch/combine on one GB300 (sm_103a).
 *
 * Model.  W logical ranks live in ONE device allocation that the caller owns:
 * W equal "regions" (rank r's symmetric heap) followed by W signal areas and
 * a small status block.  "Communication" moves tiles between regions inside
 * HBM; every tile carries its own signal.  This follows the programming model
 * of the Triton-distributed paper summary (hyper.ai, arXiv 2504.19442, section
 * 方法: symmetric memory, signal exchange, asynchronous tasks) and of
 * "Triton-distributed 语义" (sections 生产者-消费者模型, 基于信号的同步,
 * 对称内存模型, 内核设计模式, 线程块交织, 基于令牌的数据依赖).
 *
 * Conventions for every entry point:
 *   - All pointers named dev_* / device are device pointers; host pointers are
 *     named host_*.  Streams are passed as void* and are cudaStream_t values
 *     (NULL = the legacy default stream).
 *   - bf16 = IEEE bfloat16, row-major, no padding between rows.
 *   - Calls are asynchronous on the given stream(s).  Inputs must stay
 *     unchanged and outputs untouched until the stream has completed the call.
 *   - Return value: TDG_OK (0) or a negative TDG_ERR_* code from host-side
 *     validation; nothing is launched when validation fails.  Faults found on
 *     the device (a signal wait that ran out of time, an out-of-range index)
 *     are recorded in the handle's status block and read with tdg_status().
 *   - The library allocates no device memory.  Each entry point documents
 *     which caller-provided buffers it uses.
 *   - A handle is thread-compatible, not thread-safe: do not call into the
 *     same handle from two host threads at once.  Different handles may be
 *     used from different threads.
 *   - Every operation runs on the device the heap was allocated on
 *     (tdg_symm_alloc records the current device); calling it while another
 *     device is current returns TDG_ERR_INVALID.  Any host thread may call:
 *     the call makes that device's context current in the calling thread.
 *
 * Schedules.  Several args fields choose among schedules of the same
 * computation (GEMM cluster shape, ring stages, tile order, producer shape,
 * push or pull); 0 always means the library's default for the shape, and the
 * tests check every setting against the oracle.  They are per call, so two
 * threads or two shapes in one process may use different schedules.
 *
 * Environment variable:
 *   TDG_LOG=1             print host-side failures (tensor-map encoding,
 *                         MoE workspace) to stderr.
 */
#ifndef TDG_H_
#define TDG_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TDG_API __attribute__((visibility("default")))
#else
#define TDG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes -------------------------------------------------------- */
#define TDG_OK 0
#define TDG_ERR_INVALID -1     /* bad argument: shape, alignment, range, NULL */
#define TDG_ERR_CUDA -2        /* a CUDA runtime/driver call failed           */
#define TDG_ERR_NOMEM -3       /* a caller buffer / region / signal area is too small */
#define TDG_ERR_TIMEOUT -4     /* device: a bounded signal wait ran out of time */
#define TDG_ERR_UNSUPPORTED -5 /* device or mode not supported here           */
#define TDG_ERR_DEVICE -6      /* device: a kernel found an out-of-range index  */

/* ---- modes -------------------------------------------------------------- */
/* SM: producer CTAs and consumer CTAs in one persistent launch (overlapped). */
#define TDG_MODE_SM 0
/* CE: copies on the copy engine (side stream) + stream-ordered flag writes;
 *     the GEMM runs on the main stream and waits on the flags.              */
#define TDG_MODE_CE 1
/* LL: low-latency path: 8-byte {payload, flag} words, for small shards.     */
#define TDG_MODE_LL 2
/* SERIAL: same kernels, one after the other with no overlap (copy, then
 *     GEMM, then reduce) -- the measurement twin and the "barrier between
 *     phases" debugging mode.                                               */
#define TDG_MODE_SERIAL 3

/* layout of B for the GEMMs */
#define TDG_B_KN 0 /* B is K x N row-major (N contiguous)  */
#define TDG_B_NK 1 /* B is N x K row-major (K contiguous)  */

/* ---- symmetric heap ------------------------------------------------------ */
typedef struct tdg_symm tdg_symm; /* opaque, owned by the library */

/*
 * Bytes the caller must provide for a symmetric heap of `world` regions of
 * `region_bytes` each, with `signals_per_rank` 32-bit flag words and as many
 * 32-bit counter words per rank.  region_bytes must be a multiple of 1024.
 */
TDG_API size_t tdg_symm_bytes(int world, size_t region_bytes, size_t signals_per_rank);

/*
 * Carve caller memory [dev_base, dev_base + bytes) into the heap described
 * above.  Layout: region r at dev_base + r*region_bytes; then the flag words
 * of every rank; then the counter words of every rank; then the status block.
 * The signal areas and the status block are zeroed here (synchronously, with
 * cudaMemset on the current device).  dev_base must be 1024-byte aligned.
 * The caller keeps ownership of the memory; tdg_symm_free never frees it.
 * The handle owns two CUDA events (created by its first CE-mode call, for the
 * fork to and join from the side stream); tdg_symm_free destroys them.
 * Returns TDG_OK and *out, or TDG_ERR_INVALID / TDG_ERR_NOMEM / TDG_ERR_CUDA.
 */
TDG_API int tdg_symm_alloc(void *dev_base, size_t bytes, int world, size_t region_bytes,
                   size_t signals_per_rank, tdg_symm **out);

/* Release the handle (host memory only). */
TDG_API int tdg_symm_free(tdg_symm *h);

/* Base of rank `rank`'s region, or NULL if rank is out of range. */
TDG_API void *tdg_symm_region(const tdg_symm *h, int rank);

/*
 * symm_at: translate a pointer inside any region to the same offset inside
 * region `rank` ("Triton-distributed 语义", 对称内存模型: symm_at(ptr, rank)).
 * Returns NULL if local_ptr is not inside a region or rank is out of range.
 */
TDG_API void *tdg_symm_at(const tdg_symm *h, const void *local_ptr, int rank);

/* Device address of rank `rank`'s flag words / counter words (NULL if out of range). */
TDG_API uint32_t *tdg_symm_flags(const tdg_symm *h, int rank);
TDG_API uint32_t *tdg_symm_counters(const tdg_symm *h, int rank);

/* The epoch the next call will take when no other call comes first.  Epochs
 * come from one counter shared by every handle of the process, in [1, 2^31),
 * so no two calls share one: flags compare against it, and words that an
 * earlier call left in memory never carry a later call's epoch. */
TDG_API uint32_t tdg_symm_epoch(const tdg_symm *h);

/* ---- device status ------------------------------------------------------- */
typedef struct {
    int32_t code;   /* TDG_OK, TDG_ERR_TIMEOUT or TDG_ERR_DEVICE              */
    uint32_t where; /* which wait / check: see TDG_WHERE_*                   */
    uint32_t index; /* signal or tile index involved                          */
    uint32_t epoch; /* epoch of the call that failed                          */
} tdg_fault;

#define TDG_WHERE_AG_FLAG 1    /* consumer waiting on an AllGather tile flag */
#define TDG_WHERE_PIPE 2       /* an intra-CTA pipeline barrier ran out of time */
#define TDG_WHERE_LL 3         /* LL receiver waiting on a data+flag word     */
#define TDG_WHERE_MOE_EXPERT 4 /* an expert id outside [0, E)                 */
#define TDG_WHERE_RING 5       /* ring AllReduce waiting on a tile of a step   */
#define TDG_WHERE_RS_SIGNAL 6  /* GEMM-RS arrival counter update did not settle */

/*
 * Copy the status block to *out (may be NULL) after synchronising `stream`,
 * and clear it when clear != 0.  Returns the status code (TDG_OK if no device
 * fault was recorded since the last clear), or TDG_ERR_CUDA.
 */
TDG_API int tdg_status(tdg_symm *h, void *stream, tdg_fault *out, int clear);

/* Human-readable text for a TDG_* code (static storage). */
TDG_API const char *tdg_strerror(int code);

/* Number of SMs and whether the current device runs these kernels (sm_103). */
TDG_API int tdg_device_info(int *sm_count, int *supported);

/* ---- AllGather + GEMM ----------------------------------------------------- */
/*
 * C = concat_rows(A_0, ..., A_{W-1}) @ B, computed by rank `rank`
 * ("Triton-distributed 语义", 内核设计模式 "AllGather + GEMM 重叠"; paper
 * summary, 方法: intra-node AllGather on SMs or the copy engine).
 *
 * Shard s (Ms x K bf16) sits at region(s) + a_off.  The AllGather writes the
 * gathered M x K matrix (M = W*Ms) into region(rank) + g_off, shard s at rows
 * [s*Ms, (s+1)*Ms) -- every shard reaches it, its own included (pulled by
 * rank `rank`, or in push mode delivered by the senders in their order).
 * Producers signal per group of `signal_rows` gathered rows (flag word
 * g = row / signal_rows of rank `rank`'s flags, set to the call's epoch with
 * release semantics); the GEMM waits on every group its A tile needs
 * (bounded acquire spin), so it computes on tiles that have arrived while
 * others are still in flight.  Tiles are visited in the rank-swizzled order
 * pid_m = (pid_m + rank*Ms/BM) % m_tiles ("Triton-distributed 语义", 线程块交织;
 * mirrored in push mode, so the tiles follow the shards' arrival order)
 * when swizzle != 0; when Ms is a multiple of BM the local shard is read in
 * place, with no wait.
 *
 * B: K x N (TDG_B_KN) or N x K (TDG_B_NK) bf16, device pointer.
 * C: M x N output, device pointer: bf16 (each fp32 accumulator rounded to
 * nearest even), or with c_f32 = 1 float32 (the fp32 accumulator itself, no
 * rounding; M*N*4 bytes).  The caller owns B and C.
 * Requirements: 1 <= world <= 64; 0 <= rank < world; K % 8 == 0; N % 8 ==
 * 0; a_off, g_off, B, C 16-byte aligned; the gathered buffer not overlapping
 * the shard; signal_rows dividing Ms; source_order and c_f32 0 or 1; CE mode needs a
 * side_stream other than stream; LL mode an aligned LL buffer that overlaps
 * neither the shard nor the gathered buffer; SM / LL producer CTAs fewer than
 * the GEMM's grid (TDG_ERR_INVALID otherwise).  g_off + M*K*2, a_off + Ms*K*2
 * (and ll_off + M*K*4) <= region_bytes and M / signal_rows <=
 * signals_per_rank (TDG_ERR_NOMEM otherwise).  M == 0 is a no-op; N == 0
 * runs the AllGather alone (the gathered buffer and the flags, in the given
 * mode; B and C may be NULL); K == 0 writes C = 0.
 */
typedef struct {
    int world, rank;
    int64_t Ms, K, N;
    size_t a_off, g_off;
    const void *B;
    void *C;
    int b_layout;        /* TDG_B_KN or TDG_B_NK                            */
    int mode;            /* TDG_MODE_SM / CE / LL / SERIAL                  */
    int producers;       /* producer CTAs in SM / LL mode (0 = default: SM
                            mode enough to copy the shards within the GEMM's
                            time at about 50 GB/s each, 4..32; LL 8 senders),
                            copy CTAs of the SERIAL copy launch (0 = every SM) */
    int64_t signal_rows; /* rows per signal; 0 = Ms (one per shard) in CE
                            mode, else 32 when Ms is a multiple of the GEMM's
                            rows per tile and of 32, else Ms                */
    int swizzle;         /* 1 = rank-swizzled tile order, 0 = linear        */
    uint64_t timeout_ns; /* bound of every device wait; 0 = 2 s             */
    size_t ll_off;       /* LL mode: LL buffer (M*K*4 bytes) in region(rank);
                          * a word counts as delivered when its upper half is
                          * the call's epoch, so memory that last held
                          * anything but this process's LL words must be
                          * zeroed once before its first LL call               */
    uint64_t test_skip_notify; /* tests only: producers skip the notify of
                                  signal groups whose bit (g % 64) is set   */
    int source_order;    /* 0: one source at a time, rank+1, rank+2, ... (the
                            published NVSwitch swizzle); 1: all sources at once,
                            round robin over sources (their full-mesh order) */
    int c_f32;           /* 1: C is float32; 0: bf16                         */
    /* schedule (0 = default for the shape) */
    int cluster;         /* CTAs per GEMM cluster: 1 (128-row tiles), 2 (a CTA
                            pair, cta_group::2, 256-row tiles; needs M > 128)
                            or 4 (two pairs sharing each B slice by TMA
                            multicast, 512-row tiles; needs Ms % 512 == 0).
                            Default: the largest the shape allows            */
    int stages;          /* operand ring stages of the GEMM: 2 .. 4 (cluster
                            1) or 2 .. 6 (clusters 2 and 4); default all     */
    int split_tail;      /* 1: cut the tiles of the last, partial wave of the
                            persistent GEMM into 128-column halves (not with
                            SM-mode producer items)                          */
    int producer_items;  /* SM mode: GEMM items the producer CTAs take from
                            the end of the order once their copies are done:
                            0 = balanced on the host from the copy and tile
                            times, -1 = none, n > 0 = the last n items       */
    int producer_warps;  /* SM / SERIAL mode: copy workers (warps) per
                            producer CTA, 1..4 (default 2)                   */
    int producer_chunk;  /* SM / SERIAL mode: bytes per TMA bulk copy, a
                            multiple of 1024 in [4096, 65536] (default 32768) */
    int push;            /* 1: push-mode AllGather: the senders order the
                            transfers (sender s reaches destination
                            (s + j) mod W at step j), so rank `rank` receives
                            the shards in the order rank-1, rank-2, ... (all
                            at once with source_order 1) and its GEMM visits
                            the m tiles in that order; 0: pull (rank+1,
                            rank+2, ...)                                     */
} tdg_ag_gemm_args;

TDG_API int tdg_ag_gemm(tdg_symm *h, const tdg_ag_gemm_args *args, void *stream,
                void *side_stream);

/* ---- AllGather + GEMM for every rank at once ------------------------------ */
/*
 * For every rank r: C_r = concat_rows(A_0, ..., A_{W-1}) @ B_r -- the
 * AllGather+GEMM of the previous entry point run by all W ranks in one call
 * ("Triton-distributed 语义", 内核设计模式 "AllGather + GEMM 重叠", every PE;
 * paper summary, 方法: intra-node AllGather on the copy engine), W times the
 * work of one rank's call.
 *
 * Shard A_r (Ms x K bf16) at region(r) + a_off; rank r's gathered M x K
 * buffer (M = W*Ms) at region(r) + g_off, shard s at rows [s*Ms, (s+1)*Ms);
 * B_r (K x N with TDG_B_KN, N x K with TDG_B_NK) at region(r) + b_off; C_r
 * (M x N bf16) at region(r) + c_off.  Rank r's flag words g = row /
 * signal_rows of its gathered rows are set to the call's epoch.
 * CE mode: one persistent GEMM launch on `stream` runs every rank's tiles,
 * rank after rank, each rank's m tiles in the swizzled order (its own shard
 * first, read in place when Ms is a whole number of tiles) and waits (bounded)
 * on the flags of the rows it reads; the W x W shard copies run on
 * `side_stream` (cudaMemcpyAsync, then a stream-ordered flag write), rank by
 * rank.  The copies and flag writes are queued before the GEMM, so the call
 * completes even when the two streams run one after the other; the GEMM does
 * not wait behind the copies (the tiles of each rank's own shard start at
 * once).  SERIAL mode: the copies, then the GEMM, on `stream`.
 * Requirements: 1 <= world <= 64; K % 8 == 0; N % 8 == 0; c_f32 0 or 1; offsets 16-byte
 * aligned; every buffer inside its region (else TDG_ERR_NOMEM); the gathered
 * buffers and C_r overlapping no other buffer (else TDG_ERR_INVALID);
 * signal_rows dividing Ms; M / signal_rows <= signals_per_rank.  M == 0 or
 * N == 0 is a no-op; K == 0 writes C_r = 0.
 */
typedef struct {
    int world;
    int64_t Ms, K, N;
    size_t a_off, g_off, b_off, c_off;
    int b_layout;        /* TDG_B_KN or TDG_B_NK                              */
    int mode;            /* TDG_MODE_CE or TDG_MODE_SERIAL                    */
    int64_t signal_rows; /* rows per signal; 0 = Ms (one per shard)           */
    uint64_t timeout_ns; /* bound of every device wait; 0 = 2 s               */
    uint64_t test_skip_notify; /* tests only: rank 0's flag of signal group g
                                  is not written when bit (g % 64) is set     */
    int c_f32;           /* 1: C_r is float32 (M*N*4 bytes, the fp32
                            accumulator unrounded); 0: bf16                   */
    /* schedule (0 = default for the shape) */
    int cluster;         /* as in tdg_ag_gemm_args                            */
    int stages;          /* as in tdg_ag_gemm_args                            */
    int push;            /* 1: push-mode AllGather: the copies go step by
                            step, sender s to destination (s + j) mod W at
                            step j = 1 .. W-1, so every destination receives
                            one shard per step from a different sender; the
                            GEMM follows the same steps (each rank's own
                            shard first, then the shard each step brings).
                            0: pull, rank by rank (rank r's shards r+1,
                            r+2, ...), the GEMM rank by rank                 */
} tdg_ag_gemm_all_args;

TDG_API int tdg_ag_gemm_all_ranks(tdg_symm *h, const tdg_ag_gemm_all_args *args, void *stream,
                                  void *side_stream);

/* ---- GEMM + ReduceScatter -------------------------------------------------- */
/*
 * out_o = rows [o*Mo, (o+1)*Mo) of sum_r A_r @ B_r, Mo = M / W, for every
 * owner o ("Triton-distributed 语义", 内核设计模式 "GEMM + ReduceScatter 重叠";
 * paper summary, 方法: push-mode ReduceScatter, reduction in parallel,
 * synchronised by signals).
 *
 * A_r (M x K bf16) at region(r) + a_off, B_r (K x N, or N x K with
 * TDG_B_NK) at region(r) + b_off, out_o (Mo x N bf16) at region(o) + out_off.
 * Every rank's GEMM pushes each bf16 partial tile (BM x BN, tile-contiguous)
 * into the owner's staging area, region(o) + stage_off (see
 * tdg_gemm_rs_stage_bytes), then increments the owner's per-tile arrival
 * counter with release semantics.  The CTA whose increment completes the
 * count of W acquires it, sums the W partials in fixed rank order in fp32
 * and writes the bf16 result.  Each counter word carries the call's epoch
 * next to its count, so a count left by an earlier call (one that ended on
 * a fault) is ignored.  SERIAL mode runs the GEMM for all partials first
 * and the reduction after it.
 * partial_f32 = 1 pushes the partial tiles as fp32 instead of bf16: the
 * staging area is twice tdg_gemm_rs_stage_bytes(), and the only rounding is
 * the final one of the fp32 sum to bf16 (the published design leaves the
 * partial type open; bf16 is the default).
 * Requirements: M % W == 0, (M/W) % 128 == 0, K % 8 == 0, N % 8 == 0, the
 * offsets 16-byte aligned, 4*(M/W/128)*ceil(N/256) <= signals_per_rank
 * (one counter word per 32-row quarter of each of an owner's tiles),
 * partial_f32 0 or 1, and the staging area and out_o overlapping neither
 * each other nor A_r / B_r.  TDG_ERR_NOMEM when a buffer runs past its
 * region or the counter words are too few; TDG_ERR_INVALID for the rest.
 */
typedef struct {
    int world;
    int64_t M, K, N;
    size_t a_off, b_off, stage_off, out_off;
    int b_layout;
    int mode;            /* TDG_MODE_SM (overlapped) or TDG_MODE_SERIAL      */
    uint64_t timeout_ns; /* bound of every device wait; 0 = 2 s             */
    int owner_block;     /* tile order: owners per block, each rank's tiles of
                            a block back to back (must divide world; 0 =
                            world with bf16 partials, 2 with fp32 partials
                            (1 for an odd world))                            */
    int partial_f32;     /* 1: fp32 partials (twice the staging), 0: bf16     */
    /* schedule (0 = default for the shape) */
    int cluster;         /* CTAs per GEMM cluster: 1, 2 (needs (M/W) % 256
                            == 0) or 4 (needs (M/W) % 512 == 0); default the
                            largest the shape allows                         */
    int stages;          /* as in tdg_ag_gemm_args                            */
    int order;           /* 0: owner blocks (owner_block); 1: rank fastest   */
    int red_rows;        /* rows of an owed reduction an epilogue warp works
                            off after each tile: 4, 8, 16 or 32 (default 32
                            for bf16 partials, 4 for fp32); a warp holds up
                            to three owed quarters, and a fourth makes it
                            finish the oldest at once                        */
    int spare;           /* the SMs that 4-CTA clusters leave idle (order 0,
                            TDG_B_KN): a second launch of CTA pairs on them
                            takes the last `spare` of the W*W (owner block,
                            rank, owner) groups of tiles, starting as soon as
                            every CTA of the first launch runs.  0 = none
                            (default), at most W*W - 1; ignored where it
                            does not apply                                  */
} tdg_gemm_rs_args;

/* Bytes of one owner's staging area for the given shape (all W partials),
 * with bf16 partials; fp32 partials need twice as many. */
TDG_API size_t tdg_gemm_rs_stage_bytes(int world, int64_t M, int64_t N);

TDG_API int tdg_gemm_rs(tdg_symm *h, const tdg_gemm_rs_args *args, void *stream);

/* ---- ring AllReduce --------------------------------------------------------- */
/*
 * Tile-centric ring AllReduce over the W logical ranks ("Triton-distributed
 * 语义", 示例：带重叠的环形 AllReduce): a reduce-scatter ring (W-1 steps) followed
 * by an all-gather ring (W-1 steps); every tile of every step carries its own
 * signal, so a tile is reduced or forwarded as soon as it arrives.
 *
 * x_r (count float32) at region(r) + x_off is reduced in place: afterwards
 * every rank holds sum_r x_r.  Each buffer is split into W chunks of count/W;
 * at reduce-scatter step s rank r sends chunk (r - s) mod W to rank r+1, which
 * adds its own copy (local + incoming, float32) -- the textbook ring, since
 * the tile indices printed in the published example are inconsistent -- and at
 * all-gather step s rank r forwards chunk (r + 1 - s) mod W.
 * recv_r at region(r) + recv_off holds W-1 chunk-sized float32 slots
 * (tdg_allreduce_recv_bytes).  Signals: rank r's flag words
 * [0, (2W-2) * tiles_per_chunk).
 * Requirements: count % (4 * world) == 0, tile_elems % 4 == 0 (0 = default),
 * offsets 16-byte aligned, the receive slots not overlapping x, and no more
 * CTAs than can be resident at once (TDG_ERR_INVALID otherwise); x and the
 * receive slots inside their region and (2W-2) * ceil(count/W / tile_elems)
 * <= signals_per_rank (TDG_ERR_NOMEM otherwise).  count == 0 or world == 1
 * is a no-op.
 */
typedef struct {
    int world;
    int64_t count;       /* float32 elements per rank                          */
    size_t x_off;        /* data, reduced in place                             */
    size_t recv_off;     /* W-1 receive slots of count/W float32               */
    int64_t tile_elems;  /* elements per signalled tile (0 = 65536)            */
    int ctas_per_rank;   /* 0 = default                                        */
    uint64_t timeout_ns; /* bound of every device wait; 0 = 2 s                */
    uint64_t test_skip_signal; /* tests only: when nonzero, the notify of rank
                                  0's signal test_skip_signal - 1 is skipped,
                                  so rank 0's wait on it runs out            */
} tdg_allreduce_args;

TDG_API size_t tdg_allreduce_recv_bytes(int world, int64_t count);
TDG_API int tdg_allreduce(tdg_symm *h, const tdg_allreduce_args *args, void *stream);

/* ---- distributed flash decoding -------------------------------------------- */
/*
 * Decode attention with the KV cache split over the W logical ranks (paper
 * summary, 实验: distributed flash decoding; "Triton-distributed完全指南", §5.2).
 * out[b][h] = softmax_t(scale * q[b][h] . k_t) v_t over all S cached tokens,
 * kv head g = h / (Hq/Hkv).  Rank r holds tokens [r*S/W, (r+1)*S/W): K_r and
 * V_r (B x Hkv x S/W x D bf16) at region(r) + k_off / v_off.  Every CTA
 * reduces `chunk` tokens of one rank for one (batch, kv head) to a partial
 * (row max, row sum, normalised output, fp32) and pushes it into region(root)
 * + part_off; a second, stream-ordered launch on the root merges all partials
 * by log-sum-exp and writes out (bf16).
 * q, out: B x Hq x D bf16 device pointers.  Requirements: D == 128,
 * Hq % Hkv == 0, Hq/Hkv <= 16, B*Hkv <= 65535, S % world == 0, S > 0,
 * 0 <= root < world, chunk % 64 == 0 (0 = 2048 tokens), world *
 * ceil(S/world/chunk) <= 12000, offsets and pointers 16-byte aligned, the
 * partials overlapping neither K nor V (TDG_ERR_INVALID otherwise); K, V and
 * the partials (tdg_flash_decode_part_bytes) inside their regions
 * (TDG_ERR_NOMEM otherwise).
 */
typedef struct {
    int world, root;
    int64_t B, Hq, Hkv, D, S;
    size_t k_off, v_off, part_off;
    const void *q;
    void *out;
    int64_t chunk;
    float scale; /* 0 = 1/sqrt(D) */
} tdg_flash_decode_args;

TDG_API size_t tdg_flash_decode_part_bytes(int world, int64_t B, int64_t Hq, int64_t D, int64_t S,
                                           int64_t chunk);
TDG_API int tdg_flash_decode(tdg_symm *h, const tdg_flash_decode_args *args, void *stream);

/* ---- MoE dispatch / combine ------------------------------------------------ */
/*
 * Expert-parallel AllToAll as a permutation (paper summary, 实验: AllToAll
 * dispatch / combine; "Triton-distributed 正把通信纳入编译器的职责范围",
 * "DITRON 加入三级分块": per-expert sizes known only at run time).
 *
 * Rank src holds x_src (T x H bf16) at region(src) + x_off, its routing
 * topk_src (T x k int32 expert ids) at region(src) + topk_off and gates
 * (T x k float32) at region(src) + gate_off.  Experts are split evenly:
 * rank d owns experts [d*E/W, (d+1)*E/W).
 *
 * Routing (phase bit TDG_MOE_ROUTE): counts[src*E+e] (int64), the
 * expert-major exclusive scan base[0..E] (int64, base[E] = W*T*k) and
 * slot[(src*T+t)*k+kk] (int64): receive row of (src, t, kk); inside one
 * expert the rows follow (src, t, kk) order.  Optional row_src / row_tok /
 * row_k (int32 per receive row, may be NULL).
 * Dispatch (TDG_MOE_DISPATCH): recv[slot(src,t,kk)] = x_src[t] (bit copy).
 * recv is one expert-major array of W*T*k rows of H bf16; rank d's receive
 * buffer is rows [base[d*E/W], base[(d+1)*E/W]).
 * Combine (TDG_MOE_COMBINE): out_src[t] = bf16(sum_kk gate[t][kk] *
 * y[slot(src,t,kk)]) with an fp32 sum in kk order, written to region(src) +
 * out_off.  y has the receive layout; y == NULL means y = recv.
 * workspace: device scratch of tdg_moe_workspace_bytes() bytes.
 * Requirements: E % W == 0, E <= 4096, 1 <= k <= 32, k <= E, H % 8 == 0,
 * W*T*k < 2^31, phases a nonzero OR of the bits; x_off, out_off, recv and y
 * 16-byte aligned, topk_off and gate_off 4-byte aligned; slot always, counts
 * and base when routing, recv when dispatching (or combining with y NULL);
 * row_src / row_tok / row_k all or none; when combining, out not
 * overlapping the gates (TDG_ERR_INVALID otherwise).  The
 * per-rank inputs inside their region and, when routing, a workspace of
 * tdg_moe_workspace_bytes() (TDG_ERR_NOMEM otherwise).  T == 0 is a no-op.
 * An expert id outside [0, E) is reported as TDG_ERR_DEVICE by tdg_status
 * and that (t, kk) gets slot -1.
 */
#define TDG_MOE_ROUTE 1
#define TDG_MOE_DISPATCH 2
#define TDG_MOE_COMBINE 4
#define TDG_MOE_ALL 7

typedef struct {
    int world;
    int64_t T;
    int64_t H;
    int E, k;
    size_t x_off, topk_off, gate_off, out_off;
    void *recv;
    const void *y;
    int64_t *counts, *base, *slot;
    int32_t *row_src, *row_tok, *row_k;
    void *workspace;
    size_t workspace_bytes;
    int phases; /* OR of TDG_MOE_ROUTE / DISPATCH / COMBINE */
} tdg_moe_args;

TDG_API size_t tdg_moe_workspace_bytes(int world, int64_t T, int E);

TDG_API int tdg_moe_dispatch_combine(tdg_symm *h, const tdg_moe_args *args, void *stream);

/*
 * Allocation-free variant of tdg_moe_dispatch_combine.  The published design
 * has no counterpart: this entry point exists for callers that cannot allocate
 * device memory at the moment they call -- for example code running inside
 * a memory-budgeted runtime or a pool that forbids cudaMalloc after start-up,
 * or a caller with no allocator of its own -- and so cannot hand over the
 * routing workspace.
 *
 * It behaves exactly like tdg_moe_dispatch_combine, except that args->workspace
 * and args->workspace_bytes are ignored: the routing scratch (two int32 tables
 * of W * ceil(T/64) * E entries) lives in a fixed device array inside the
 * library, TDG_MOE_STATIC_WORKSPACE_BYTES (2 MiB) in size, which every GPU that
 * loads the library keeps until the process exits.  Inputs and outputs are
 * still the caller's.  Nothing is allocated or freed by this call.
 *   - Arguments are checked first, exactly as tdg_moe_dispatch_combine does
 *     (the same TDG_ERR_INVALID / TDG_ERR_NOMEM codes).  Then it returns
 *     TDG_ERR_NOMEM, launching nothing, when the routing phase is requested
 *     and tdg_moe_workspace_bytes(world, T, E) exceeds 2 MiB (that is, when
 *     W * ceil(T/64) * E > 262144).
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it for that device's context; a context
 *     created anew (after cudaDeviceReset) looks it up again on its first
 *     call.  Make that first call before any stream capture.
 *   - All calls on one device share the array and it keeps the last call's
 *     contents; nothing in it needs to start at zero (every entry a call reads
 *     is written earlier in the same call).  Calls that overlap on the GPU
 *     (for example on two streams at once) race on it: serialise them.
 */
#define TDG_MOE_STATIC_WORKSPACE_BYTES (2u * 1024u * 1024u)
TDG_API int tdg_moe_dispatch_combine_noalloc(tdg_symm *h, const tdg_moe_args *args, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TDG_H_ */
