/*
 * tdg_oracle.c -- the CPU oracle for the tile-centric overlapped
 * AllGather+GEMM, GEMM+ReduceScatter and MoE dispatch/combine path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library under tile_centric_comm_gb300/) never calls it, links it
 * or shares a line of code with it.
 *
 * Every function here is the plain definition of what the method computes,
 * written as explicit loops in double precision with no blocking, fusion or
 * reordering beyond what the definition states.  A reader can check each
 * loop nest against the passage it cites:
 *
 *   [P1 方法]    "Triton-distributed" paper summary (hyper.ai, arXiv 2504.19442),
 *                section 方法 (method): symmetric memory, signal exchange,
 *                intra-node AllGather / push-mode ReduceScatter, and the
 *                low-latency (LL) protocol with data and flag in one 8-byte word.
 *   [P1 实验]    same page, section 实验 (experiments): expert-parallel
 *                AllToAll dispatch / combine.
 *   [P2 AG+GEMM] "Triton-distributed 语义" (triton-distributed-ascend docs),
 *                section 内核设计模式, "AllGather + GEMM 重叠".
 *   [P2 GEMM+RS] same page, "GEMM + ReduceScatter 重叠".
 *   [P2 交织]    same page, section 线程块交织 (threadblock swizzle).
 *   [P4 DITRON]  "Triton-distributed 正把通信纳入编译器的职责范围" (cronfeed),
 *                section "DITRON 加入三级分块": per-expert token counts are
 *                only known at run time.
 *
 * Readings where the cited pages are silent (each one is listed with its reason in
 * the design notes of this repository):
 *   - bf16 is IEEE-754 binary16-brain (1 sign, 8 exponent, 7 fraction bits);
 *     outputs are rounded once, from the exact double-precision sum, to the
 *     nearest bf16 value with ties to even.
 *   - AllGather concatenates the W shards along rows, in rank order.
 *   - ReduceScatter gives owner o the rows [o*M/W, (o+1)*M/W) of the sum of
 *     the W partial products.
 *   - MoE receive rows are expert-major; inside one expert the rows are in
 *     (source rank, token) order; rank d owns experts [d*E/W, (d+1)*E/W).
 *   - combine: out[src][t] = sum over k of gate[src][t][k] * y[slot(src,t,k)].
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (OpenMP only parallelises the
 * independent output rows; every sum is still taken in the order written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* bf16 <-> double                                                          */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern -> double (exact: every bf16 value is a double). */
ORC_EXPORT double orc_bf16_to_f64(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * double -> bf16 bit pattern, round to nearest, ties to even (IEEE 754
 * roundTiesToEven), applied once to the exact double value.
 *
 * bf16 carries 8 significant bits.  For |x| = m * 2^e with m in [0.5, 1)
 * (frexp), the spacing of bf16 values around x is 2^(e-8); below the
 * smallest normal (2^-126) the spacing is fixed at 2^-133.  Scaling by a
 * power of two is exact, so nearbyint() on the scaled value (default
 * rounding mode: to nearest, ties to even) performs exactly one rounding.
 * Values that round past the largest finite bf16 become infinity.
 */
ORC_EXPORT uint16_t orc_f64_to_bf16(double x)
{
    if (isnan(x))
        return (uint16_t)0x7FC0u;
    uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0u;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    int e = 0;
    (void)frexp(a, &e);
    int ulp_exp = e - 8;
    if (ulp_exp < -133)
        ulp_exp = -133;
    double r = nearbyint(ldexp(a, -ulp_exp));
    double v = ldexp(r, ulp_exp);
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (v > bf16_max)
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)v; /* exact: v has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)((bits >> 16) & 0x7FFFu));
}

ORC_EXPORT void orc_f64_to_bf16_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f64_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* AllGather + GEMM                                                          */
/* ------------------------------------------------------------------------ */

/*
 * [P2 AG+GEMM], [P1 方法]: the producer gathers every rank's shard of A and
 * the consumer multiplies the gathered matrix by B.  The overlap, the tile
 * order and the signals do not change the result, so the oracle is the
 * definition itself:
 *
 *   G = concat_rows(A_0, ..., A_{W-1})          (M = W*Ms rows, K columns)
 *   C[i][j] = sum_{k=0}^{K-1} G[i][k] * B[k][j]  (exact in double for the
 *                                                 sizes used; one rounding)
 *
 * A[s] points to shard s, Ms x K row-major bf16.  B is K x N row-major bf16.
 * Outputs: C64 (M x N double, may be NULL) and C16 (M x N bf16, may be NULL).
 */
ORC_EXPORT void orc_ag_gemm(int W, int64_t Ms, int64_t K, int64_t N,
                            const uint16_t *const *A, const uint16_t *B,
                            double *C64, uint16_t *C16)
{
    const int64_t M = (int64_t)W * Ms;
    /* the AllGather: row i of G is row (i mod Ms) of shard (i div Ms) */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        const uint16_t *g_row = A[i / Ms] + (i % Ms) * K;
        for (int64_t j = 0; j < N; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += orc_bf16_to_f64(g_row[k]) * orc_bf16_to_f64(B[k * N + j]);
            if (C64)
                C64[i * N + j] = s;
            if (C16)
                C16[i * N + j] = orc_f64_to_bf16(s);
        }
    }
}

/* Same definition, evaluated only at the n given (row, col) positions. */
ORC_EXPORT void orc_ag_gemm_sampled(int W, int64_t Ms, int64_t K, int64_t N,
                                    const uint16_t *const *A, const uint16_t *B,
                                    int64_t n, const int64_t *rows,
                                    const int64_t *cols, double *out64)
{
    (void)W;
#pragma omp parallel for schedule(static)
    for (int64_t q = 0; q < n; ++q) {
        const int64_t i = rows[q], j = cols[q];
        const uint16_t *g_row = A[i / Ms] + (i % Ms) * K;
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += orc_bf16_to_f64(g_row[k]) * orc_bf16_to_f64(B[k * N + j]);
        out64[q] = s;
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM + ReduceScatter                                                      */
/* ------------------------------------------------------------------------ */

/*
 * [P2 GEMM+RS], [P1 方法] (push-mode ReduceScatter): every rank r produces
 * the partial product P_r = A_r * B_r (M x N); the ReduceScatter sums the W
 * partials and gives owner o the rows [o*Mo, (o+1)*Mo), Mo = M / W:
 *
 *   out_o[i][j] = sum_{r=0}^{W-1} sum_{k=0}^{K-1} A_r[o*Mo+i][k] * B_r[k][j]
 *
 * A[r]: M x K row-major bf16, B[r]: K x N row-major bf16.
 * out64 / out16: W blocks of Mo x N (owner-major), either may be NULL.
 */
ORC_EXPORT void orc_gemm_rs(int W, int64_t M, int64_t K, int64_t N,
                            const uint16_t *const *A, const uint16_t *const *B,
                            double *out64, uint16_t *out16)
{
    const int64_t Mo = M / W;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t row = 0; row < M; ++row) {
        const int64_t o = row / Mo, i = row % Mo;
        for (int64_t j = 0; j < N; ++j) {
            double s = 0.0;
            for (int r = 0; r < W; ++r) {
                double p = 0.0; /* the partial of rank r */
                for (int64_t k = 0; k < K; ++k)
                    p += orc_bf16_to_f64(A[r][row * K + k]) *
                         orc_bf16_to_f64(B[r][k * N + j]);
                s += p;
            }
            const int64_t at = (o * Mo + i) * N + j;
            if (out64)
                out64[at] = s;
            if (out16)
                out16[at] = orc_f64_to_bf16(s);
        }
    }
}

/* Same definition at n sampled (global row, col) positions of the output. */
ORC_EXPORT void orc_gemm_rs_sampled(int W, int64_t M, int64_t K, int64_t N,
                                    const uint16_t *const *A,
                                    const uint16_t *const *B, int64_t n,
                                    const int64_t *rows, const int64_t *cols,
                                    double *out64)
{
    (void)M;
#pragma omp parallel for schedule(static)
    for (int64_t q = 0; q < n; ++q) {
        const int64_t row = rows[q], j = cols[q];
        double s = 0.0;
        for (int r = 0; r < W; ++r) {
            double p = 0.0;
            for (int64_t k = 0; k < K; ++k)
                p += orc_bf16_to_f64(A[r][row * K + k]) *
                     orc_bf16_to_f64(B[r][k * N + j]);
            s += p;
        }
        out64[q] = s;
    }
}

/* Partial product of one rank, P_r = A_r * B_r (M x N double). */
ORC_EXPORT void orc_gemm_partial(int64_t M, int64_t K, int64_t N,
                                 const uint16_t *A, const uint16_t *B,
                                 double *P)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += orc_bf16_to_f64(A[i * K + k]) * orc_bf16_to_f64(B[k * N + j]);
            P[i * N + j] = s;
        }
}

/* ------------------------------------------------------------------------ */
/* MoE dispatch / combine                                                    */
/* ------------------------------------------------------------------------ */

/*
 * [P1 实验] expert-parallel AllToAll, [P4 DITRON] per-expert sizes known
 * only at run time.  Routing metadata as an explicit per-token loop.
 *
 * topk: W x T x KK expert ids (each in [0, E)).  Outputs:
 *   counts[src*E + e] : number of (t, k) of rank src routed to expert e
 *   base[e]           : first receive row of expert e (E+1 entries; base[E]
 *                       is the total row count) -- expert-major exclusive scan
 *   off[src*E + e]    : rows of expert e that come from ranks before src
 *   slot[(src*T+t)*KK+k] = base[e] + off[src][e]
 *                          + #{ earlier (t', k') of src, in (t, k) order,
 *                               routed to e }
 *   row_src / row_tok / row_k : inverse map, one entry per receive row.
 * Returns 0, or -1 if an expert id is out of range (nothing is written then).
 */
ORC_EXPORT int orc_moe_route(int W, int64_t T, int KK, int E,
                             const int32_t *topk, int64_t *counts,
                             int64_t *base, int64_t *off, int64_t *slot,
                             int32_t *row_src, int32_t *row_tok,
                             int32_t *row_k)
{
    for (int64_t q = 0; q < (int64_t)W * T * KK; ++q)
        if (topk[q] < 0 || topk[q] >= E)
            return -1;
    /* 1. histogram */
    memset(counts, 0, sizeof(int64_t) * (size_t)W * (size_t)E);
    for (int src = 0; src < W; ++src)
        for (int64_t t = 0; t < T; ++t)
            for (int k = 0; k < KK; ++k)
                counts[(int64_t)src * E + topk[((int64_t)src * T + t) * KK + k]] += 1;
    /* 2. expert-major exclusive scan */
    int64_t running = 0;
    for (int e = 0; e < E; ++e) {
        base[e] = running;
        for (int src = 0; src < W; ++src) {
            off[(int64_t)src * E + e] = running - base[e];
            running += counts[(int64_t)src * E + e];
        }
    }
    base[E] = running;
    /* 3. second pass in the same loop order assigns the slots */
    int64_t *cursor = (int64_t *)calloc((size_t)W * (size_t)E, sizeof(int64_t));
    if (!cursor)
        return -2;
    for (int src = 0; src < W; ++src)
        for (int64_t t = 0; t < T; ++t)
            for (int k = 0; k < KK; ++k) {
                const int64_t q = ((int64_t)src * T + t) * KK + k;
                const int e = topk[q];
                const int64_t s = base[e] + off[(int64_t)src * E + e] +
                                  cursor[(int64_t)src * E + e]++;
                slot[q] = s;
                if (row_src) row_src[s] = src;
                if (row_tok) row_tok[s] = (int32_t)t;
                if (row_k) row_k[s] = k;
            }
    free(cursor);
    return 0;
}

/* Dispatch: recv[slot(src,t,k)] = x[src][t] (rows of H bf16, bit copy). */
ORC_EXPORT void orc_moe_dispatch(int W, int64_t T, int KK, int64_t H,
                                 const uint16_t *x, const int64_t *slot,
                                 uint16_t *recv)
{
    for (int src = 0; src < W; ++src)
        for (int64_t t = 0; t < T; ++t)
            for (int k = 0; k < KK; ++k) {
                const int64_t s = slot[((int64_t)src * T + t) * KK + k];
                memcpy(recv + s * H, x + ((int64_t)src * T + t) * H,
                       sizeof(uint16_t) * (size_t)H);
            }
}

/*
 * Combine: out[src][t][h] = bf16( sum_{k=0}^{KK-1} gate[src][t][k] *
 *                                 y[slot(src,t,k)][h] ), sum in double.
 * y has the receive layout (one row per slot).  gate is float32.
 */
ORC_EXPORT void orc_moe_combine(int W, int64_t T, int KK, int64_t H,
                                const uint16_t *y, const int64_t *slot,
                                const float *gate, uint16_t *out16,
                                double *out64)
{
#pragma omp parallel for schedule(static)
    for (int64_t st = 0; st < (int64_t)W * T; ++st)
        for (int64_t h = 0; h < H; ++h) {
            double s = 0.0;
            for (int k = 0; k < KK; ++k) {
                const int64_t q = st * KK + k;
                s += (double)gate[q] * orc_bf16_to_f64(y[slot[q] * H + h]);
            }
            if (out16)
                out16[st * H + h] = orc_f64_to_bf16(s);
            if (out64)
                out64[st * H + h] = s;
        }
}

/* ------------------------------------------------------------------------ */
/* Low-latency (LL) words and the threadblock swizzle                        */
/* ------------------------------------------------------------------------ */

/*
 * [P1 方法] LL protocol: data and flag share one 8-byte block.  Reading:
 * word = payload (low 32 bits) | flag (high 32 bits), flag = the call's
 * nonzero epoch.  pack: n payload words -> n LL words.
 */
ORC_EXPORT void orc_ll_pack(const uint32_t *payload, int64_t n, uint32_t flag,
                            uint64_t *words)
{
    for (int64_t i = 0; i < n; ++i)
        words[i] = (uint64_t)payload[i] | ((uint64_t)flag << 32);
}

/* unpack: returns the number of words whose flag differs from `flag`
 * (those payloads are not written). */
ORC_EXPORT int64_t orc_ll_unpack(const uint64_t *words, int64_t n,
                                 uint32_t flag, uint32_t *payload)
{
    int64_t missing = 0;
    for (int64_t i = 0; i < n; ++i) {
        if ((uint32_t)(words[i] >> 32) != flag) {
            ++missing;
            continue;
        }
        payload[i] = (uint32_t)(words[i] & 0xFFFFFFFFu);
    }
    return missing;
}

/*
 * [P2 交织] threadblock swizzle: pid_m = (pid_m + rank * tiles_per_pe) %
 * total_tiles.  Writes, for linear tile ids 0 .. total_m*n_tiles-1 taken in
 * m-major order (all n tiles of one m row before the next), the swizzled
 * (pid_m, pid_n) pair.
 */
ORC_EXPORT void orc_swizzle_order(int rank, int64_t tiles_per_pe,
                                  int64_t total_m, int64_t n_tiles,
                                  int64_t *pid_m_out, int64_t *pid_n_out)
{
    for (int64_t id = 0; id < total_m * n_tiles; ++id) {
        const int64_t pid_m = id / n_tiles, pid_n = id % n_tiles;
        pid_m_out[id] = (pid_m + (int64_t)rank * tiles_per_pe) % total_m;
        pid_n_out[id] = pid_n;
    }
}

/* ------------------------------------------------------------------------ */
/* AllReduce                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * "Triton-distributed 语义", 示例：带重叠的环形 AllReduce: after the ring's
 * reduce-scatter and all-gather phases every rank holds the element-wise sum
 * of all ranks' buffers.  The oracle is that sum:
 *
 *   out[i] = sum_{r=0}^{W-1} x_r[i]      (double precision, rank order)
 *
 * x[r] points to rank r's buffer of n float32 values; out has n doubles.
 */
ORC_EXPORT void orc_allreduce(int W, int64_t n, const float *const *x, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int r = 0; r < W; ++r)
            s += (double)x[r][i];
        out[i] = s;
    }
}

/* ------------------------------------------------------------------------ */
/* Decode attention (the distributed flash-decoding workload)                */
/* ------------------------------------------------------------------------ */

/*
 * Paper summary (hyper.ai, arXiv 2504.19442), section 实验: distributed flash
 * decoding over long KV caches; "Triton-distributed完全指南", §5.2 (Fig. 5):
 * flash-decode scaling over GPU count and KV length.  Splitting the KV cache
 * over ranks and merging the partial results changes only the rounding, so the
 * oracle is plain softmax attention of one query token over the whole cache:
 *
 *   s_t = scale * sum_d q[b][h][d] * k[b][g][t][d],   g = h / (Hq / Hkv)
 *   out[b][h][d] = sum_t exp(s_t - max_t s) * v[b][g][t][d] / sum_t exp(s_t - max_t s)
 *
 * q: B x Hq x D, k and v: B x Hkv x S x D (bf16 bits); out64: B x Hq x D.
 */
ORC_EXPORT void orc_attention_decode(int64_t B, int64_t Hq, int64_t Hkv, int64_t D, int64_t S,
                                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                     double scale, double *out64)
{
    const int64_t G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * Hq; ++bh) {
        const int64_t b = bh / Hq, h = bh % Hq, g = h / G;
        const uint16_t *qq = q + (b * Hq + h) * D;
        const uint16_t *kk = k + (b * Hkv + g) * S * D;
        const uint16_t *vv = v + (b * Hkv + g) * S * D;
        double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        double mx = -INFINITY;
        for (int64_t t = 0; t < S; ++t) {
            double a = 0.0;
            for (int64_t d = 0; d < D; ++d)
                a += orc_bf16_to_f64(qq[d]) * orc_bf16_to_f64(kk[t * D + d]);
            s[t] = scale * a;
            if (s[t] > mx)
                mx = s[t];
        }
        double den = 0.0;
        for (int64_t t = 0; t < S; ++t) {
            s[t] = exp(s[t] - mx);
            den += s[t];
        }
        for (int64_t d = 0; d < D; ++d) {
            double num = 0.0;
            for (int64_t t = 0; t < S; ++t)
                num += s[t] * orc_bf16_to_f64(vv[t * D + d]);
            out64[bh * D + d] = num / den;
        }
        free(s);
    }
}
