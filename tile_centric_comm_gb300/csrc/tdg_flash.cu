// tdg_flash.cu -- distributed flash decoding over W logical ranks (paper
// summary, 实验: distributed flash decoding; "Triton-distributed完全指南" §5.2).
//
// The KV cache is split by tokens over the ranks.  CTA (j, b, g) reduces
// `chunk` tokens of rank j / splits_per_rank for batch b and kv head g: its 4
// warps walk 16-token groups, staged through shared memory with cp.async
// (double buffered), compute S = Q K^T and O += P V with bf16 mma.sync
// (m16n8k16, fp32 accumulate; the G = Hq/Hkv query heads of the kv head are
// the M rows) and keep an online softmax in fp32 (base-2 exponent).  The warps
// merge in shared memory; the CTA pushes (max, sum, normalised output) into
// the root rank's partial buffer.  A second, stream-ordered launch on the root
// merges every partial by log-sum-exp (one CTA per (batch, query head), one
// thread per dimension) and writes the bf16 output.  Nothing spins.
// Decode attention is bound by HBM (about 8 FLOP per cached byte), so the
// register-level mma.sync suffices for the arithmetic.
#include "tdg_internal.h"

namespace tdg {

namespace fd {
constexpr int D = 128;
constexpr int WARPS = 4;
constexpr int GT = 16;                 // tokens per warp group
constexpr int ROW = D + 8;             // smem row pitch in bf16 (272 B, conflict-free ldmatrix)
constexpr int BUF = GT * ROW;          // one 16-token tile, elements
constexpr int WARP_SMEM = 2 * 2 * BUF; // K and V, double buffered
constexpr int SMEM = WARPS * WARP_SMEM * 2;
} // namespace fd

struct FlashParams {
    int W, G, splits; // splits per rank
    int64_t B, Hq, Hkv, S, Sr, chunk;
    float scale_log2;
    const uint8_t *regions;
    uint64_t region_bytes;
    uint64_t k_off, v_off;
    float *part_o;  // [W*splits][B][Hq][D]
    float *part_ml; // [W*splits][B][Hq][2]
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t ld_u32_bf16pair(const __nv_bfloat16 *p)
{
    return *reinterpret_cast<const uint32_t *>(p);
}

// stage one 16-token tile of K and V (rows beyond n_valid are zero-filled)
__device__ __forceinline__ void fd_stage(const __nv_bfloat16 *kg, const __nv_bfloat16 *vg, int n_valid,
                                         uint32_t ks, uint32_t vs, int lane)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i; // 256 pieces of 16 B per tile
        const int tok = e >> 4, piece = e & 15;
        const bool ok = tok < n_valid;
        const size_t go = ok ? (size_t)tok * fd::D + piece * 8 : 0;
        const uint32_t so = (uint32_t)(tok * fd::ROW + piece * 8) * 2;
        cp_async16(ks + so, kg + go, ok ? 16u : 0u);
        cp_async16(vs + so, vg + go, ok ? 16u : 0u);
    }
}

__global__ void __launch_bounds__(fd::WARPS * 32) flash_decode_kernel(const __grid_constant__ FlashParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __nv_bfloat16 *sm = reinterpret_cast<__nv_bfloat16 *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int j = blockIdx.x;                       // global split
    const int b = (int)(blockIdx.y / p.Hkv), g = (int)(blockIdx.y % p.Hkv);
    const int rank = j / p.splits, lsplit = j % p.splits;
    const int64_t t0 = (int64_t)lsplit * p.chunk;
    const int64_t t1 = min(p.Sr, t0 + p.chunk);
    const size_t kv_head = ((size_t)b * p.Hkv + g) * (size_t)p.Sr * fd::D;
    const __nv_bfloat16 *K = reinterpret_cast<const __nv_bfloat16 *>(p.regions + (uint64_t)rank * p.region_bytes + p.k_off) + kv_head;
    const __nv_bfloat16 *V = reinterpret_cast<const __nv_bfloat16 *>(p.regions + (uint64_t)rank * p.region_bytes + p.v_off) + kv_head;

    // Q fragments (A operand, rows = the G query heads, zero beyond G)
    uint32_t qa[8][4];
    const __nv_bfloat16 *Q = p.q + ((size_t)b * p.Hq + (size_t)g * p.G) * fd::D;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int c = ks * 16 + tig * 2;
        qa[ks][0] = gid < p.G ? ld_u32_bf16pair(Q + gid * fd::D + c) : 0u;
        qa[ks][1] = gid + 8 < p.G ? ld_u32_bf16pair(Q + (gid + 8) * fd::D + c) : 0u;
        qa[ks][2] = gid < p.G ? ld_u32_bf16pair(Q + gid * fd::D + c + 8) : 0u;
        qa[ks][3] = gid + 8 < p.G ? ld_u32_bf16pair(Q + (gid + 8) * fd::D + c + 8) : 0u;
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n)
        o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    __nv_bfloat16 *wsm = sm + warp * fd::WARP_SMEM;
    const uint32_t wbase = smem_u32(wsm);
    const int64_t ngroups = (t1 - t0 + fd::GT - 1) / fd::GT;
    // this warp takes groups warp, warp + WARPS, ...
    int64_t grp = warp;
    if (grp < ngroups) {
        const int64_t tt = t0 + grp * fd::GT;
        fd_stage(K + tt * fd::D, V + tt * fd::D, (int)min((int64_t)fd::GT, t1 - tt), wbase, wbase + fd::BUF * 2, lane);
    }
    cp_async_commit();
    int buf = 0;
    for (; grp < ngroups; grp += fd::WARPS) {
        const int64_t nxt = grp + fd::WARPS;
        if (nxt < ngroups) {
            const int64_t tt = t0 + nxt * fd::GT;
            const uint32_t kb = wbase + (uint32_t)((buf ^ 1) * 2 * fd::BUF) * 2;
            fd_stage(K + tt * fd::D, V + tt * fd::D, (int)min((int64_t)fd::GT, t1 - tt), kb, kb + fd::BUF * 2, lane);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        const uint32_t ks_base = wbase + (uint32_t)(buf * 2 * fd::BUF) * 2;
        const uint32_t vs_base = ks_base + fd::BUF * 2;
        const int64_t tt = t0 + grp * fd::GT;
        const int nval = (int)min((int64_t)fd::GT, t1 - tt);

        // S = Q K^T: two n8 tiles (tokens 0-7, 8-15), eight k steps of 16 dims
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int tok = (mi >= 2 ? 8 : 0) + ri;
            const int dim = ks * 16 + (mi & 1) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ks_base + (uint32_t)(tok * fd::ROW + dim) * 2, b0, b1, b2, b3);
            mma_bf16_16816(s[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
            mma_bf16_16816(s[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
        // scale to the base-2 domain and mask tokens past the chunk's end
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int tok = nt * 8 + tig * 2 + (c & 1);
                s[nt][c] = tok < nval ? s[nt][c] * p.scale_log2 : -INFINITY;
            }
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2f(m0 - ms0), al1 = exp2f(m1 - ms1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            s[nt][0] = exp2f(s[nt][0] - ms0);
            s[nt][1] = exp2f(s[nt][1] - ms0);
            s[nt][2] = exp2f(s[nt][2] - ms1);
            s[nt][3] = exp2f(s[nt][3] - ms1);
            ps0 += s[nt][0] + s[nt][1];
            ps1 += s[nt][2] + s[nt][3];
        }
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            o[n][0] *= al0;
            o[n][1] *= al0;
            o[n][2] *= al1;
            o[n][3] *= al1;
        }
        // P as the A operand (the accumulator layout of two n8 tiles)
        const uint32_t pa0 = pack_bf16x2(s[0][0], s[0][1]);
        const uint32_t pa1 = pack_bf16x2(s[0][2], s[0][3]);
        const uint32_t pa2 = pack_bf16x2(s[1][0], s[1][1]);
        const uint32_t pa3 = pack_bf16x2(s[1][2], s[1][3]);
        // O += P V: 16 n8 tiles of dims, one k step of 16 tokens
#pragma unroll
        for (int nd = 0; nd < 16; nd += 2) {
            const int tok = (mi & 1) * 8 + ri;
            const int dim = (nd + (mi >> 1)) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vs_base + (uint32_t)(tok * fd::ROW + dim) * 2, b0, b1, b2, b3);
            mma_bf16_16816(o[nd], pa0, pa1, pa2, pa3, b0, b1);
            mma_bf16_16816(o[nd + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
        __syncwarp();
        buf ^= 1;
    }
    cp_async_wait<0>();
    __syncthreads();

    // merge the warps: each writes (m, l, o) rows g and g+8 to shared memory
    float *ms = reinterpret_cast<float *>(smem_raw);          // [WARPS][16]
    float *ls = ms + fd::WARPS * 16;                          // [WARPS][16]
    float *os = ls + fd::WARPS * 16;                          // [WARPS][16][D]
    if (tig == 0) {
        ms[warp * 16 + gid] = m0;
        ms[warp * 16 + gid + 8] = m1;
        ls[warp * 16 + gid] = l0;
        ls[warp * 16 + gid + 8] = l1;
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int c = n * 8 + tig * 2;
        os[(warp * 16 + gid) * fd::D + c] = o[n][0];
        os[(warp * 16 + gid) * fd::D + c + 1] = o[n][1];
        os[(warp * 16 + gid + 8) * fd::D + c] = o[n][2];
        os[(warp * 16 + gid + 8) * fd::D + c + 1] = o[n][3];
    }
    __syncthreads();
    const size_t part_row0 = ((size_t)j * p.B + b) * p.Hq + (size_t)g * p.G;
    for (int idx = threadIdx.x; idx < p.G * fd::D; idx += blockDim.x) {
        const int h = idx / fd::D, d = idx % fd::D;
        float M = -INFINITY;
        for (int w = 0; w < fd::WARPS; ++w)
            M = fmaxf(M, ms[w * 16 + h]);
        const float Ms = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
        for (int w = 0; w < fd::WARPS; ++w) {
            const float e = exp2f(ms[w * 16 + h] - Ms);
            L += ls[w * 16 + h] * e;
            O += os[(w * 16 + h) * fd::D + d] * e;
        }
        __stcg(p.part_o + (part_row0 + h) * fd::D + d, L > 0.f ? O / L : 0.f);
        if (d == 0) {
            __stcg(p.part_ml + (part_row0 + h) * 2, M);
            __stcg(p.part_ml + (part_row0 + h) * 2 + 1, L);
        }
    }
}

// The root merges every split's partial by log-sum-exp: one CTA per
// (batch, query head), one thread per output dimension.  The split weights
// l_j * 2^(m_j - M) are computed once per CTA in shared memory.
__global__ void __launch_bounds__(fd::D) flash_combine_kernel(const __grid_constant__ FlashParams p)
{
    extern __shared__ float wsh[]; // [nsplit] weights, then [32] reduction scratch
    const size_t row = blockIdx.x; // b * Hq + h
    const int nsplit = p.W * p.splits;
    const size_t stride = (size_t)p.B * p.Hq;
    float mloc = -INFINITY;
    for (int j = threadIdx.x; j < nsplit; j += blockDim.x)
        mloc = fmaxf(mloc, __ldcg(p.part_ml + ((size_t)j * stride + row) * 2));
    float *red = wsh + nsplit;
    for (int o = 16; o > 0; o >>= 1)
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = mloc;
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
        M = fmaxf(M, red[w]);
    const float Ms = M == -INFINITY ? 0.f : M;
    for (int j = threadIdx.x; j < nsplit; j += blockDim.x) {
        const size_t pr = (size_t)j * stride + row;
        wsh[j] = __ldcg(p.part_ml + pr * 2 + 1) * exp2f(__ldcg(p.part_ml + pr * 2) - Ms);
    }
    __syncthreads();
    const int d = threadIdx.x;
    float L = 0.f, O = 0.f;
    int j = 0;
    for (; j + 8 <= nsplit; j += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            v[u] = __ldcg(p.part_o + ((size_t)(j + u) * stride + row) * fd::D + d);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            L += wsh[j + u];
            O += v[u] * wsh[j + u];
        }
    }
    for (; j < nsplit; ++j) {
        L += wsh[j];
        O += __ldcg(p.part_o + ((size_t)j * stride + row) * fd::D + d) * wsh[j];
    }
    p.out[row * fd::D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
}

} // namespace tdg

using namespace tdg;
using namespace tdg_host;

namespace {
int64_t fd_chunk(int64_t c) { return c > 0 ? c : 2048; }
} // namespace

extern "C" size_t tdg_flash_decode_part_bytes(int world, int64_t B, int64_t Hq, int64_t D, int64_t S,
                                              int64_t chunk)
{
    if (world <= 0 || B <= 0 || Hq <= 0 || D <= 0 || S <= 0 || S % world)
        return 0;
    const int64_t Sr = S / world, c = fd_chunk(chunk);
    const int64_t splits = (Sr + c - 1) / c;
    return (size_t)world * splits * B * Hq * (D + 2) * sizeof(float);
}

extern "C" int tdg_flash_decode(tdg_symm *h, const tdg_flash_decode_args *a, void *stream)
{
    if (!h || !a)
        return TDG_ERR_INVALID;
    if (const int drc = check_device(h))
        return drc;
    const int W = a->world;
    if (W != h->world || a->root < 0 || a->root >= W || a->B <= 0 || a->Hq <= 0 || a->Hkv <= 0 ||
        a->D != fd::D || a->S <= 0 || a->S % W || a->Hq % a->Hkv || a->Hq / a->Hkv > 16)
        return TDG_ERR_INVALID;
    const int64_t chunk = fd_chunk(a->chunk);
    if (chunk % 64 || !a->q || !a->out || !aligned16(a->q) || !aligned16(a->out) || !aligned16(a->k_off) ||
        !aligned16(a->v_off) || !aligned16(a->part_off))
        return TDG_ERR_INVALID;
    const int64_t Sr = a->S / W, splits = (Sr + chunk - 1) / chunk;
    const uint64_t kv_bytes = (uint64_t)a->B * a->Hkv * Sr * fd::D * 2;
    const size_t part = tdg_flash_decode_part_bytes(W, a->B, a->Hq, a->D, a->S, chunk);
    const uint64_t R = h->region_bytes;
    if (a->k_off + kv_bytes > R || a->v_off + kv_bytes > R || a->part_off + part > R)
        return TDG_ERR_NOMEM;
    // the partials (written) overlap neither K nor V
    if ((a->part_off < a->k_off + kv_bytes && a->k_off < a->part_off + part) ||
        (a->part_off < a->v_off + kv_bytes && a->v_off < a->part_off + part))
        return TDG_ERR_INVALID;
    if (a->B * a->Hkv > 65535 || (int64_t)W * splits * 4 + 128 > 48 * 1024)
        return TDG_ERR_INVALID;
    FlashParams p;
    memset(&p, 0, sizeof p);
    p.W = W;
    p.G = (int)(a->Hq / a->Hkv);
    p.splits = (int)splits;
    p.B = a->B;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.S = a->S;
    p.Sr = Sr;
    p.chunk = chunk;
    const float scale = a->scale > 0.f ? a->scale : 1.0f / sqrtf((float)fd::D);
    p.scale_log2 = scale * 1.4426950408889634f; // log2(e): scores live in the base-2 domain
    p.regions = h->base;
    p.region_bytes = R;
    p.k_off = a->k_off;
    p.v_off = a->v_off;
    uint8_t *root = h->base + (uint64_t)a->root * R + a->part_off;
    p.part_o = reinterpret_cast<float *>(root);
    p.part_ml = p.part_o + (size_t)W * splits * a->B * a->Hq * fd::D;
    p.q = static_cast<const __nv_bfloat16 *>(a->q);
    p.out = static_cast<__nv_bfloat16 *>(a->out);
    if (cudaError_t e = set_smem(reinterpret_cast<const void *>(&flash_decode_kernel), fd::SMEM);
        e != cudaSuccess)
        return cuda_err(e, "flash smem");
    void *args[] = {&p};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = cuda_err(launch(reinterpret_cast<const void *>(&flash_decode_kernel),
                             dim3((unsigned)(W * splits), (unsigned)(a->B * a->Hkv)), dim3(fd::WARPS * 32),
                             fd::SMEM, st, args, false),
                      "flash launch");
    if (rc != TDG_OK)
        return rc;
    return cuda_err(launch(reinterpret_cast<const void *>(&flash_combine_kernel), dim3((unsigned)(a->B * a->Hq)),
                           dim3(fd::D), (size_t)(W * splits + 32) * sizeof(float), st, args, false),
                    "flash combine launch");
}
