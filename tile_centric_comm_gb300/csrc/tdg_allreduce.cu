// tdg_allreduce.cu -- tile-centric ring AllReduce over W logical ranks
// ("Triton-distributed 语义", 示例：带重叠的环形 AllReduce: a reduce-scatter ring
// then an all-gather ring, each tile signalled on its own so it is reduced or
// forwarded the moment it arrives).
//
// One cooperative launch of W * G CTAs: CTA (r, g) acts for rank r on the
// tiles t = g, g + G, ... of every step.  A step of rank r waits only on the
// same tiles of the previous step of rank r-1, so the dependency graph is
// acyclic and, with every CTA resident, every wait ends.
//   reduce-scatter, s = 0 .. W-2:  chunk c = (r - s) mod W,
//       v = x_r[c] (+ recv_r[s-1] when s > 0)  -> recv_{r+1}[s], signal (s)
//   final, s = W-1:                 chunk f = (r + 1) mod W,
//       v = x_r[f] + recv_r[W-2]    -> x_r[f] and x_{r+1}[f], signal (W-1)
//   all-gather, s = W .. 2W-3:      chunk c = (r + 1 - (s - W + 1)) mod W,
//       x_r[c] (arrived at step s-1) -> x_{r+1}[c], signal (s)
// Data written by another CTA is read with ld.global.cg (through L2 only).
#include "tdg_internal.h"

namespace tdg {

struct RingParams {
    DevStatus *status;
    uint32_t epoch;
    uint64_t timeout_ns;
    int W, G;
    int64_t chunk;   // elements per chunk (count / W)
    int64_t tile;    // elements per tile
    int64_t tiles;   // tiles per chunk
    uint8_t *regions;
    uint64_t region_bytes;
    uint64_t x_off, recv_off;
    uint32_t *flags;  // rank 0's flag words
    uint64_t nsig;    // flag words per rank
    uint64_t skip;    // tests only: rank 0's signal skip - 1 is never notified (0: none)
};

__device__ __forceinline__ float *ring_x(const RingParams &p, int r, int c)
{
    return reinterpret_cast<float *>(p.regions + (uint64_t)r * p.region_bytes + p.x_off) + (int64_t)c * p.chunk;
}
__device__ __forceinline__ float *ring_recv(const RingParams &p, int r, int slot)
{
    return reinterpret_cast<float *>(p.regions + (uint64_t)r * p.region_bytes + p.recv_off) +
           (int64_t)slot * p.chunk;
}
__device__ __forceinline__ uint32_t *ring_flag(const RingParams &p, int r, int step, int64_t t)
{
    return p.flags + (uint64_t)r * p.nsig + (uint64_t)step * p.tiles + t;
}

// thread 0 waits (bounded) for the tile's signal; the CTA follows it
__device__ __forceinline__ void ring_wait(const RingParams &p, int r, int step, int64_t t, bool &gave_up)
{
    if (threadIdx.x == 0 && !gave_up) {
        if (!wait_flag(ring_flag(p, r, step, t), p.epoch, p.timeout_ns)) {
            report_fault(p.status, TDG_ERR_TIMEOUT, TDG_WHERE_RING, (uint32_t)(step * p.tiles + t), p.epoch);
            gave_up = true;
        }
    }
    __syncthreads();
}

// every thread's writes of the tile are done before thread 0 publishes it
__device__ __forceinline__ void ring_notify(const RingParams &p, int r, int step, int64_t t)
{
    __syncthreads();
    if (threadIdx.x == 0 && !(p.skip && r == 0 && (uint64_t)step * p.tiles + t == p.skip - 1)) {
        __threadfence();
        st_release_gpu(ring_flag(p, r, step, t), p.epoch);
    }
}

// Element-wise body of one tile: UNROLL float4 loads of each operand are in
// flight before any add or store (the loop is bound by memory latency).
constexpr int UNROLL = 4;

template <int KIND> // 0: out = a (+ b if has_b); 1: a = out2 = a + b; 2: out = a
__device__ __forceinline__ void ring_tile(const float4 *a, const float4 *b, float4 *out, float4 *out2,
                                          int64_t nv, bool has_b)
{
    const int64_t stride = (int64_t)blockDim.x * UNROLL;
    for (int64_t i0 = threadIdx.x; i0 < nv; i0 += stride) {
        float4 va[UNROLL], vb[UNROLL];
#pragma unroll
        for (int j = 0; j < UNROLL; ++j) {
            const int64_t i = i0 + (int64_t)j * blockDim.x;
            if (i < nv) {
                va[j] = __ldcg(a + i);
                if (has_b)
                    vb[j] = __ldcg(b + i);
            }
        }
#pragma unroll
        for (int j = 0; j < UNROLL; ++j) {
            const int64_t i = i0 + (int64_t)j * blockDim.x;
            if (i < nv) {
                float4 v = va[j];
                if (has_b) { // local + incoming
                    v.x += vb[j].x;
                    v.y += vb[j].y;
                    v.z += vb[j].z;
                    v.w += vb[j].w;
                }
                if (KIND == 1)
                    __stcg(out2 + i, v);
                __stcg(out + i, v);
            }
        }
    }
}

__global__ void __launch_bounds__(256, 2) ring_allreduce_kernel(const __grid_constant__ RingParams p)
{
    const int r = blockIdx.x / p.G, g = blockIdx.x % p.G;
    const int W = p.W, nxt = (r + 1) % W;
    bool gave_up = false;
    for (int s = 0; s <= 2 * W - 3; ++s) {
        for (int64_t t = g; t < p.tiles; t += p.G) {
            const int64_t e0 = t * p.tile;
            const int64_t ne = min(p.tile, p.chunk - e0);
            const int64_t nv = ne / 4;
            if (s > 0)
                ring_wait(p, r, s - 1, t, gave_up);
            if (s <= W - 2) { // reduce-scatter push
                const int c = ((r - s) % W + W) % W;
                ring_tile<0>(reinterpret_cast<const float4 *>(ring_x(p, r, c) + e0),
                             reinterpret_cast<const float4 *>(ring_recv(p, r, s - 1) + e0),
                             reinterpret_cast<float4 *>(ring_recv(p, nxt, s) + e0), nullptr, nv, s > 0);
            } else if (s == W - 1) { // final reduction of chunk r+1, then the first all-gather push
                const int f = nxt;
                float4 *xl = reinterpret_cast<float4 *>(ring_x(p, r, f) + e0);
                ring_tile<1>(xl, reinterpret_cast<const float4 *>(ring_recv(p, r, W - 2) + e0),
                             reinterpret_cast<float4 *>(ring_x(p, nxt, f) + e0), xl, nv, true);
            } else { // all-gather forward of the chunk that arrived at step s-1
                const int c = ((r + 1 - (s - (W - 1))) % W + W) % W;
                ring_tile<2>(reinterpret_cast<const float4 *>(ring_x(p, r, c) + e0), nullptr,
                             reinterpret_cast<float4 *>(ring_x(p, nxt, c) + e0), nullptr, nv, false);
            }
            ring_notify(p, nxt, s, t);
        }
    }
}

} // namespace tdg

using namespace tdg;
using namespace tdg_host;

extern "C" size_t tdg_allreduce_recv_bytes(int world, int64_t count)
{
    if (world <= 1 || count <= 0)
        return 0;
    return (size_t)(world - 1) * (size_t)(count / world) * sizeof(float);
}

extern "C" int tdg_allreduce(tdg_symm *h, const tdg_allreduce_args *a, void *stream)
{
    if (!h || !a)
        return TDG_ERR_INVALID;
    if (const int drc = check_device(h))
        return drc;
    const int W = a->world;
    if (W != h->world || a->count < 0)
        return TDG_ERR_INVALID;
    if (a->count == 0 || W == 1)
        return TDG_OK;
    if (a->count % (4 * W) || !aligned16(a->x_off) || !aligned16(a->recv_off))
        return TDG_ERR_INVALID;
    const int64_t chunk = a->count / W;
    int64_t tile = a->tile_elems > 0 ? a->tile_elems : 65536;
    if (tile % 4)
        return TDG_ERR_INVALID;
    if (tile > chunk)
        tile = chunk;
    const int64_t tiles = (chunk + tile - 1) / tile;
    const uint64_t R = h->region_bytes;
    if (a->x_off + (uint64_t)a->count * 4 > R || a->recv_off + tdg_allreduce_recv_bytes(W, a->count) > R)
        return TDG_ERR_NOMEM;
    if (a->x_off < a->recv_off + tdg_allreduce_recv_bytes(W, a->count) && a->recv_off < a->x_off + (uint64_t)a->count * 4)
        return TDG_ERR_INVALID; // the receive slots overlap the data
    if ((uint64_t)(2 * W - 2) * tiles > h->nsig)
        return TDG_ERR_NOMEM;
    int per_sm = 0;
    const void *fn = reinterpret_cast<const void *>(&ring_allreduce_kernel);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 256, 0) != cudaSuccess || per_sm < 1)
        return TDG_ERR_CUDA;
    // default: as many CTAs per rank as can all be resident (every wait relies on it)
    int G = a->ctas_per_rank > 0 ? a->ctas_per_rank : (per_sm * h->sm_count) / W;
    if (G < 1)
        G = 1;
    if ((int64_t)G > tiles)
        G = (int)tiles;
    if ((int64_t)G * W > (int64_t)per_sm * h->sm_count)
        return TDG_ERR_INVALID; // every CTA must be resident at once
    RingParams p;
    memset(&p, 0, sizeof p);
    p.status = h->status;
    p.epoch = next_epoch(h);
    p.timeout_ns = timeout_or_default(a->timeout_ns);
    p.W = W;
    p.G = G;
    p.chunk = chunk;
    p.tile = tile;
    p.tiles = tiles;
    p.regions = h->base;
    p.region_bytes = R;
    p.x_off = a->x_off;
    p.recv_off = a->recv_off;
    p.flags = h->flags;
    p.nsig = h->nsig;
    p.skip = a->test_skip_signal;
    void *args[] = {&p};
    return cuda_err(launch(fn, dim3(W * G), dim3(256), 0, static_cast<cudaStream_t>(stream), args, true),
                    "allreduce launch");
}
