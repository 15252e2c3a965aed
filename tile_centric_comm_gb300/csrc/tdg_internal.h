// tdg_internal.h -- host-side declarations shared by the translation units of
// libtdg (the handle layout, tensor-map encoding through the driver entry
// point, launch helpers).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "tdg.h"
#include "tdg_ptx.cuh"

struct tdg_symm {
    uint8_t *base;
    size_t bytes;
    int world;
    size_t region_bytes;
    size_t nsig;            // flag words (and counter words) per rank
    uint32_t *flags;        // world * nsig
    uint32_t *counters;     // world * nsig
    tdg::DevStatus *status; // one status block
    uint32_t epoch;         // last epoch handed out
    int device;
    int sm_count;
    cudaEvent_t ce_ev[2] = {nullptr, nullptr}; // fork / join events of CE-mode calls, made once
};

namespace tdg_host {

// The handle's fork / join events for CE-mode calls, created on first use
// (timing disabled) and destroyed with the handle.  Returns false on failure.
inline bool ce_events(tdg_symm *h, cudaEvent_t &ev0, cudaEvent_t &ev1)
{
    for (int i = 0; i < 2; ++i)
        if (!h->ce_ev[i] && cudaEventCreateWithFlags(&h->ce_ev[i], cudaEventDisableTiming) != cudaSuccess) {
            h->ce_ev[i] = nullptr;
            return false;
        }
    ev0 = h->ce_ev[0];
    ev1 = h->ce_ev[1];
    return true;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The epoch of a new call: one counter for every handle of the process, so no
// two calls share an epoch.  Words that a call leaves in memory (LL words in a
// caller's region, which a later heap over the same memory may not clear) can
// then never carry a later call's epoch.  Epochs stay below 2^31, where a
// zeroed flag compares as not yet reached.
uint32_t next_epoch(tdg_symm *h);
// The epoch the next call will take (when no other call comes first).
uint32_t peek_epoch();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned16(size_t v) { return (v & 15u) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).  Returns false on failure.
bool encode_tiled(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes /* rank-1 */,
                  const uint32_t *box, CUtensorMapSwizzle swz);

// bf16 2-D map: inner (contiguous) extent, outer extent, row pitch in bytes.
bool map_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// bf16 3-D map (dim 2 stride given in bytes, e.g. the region size).
bool map_bf16_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);
// The same for fp32 elements.
bool map_f32_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
bool map_f32_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);

// cuStreamWriteValue32 (stream-ordered flag write, with the default memory
// barrier before the write).  Returns false when unavailable or failing.
bool stream_write_u32(cudaStream_t s, uint32_t *dev_addr, uint32_t value);

// Opt a kernel into the large dynamic shared memory it needs on the current
// device.  The attribute is set once per (function, device); safe to call from
// several host threads.
cudaError_t set_smem(const void *fn, int bytes);

// The calling thread's current CUDA context (cuCtxGetCurrent through the
// driver entry point), or nullptr when there is none or it cannot be read.
void *current_context();

// TDG_OK when the current device is the one the heap was allocated on (its
// context is then current in the calling thread), TDG_ERR_INVALID when it is
// another, TDG_ERR_CUDA when it cannot be read or made current.
int check_device(const tdg_symm *h);

// Launch with the cooperative attribute (all CTAs co-resident, which the
// cross-CTA signal waits rely on).  `after_prev`: the programmatic
// serialisation attribute, so that the kernel may start while the previous
// one in the stream still runs, once that one's CTAs have all run
// griddepcontrol.launch_dependents.
cudaError_t launch(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   void **args, bool cooperative, int cluster = 1, bool after_prev = false);

// Number of `cl`-CTA clusters of `fn` that can be resident at once (0 on error).
int max_clusters(const void *fn, int block, int smem, int cl);

// The GEMM cluster shape of a call: `req` (0 = the default, the largest the
// shape allows) against what the shape allows -- allow2: CTA pairs
// (cta_group::2), allow4: clusters of two pairs sharing B.  Returns 1, 2 or 4,
// or 0 when the request is not allowed.
inline int pick_cluster(int req, bool allow2, bool allow4)
{
    allow4 = allow4 && allow2;
    switch (req) {
    case 0: return allow4 ? 4 : (allow2 ? 2 : 1);
    case 1: return 1;
    case 2: return allow2 ? 2 : 0;
    case 4: return allow4 ? 4 : 0;
    default: return 0;
    }
}

// Operand ring stages of the GEMM: `req` (0 = all that fit the ring: 4 of
// 48 KB with one CTA per tile, 6 of 32 KB with pairs), or 0 when out of range.
inline int pick_stages(int req, int cl)
{
    const int mx = cl == 1 ? 4 : 6;
    if (req == 0)
        return mx;
    return (req >= 2 && req <= mx) ? req : 0;
}

inline int cuda_err(cudaError_t e, const char *what)
{
    if (e == cudaSuccess)
        return TDG_OK;
    if (getenv("TDG_LOG"))
        fprintf(stderr, "[tdg] %s: %s\n", what, cudaGetErrorString(e));
    return TDG_ERR_CUDA;
}

inline uint64_t timeout_or_default(uint64_t t) { return t ? t : 2000000000ull; }

// Intra-CTA pipeline waits sit downstream of at most one signal wait that runs
// out (a CTA stops waiting on signals after its first timeout), so their
// bound is twice the signal bound plus a second.
inline uint64_t pipe_timeout(uint64_t signal_timeout) { return 2 * signal_timeout + 1000000000ull; }

} // namespace tdg_host
