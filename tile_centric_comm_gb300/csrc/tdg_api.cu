// tdg_api.cu -- the symmetric heap (W regions + per-rank signal words + a
// status block carved out of one caller allocation), the device status, and
// the host helpers every operation shares.
//
// The heap realises Triton-distributed's symmetric memory ("Triton-distributed 语义",
// 对称内存模型: every PE allocates at the same virtual address; symm_at maps a
// local pointer to the peer's) on one GPU: region r stands for rank r's heap,
// and symm_at is pointer arithmetic between regions.
#include <new>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "tdg_internal.h"

using namespace tdg_host;

namespace {

size_t flags_offset(int world, size_t region_bytes) { return align_up((size_t)world * region_bytes, 256); }
size_t words_bytes(int world, size_t nsig) { return align_up((size_t)world * nsig * 4, 256); }

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                      const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                      const cuuint32_t *, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);
typedef CUresult (*PFN_writeValue32_t)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

void *driver_fn(const char *name)
{
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return fn;
}

} // namespace

namespace tdg_host {

bool encode_tiled(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                  CUtensorMapSwizzle swz)
{
    static PFN_encodeTiled_t fn = reinterpret_cast<PFN_encodeTiled_t>(driver_fn("cuTensorMapEncodeTiled"));
    if (!fn)
        return false;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i)
        s[i] = strides_bytes[i];
    CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void *>(base), d, s, b, e,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && getenv("TDG_LOG"))
        fprintf(stderr, "[tdg] cuTensorMapEncodeTiled failed (%d)\n", (int)r);
    return r == CUDA_SUCCESS;
}

bool map_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer)
{
    const uint64_t dims[2] = {inner, outer};
    const uint64_t str[1] = {row_bytes};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool map_bf16_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2)
{
    const uint64_t dims[3] = {d0, d1, d2};
    const uint64_t str[2] = {s1_bytes, s2_bytes};
    const uint32_t box[3] = {b0, b1, b2};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool map_f32_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer)
{
    const uint64_t dims[2] = {inner, outer};
    const uint64_t str[1] = {row_bytes};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool map_f32_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2)
{
    const uint64_t dims[3] = {d0, d1, d2};
    const uint64_t str[2] = {s1_bytes, s2_bytes};
    const uint32_t box[3] = {b0, b1, b2};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

bool stream_write_u32(cudaStream_t s, uint32_t *dev_addr, uint32_t value)
{
    static PFN_writeValue32_t fn = reinterpret_cast<PFN_writeValue32_t>(driver_fn("cuStreamWriteValue32"));
    if (!fn)
        return false;
    return fn(reinterpret_cast<CUstream>(s), reinterpret_cast<CUdeviceptr>(dev_addr), value, 0) ==
           CUDA_SUCCESS;
}

cudaError_t set_smem(const void *fn, int bytes)
{
    struct Done {
        const void *fn;
        int dev, bytes;
    };
    static std::mutex mu;
    static std::vector<Done> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const Done &d : done)
        if (d.fn == fn && d.dev == dev && d.bytes >= bytes)
            return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        done.push_back({fn, dev, bytes});
    return e;
}

void *current_context()
{
    typedef CUresult (*PFN_ctxGetCurrent_t)(CUcontext *);
    static PFN_ctxGetCurrent_t fn = reinterpret_cast<PFN_ctxGetCurrent_t>(driver_fn("cuCtxGetCurrent"));
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS)
        return nullptr;
    return c;
}

int check_device(const tdg_symm *h)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return TDG_ERR_CUDA;
    if (dev != h->device)
        return TDG_ERR_INVALID;
    // The driver calls that follow (tensor-map encoding, stream memory
    // operations) need the device's context current in this thread; a thread
    // whose first CUDA call this is may not have it yet.
    return cudaSetDevice(dev) == cudaSuccess ? TDG_OK : TDG_ERR_CUDA;
}

cudaError_t launch(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   void **args, bool cooperative, int cluster, bool after_prev)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[3];
    int n = 0;
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = cooperative ? 1 : 0;
    ++n;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (after_prev) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

namespace {
std::atomic<uint32_t> g_epoch{0};
constexpr uint32_t EPOCH_LIMIT = 0x7FFFFFFFu;
uint32_t epoch_after(uint32_t e) { return e >= EPOCH_LIMIT ? 1u : e + 1u; }
} // namespace

uint32_t next_epoch(tdg_symm *h)
{
    uint32_t cur = g_epoch.load(std::memory_order_relaxed);
    while (!g_epoch.compare_exchange_weak(cur, epoch_after(cur), std::memory_order_relaxed)) {
    }
    h->epoch = epoch_after(cur);
    return h->epoch;
}

uint32_t peek_epoch() { return epoch_after(g_epoch.load(std::memory_order_relaxed)); }

int max_clusters(const void *fn, int block, int smem, int cl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess)
        return 0;
    return n;
}

} // namespace tdg_host

extern "C" {

size_t tdg_symm_bytes(int world, size_t region_bytes, size_t signals_per_rank)
{
    if (world <= 0)
        return 0;
    return flags_offset(world, region_bytes) + 2 * words_bytes(world, signals_per_rank) + 256;
}

int tdg_symm_alloc(void *dev_base, size_t bytes, int world, size_t region_bytes,
                   size_t signals_per_rank, tdg_symm **out)
{
    if (!out || !dev_base || world < 1 || world > 64 || region_bytes == 0 ||
        (region_bytes % 1024) != 0 || (reinterpret_cast<uintptr_t>(dev_base) % 1024) != 0)
        return TDG_ERR_INVALID;
    *out = nullptr;
    if (bytes < tdg_symm_bytes(world, region_bytes, signals_per_rank))
        return TDG_ERR_NOMEM;
    tdg_symm *h = new (std::nothrow) tdg_symm();
    if (!h)
        return TDG_ERR_NOMEM;
    h->base = static_cast<uint8_t *>(dev_base);
    h->bytes = bytes;
    h->world = world;
    h->region_bytes = region_bytes;
    h->nsig = signals_per_rank;
    const size_t fo = flags_offset(world, region_bytes);
    const size_t wb = words_bytes(world, signals_per_rank);
    h->flags = reinterpret_cast<uint32_t *>(h->base + fo);
    h->counters = reinterpret_cast<uint32_t *>(h->base + fo + wb);
    h->status = reinterpret_cast<tdg::DevStatus *>(h->base + fo + 2 * wb);
    h->epoch = 0;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
        delete h;
        return TDG_ERR_CUDA;
    }
    cudaError_t e = cudaMemset(h->base + fo, 0, 2 * wb + 256);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        delete h;
        return cuda_err(e, "symm_alloc memset");
    }
    *out = h;
    return TDG_OK;
}

int tdg_symm_free(tdg_symm *h)
{
    if (h) {
        for (cudaEvent_t e : h->ce_ev)
            if (e)
                cudaEventDestroy(e); // pending work on an event may still finish; its resources go then
    }
    delete h;
    return TDG_OK;
}

void *tdg_symm_region(const tdg_symm *h, int rank)
{
    if (!h || rank < 0 || rank >= h->world)
        return nullptr;
    return h->base + (size_t)rank * h->region_bytes;
}

void *tdg_symm_at(const tdg_symm *h, const void *local_ptr, int rank)
{
    if (!h || rank < 0 || rank >= h->world)
        return nullptr;
    const uint8_t *p = static_cast<const uint8_t *>(local_ptr);
    if (p < h->base || p >= h->base + (size_t)h->world * h->region_bytes)
        return nullptr;
    const size_t off = (size_t)(p - h->base) % h->region_bytes;
    return h->base + (size_t)rank * h->region_bytes + off;
}

uint32_t *tdg_symm_flags(const tdg_symm *h, int rank)
{
    if (!h || rank < 0 || rank >= h->world)
        return nullptr;
    return h->flags + (size_t)rank * h->nsig;
}

uint32_t *tdg_symm_counters(const tdg_symm *h, int rank)
{
    if (!h || rank < 0 || rank >= h->world)
        return nullptr;
    return h->counters + (size_t)rank * h->nsig;
}

uint32_t tdg_symm_epoch(const tdg_symm *h)
{
    if (!h)
        return 0;
    return tdg_host::peek_epoch();
}

int tdg_status(tdg_symm *h, void *stream, tdg_fault *out, int clear)
{
    if (!h)
        return TDG_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    tdg::DevStatus st;
    cudaError_t e = cudaMemcpyAsync(&st, h->status, sizeof st, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && clear)
        e = cudaMemsetAsync(h->status, 0, sizeof st, s);
    if (e == cudaSuccess && clear)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_err(e, "status");
    if (out) {
        out->code = st.code;
        out->where = st.where;
        out->index = st.index;
        out->epoch = st.epoch;
    }
    return st.code;
}

const char *tdg_strerror(int code)
{
    switch (code) {
    case TDG_OK: return "ok";
    case TDG_ERR_INVALID: return "invalid argument (shape, alignment, range or NULL)";
    case TDG_ERR_CUDA: return "a CUDA call failed";
    case TDG_ERR_NOMEM: return "caller buffer, region or signal area too small";
    case TDG_ERR_TIMEOUT: return "a device signal wait ran out of time";
    case TDG_ERR_UNSUPPORTED: return "not supported on this device or in this mode";
    case TDG_ERR_DEVICE: return "a kernel found an out-of-range index";
    default: return "unknown tdg error";
    }
}

int tdg_device_info(int *sm_count, int *supported)
{
    int dev = 0, major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return cuda_err(e, "device_info");
    if (sm_count)
        *sm_count = sms;
    if (supported)
        *supported = (major == 10 && minor == 3) ? 1 : 0;
    return TDG_OK;
}

} // extern "C"
