// gma_noalloc.cu -- gma_forward_causal_noalloc: the causal forward pass for callers that cannot
// allocate device memory, and gma_noalloc_check, which reports what its kernels found.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they run GMA: code
// inside a custom allocator or memory-pool callback, a plugin whose host application owns every
// device allocation, or a real-time loop that must not touch the allocator after start-up.  They
// can still pass their inputs and outputs, but not a workspace.  This entry point supplies the
// workspace itself from a fixed-size array that lives in the library's device image.
//
// The array is a file-scope __device__ variable: every GPU that loads this library holds
// GMA_NOALLOC_SCRATCH_BYTES of it until the process exits.  Host code cannot use the array's
// name as a device address (in host code the name is only a host-side stand-in), so the first
// call on each device, with that device current, asks the runtime for the array's device
// address with cudaGetSymbolAddress and caches it together with the identity of the CUDA context
// it belongs to.  A call made under another context (after cudaDeviceReset, for instance, which
// unloads the module so that the array may move) looks the address up again.
#include <mutex>

#include <cuda.h>

#include "gma_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)GMA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

std::mutex g_setup_mutex;
struct Entry {
    void *ptr = nullptr;
    unsigned long long ctx_id = 0;
};
Entry g_entry[kMaxDevices];

// The unique id of the CUDA context current on this thread (0 if it cannot be read).  Context ids
// are never reused within a process, so a changed id means the array must be looked up again.
unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = (CtxGetCurrentFn)p;
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = (CtxGetIdFn)p;
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of this device's copy of the scratch array, looked up once per device and
// context.
gma_status_t scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_NO_DEVICE;
    if (dev < 0 || dev >= kMaxDevices) return GMA_ERR_NO_DEVICE;
    const unsigned long long id = current_context_id();   // 0 before the runtime made one
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    Entry &e = g_entry[dev];
    if (!e.ptr || id == 0 || e.ctx_id != id) {
        // (the lookup also makes the device's primary context current if none was)
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GMA_ERR_CUDA;
        e.ptr = p;
        e.ctx_id = current_context_id();
    }
    *out = e.ptr;
    return GMA_OK;
}

}  // namespace

extern "C" gma_status_t gma_forward_causal_noalloc(const gma_shape_t *shape, const void *QX,
                                                   const void *KX, const void *V,
                                                   const float *mu, const float *raw_var,
                                                   const float *prior_logits, void *O,
                                                   gma_stream_t stream)
{
    const size_t need = gma_workspace_size(shape, GMA_VARIANT_CAUSAL);
    if (need == 0)   // invalid shape: the regular entry point names the error, enqueuing nothing
        return gma_forward_causal(shape, QX, KX, V, mu, raw_var, prior_logits, O, nullptr, 0,
                                  stream);
    gma_shape_t s = *shape;
    if (need > kScratchBytes) {
        // the smaller workspace of the same computation, if that one fits
        s.flags |= GMA_FLAG_RECOMPUTE_KEYS;
        if (gma_workspace_size(&s, GMA_VARIANT_CAUSAL) > kScratchBytes) return GMA_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    const gma_status_t r = scratch_for_current_device(&scratch);
    if (r != GMA_OK) return r;
    return gma_forward_causal(&s, QX, KX, V, mu, raw_var, prior_logits, O, scratch, kScratchBytes,
                              stream);
}

extern "C" gma_status_t gma_noalloc_check(gma_stream_t stream)
{
    void *scratch = nullptr;
    const gma_status_t r = scratch_for_current_device(&scratch);
    if (r != GMA_OK) return r;
    return gma_check_workspace(scratch, stream);
}
