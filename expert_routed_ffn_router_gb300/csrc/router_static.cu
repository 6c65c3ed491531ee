// router_static.cu -- moe_router_topk_noalloc: the router with its scratch memory in a
// fixed array that the library itself holds on every GPU, for callers that cannot hand
// the library a workspace.
//
// Who needs it: code that runs where device allocation is not available or not allowed
// -- for instance a plug-in loaded by a host application that owns all device memory and
// gives out only input and output buffers, or a real-time path whose allocator is frozen
// after start-up.  Such a caller cannot call cudaMalloc (or a framework allocator) to
// obtain the workspace that moe_router_topk requires.
//
// How: the scratch (split-K partial logits, squared norms, completion counters and a
// status word) lives in `g_router_scratch`, a file-scope __device__ array of
// kRouterScratchBytes bytes.  In host code the array's name is only a stand-in for the
// device object, so its device address is looked up with cudaGetSymbolAddress, once per
// device, with that device current, on the first call made on that device; the kernel is
// then given that address.  The address belongs to the device's current CUDA context: if
// the context is destroyed and created again (cudaDeviceReset), the module is loaded again
// and the array may move, so the cache also remembers the context's unique id and repeats
// the lookup when it changes.  No call here allocates or frees memory.
#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {
namespace {

constexpr size_t kRouterScratchBytes = size_t(16) << 20;  // 16 MiB per GPU
constexpr size_t kStatusBytes = 256;                      // status word + padding
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_router_scratch[kRouterScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current context (driver entry points looked up once).
bool current_context_id(unsigned long long *id)
{
    static const CtxGetCurrentFn get_current = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                                 &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
                   ? reinterpret_cast<CtxGetCurrentFn>(p) : nullptr;
    }();
    static const CtxGetIdFn get_id = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault,
                                                 &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
                   ? reinterpret_cast<CtxGetIdFn>(p) : nullptr;
    }();
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

std::mutex g_setup_mutex;
struct ScratchAddr {
    unsigned long long ctx_id = 0;
    unsigned char *addr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];

// Device address of g_router_scratch on the current device (looked up on first use, and
// again whenever the device's context changed since).
cudaError_t scratch_address(unsigned char **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);   // false before the runtime set up the context
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchAddr &sa = g_scratch[dev];
    if (!have_id || !sa.addr || sa.ctx_id != id) {
        void *p = nullptr;
        // (also makes the device's primary context current when the runtime has not yet)
        e = cudaGetSymbolAddress(&p, g_router_scratch);
        if (e != cudaSuccess) return e;
        if (!current_context_id(&id)) return cudaErrorDeviceUninitialized;
        sa.addr = static_cast<unsigned char *>(p);
        sa.ctx_id = id;
    }
    *out = sa.addr;
    return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" int moe_router_topk_noalloc(const void *X, const void *W_gate, const float *bias,
                                       int T, int H, int E, int K, int32_t *topk_idx,
                                       float *topk_w, void *stream)
{
    using namespace moe;
    if (T < 0 || H <= 0 || E <= 0 || K <= 0 || K > E) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || K > 32 || H % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    const void *ptrs[] = {X, W_gate, bias, topk_idx, topk_w};
    for (const void *p : ptrs) {
        if (!p) return MOE_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return MOE_ERR_MISALIGNED;
    }
    if (T == 0) return MOE_OK;
    const RouterPlan plan = router_plan(T, H, E);
    if (kStatusBytes + plan.total() > kRouterScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;

    unsigned char *base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
    RouterScratch scr{};
    size_t o = kStatusBytes;
    scr.part = reinterpret_cast<float *>(base + o); o += plan.part_bytes;
    scr.xsq = reinterpret_cast<float *>(base + o); o += plan.xsq_bytes;
    scr.wsq = reinterpret_cast<float *>(base + o); o += plan.wsq_bytes;
    scr.cnt = reinterpret_cast<unsigned *>(base + o);
    // the completion counters must start at zero; launch_router clears them on `stream`
    // before the kernel, so whatever an earlier call left in the array does not matter
    const cudaError_t e = launch_router(X, W_gate, bias, T, H, E, K, topk_idx, topk_w, plan, scr,
                                        reinterpret_cast<int *>(base),
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_router_topk_noalloc_status(void *stream)
{
    using namespace moe;
    unsigned char *base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, base, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(base, 0, sizeof v, s) != cudaSuccess) return MOE_ERR_CUDA;
    return v;
}
