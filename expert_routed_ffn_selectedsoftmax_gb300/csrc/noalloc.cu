// noalloc.cu -- moe_forward for callers that cannot allocate device memory.
//
// Some hosts of this layer hand it only its inputs and outputs: serving
// runtimes and audio-plugin hosts that own every byte of device memory through
// their own pool and forbid cudaMalloc while serving (cudaMalloc synchronises
// the device and can fail under a fixed memory budget).  For them,
// moe_forward_noalloc runs the same kernels as moe_forward with its scratch in
// one static device array defined in this file.  The array is part of the
// library image: every GPU that loads the library holds it until the process
// exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;   // 8 MiB

// The scratch area itself.  In host code this name is only a host-side
// stand-in; kernels receive the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// cuCtxGetCurrent through the runtime's driver entry point (the library does
// not link the driver library directly).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current()
{
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load();
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f);
    }
    return reinterpret_cast<CtxGetCurrentFn>(f);
}

// Per device: the context the address was looked up in, and the address.
// A new context on the device (after cudaDeviceReset, or a context torn down
// and re-created by the host) loads the library's module again, possibly at
// another address, so the lookup is repeated then.
std::mutex g_setup_mutex;
CUcontext g_scratch_ctx[moe::kCachedDevices] = {};
void *g_scratch_addr[moe::kCachedDevices] = {};

// Device address of the scratch array in the current device's current
// context: looked up (cudaGetSymbolAddress, return code checked) the first
// time a device / context is seen, with that device current.  nullptr on
// failure.
void *scratch_on_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current();
    if (get && get(&ctx) != CUDA_SUCCESS) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (ctx && dev < moe::kCachedDevices && g_scratch_addr[dev] && g_scratch_ctx[dev] == ctx)
        return g_scratch_addr[dev];
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    // (the lookup makes the device's primary context current if none was)
    if (get && !ctx && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    if (dev < moe::kCachedDevices) {
        g_scratch_addr[dev] = ptr;
        g_scratch_ctx[dev] = ctx;
    }
    return ptr;
}

}  // namespace

extern "C" {

moe_status moe_forward_noalloc(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                               const float *sel_bias, int E, int k, const void *w_gate,
                               const void *w_up, const void *w_down, moe_dtype w_dt, int F,
                               float *out, int path, moe_stream stream)
{
    // moe_forward's own argument checks first, then the size of the static area
    moe_status st = moe::forward_args_check(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up,
                                            w_down, w_dt, F, out, path, MOE_SCORE_SELECTED_SOFTMAX,
                                            false);
    if (st != MOE_OK || T == 0) return st;
    const size_t need = moe_workspace_size(T, d, E, k, F, act_dt, w_dt);
    if (need == 0) return MOE_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;   // beyond the static area
    void *scratch = scratch_on_current_device();
    if (!scratch) return MOE_ERR_CUDA;
    return moe_forward(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up, w_down, w_dt, F,
                       out, scratch, kNoAllocScratchBytes, path, stream);
}

moe_status moe_check_noalloc(uint32_t *device_word, moe_stream stream)
{
    void *scratch = scratch_on_current_device();
    if (!scratch) return MOE_ERR_CUDA;
    return moe_check(scratch, device_word, stream);
}

}  // extern "C"
