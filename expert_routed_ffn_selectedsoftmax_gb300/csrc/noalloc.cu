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
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;   // 8 MiB

// The scratch area itself.  In host code this name is only a host-side
// stand-in; kernels receive the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).  Returns nullptr on failure.
void *scratch_on_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

moe_status moe_forward_noalloc(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                               const float *sel_bias, int E, int k, const void *w_gate,
                               const void *w_up, const void *w_down, moe_dtype w_dt, int F,
                               float *out, int path, moe_stream stream)
{
    // Argument errors first, exactly as moe_forward reports them (a NULL
    // workspace with size 0 never passes the later checks, so probe sizes here).
    if (T < 0) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_workspace_size(T, d, E, k, F, act_dt, w_dt);
    if (need == 0) {
        // invalid sizes or dtype combination: let moe_forward name the error
        return moe_forward(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up, w_down, w_dt,
                           F, out, nullptr, 0, path, stream);
    }
    if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;   // beyond the static area
    if (T == 0)
        return moe_forward(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up, w_down, w_dt,
                           F, out, nullptr, 0, path, stream);
    void *scratch = scratch_on_current_device();
    if (!scratch) return MOE_ERR_CUDA;
    return moe_forward(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up, w_down, w_dt, F,
                       out, scratch, kNoAllocScratchBytes, path, stream);
}

}  // extern "C"
