// layout_static.cu -- ep_get_layout_static_scratch: the layout computation for callers
// that cannot allocate device memory.
//
// ep_get_layout needs a caller-provided device workspace for its per-channel partial
// counts. Some callers have no way to provide one: for example a plugin whose host
// framework owns every byte of device memory through its own pool and forbids side
// allocations, or a latency-critical loop where cudaMalloc / cudaFree would
// synchronise the device or fragment the pool. This entry point keeps that workspace in
// a fixed-size array compiled into the library instead, so the caller passes only
// inputs and outputs.
//
// The array lives in device memory of every GPU that loads the library, for the life
// of the process, whether or not this entry point is ever called.
#include <cuda.h>   // driver types only (the driver functions are looked up at run time)

#include <mutex>

#include "ep_internal.cuh"

// The scratch shared by every call on a device. Only its device address (looked up
// below) may be handed to kernels; in host code this name is a host-side stand-in.
static __device__ __align__(256) unsigned char g_layout_scratch[EP_LAYOUT_STATIC_SCRATCH_BYTES];

namespace {

// The array's device address belongs to the module loaded into one CUDA context. After
// cudaDeviceReset (or any new primary context) the module is loaded again, possibly at
// another address, so the cached address is keyed by the context's unique id.
struct ScratchAddr {
    unsigned long long ctx_id;
    void* addr;
};

std::mutex g_scratch_mutex;
ScratchAddr g_scratch_addr[128] = {};        // per device ordinal

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Looks up the two driver functions once (no link-time dependency on libcuda).
bool driver_functions() {
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    return g_ctx_get_current != nullptr && g_ctx_get_id != nullptr;
}

// Id of the current context (0 if there is none yet).
bool current_ctx_id(unsigned long long* id) {
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return false;
    *id = 0;
    if (ctx == nullptr) return true;
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

extern "C" ep_status ep_get_layout_static_scratch(const ep_shape* shape, const int64_t* topk_idx,
                                                  ep_layout* layout, ep_handle* handle,
                                                  const ep_launch* launch) {
    ep_status st = ep::check_shape(shape);
    if (st != EP_OK) return st;
    if (ep_layout_workspace_size(shape) > (size_t)EP_LAYOUT_STATIC_SCRATCH_BYTES)
        return EP_ERR_UNSUPPORTED;   // shape needs more scratch than the fixed array holds

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ep::cuda_fail(e);
    if (dev < 0 || dev >= 128) return EP_ERR_UNSUPPORTED;
    if (!driver_functions()) return EP_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    {
        // Set-up once per context, with the device current: resolve the array's device
        // address. A context seen for the first time (the first call, or the first after
        // a device reset) repeats the lookup.
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        unsigned long long id = 0;
        if (!current_ctx_id(&id)) return EP_ERR_UNSUPPORTED;
        ScratchAddr& c = g_scratch_addr[dev];
        if (id == 0 || c.addr == nullptr || c.ctx_id != id) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_layout_scratch);   // creates the context if needed
            if (e != cudaSuccess) return ep::cuda_fail(e);
            if (!current_ctx_id(&id) || id == 0) return EP_ERR_UNSUPPORTED;
            c.ctx_id = id;
            c.addr = p;
        }
        scratch = c.addr;
    }
    // The layout kernels overwrite every scratch word they later read, so the contents
    // left by an earlier call need no clearing.
    return ep_get_layout(shape, topk_idx, layout, handle, scratch,
                         (size_t)EP_LAYOUT_STATIC_SCRATCH_BYTES, launch);
}
