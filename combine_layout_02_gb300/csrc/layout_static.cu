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
#include <mutex>

#include "ep_internal.cuh"

// The scratch shared by every call on a device. Only its device address (looked up
// below) may be handed to kernels; in host code this name is a host-side stand-in.
static __device__ __align__(256) unsigned char g_layout_scratch[EP_LAYOUT_STATIC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mutex;
void* g_scratch_addr[128] = {nullptr};   // device address of g_layout_scratch, per device
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
    void* scratch = nullptr;
    {
        // One-time set-up per device, with that device current: resolve the array's
        // device address.
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        if (g_scratch_addr[dev] == nullptr) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_layout_scratch);
            if (e != cudaSuccess) return ep::cuda_fail(e);
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    // The layout kernels overwrite every scratch word they later read, so the contents
    // left by an earlier call need no clearing.
    return ep_get_layout(shape, topk_idx, layout, handle, scratch,
                         (size_t)EP_LAYOUT_STATIC_SCRATCH_BYTES, launch);
}
