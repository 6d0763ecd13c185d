// ep_api.cu -- host plumbing shared by every libep entry point: shape validation,
// event ordering ([OVERLAP] previous_event / async_finish), SM-count cache, launch
// accounting, status strings, and the synchronous read-back helpers.
//
// [OVERLAP] = "How DeepEP Achieves Communication-Computation Overlapping with
// EventOverlap"; [README] = "DeepEP", README of the EnflameTechnology/DeepEP port.
#include <atomic>
#include <mutex>

#include "ep_internal.cuh"

namespace ep {

namespace {
std::atomic<uint64_t> g_launches{0};
thread_local char g_last_error[256] = "";
std::mutex g_sm_mutex;
int g_sm_cache[128] = {0};
}  // namespace

ep_status cuda_fail(cudaError_t e) {
    const char* s = cudaGetErrorString(e);
    size_t i = 0;
    for (; s && s[i] && i + 1 < sizeof(g_last_error); ++i) g_last_error[i] = s[i];
    g_last_error[i] = '\0';
    return EP_ERR_CUDA;
}

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

ep_status check_shape(const ep_shape* sh) {
    if (sh == nullptr) return EP_ERR_INVALID_ARG;
    if (sh->num_ranks < 1 || sh->num_tokens < 0 || sh->hidden < 1 || sh->num_experts < 1 ||
        sh->num_topk < 1 || sh->num_channels < 1 || sh->num_sms < 0 ||
        sh->num_max_dispatch_tokens_per_rank < 0)
        return EP_ERR_INVALID_ARG;
    if (sh->num_experts % sh->num_ranks != 0) return EP_ERR_INVALID_ARG;
    if (sh->hidden % EP_FP8_GROUP != 0) return EP_ERR_INVALID_ARG;
    if (sh->num_ranks > EP_MAX_RANKS || sh->num_topk > EP_MAX_TOPK ||
        sh->num_experts > EP_MAX_EXPERTS)
        return EP_ERR_UNSUPPORTED;
    // Row and element indices stay within int32 / int64 ranges used by the kernels.
    if ((int64_t)sh->num_ranks * sh->num_tokens > (int64_t)1 << 30) return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 1;
    std::lock_guard<std::mutex> lock(g_sm_mutex);
    if (g_sm_cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        g_sm_cache[dev] = n;
    }
    return g_sm_cache[dev];
}

ep_status begin_call(const ep_launch* launch) {
    if (launch == nullptr) return EP_ERR_INVALID_ARG;
    if (launch->wait_event != nullptr) {
        cudaError_t e = cudaStreamWaitEvent(launch->stream, launch->wait_event, 0);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return EP_OK;
}

ep_status end_call(const ep_launch* launch) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    if (launch->record_event != nullptr) {
        e = cudaEventRecord(launch->record_event, launch->stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return EP_OK;
}

ep_status load_row_offsets(const int64_t* host, int R, RowOffsets* out) {
    if (host == nullptr) return EP_ERR_INVALID_ARG;
    if (host[0] < 0) return EP_ERR_INVALID_ARG;
    for (int d = 0; d <= R; ++d) {
        if (d > 0 && host[d] < host[d - 1]) return EP_ERR_INVALID_ARG;
        out->v[d] = host[d];
    }
    for (int d = R + 1; d <= EP_MAX_RANKS; ++d) out->v[d] = host[R];
    return EP_OK;
}

}  // namespace ep

extern "C" {

ep_status ep_read_recv_counts_sync(const ep_shape* shape, const ep_handle* handle,
                                   int32_t* host_counts, cudaStream_t stream) {
    ep_status st = ep::check_shape(shape);
    if (st != EP_OK) return st;
    if (handle == nullptr || handle->rank_prefix_matrix == nullptr || host_counts == nullptr)
        return EP_ERR_INVALID_ARG;
    const int R = shape->num_ranks;
    cudaError_t e = cudaMemcpyAsync(host_counts, handle->rank_prefix_matrix + (size_t)(R - 1) * R,
                                    sizeof(int32_t) * R, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return ep::cuda_fail(e);
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return ep::cuda_fail(e);
    return EP_OK;
}

ep_status ep_read_error_flags_sync(const uint32_t* error_flags, uint32_t* host_flags,
                                   cudaStream_t stream) {
    if (error_flags == nullptr || host_flags == nullptr) return EP_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(host_flags, error_flags, sizeof(uint32_t),
                                    cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return ep::cuda_fail(e);
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return ep::cuda_fail(e);
    return EP_OK;
}

const char* ep_status_string(ep_status status) {
    switch (status) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG: bad argument or shape";
        case EP_ERR_CUDA: return "EP_ERR_CUDA: a CUDA call failed (see ep_last_cuda_error)";
        case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED: shape beyond the library limits";
        default: return "unknown ep_status";
    }
}

const char* ep_last_cuda_error(void) { return ep::g_last_error; }

uint64_t ep_kernel_launch_count(void) { return ep::g_launches.load(std::memory_order_relaxed); }

int32_t ep_abi_version(void) { return 101; }

}  // extern "C"
