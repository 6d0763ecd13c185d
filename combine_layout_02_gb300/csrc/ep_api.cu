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

namespace ep {
namespace {

// One thread arms a barrier for 32 bytes and bulk-copies only 16 into shared memory, so
// the barrier phase never completes and the bounded wait has to give up.
__global__ void wait_timeout_probe_kernel(const void* src16, uint64_t timeout_ns, uint32_t* err,
                                          uint32_t* elapsed_us) {
    __shared__ __align__(128) unsigned char buf[32];
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    pdl_wait();
    mbar_init(&bar, 1);
    mbar_expect_bytes(&bar, 32);
    bulk_load(buf, src16, 16, &bar);
    const uint64_t t0 = global_ns();
    const bool done = mbar_wait_bounded(&bar, 0, timeout_ns);
    const uint64_t t1 = global_ns();
    if (!done) raise_flag(err, EP_DEVERR_TIMEOUT);
    if (elapsed_us != nullptr) *elapsed_us = (uint32_t)((t1 - t0) / 1000u);
}

}  // namespace
}  // namespace ep

extern "C" {

ep_status ep_selftest_wait_timeout(const void* src16, int32_t timeout_ms, uint32_t* elapsed_us,
                                   const ep_launch* launch) {
    using namespace ep;
    if (launch == nullptr || launch->error_flags == nullptr || src16 == nullptr) return EP_ERR_INVALID_ARG;
    if (((uintptr_t)src16 & 15) != 0 || timeout_ms < 1 || timeout_ms > 10000) return EP_ERR_INVALID_ARG;
    ep_status st = begin_call(launch);
    if (st != EP_OK) return st;
    cudaError_t e = launch_pdl(wait_timeout_probe_kernel, dim3(1), dim3(32), 0, launch->stream, src16,
                               (uint64_t)timeout_ms * 1000000ull, launch->error_flags, elapsed_us);
    if (e != cudaSuccess) return cuda_fail(e);
    return end_call(launch);
}

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

ep_status ep_buffer_size_hint(const ep_shape* sh, ep_dtype recv_dtype, int32_t fp8_scale_format,
                              ep_size_hint* out) {
    ep_status st = ep::check_shape(sh);
    if (st != EP_OK) return st;
    if (out == nullptr) return EP_ERR_INVALID_ARG;
    if (recv_dtype != EP_BF16 && recv_dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
    if (fp8_scale_format < EP_FP8_SCALE_FP32 || fp8_scale_format > EP_FP8_SCALE_TENSOR)
        return EP_ERR_INVALID_ARG;
    const uint64_t R = (uint64_t)sh->num_ranks, T = (uint64_t)sh->num_tokens,
                   H = (uint64_t)sh->hidden, k = (uint64_t)sh->num_topk,
                   E = (uint64_t)sh->num_experts, E_loc = E / R,
                   nmax = (uint64_t)sh->num_max_dispatch_tokens_per_rank, G = H / EP_FP8_GROUP;
    const bool fp8 = recv_dtype == EP_FP8_E4M3;
    const uint64_t elem = fp8 ? 1 : 2;
    const uint64_t scale = fp8 ? (fp8_scale_format == EP_FP8_SCALE_UE8M0 ? 1 : 4) : 0;
    bool bad = false;
    auto mul = [&bad](uint64_t a, uint64_t b) {
        uint64_t r = 0;
        if (__builtin_mul_overflow(a, b, &r)) bad = true;
        return r;
    };
    ep_size_hint h{};
    const uint64_t rows = mul(mul(R, R), T);
    h.recv_rows = (int64_t)rows;
    h.recv_x_bytes = mul(mul(rows, H), elem);
    h.recv_x_scales_bytes = mul(mul(rows, G), scale);
    h.recv_topk_idx_bytes = mul(mul(rows, k), 8);
    h.recv_topk_weights_bytes = mul(mul(rows, k), 4);
    h.recv_src_idx_bytes = mul(rows, 4);
    const uint64_t em_rows = mul(rows, k < E_loc ? k : E_loc);
    h.expert_major_rows = (int64_t)em_rows;
    h.expert_major_x_bytes = mul(mul(em_rows, H), elem);
    const uint64_t slots = mul(mul(mul(R, E_loc), R), nmax);
    h.ll_slots = slots;
    h.ll_recv_x_bytes = mul(mul(slots, H), elem);
    h.ll_recv_x_scales_bytes = mul(mul(slots, G), scale);
    h.ll_src_info_bytes = mul(slots, 4);
    h.ll_slot_bytes = mul(mul(mul(R, T), k), 4);
    h.ll_send_count_bytes = mul(mul(E, R), 4);
    h.ll_recv_expert_count_bytes = mul(E, 4);
    h.ll_layout_range_bytes = mul(mul(E, R), 8);
    h.layout_workspace_bytes = ep_layout_workspace_size(sh);
    if (bad || rows > (uint64_t)INT64_MAX || em_rows > (uint64_t)INT64_MAX) return EP_ERR_UNSUPPORTED;
    *out = h;
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

int32_t ep_abi_version(void) { return 103; }

}  // extern "C"
