// ll.cu -- low-latency dispatch / combine into fixed per-(expert, source) slots, with
// the send / receive phase split.
//
// [README] "DeepEP" README (EnflameTechnology/DeepEP), low-latency example:
//          low_latency_dispatch(x, topk_idx, num_max_dispatch_tokens_per_rank,
//          num_experts, async_finish, return_recv_hook) -> recv_hidden_states,
//          recv_expert_count (int32 in the port), handle, event, hook;
//          low_latency_combine(x, topk_idx, topk_weights, handle, ...) ->
//          combined_hidden_states.
// [HOOK]   "How DeepEP Enables Hook-Based Overlapping Without SM Occupation",
//          "Two-Phase Kernel Architecture": the send phase runs at once, the receive
//          phase when the hook is called.
//
// Reading of the receive format: rank d keeps, for each local expert el, R*Nmax
// slots; source s owns [s*Nmax, (s+1)*Nmax) and fills them in the order of its
// (token, k) entries: entry (t, j) of source s with expert e takes slot
//   s*Nmax + #{(t', j') before (t, j) in source s with expert e}.
// The send kernel computes that count by a block-wide scan of the source's earlier
// entries (at most Nmax*k of them), so no block waits on another. Extra blocks write
// the per-(destination, expert, source) count signals; the receive kernel only
// reads those signals.
#include "rowops.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;

struct LLArgs {
    const char* x;
    const int64_t* topk_idx;
    const float* topk_weights;
    char* recv_x;
    float* recv_x_scales;
    int32_t* src_info;
    int32_t* slot;
    int32_t* send_count;
    int32_t* recv_expert_count;
    int32_t* layout_range;
    const char* y;
    char* out;
    int R, T, H, E, k, E_loc, nmax, use_fp8;
    uint32_t* err;
};

// Blocks [0, R*T): one per source token. Blocks [R*T, R*T + R): count signal of one
// source rank.
__global__ void __launch_bounds__(kThreads) ll_send_kernel(LLArgs a) {
    __shared__ int64_t s_e[EP_MAX_TOPK];
    __shared__ int s_cnt[EP_MAX_TOPK];
    __shared__ int64_t s_rows[EP_MAX_TOPK];
    __shared__ int s_nv;
    extern __shared__ int hist[];   // [E], count blocks only
    const int b = blockIdx.x;
    const int64_t slots = (int64_t)a.R * a.nmax;
    pdl_wait();

    if (b >= a.R * a.T) {
        const int s = b - a.R * a.T;
        for (int e = threadIdx.x; e < a.E; e += kThreads) hist[e] = 0;
        __syncthreads();
        const int64_t* tk = a.topk_idx + (int64_t)s * a.T * a.k;
        for (int i = threadIdx.x; i < a.T * a.k; i += kThreads) {
            const int64_t e = tk[i];
            if (e >= 0 && e < a.E) atomicAdd(&hist[(int)e], 1);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < a.E; e += kThreads)
            a.send_count[(int64_t)e * a.R + s] = min(hist[e], a.nmax);   // e = d*E_loc + el
        pdl_trigger();
        return;
    }

    const int s = b / a.T, t = b - s * a.T;
    const int64_t tok = (int64_t)s * a.T + t;
    if (threadIdx.x < a.k) {
        s_e[threadIdx.x] = a.topk_idx[tok * a.k + threadIdx.x];
        s_cnt[threadIdx.x] = 0;
    }
    __syncthreads();

    // Rank of each entry among the source's earlier entries with the same expert.
    const int64_t* tk = a.topk_idx + (int64_t)s * a.T * a.k;
    const int lim = t * a.k + a.k;
    for (int i = threadIdx.x; i < lim; i += kThreads) {
        const int64_t e = tk[i];
        if (e < 0) continue;
        for (int j = 0; j < a.k; ++j)
            if (e == s_e[j] && i < t * a.k + j) atomicAdd(&s_cnt[j], 1);
    }
    __syncthreads();

    if (threadIdx.x < a.k) {
        const int j = threadIdx.x;
        const int64_t e = s_e[j];
        int64_t row = -1;
        int32_t pos = -1;
        if (e >= a.E || e < -1) {
            raise_flag(a.err, EP_DEVERR_BAD_EXPERT);
        } else if (e >= 0) {
            if (s_cnt[j] >= a.nmax) {
                raise_flag(a.err, EP_DEVERR_SLOT_OVERFLOW);
            } else {
                const int d = (int)(e / a.E_loc), el = (int)(e - (int64_t)d * a.E_loc);
                pos = s * a.nmax + s_cnt[j];
                row = ((int64_t)d * a.E_loc + el) * slots + pos;
                a.src_info[row] = t;
            }
        }
        a.slot[tok * a.k + j] = pos;
        s_rows[j] = row;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int n = 0;
        for (int j = 0; j < a.k; ++j)
            if (s_rows[j] >= 0) s_rows[n++] = s_rows[j];
        s_nv = n;
    }
    __syncthreads();

    const char* src = a.x + tok * (int64_t)a.H * 2;
    if (a.use_fp8)
        scatter_quant_row<1>(src, reinterpret_cast<uint8_t*>(a.recv_x), a.recv_x_scales, s_rows, s_nv,
                             a.H, threadIdx.x, kThreads);
    else
        scatter_copy_row<2>(src, a.recv_x, s_rows, s_nv, (int64_t)a.H * 2, threadIdx.x, kThreads);
    pdl_trigger();
}

// One thread per (destination rank, local expert) = expert e.
__global__ void __launch_bounds__(kThreads) ll_recv_kernel(LLArgs a) {
    const int e = blockIdx.x * kThreads + threadIdx.x;
    pdl_trigger();
    pdl_wait();
    if (e >= a.E) return;
    int total = 0;
    for (int s = 0; s < a.R; ++s) {
        const int c = a.send_count[(int64_t)e * a.R + s];
        total += c;
        a.layout_range[((int64_t)e * a.R + s) * 2 + 0] = s * a.nmax;
        a.layout_range[((int64_t)e * a.R + s) * 2 + 1] = c;
    }
    a.recv_expert_count[e] = total;
}

// One block per output token: weighted sum over the token's valid entries.
__global__ void __launch_bounds__(kThreads) ll_combine_kernel(LLArgs a) {
    __shared__ int64_t s_rows[EP_MAX_TOPK];
    __shared__ float s_w[EP_MAX_TOPK];
    __shared__ int s_nv;
    const int64_t tok = blockIdx.x;
    const int64_t slots = (int64_t)a.R * a.nmax;
    pdl_wait();
    if (threadIdx.x < a.k) {
        const int j = threadIdx.x;
        const int64_t e = a.topk_idx[tok * a.k + j];
        const int32_t pos = a.slot[tok * a.k + j];
        int64_t row = -1;
        if (e >= 0 && e < a.E && pos >= 0 && pos < slots) {
            const int d = (int)(e / a.E_loc), el = (int)(e - (int64_t)d * a.E_loc);
            row = ((int64_t)d * a.E_loc + el) * slots + pos;
        }
        s_rows[j] = row;
        s_w[j] = a.topk_weights[tok * a.k + j];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int n = 0;
        for (int j = 0; j < a.k; ++j)
            if (s_rows[j] >= 0) {
                s_rows[n] = s_rows[j];
                s_w[n] = s_w[j];
                ++n;
            }
        s_nv = n;
    }
    __syncthreads();
    gather_reduce_row<1>(a.y, s_rows, s_w, s_nv, a.H, a.out + tok * (int64_t)a.H * 2, threadIdx.x, kThreads);
    pdl_trigger();
}

ep_status ll_common_checks(const ep_shape* sh, const ep_launch* launch) {
    ep_status st = check_shape(sh);
    if (st != EP_OK) return st;
    if (launch == nullptr) return EP_ERR_INVALID_ARG;
    if (sh->num_max_dispatch_tokens_per_rank < 1) return EP_ERR_INVALID_ARG;
    if (sh->num_tokens > sh->num_max_dispatch_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if ((int64_t)sh->num_ranks * sh->num_max_dispatch_tokens_per_rank > (int64_t)1 << 30)
        return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

}  // namespace
}  // namespace ep

extern "C" {

ep_status ep_ll_dispatch(const ep_shape* sh, const void* x, const int64_t* topk_idx, int use_fp8,
                         ep_phase phase, ep_ll_buffer* buf, const ep_launch* launch) {
    using namespace ep;
    ep_status st = ll_common_checks(sh, launch);
    if (st != EP_OK) return st;
    if (buf == nullptr || (phase & EP_PHASE_BOTH) == 0 || (phase & ~EP_PHASE_BOTH) != 0)
        return EP_ERR_INVALID_ARG;
    if (buf->send_count == nullptr) return EP_ERR_INVALID_ARG;
    if (phase & EP_PHASE_SEND) {
        if (buf->recv_x == nullptr || buf->src_info == nullptr || buf->slot == nullptr)
            return EP_ERR_INVALID_ARG;
        if (sh->num_tokens > 0 && (x == nullptr || topk_idx == nullptr)) return EP_ERR_INVALID_ARG;
        if (use_fp8 && buf->recv_x_scales == nullptr) return EP_ERR_INVALID_ARG;
        if (((uintptr_t)x & 15) != 0 || ((uintptr_t)buf->recv_x & 15) != 0) return EP_ERR_INVALID_ARG;
    }
    if ((phase & EP_PHASE_RECV) && (buf->recv_expert_count == nullptr || buf->layout_range == nullptr))
        return EP_ERR_INVALID_ARG;

    LLArgs a{};
    a.x = reinterpret_cast<const char*>(x);
    a.topk_idx = topk_idx;
    a.recv_x = reinterpret_cast<char*>(buf->recv_x);
    a.recv_x_scales = buf->recv_x_scales;
    a.src_info = buf->src_info;
    a.slot = buf->slot;
    a.send_count = buf->send_count;
    a.recv_expert_count = buf->recv_expert_count;
    a.layout_range = buf->layout_range;
    a.R = sh->num_ranks;
    a.T = sh->num_tokens;
    a.H = sh->hidden;
    a.E = sh->num_experts;
    a.k = sh->num_topk;
    a.E_loc = a.E / a.R;
    a.nmax = sh->num_max_dispatch_tokens_per_rank;
    a.use_fp8 = use_fp8 ? 1 : 0;
    a.err = launch->error_flags;

    if ((st = begin_call(launch)) != EP_OK) return st;
    if (phase & EP_PHASE_SEND) {
        const unsigned blocks = (unsigned)(a.R * a.T + a.R);
        cudaError_t e = launch_pdl(ll_send_kernel, dim3(blocks), dim3(kThreads),
                                   sizeof(int) * (size_t)a.E, launch->stream, a);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (phase & EP_PHASE_RECV) {
        cudaError_t e = launch_pdl(ll_recv_kernel, dim3((unsigned)ceil_div(a.E, kThreads)),
                                   dim3(kThreads), 0, launch->stream, a);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return end_call(launch);
}

ep_status ep_ll_combine(const ep_shape* sh, const void* y, const int64_t* topk_idx,
                        const float* topk_weights, const ep_ll_buffer* handle, ep_phase phase,
                        void* out, const ep_launch* launch) {
    using namespace ep;
    ep_status st = ll_common_checks(sh, launch);
    if (st != EP_OK) return st;
    if ((phase & EP_PHASE_BOTH) == 0 || (phase & ~EP_PHASE_BOTH) != 0) return EP_ERR_INVALID_ARG;
    if (phase & EP_PHASE_RECV) {
        if (handle == nullptr || handle->slot == nullptr) return EP_ERR_INVALID_ARG;
        if (sh->num_tokens > 0 && (y == nullptr || topk_idx == nullptr || topk_weights == nullptr || out == nullptr))
            return EP_ERR_INVALID_ARG;
        if (((uintptr_t)y & 15) != 0 || ((uintptr_t)out & 15) != 0) return EP_ERR_INVALID_ARG;
    }
    LLArgs a{};
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.slot = handle ? handle->slot : nullptr;
    a.y = reinterpret_cast<const char*>(y);
    a.out = reinterpret_cast<char*>(out);
    a.R = sh->num_ranks;
    a.T = sh->num_tokens;
    a.H = sh->hidden;
    a.E = sh->num_experts;
    a.k = sh->num_topk;
    a.E_loc = a.E / a.R;
    a.nmax = sh->num_max_dispatch_tokens_per_rank;
    a.err = launch->error_flags;

    if ((st = begin_call(launch)) != EP_OK) return st;
    // Send phase: in one device memory the return transfer is nothing; the call only
    // orders the stream (wait_event) and records the completion event.
    if ((phase & EP_PHASE_RECV) && a.R * a.T > 0) {
        cudaError_t e = launch_pdl(ll_combine_kernel, dim3((unsigned)(a.R * a.T)), dim3(kThreads), 0,
                                   launch->stream, a);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return end_call(launch);
}

ep_status ep_clean_ll_buffer(const ep_shape* sh, ep_ll_buffer* buf, const ep_launch* launch) {
    using namespace ep;
    ep_status st = check_shape(sh);
    if (st != EP_OK) return st;
    if (buf == nullptr || launch == nullptr) return EP_ERR_INVALID_ARG;
    if ((st = begin_call(launch)) != EP_OK) return st;
    const size_t E = (size_t)sh->num_experts, R = (size_t)sh->num_ranks;
    cudaError_t e = cudaSuccess;
    if (buf->send_count) e = cudaMemsetAsync(buf->send_count, 0, sizeof(int32_t) * E * R, launch->stream);
    if (e == cudaSuccess && buf->recv_expert_count)
        e = cudaMemsetAsync(buf->recv_expert_count, 0, sizeof(int32_t) * E, launch->stream);
    if (e == cudaSuccess && buf->layout_range)
        e = cudaMemsetAsync(buf->layout_range, 0, sizeof(int32_t) * E * R * 2, launch->stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return end_call(launch);
}

}  // extern "C"
