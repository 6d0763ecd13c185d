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
// The send kernel computes that count by a block-wide scan of the source's entries in
// earlier tokens (at most Nmax*k of them; one shared-memory lookup each, in a table from
// expert to the token's entry), plus the token's own earlier entries with the same
// expert (a match-any vote), so no block waits on another.
//
// Packed variant (no gaps between the sources): entry (t, j) of source s takes
//   sum over s' < s of count[s'][e] + (the same in-source rank),
// so the per-source counts must exist before any row is placed.
//
// Send phase, both layouts: a small kernel with one block per source writes the per-
// (destination, expert, source) counts (the count signals the receive phase reads) and
// lets the send kernel start at once; the send kernel loads its row and ranks its
// entries, then waits for the counts (programmatic dependent launch) before it writes
// anything. With the receive phase in the same call, R extra blocks of the send kernel
// turn the signals into recv_expert_count / layout_range.
#include "rowops.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;
constexpr int kCombineU = 1;        // units per thread per batch in the LL combine
constexpr int kSendThreads = 128;   // threads per token block of the send kernel
constexpr int kSendPre = 8;         // 16-byte row pieces per thread loaded before the scan
constexpr int kSendScanPre = 8;     // earlier entries per thread loaded up front

__device__ __forceinline__ int ceil_div_dev(int a, int b) { return (a + b - 1) / b; }

struct LLArgs {
    const char* x;
    const int64_t* topk_idx;
    const float* topk_weights;
    char* recv_x;
    void* recv_x_scales;
    int32_t* src_info;
    int32_t* slot;
    int32_t* send_count;
    int32_t* recv_expert_count;
    int32_t* layout_range;
    const char* y;
    char* out;
    int R, T, H, E, k, E_loc, nmax, use_fp8, write_recv, packed;
    int col_split;                  // combine: blocks per token (column ranges)
    QuantMode qm;                   // send phase with use_fp8: scale format
    uint32_t* err;
};

// Receive outputs of expert e, by one warp: lane s (and s + 32) loads the count signal of
// source s, so all of them go out at once; a shuffle scan over the lanes gives the packed
// layout's starts. layout_range[e][s] = (first slot of source s, count), recv_expert_count[e]
// = the sum.
__device__ __forceinline__ void expert_ranges_warp(const LLArgs& a, int64_t e, int lane) {
    const int c0 = lane < a.R ? a.send_count[e * a.R + lane] : 0;
    const int c1 = lane + 32 < a.R ? a.send_count[e * a.R + lane + 32] : 0;
    int i0 = c0, i1 = c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(0xFFFFFFFFu, i0, o);
        const int y1 = __shfl_up_sync(0xFFFFFFFFu, i1, o);
        if (lane >= o) {
            i0 += y0;
            i1 += y1;
        }
    }
    const int t0 = __shfl_sync(0xFFFFFFFFu, i0, 31), t1 = __shfl_sync(0xFFFFFFFFu, i1, 31);
    if (lane < a.R) {
        a.layout_range[(e * a.R + lane) * 2 + 0] = a.packed ? i0 - c0 : lane * a.nmax;
        a.layout_range[(e * a.R + lane) * 2 + 1] = c0;
    }
    if (lane + 32 < a.R) {
        a.layout_range[(e * a.R + lane + 32) * 2 + 0] = a.packed ? t0 + i1 - c1 : (lane + 32) * a.nmax;
        a.layout_range[(e * a.R + lane + 32) * 2 + 1] = c1;
    }
    if (lane == 0) a.recv_expert_count[e] = t0 + t1;
}

// Send phase, first kernel: block s counts source s's entries per expert (capped at
// Nmax, as the send kernel caps them) into send_count[e][s]. It waits for everything
// earlier, then lets the send kernel launch: that kernel reads only inputs before its
// own wait.
__global__ void __launch_bounds__(kThreads) ll_count_kernel(LLArgs a) {
    extern __shared__ int hist[];   // [E]
    const int s = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i < a.E; i += kThreads) hist[i] = 0;
    __syncthreads();
    const int64_t* tk = a.topk_idx + (int64_t)s * a.T * a.k;
#pragma unroll 4
    for (int i = threadIdx.x; i < a.T * a.k; i += kThreads) {
        const int64_t e = __ldg(tk + i);
        if (e >= 0 && e < a.E) atomicAdd(&hist[(int)e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += kThreads)
        a.send_count[(int64_t)e * a.R + s] = min(hist[e], a.nmax);
}

// Blocks [0, R*T): one per source token. With the receive phase in the same call
// (write_recv), blocks [R*T, R*T + R): destination d's recv_expert_count and
// layout_range from the count kernel's signals.
__global__ void __launch_bounds__(kSendThreads) ll_send_kernel(LLArgs a) {
    __shared__ int64_t s_e[EP_MAX_TOPK];
    __shared__ int s_cnt[EP_MAX_TOPK];
    __shared__ int64_t s_rows[EP_MAX_TOPK];
    __shared__ int s_nv;
    extern __shared__ int hist[];   // [E]: expert -> one of the token's entries
    const int b = blockIdx.x;
    const int64_t slots = (int64_t)a.R * a.nmax;

    if (b >= a.R * a.T) {
        const int d = b - a.R * a.T;
        pdl_wait();
        for (int el = threadIdx.x >> 5; el < a.E_loc; el += kSendThreads / 32)
            expert_ranges_warp(a, (int64_t)d * a.E_loc + el, threadIdx.x & 31);
        pdl_trigger();
        return;
    }

    const int s = b / a.T, t = b - s * a.T;
    const int64_t tok = (int64_t)s * a.T + t;
    const char* src = a.x + tok * (int64_t)a.H * 2;
    // The token's row does not depend on the slot ranks: load its first batch now, so the
    // load overlaps the rank scan below.
    const int qunits = a.H >> 4;                 // fp8: 16 channels per unit
    const int cunits = a.H >> 3;                 // bf16 copy: 8 channels per unit
    uint4 pre[kSendPre];
#pragma unroll
    for (int i = 0; i < kSendPre; ++i) {
        pre[i] = make_uint4(0, 0, 0, 0);
        if (a.use_fp8) {
            const int u = threadIdx.x + (i >> 1) * kSendThreads;
            if (u < qunits) pre[i] = ld_stream_v4(src + (int64_t)u * 32 + (i & 1) * 16);
        } else {
            const int u = threadIdx.x + i * kSendThreads;
            if (u < cunits) pre[i] = ld_stream_v4(src + (int64_t)u * 16);
        }
    }
    // The source's entries in earlier tokens (for the slot ranks) do not depend on this
    // token either: each thread loads its first kScanPre of them now, with the row and
    // the token's own ids, so all three share one memory round trip.
    const int64_t* tk = a.topk_idx + (int64_t)s * a.T * a.k;
    const int lim = t * a.k;
    int64_t pre_e[kSendScanPre];
#pragma unroll
    for (int q = 0; q < kSendScanPre; ++q) {
        const int i = threadIdx.x + q * kSendThreads;
        pre_e[q] = i < lim ? __ldg(tk + i) : -1;
    }
    // hist[e] (the block's E ints, not cleared): one of this token's entries with
    // expert e. A value left by another block is never used for an expert outside this
    // token: a lookup counts only if the entry it names has that very expert.
    if (threadIdx.x < a.k) {
        const int64_t e = a.topk_idx[tok * a.k + threadIdx.x];
        s_e[threadIdx.x] = e;
        s_cnt[threadIdx.x] = 0;
        if (e >= 0 && e < a.E) hist[(int)e] = threadIdx.x;
    }
    __syncthreads();

    // Count of the source's entries in earlier tokens with each of this token's experts,
    // booked on the entry the table names (one shared-memory lookup per entry).
#pragma unroll
    for (int q = 0; q < kSendScanPre; ++q) {
        const int64_t e = pre_e[q];
        if (e < 0 || e >= a.E) continue;
        const int j = hist[(int)e];
        if ((unsigned)j < (unsigned)a.k && s_e[j] == e) atomicAdd(&s_cnt[j], 1);
    }
    for (int i = threadIdx.x + kSendScanPre * kSendThreads; i < lim; i += kSendThreads) {
        const int64_t e = __ldg(tk + i);
        if (e < 0 || e >= a.E) continue;
        const int j = hist[(int)e];
        if ((unsigned)j < (unsigned)a.k && s_e[j] == e) atomicAdd(&s_cnt[j], 1);
    }
    __syncthreads();
    // Nothing before this wait wrote: the count kernel's signals (the packed layout's
    // earlier-source counts) are complete after it.
    pdl_wait();

    // Warp 0 (k <= 32 lanes) places the entries and compacts the valid rows in entry
    // order with a ballot.
    if (threadIdx.x < 32) {
        const int j = threadIdx.x;
        int64_t row = -1;
        // Rank = count in earlier tokens + this token's earlier entries with the same
        // expert (lanes >= k hold distinct values that match nothing).
        const int64_t ej = j < a.k ? s_e[j] : -2 - (int64_t)j;
        const unsigned same = __match_any_sync(0xFFFFFFFFu, (unsigned long long)ej);
        if (j < a.k) {
            const int64_t e = ej;
            int32_t pos = -1;
            if (e >= a.E || e < -1) {
                raise_flag(a.err, EP_DEVERR_BAD_EXPERT);
            } else if (e >= 0) {
                const int rank = s_cnt[hist[(int)e]] + __popc(same & lanemask_lt());
                if (rank >= a.nmax) {
                    raise_flag(a.err, EP_DEVERR_SLOT_OVERFLOW);
                } else {
                    const int d = (int)(e / a.E_loc), el = (int)(e - (int64_t)d * a.E_loc);
                    int start = s * a.nmax;
                    if (a.packed) {
                        start = 0;
                        for (int src = 0; src < s; ++src) start += a.send_count[e * a.R + src];
                    }
                    pos = start + rank;
                    row = ((int64_t)d * a.E_loc + el) * slots + pos;
                    a.src_info[row] = t;
                }
            }
            a.slot[tok * a.k + j] = pos;
        }
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, row >= 0);
        if (row >= 0) s_rows[__popc(bal & lanemask_lt())] = row;
        if (j == 0) s_nv = __popc(bal);
    }
    __syncthreads();
    const int nv = s_nv;

    if (a.use_fp8) {
        uint8_t* q_base = reinterpret_cast<uint8_t*>(a.recv_x);
#pragma unroll
        for (int i = 0; i < kSendPre / 2; ++i) { // the prefetched units (all lanes shuffle)
            const int u = threadIdx.x + i * kSendThreads;
            float scale;
            uint32_t sbyte;
            const uint4 q = quant_unit(pre[2 * i], pre[2 * i + 1], a.qm, scale, sbyte);
            if (u < qunits)
                store_quant_unit(q_base, a.recv_x_scales, s_rows, nv, a.H, u, q, scale, sbyte, a.qm.mode);
        }
        scatter_quant_row<1>(src, q_base, a.recv_x_scales, s_rows, nv, a.H, a.qm, threadIdx.x,
                             kSendThreads, kSendPre / 2 * kSendThreads);
    } else {
        for (int p = 0; p < nv; ++p) {
            char* dst = a.recv_x + s_rows[p] * (int64_t)a.H * 2;
#pragma unroll
            for (int i = 0; i < kSendPre; ++i) {
                const int u = threadIdx.x + i * kSendThreads;
                if (u < cunits) st_v4(dst + (int64_t)u * 16, pre[i]);
            }
        }
        for (int u = threadIdx.x + kSendPre * kSendThreads; u < cunits; u += kSendThreads) {
            const uint4 v = ld_stream_v4(src + (int64_t)u * 16);
            for (int p = 0; p < nv; ++p) st_v4(a.recv_x + s_rows[p] * (int64_t)a.H * 2 + (int64_t)u * 16, v);
        }
    }
    pdl_trigger();
}

// One warp per (destination rank, local expert) = expert e.
__global__ void __launch_bounds__(kThreads) ll_recv_kernel(LLArgs a) {
    const int64_t e = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    pdl_trigger();
    pdl_wait();
    if (e < a.E) expert_ranges_warp(a, e, threadIdx.x & 31);
}

// One block per output token: weighted sum over the token's valid entries.
// Block (token, column part): blockIdx.y selects a contiguous range of 16-byte units so
// that each thread's loads for the part are issued in one batch.
__global__ void __launch_bounds__(kThreads) ll_combine_kernel(LLArgs a) {
    __shared__ int64_t s_rows[EP_MAX_TOPK];
    __shared__ float s_w[EP_MAX_TOPK];
    __shared__ int s_nv;
    const int64_t tok = blockIdx.x;
    const int64_t slots = (int64_t)a.R * a.nmax;
    pdl_wait();
    if (threadIdx.x < 32) {                     // warp 0: rows and weights, compacted
        const int j = threadIdx.x;
        int64_t row = -1;
        float w = 0.0f;
        if (j < a.k) {
            const int64_t e = a.topk_idx[tok * a.k + j];
            const int32_t pos = a.slot[tok * a.k + j];
            w = a.topk_weights[tok * a.k + j];
            if (e >= 0 && e < a.E && pos >= 0 && pos < slots) {
                const int d = (int)(e / a.E_loc), el = (int)(e - (int64_t)d * a.E_loc);
                row = ((int64_t)d * a.E_loc + el) * slots + pos;
            }
        }
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, row >= 0);
        if (row >= 0) {
            const int p = __popc(bal & lanemask_lt());
            s_rows[p] = row;
            s_w[p] = w;
        }
        if (j == 0) s_nv = __popc(bal);
    }
    __syncthreads();
    const int units = a.H >> 3;
    const int per = ceil_div_dev(units, a.col_split);
    const int u_begin = blockIdx.y * per;
    gather_reduce_row<kCombineU>(a.y, s_rows, s_w, s_nv, a.H, a.out + tok * (int64_t)a.H * 2,
                                 threadIdx.x, kThreads, u_begin, min(units, u_begin + per));
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
        if (buf->recv_x == nullptr || buf->src_info == nullptr ||
            (sh->num_tokens > 0 && buf->slot == nullptr))
            return EP_ERR_INVALID_ARG;
        if (sh->num_tokens > 0 && (x == nullptr || topk_idx == nullptr)) return EP_ERR_INVALID_ARG;
        if (use_fp8 && sh->num_tokens > 0 && buf->recv_x_scales == nullptr) return EP_ERR_INVALID_ARG;
        const int fmt = buf->fp8.scale_format;
        if (fmt < EP_FP8_SCALE_FP32 || fmt > EP_FP8_SCALE_TENSOR) return EP_ERR_INVALID_ARG;
        if (fmt != EP_FP8_SCALE_FP32 && !use_fp8) return EP_ERR_INVALID_ARG;
        if (fmt == EP_FP8_SCALE_TENSOR &&
            !(buf->fp8.tensor_scale > 0.0f && buf->fp8.tensor_scale <= 3.4028234e38f))
            return EP_ERR_INVALID_ARG;
        if (((uintptr_t)x & 15) != 0 || ((uintptr_t)buf->recv_x & 15) != 0) return EP_ERR_INVALID_ARG;
    }
    if ((phase & EP_PHASE_RECV) && (buf->recv_expert_count == nullptr || buf->layout_range == nullptr))
        return EP_ERR_INVALID_ARG;
    if (buf->layout != EP_LL_LAYOUT_SLOTS && buf->layout != EP_LL_LAYOUT_PACKED) return EP_ERR_INVALID_ARG;

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
    a.write_recv = (phase & EP_PHASE_RECV) ? 1 : 0;
    a.packed = buf->layout == EP_LL_LAYOUT_PACKED ? 1 : 0;
    a.qm.mode = buf->fp8.scale_format;
    a.qm.tscale = buf->fp8.tensor_scale;
    a.qm.tinv = a.qm.mode == EP_FP8_SCALE_TENSOR ? 1.0f / buf->fp8.tensor_scale : 0.0f;
    a.err = launch->error_flags;

    if ((st = begin_call(launch)) != EP_OK) return st;
    if (phase & EP_PHASE_SEND) {
        cudaError_t e = launch_pdl(ll_count_kernel, dim3((unsigned)a.R), dim3(kThreads),
                                   sizeof(int) * (size_t)a.E, launch->stream, a);
        if (e == cudaSuccess) {
            // Token blocks, plus one receive-output block per destination with BOTH.
            const unsigned blocks = (unsigned)(a.R * a.T + (a.write_recv ? a.R : 0));
            if (blocks > 0)
                e = launch_pdl(ll_send_kernel, dim3(blocks), dim3(kSendThreads), sizeof(int) * (size_t)a.E,
                               launch->stream, a);
        }
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (phase == EP_PHASE_RECV) {
        // Receive phase launched on its own (the hook): turn the count signals written
        // by the send phase into counts and layout ranges. With EP_PHASE_BOTH the send
        // kernel's extra blocks already wrote them.
        cudaError_t e = launch_pdl(ll_recv_kernel, dim3((unsigned)ceil_div(a.E, kThreads / 32)),
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
        if (handle == nullptr || (sh->num_tokens > 0 && handle->slot == nullptr)) return EP_ERR_INVALID_ARG;
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
        a.col_split = 1;
        cudaError_t e = launch_pdl(ll_combine_kernel, dim3((unsigned)(a.R * a.T), (unsigned)a.col_split),
                                   dim3(kThreads), 0, launch->stream, a);
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
