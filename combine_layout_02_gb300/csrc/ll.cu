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
//   s*Nmax + #{(t', j') before (t, j) in source s with expert e}   (its in-source rank).
//
// Packed variant (no gaps between the sources): entry (t, j) of source s takes
//   sum over s' < s of count[s'][e] + (the same in-source rank),
// so the per-source counts must exist before any row is placed.
//
// Send phase, both layouts, two kernels:
//   ll_rank_kernel -- one block per source: the in-source rank of every entry, in entry
//       order, chunk by chunk (a match-any vote within each warp, a table of per-warp
//       counts per expert scanned across the warps, a running count per expert across
//       chunks): linear in the source's T*k entries. It writes the slot array (the final
//       slot, or the in-source rank for the packed layout) and the per-(destination,
//       expert, source) counts, the signals the receive phase reads. It waits for
//       everything earlier before it triggers the send kernel's launch.
//   ll_send_kernel -- one block per source token: loads its row and its expert ids and
//       quantises the row while the rank kernel runs, waits for it (programmatic
//       dependent launch), reads its slots (adding the earlier sources' counts for the
//       packed layout), then stores the row to every destination slot.
// With the receive phase in the same call, R extra blocks of the send kernel turn the
// signals into recv_expert_count / layout_range.
#include <mutex>

#include "rowops.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;
constexpr int kCombineU = 1;        // units per thread per batch in the LL combine
constexpr int kSendThreads = 128;   // threads per token block of the send kernel
constexpr int kSendPre = 8;         // 16-byte row pieces per thread loaded before the wait
constexpr int kSendBlocksPerSm = 7; // the decode shape's 1024 token blocks in one wave
constexpr int kRankThreads = 1024;  // rank kernel: one block per source
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kRankSmemMax = 96 * 1024;       // [warps per chunk][E] table + [E] counts

// Warps (of 32 entries each) per chunk of the rank kernel, so that its table and the
// running counts fit (at least one warp: 64 KB at the largest E).
inline int rank_chunk_warps(int E) {
    const int w = kRankSmemMax / (int)(sizeof(int) * E) - 1;
    return w < 1 ? 1 : (w > kRankWarps ? kRankWarps : w);
}

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
    int cw;                         // rank kernel: warps per chunk
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

// An expert id as int32: ids in [-1, E) unchanged, anything else -2 (a bad entry).
__device__ __forceinline__ int ll_id32(int64_t e, int E) { return (e >= -1 && e < E) ? (int)e : -2; }

// Send phase, first kernel: block s ranks source s's entries (see the file header). The
// entries go through in chunks of cw warps x 32 entries, in entry order: within a warp
// the rank is the number of earlier lanes with the same expert (match-any vote); the
// warp's count per expert goes into a [cw][E] table, whose exclusive scan over the warps,
// started at the expert's running count of the earlier chunks, gives each warp's base.
__global__ void __launch_bounds__(kRankThreads) ll_rank_kernel(LLArgs a) {
    extern __shared__ int rsm[];
    int* wtab = rsm;                  // [cw][E]
    int* carry = rsm + a.cw * a.E;    // [E] running count per expert
    const int s = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = a.T * a.k, chunk = a.cw * 32;
    const bool act = warp < a.cw;
    const int64_t* tk = a.topk_idx + (int64_t)s * n;
    int32_t* slot = a.slot + (int64_t)s * n;
    // Everything earlier in the stream is complete past this wait, so the send kernel may
    // read the call's inputs as soon as it starts.
    pdl_wait();
    pdl_trigger();
    int cur = (act && warp * 32 + lane < n) ? ll_id32(__ldg(tk + warp * 32 + lane), a.E) : -1;
    for (int e = threadIdx.x; e < a.E; e += kRankThreads) carry[e] = 0;
    for (int c0 = 0; c0 < n; c0 += chunk) {              // block-uniform trip count
        const int i = c0 + warp * 32 + lane;
        const int in = i + chunk;
        const int nxt = (act && in < n) ? ll_id32(__ldg(tk + in), a.E) : -1;   // next chunk
        for (int x = threadIdx.x; x < a.cw * a.E; x += kRankThreads) wtab[x] = 0;
        __syncthreads();
        const int e = cur;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, e >= 0 ? e : -1 - lane);
        const int rw = __popc(peers & lanemask_lt());
        if (act && e >= 0 && rw == 0) wtab[warp * a.E + e] = __popc(peers);
        __syncthreads();
        for (int ee = threadIdx.x; ee < a.E; ee += kRankThreads) {
            int v[kRankWarps];
#pragma unroll
            for (int w = 0; w < kRankWarps; ++w) v[w] = w < a.cw ? wtab[w * a.E + ee] : 0;
            int c = carry[ee];
#pragma unroll
            for (int w = 0; w < kRankWarps; ++w) {
                if (w < a.cw) wtab[w * a.E + ee] = c;
                c += v[w];
            }
            carry[ee] = c;
        }
        __syncthreads();
        if (act && i < n) {
            int32_t pos = -1;
            if (e == -2) {
                raise_flag(a.err, EP_DEVERR_BAD_EXPERT);
            } else if (e >= 0) {
                const int rank = wtab[warp * a.E + e] + rw;
                if (rank >= a.nmax) raise_flag(a.err, EP_DEVERR_SLOT_OVERFLOW);
                else pos = a.packed ? rank : s * a.nmax + rank;
            }
            slot[i] = pos;
        }
        cur = nxt;
        __syncthreads();                                 // the table is reused
    }
    for (int e = threadIdx.x; e < a.E; e += kRankThreads)
        a.send_count[(int64_t)e * a.R + s] = min(carry[e], a.nmax);
}

// Blocks [0, R*T): one per source token. With the receive phase in the same call
// (write_recv), blocks [R*T, R*T + R): destination d's recv_expert_count and
// layout_range from the rank kernel's signals.
__global__ void __launch_bounds__(kSendThreads, kSendBlocksPerSm) ll_send_kernel(LLArgs a) {
    __shared__ int64_t s_e[EP_MAX_TOPK];
    __shared__ int64_t s_rows[EP_MAX_TOPK];
    __shared__ int s_nv;
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
    // The token's row and expert ids are inputs of the call: they are loaded while the
    // rank kernel runs.
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
    if (threadIdx.x < a.k) s_e[threadIdx.x] = a.topk_idx[tok * a.k + threadIdx.x];
    // The quantised units do not depend on where they go: quantise them while the rank
    // kernel still runs (block-uniform branch: every lane takes part in the shuffles).
    uint4 qv[kSendPre / 2];
    float qs[kSendPre / 2];
    uint32_t qb[kSendPre / 2];
    if (a.use_fp8) {
#pragma unroll
        for (int i = 0; i < kSendPre / 2; ++i) qv[i] = quant_unit(pre[2 * i], pre[2 * i + 1], a.qm, qs[i], qb[i]);
    }
    __syncthreads();
    // Nothing before this wait wrote: the rank kernel's slots and counts are complete
    // after it.
    pdl_wait();

    // Warp 0 (k <= 32 lanes) places the entries and compacts the valid rows in entry
    // order with a ballot.
    if (threadIdx.x < 32) {
        const int j = threadIdx.x;
        int64_t row = -1;
        if (j < a.k) {
            // The rank kernel flagged bad ids and overflows and gave them slot -1.
            const int32_t got = a.slot[tok * a.k + j];
            if (got >= 0) {
                const int64_t e = s_e[j];
                const int d = (int)(e / a.E_loc), el = (int)(e - (int64_t)d * a.E_loc);
                int32_t pos = got;
                if (a.packed) {          // got = in-source rank; add the earlier sources' counts
                    for (int src = 0; src < s; ++src) pos += a.send_count[e * a.R + src];
                    a.slot[tok * a.k + j] = pos;
                }
                row = ((int64_t)d * a.E_loc + el) * slots + pos;
                a.src_info[row] = t;
            }
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
        for (int i = 0; i < kSendPre / 2; ++i) { // the units quantised before the wait
            const int u = threadIdx.x + i * kSendThreads;
            if (u < qunits)
                store_quant_unit(q_base, a.recv_x_scales, s_rows, nv, a.H, u, qv[i], qs[i], qb[i], a.qm.mode);
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

// Lets the rank kernel use up to kRankSmemMax of dynamic shared memory (once per device).
cudaError_t rank_kernel_smem_attribute() {
    static std::mutex mu;
    static bool done[128];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        e = cudaFuncSetAttribute(ll_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRankSmemMax);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    return cudaSuccess;
}

ep_status ll_common_checks(const ep_shape* sh, const ep_launch* launch) {
    ep_status st = check_shape(sh);
    if (st != EP_OK) return st;
    if (launch == nullptr) return EP_ERR_INVALID_ARG;
    if (sh->num_max_dispatch_tokens_per_rank < 1) return EP_ERR_INVALID_ARG;
    if (sh->num_tokens > sh->num_max_dispatch_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if ((int64_t)sh->num_ranks * sh->num_max_dispatch_tokens_per_rank > (int64_t)1 << 30)
        return EP_ERR_UNSUPPORTED;
    // Entry counts of one source (T*k) and of all sources (R*T*k) are int32 in the kernels.
    if ((int64_t)sh->num_ranks * sh->num_tokens * sh->num_topk > (int64_t)INT32_MAX)
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
        a.cw = rank_chunk_warps(a.E);
        cudaError_t e = rank_kernel_smem_attribute();
        if (e == cudaSuccess)
            e = launch_pdl(ll_rank_kernel, dim3((unsigned)a.R), dim3(kRankThreads),
                                   sizeof(int) * (size_t)(a.cw + 1) * a.E, launch->stream, a);
        if (e == cudaSuccess) {
            // Token blocks, plus one receive-output block per destination with BOTH.
            const unsigned blocks = (unsigned)(a.R * a.T + (a.write_recv ? a.R : 0));
            if (blocks > 0)
                e = launch_pdl(ll_send_kernel, dim3(blocks), dim3(kSendThreads), 0, launch->stream, a);
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
