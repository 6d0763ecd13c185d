// combine.cu -- normal-mode combine: rows come back from every virtual rank a token
// was sent to and are reduced into token order.
//
// [README] "DeepEP" README (EnflameTechnology/DeepEP), normal-kernel example:
//          combine_forward = combine(x, handle) -> combined_x; dispatch_backward =
//          combine(grad_recv_x, handle, topk_weights=grad_recv_topk_weights), which
//          also reduces the weight gradients.
// [REUSE]  "How DeepEP Optimizes Handle Reuse for Repeated Dispatches", "Combining
//          with Handle Reuse".
//
// One warp per output token: the warp gathers the destination rows from send_head
// (ascending rank order) and their coefficients (1, or the sum of the token's weights
// whose experts live on that rank), then accumulates in fp32 registers and stores
// bf16 once. Each received row is read exactly once, with 32-byte loads when y is
// 32-byte aligned (16-byte loads otherwise). The batch shape (units per lane U, rows
// P) and the blocks kept resident per SM follow the row length and the rows per token,
// so that enough bytes are in flight per SM (see combine_form).
#include "rowops.cuh"

namespace ep {
namespace {

constexpr int kThreads = 128;   // 4 warps: measured faster than 64, 256 or 512 threads per block
constexpr int kWarps = kThreads / 32;
// Gather batch: P rows x U 16-byte units per lane in flight (best measured on GB300
// among U in {1,2,4} x P in {4,8}).
constexpr int kU = 4, kP = 4;
// With 32-byte-aligned y: 32-byte loads, 2 units x 4 rows per lane in flight (measured
// faster than the 16-byte form: 441 vs 450 us on the DeepSeek-V3 shape).
constexpr int kU32 = 2, kP32 = 4;

struct CombineArgs {
    const char* y;
    RowOffsets off;
    const int32_t* send_head;
    const int64_t* topk_idx;
    const float* topk_weights;
    const float* recv_topk_weights;
    char* out;
    float* combined_topk_weights;
    int R, T, H, k, E_loc, weighted;
    int64_t ntok;
    uint32_t* err;
};

// Metadata of token g held by the warp's lanes: lanes < k its expert id and weight,
// lane d (and d + 32) its send_head entry for destination d.
struct TokenMeta {
    int64_t e;
    float w;
    int h0, h1;
};

__device__ __forceinline__ TokenMeta load_meta(const CombineArgs& a, int64_t g, int lane) {
    TokenMeta m{-1, 0.0f, -1, -1};
    if (a.weighted && lane < a.k) {
        m.e = a.topk_idx[g * a.k + lane];
        m.w = a.topk_weights[g * a.k + lane];
    }
    if (lane < a.R) m.h0 = a.send_head[g * a.R + lane];
    if (lane + 32 < a.R) m.h1 = a.send_head[g * a.R + lane + 32];
    return m;
}

template <int U, int P, bool V32, int MIN_BLOCKS = 0>
__global__ void __launch_bounds__(kThreads, MIN_BLOCKS) combine_kernel(CombineArgs a) {
    __shared__ int64_t s_row[kWarps][EP_MAX_RANKS];
    __shared__ float s_coef[kWarps][EP_MAX_RANKS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    pdl_wait();

    for (int64_t g = (int64_t)blockIdx.x * kWarps + warp; g < a.ntok; g += nw) {
        // Every metadata load of the token is issued at once: lanes < k read the token's
        // expert ids and weights, lanes < R its send_head entries. The coefficient of
        // rank d is then a sum over warp shuffles (entries in ascending order).
        const TokenMeta cur = load_meta(a, g, lane);
        const int rank_j = cur.e >= 0 ? (int)(cur.e / a.E_loc) : -1;
        const float w_j = cur.w;
        int nd = 0;
        for (int d0 = 0; d0 < a.R; d0 += 32) {
            const int d = d0 + lane;
            int64_t row = -1;
            if (d < a.R) {
                const int h = d0 == 0 ? cur.h0 : cur.h1;
                if (h >= 0) {
                    row = a.off.v[d] + h;
                    if (row >= a.off.v[d + 1]) {
                        raise_flag(a.err, EP_DEVERR_RECV_OVERFLOW);
                        row = -1;
                    }
                }
            }
            float coef = 1.0f;
            if (a.weighted) {
                coef = 0.0f;
                for (int j = 0; j < a.k; ++j) {
                    const int rj = __shfl_sync(0xFFFFFFFFu, rank_j, j);
                    const float wj = __shfl_sync(0xFFFFFFFFu, w_j, j);
                    if (rj == d) coef += wj;
                }
            }
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, row >= 0);
            if (row >= 0) {
                const int p = nd + __popc(bal & lanemask_lt());
                s_row[warp][p] = row;
                s_coef[warp][p] = coef;
            }
            nd += __popc(bal);
        }
        __syncwarp();

        if (a.combined_topk_weights != nullptr && lane < a.k) {
            float sum = 0.0f;
            for (int p = 0; p < nd; ++p) sum += a.recv_topk_weights[s_row[warp][p] * a.k + lane];
            a.combined_topk_weights[g * a.k + lane] = sum;
        }

        if (V32)
            gather_reduce_row32<U, P>(a.y, s_row[warp], s_coef[warp], nd, a.H,
                                      a.out + g * (int64_t)a.H * 2, lane, 32);
        else
            gather_reduce_row<U, P>(a.y, s_row[warp], s_coef[warp], nd, a.H,
                                    a.out + g * (int64_t)a.H * 2, lane, 32);
        __syncwarp();
    }
    pdl_trigger();
}

// The kernel form for a shape. Short rows leave a token's gather with few bytes per lane,
// so those forms trade load registers for resident warps (A/B on GB300, fraction of the
// copy bandwidth, 2 units x 4 rows -> the chosen form, top-8 unless noted): H = 256
// 0.33 -> 0.77, H = 512 0.61 -> 0.96, H = 1024 0.95 -> 1.04; at most two rows per token
// (k <= 2 or R <= 2, H 4096-7168) 0.95-0.97 -> 1.01-1.02. Wider rows with more rows per
// token keep 2 units x 4 rows at 126 registers (four 128-thread blocks per SM).
using CombineKernel = void (*)(CombineArgs);
CombineKernel combine_form(int H, int k, int R, bool y32) {
    if (H <= 256) return combine_kernel<1, 4, false, 10>;   // 16-byte units: one per lane
    if (!y32) return combine_kernel<kU, kP, false>;
    if (H <= 1024) return combine_kernel<1, 4, true, 8>;    // one 32-byte unit per lane per row
    if (k <= 2 || R <= 2) return combine_kernel<kU32, 2, true, 5>;
    return combine_kernel<kU32, kP32, true>;
}

}  // namespace
}  // namespace ep

extern "C" ep_status ep_combine(const ep_shape* sh, const void* y, const int64_t* y_row_offset,
                                const ep_handle* handle, ep_combine_mode mode,
                                const int64_t* topk_idx, const float* topk_weights,
                                const float* recv_topk_weights, void* out,
                                float* combined_topk_weights, const ep_launch* launch) {
    using namespace ep;
    ep_status st = check_shape(sh);
    if (st != EP_OK) return st;
    if (handle == nullptr || launch == nullptr) return EP_ERR_INVALID_ARG;
    const int64_t ntok = (int64_t)sh->num_ranks * sh->num_tokens;
    CombineArgs a{};
    if ((st = load_row_offsets(y_row_offset, sh->num_ranks, &a.off)) != EP_OK) return st;
    // With no row in any region nothing is read from y / recv_topk_weights (every token
    // gets +0 and zero weight sums), so those may be NULL.
    const bool rows = a.off.v[sh->num_ranks] > a.off.v[0];
    if (ntok > 0 && handle->send_head == nullptr) return EP_ERR_INVALID_ARG;
    if (ntok > 0 && (out == nullptr || (rows && y == nullptr))) return EP_ERR_INVALID_ARG;
    if (mode != EP_COMBINE_SUM && mode != EP_COMBINE_WEIGHTED) return EP_ERR_INVALID_ARG;
    if (mode == EP_COMBINE_WEIGHTED && ntok > 0 && (topk_idx == nullptr || topk_weights == nullptr))
        return EP_ERR_INVALID_ARG;
    if (ntok > 0 && recv_topk_weights != nullptr && combined_topk_weights == nullptr)
        return EP_ERR_INVALID_ARG;
    if (ntok > 0 && rows && combined_topk_weights != nullptr && recv_topk_weights == nullptr)
        return EP_ERR_INVALID_ARG;
    if (((uintptr_t)y & 15) != 0 || ((uintptr_t)out & 15) != 0) return EP_ERR_INVALID_ARG;

    a.y = reinterpret_cast<const char*>(y);
    a.send_head = handle->send_head;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.recv_topk_weights = recv_topk_weights;
    a.out = reinterpret_cast<char*>(out);
    a.combined_topk_weights = combined_topk_weights;
    a.R = sh->num_ranks;
    a.T = sh->num_tokens;
    a.H = sh->hidden;
    a.k = sh->num_topk;
    a.E_loc = sh->num_experts / sh->num_ranks;
    a.weighted = mode == EP_COMBINE_WEIGHTED;
    a.ntok = ntok;
    a.err = launch->error_flags;

    if ((st = begin_call(launch)) != EP_OK) return st;
    if (ntok > 0) {
        const CombineKernel kernel = combine_form(a.H, a.k, a.R, ((uintptr_t)y & 31) == 0);
        int64_t blocks = (ntok + kWarps - 1) / kWarps;
        if (sh->num_sms > 0) {
            int per_sm = 0;
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
            if (e != cudaSuccess) return cuda_fail(e);
            const int64_t cap = (int64_t)sh->num_sms * (per_sm > 0 ? per_sm : 1);
            if (blocks > cap) blocks = cap;
        }
        cudaError_t e = launch_pdl(kernel, dim3((unsigned)blocks), dim3(kThreads), 0, launch->stream, a);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return end_call(launch);
}
