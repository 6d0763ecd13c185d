// expert_major.cu -- dispatch and combine in the expert-major packed layout: rank d's
// region holds one row per valid (token, k) entry whose expert lives on d, grouped by
// local expert (the handle's expert_rows / expert_prefix from ep_get_layout).
//
// [README] "DeepEP" README (EnflameTechnology/DeepEP), low-latency example: the
//          received rows come in a "specific format" for a grouped GEMM. Here the same
//          idea for the normal kernels: each local expert's rows are contiguous, so a
//          grouped GEMM can consume the region without a permutation.
//
// One warp per source token, like the rank-major kernels, but the destinations are the
// token's valid entries (one row each, ascending entry order) instead of its ranks.
#include "rowops.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCopyU = 8, kQuantU = 2, kGatherU = 4, kGatherP = 4;
constexpr int kCombineThreads = 128;    // combine: 4 warps per block, as the rank-major one
constexpr int kCombineWarps = kCombineThreads / 32;

struct EmArgs {
    const char* x;
    const int64_t* topk_idx;
    const float* topk_weights;   // nullable
    const int32_t* expert_rows;
    char* recv_x;
    void* recv_x_scales;
    float* recv_weights;         // nullable, [rows]
    int32_t* recv_src_idx;       // nullable, [rows]
    const char* y;
    char* out;
    RowOffsets off;
    int R, T, H, k, E, E_loc, weighted;
    int64_t ntok;
    QuantMode qm;
    uint32_t* err;
};

// Rows of token g's valid entries (ascending j) into s_row / s_coef; returns how many.
// coef = the entry's weight when weights are given, else 1.
__device__ __forceinline__ int entry_rows(const EmArgs& a, int64_t g, int lane, int64_t* s_row,
                                          float* s_coef) {
    int64_t row = -1;
    float w = 1.0f;
    if (lane < a.k) {
        const int64_t e = a.topk_idx[g * a.k + lane];
        const int r = a.expert_rows[g * a.k + lane];
        if (e >= 0 && e < a.E && r >= 0) {
            const int d = (int)(e / a.E_loc);
            row = a.off.v[d] + r;
            if (row >= a.off.v[d + 1]) {
                raise_flag(a.err, EP_DEVERR_RECV_OVERFLOW);
                row = -1;
            }
            if (a.topk_weights != nullptr) w = a.topk_weights[g * a.k + lane];
        }
    }
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, row >= 0);
    if (row >= 0) {
        const int p = __popc(bal & lanemask_lt());
        s_row[p] = row;
        s_coef[p] = w;
    }
    return __popc(bal);
}

// QUANT: fused e4m3, by units (PAIRS false) or by pairs of units with 32-byte stores
// (PAIRS true: x and the receive rows 32-byte aligned).
template <bool QUANT, bool V32 = false, bool PAIRS = false>
__global__ void __launch_bounds__(kThreads) dispatch_em_kernel(EmArgs a) {
    __shared__ int64_t s_row[kWarps][EP_MAX_TOPK];
    __shared__ float s_coef[kWarps][EP_MAX_TOPK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    pdl_wait();
    for (int64_t g = (int64_t)blockIdx.x * kWarps + warp; g < a.ntok; g += nw) {
        const int t = (int)(g % a.T);
        const char* src = a.x + g * (int64_t)a.H * 2;
        uint4 qa[kQuantU], qb[kQuantU];   // quantising: first batch loaded with the metadata
        u32x8 qp[2];
        if (QUANT && PAIRS) pair_load(src, a.H >> 5, lane, qp);
        else if (QUANT) quant_load<kQuantU, V32>(src, a.H >> 4, 0, lane, 32, qa, qb);
        const int nd = entry_rows(a, g, lane, s_row[warp], s_coef[warp]);
        __syncwarp();
        if (lane < nd) {
            const int64_t row = s_row[warp][lane];
            if (a.recv_src_idx != nullptr) a.recv_src_idx[row] = t;
            if (a.recv_weights != nullptr) a.recv_weights[row] = s_coef[warp][lane];
        }
        if (QUANT && PAIRS)
            scatter_quant_pairs_loaded(src, reinterpret_cast<uint8_t*>(a.recv_x), a.recv_x_scales,
                                       s_row[warp], nd, a.H, a.qm, lane, qp);
        else if (QUANT)
            scatter_quant_row_loaded<kQuantU, V32>(src, reinterpret_cast<uint8_t*>(a.recv_x), a.recv_x_scales,
                                                   s_row[warp], nd, a.H, a.qm, lane, 32, 0, qa, qb);
        else
            scatter_copy_row<kCopyU>(src, a.recv_x, s_row[warp], nd, (int64_t)a.H * 2, lane, 32);
        __syncwarp();
    }
    pdl_trigger();
}

// bf16 copy with bulk copies (tma_row_load / tma_row_store, as the rank-major dispatch):
// one warp per source token, its valid entries' rows as destinations.
__global__ void __launch_bounds__(kTmaWarps * 32) dispatch_em_tma_kernel(EmArgs a) {
    extern __shared__ __align__(128) unsigned char rowbuf[];
    __shared__ int64_t s_row[kTmaWarps][EP_MAX_TOPK];
    __shared__ float s_coef[kTmaWarps][EP_MAX_TOPK];
    __shared__ __align__(8) uint64_t s_bar[kTmaWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t row_bytes = (uint32_t)a.H * 2u;
    unsigned char* buf = rowbuf + (size_t)warp * row_bytes;
    const int64_t nw = (int64_t)gridDim.x * kTmaWarps;
    if (lane == 0) mbar_init(&s_bar[warp], 1);
    __syncwarp();
    pdl_wait();
    uint32_t parity = 0;
    bool live = true;       // lane 0: false once a row load failed to land in time
    for (int64_t g = (int64_t)blockIdx.x * kTmaWarps + warp; g < a.ntok; g += nw) {
        const int t = (int)(g % a.T);
        if (lane == 0 && live) tma_row_load(buf, a.x + g * (int64_t)row_bytes, row_bytes, &s_bar[warp]);
        const int nd = entry_rows(a, g, lane, s_row[warp], s_coef[warp]);
        __syncwarp();
        if (lane < nd) {
            const int64_t row = s_row[warp][lane];
            if (a.recv_src_idx != nullptr) a.recv_src_idx[row] = t;
            if (a.recv_weights != nullptr) a.recv_weights[row] = s_coef[warp][lane];
        }
        if (lane == 0 && live)
            live = tma_row_store(buf, a.recv_x, s_row[warp], nd, row_bytes, &s_bar[warp], parity, a.err);
        __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
    pdl_trigger();
}

// The batch shape (units per lane U, rows P) and resident blocks per SM follow the row
// length and the entries per token, as in the rank-major combine (combine_em_form).
template <int U, int P, bool V32, int MIN_BLOCKS = 0>
__global__ void __launch_bounds__(kCombineThreads, MIN_BLOCKS) combine_em_kernel(EmArgs a) {
    __shared__ int64_t s_row[kCombineWarps][EP_MAX_TOPK];
    __shared__ float s_coef[kCombineWarps][EP_MAX_TOPK];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kCombineWarps;
    pdl_wait();
    for (int64_t g = (int64_t)blockIdx.x * kCombineWarps + warp; g < a.ntok; g += nw) {
        const int nd = entry_rows(a, g, lane, s_row[warp], s_coef[warp]);
        __syncwarp();
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

// Rows of at most 256 channels: 16-byte units, one per lane; up to 1024 channels: one
// 32-byte unit per lane per row; at most two entries per token: 2 rows per batch; the
// rest 2 units x 4 rows. The short-row and two-row forms keep more blocks resident.
using CombineEmKernel = void (*)(EmArgs);
CombineEmKernel combine_em_form(int H, int k, bool y32) {
    if (H <= 256) return combine_em_kernel<1, 4, false, 10>;
    if (!y32) return combine_em_kernel<kGatherU, kGatherP, false>;
    if (H <= 1024) return combine_em_kernel<1, 4, true, 8>;
    if (k <= 2) return combine_em_kernel<2, 2, true, 5>;
    return combine_em_kernel<2, 4, true>;
}

ep_status em_common(const ep_shape* sh, const ep_handle* handle, const int64_t* topk_idx,
                    const int64_t* row_offset, const ep_launch* launch, EmArgs* a) {
    ep_status st = check_shape(sh);
    if (st != EP_OK) return st;
    if (sh->num_experts > EP_EXPERT_MAJOR_MAX_EXPERTS) return EP_ERR_UNSUPPORTED;
    if (handle == nullptr || launch == nullptr) return EP_ERR_INVALID_ARG;
    const int64_t ntok = (int64_t)sh->num_ranks * sh->num_tokens;
    if (ntok > 0 && (handle->expert_rows == nullptr || topk_idx == nullptr)) return EP_ERR_INVALID_ARG;
    if ((st = load_row_offsets(row_offset, sh->num_ranks, &a->off)) != EP_OK) return st;
    a->topk_idx = topk_idx;
    a->expert_rows = handle->expert_rows;
    a->R = sh->num_ranks;
    a->T = sh->num_tokens;
    a->H = sh->hidden;
    a->k = sh->num_topk;
    a->E = sh->num_experts;
    a->E_loc = sh->num_experts / sh->num_ranks;
    a->ntok = ntok;
    a->err = launch->error_flags;
    return EP_OK;
}

}  // namespace
}  // namespace ep

extern "C" {

ep_status ep_dispatch_expert_major(const ep_shape* sh, const void* x, ep_dtype recv_dtype,
                                   const int64_t* topk_idx, const float* topk_weights,
                                   const ep_handle* handle, ep_recv* out, const ep_launch* launch) {
    using namespace ep;
    if (out == nullptr) return EP_ERR_INVALID_ARG;
    EmArgs a{};
    ep_status st = em_common(sh, handle, topk_idx, out->row_offset, launch, &a);
    if (st != EP_OK) return st;
    if (recv_dtype != EP_BF16 && recv_dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
    // Receive buffers may be NULL when the regions hold no row (nothing is written).
    const bool rows = a.off.v[a.R] > a.off.v[0];
    if (a.ntok > 0 && x == nullptr) return EP_ERR_INVALID_ARG;
    if (rows && out->recv_x == nullptr) return EP_ERR_INVALID_ARG;
    if (out->recv_topk_idx != nullptr) return EP_ERR_INVALID_ARG;   // one entry per row
    if (a.ntok > 0 && out->recv_topk_weights != nullptr && topk_weights == nullptr) return EP_ERR_INVALID_ARG;
    if (recv_dtype == EP_FP8_E4M3 && rows && out->recv_x_scales == nullptr) return EP_ERR_INVALID_ARG;
    if (((uintptr_t)x & 15) != 0 || ((uintptr_t)out->recv_x & 15) != 0) return EP_ERR_INVALID_ARG;
    const int fmt = out->fp8.scale_format;
    if (fmt < EP_FP8_SCALE_FP32 || fmt > EP_FP8_SCALE_TENSOR) return EP_ERR_INVALID_ARG;
    if (fmt != EP_FP8_SCALE_FP32 && recv_dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
    if (fmt == EP_FP8_SCALE_TENSOR &&
        !(out->fp8.tensor_scale > 0.0f && out->fp8.tensor_scale <= 3.4028234e38f))
        return EP_ERR_INVALID_ARG;
    a.x = reinterpret_cast<const char*>(x);
    a.topk_weights = topk_weights;
    a.recv_x = reinterpret_cast<char*>(out->recv_x);
    a.recv_x_scales = out->recv_x_scales;
    a.recv_weights = out->recv_topk_weights;
    a.recv_src_idx = out->recv_src_idx;
    a.qm.mode = fmt;
    a.qm.tscale = out->fp8.tensor_scale;
    a.qm.tinv = fmt == EP_FP8_SCALE_TENSOR ? 1.0f / out->fp8.tensor_scale : 0.0f;
    if ((st = begin_call(launch)) != EP_OK) return st;
    if (a.ntok > 0) {
        const size_t tma_smem = (size_t)kTmaWarps * (size_t)a.H * 2;
        cudaError_t e = cudaSuccess;
        if (recv_dtype == EP_FP8_E4M3) {
            const unsigned blocks = (unsigned)((a.ntok + kWarps - 1) / kWarps);
            const bool x32 = ((uintptr_t)x & 31) == 0, r32 = ((uintptr_t)out->recv_x & 31) == 0;
            e = x32 && r32   // 32-byte loads of the bf16 row, 32-byte stores of e4m3 pairs
                    ? launch_pdl(dispatch_em_kernel<true, true, true>, dim3(blocks), dim3(kThreads), 0, launch->stream, a)
                : x32 ? launch_pdl(dispatch_em_kernel<true, true>, dim3(blocks), dim3(kThreads), 0, launch->stream, a)
                      : launch_pdl(dispatch_em_kernel<true>, dim3(blocks), dim3(kThreads), 0, launch->stream, a);
        } else if (tma_smem <= (size_t)kTmaSmemMax) {
            e = cudaFuncSetAttribute(dispatch_em_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kTmaSmemMax);
            const unsigned blocks = (unsigned)((a.ntok + kTmaWarps - 1) / kTmaWarps);
            if (e == cudaSuccess)
                e = launch_pdl(dispatch_em_tma_kernel, dim3(blocks), dim3(kTmaWarps * 32), tma_smem,
                               launch->stream, a);
        } else {
            const unsigned blocks = (unsigned)((a.ntok + kWarps - 1) / kWarps);
            e = launch_pdl(dispatch_em_kernel<false>, dim3(blocks), dim3(kThreads), 0, launch->stream, a);
        }
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return end_call(launch);
}

ep_status ep_combine_expert_major(const ep_shape* sh, const void* y, const int64_t* y_row_offset,
                                  const ep_handle* handle, ep_combine_mode mode,
                                  const int64_t* topk_idx, const float* topk_weights, void* out,
                                  const ep_launch* launch) {
    using namespace ep;
    EmArgs a{};
    ep_status st = em_common(sh, handle, topk_idx, y_row_offset, launch, &a);
    if (st != EP_OK) return st;
    if (mode != EP_COMBINE_SUM && mode != EP_COMBINE_WEIGHTED) return EP_ERR_INVALID_ARG;
    const bool rows = a.off.v[a.R] > a.off.v[0];     // no row: y is never read
    if (a.ntok > 0 && (out == nullptr || (rows && y == nullptr))) return EP_ERR_INVALID_ARG;
    if (mode == EP_COMBINE_WEIGHTED && a.ntok > 0 && topk_weights == nullptr) return EP_ERR_INVALID_ARG;
    if (((uintptr_t)y & 15) != 0 || ((uintptr_t)out & 15) != 0) return EP_ERR_INVALID_ARG;
    a.y = reinterpret_cast<const char*>(y);
    a.out = reinterpret_cast<char*>(out);
    a.topk_weights = mode == EP_COMBINE_WEIGHTED ? topk_weights : nullptr;
    if ((st = begin_call(launch)) != EP_OK) return st;
    if (a.ntok > 0) {
        const unsigned blocks = (unsigned)((a.ntok + kCombineWarps - 1) / kCombineWarps);
        // 32-byte loads when y is 32-byte aligned (as the rank-major combine).
        cudaError_t e = launch_pdl(combine_em_form(a.H, a.k, ((uintptr_t)y & 31) == 0), dim3(blocks),
                                   dim3(kCombineThreads), 0, launch->stream, a);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return end_call(launch);
}

}  // extern "C"
