// dispatch.cu -- normal-mode dispatch: every source token row is read once and
// stored to each virtual rank it is routed to.
//
// [README] "DeepEP" README (EnflameTechnology/DeepEP), normal-kernel example:
//          dispatch(x, topk_idx, topk_weights, ...) -> recv_x, recv_topk_idx,
//          recv_topk_weights, num_recv_tokens_per_expert_list, handle; x may be bf16
//          or a pre-quantised (fp8, scales) tuple; feature notes: FP8 dispatch with
//          per-group scales; combine_backward = dispatch with the handle.
// [REUSE]  "How DeepEP Optimizes Handle Reuse for Repeated Dispatches", "Fast Path
//          Dispatch with Handle Reuse": with a handle, no topk is passed and the
//          cached layout is used directly.
//
// One warp per source token: the warp reads the token's send_head row, compacts the
// destination rows into shared memory (ballot + popc, ascending rank order), writes
// the per-row metadata, then moves the payload. In one device memory the all-to-all
// reduces to this scatter; nothing is exchanged between GPUs. Three kernels:
//   dispatch_tma_kernel      copies (bf16, or pre-quantised e4m3): one bulk copy loads
//                            the row into shared memory, one bulk copy per destination
//                            stores it (rows up to 50 KB);
//   dispatch_kernel<copy>    the same copy with 16-byte vector loads / stores (wider rows);
//   dispatch_kernel<quant>   fused e4m3 quantisation, software-pipelined row loads
//                            (32-byte loads when x is 32-byte aligned; pairs of units
//                            with 32-byte stores when the receive rows are too).
#include "rowops.cuh"

namespace ep {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

enum { kCopy = 0, kQuant = 1, kQuantPair = 2 };

struct DispatchArgs {
    const char* x;
    const float* x_scales;          // pre-quantised input only
    const int64_t* topk_idx;        // nullable (handle reuse)
    const float* topk_weights;      // nullable
    const int32_t* send_head;
    char* recv_x;
    void* recv_x_scales;
    int64_t* recv_topk_idx;
    float* recv_topk_weights;
    int32_t* recv_src_idx;
    RowOffsets off;
    int R, T, H, k, E_loc;
    int in_elem;                    // bytes per element of x
    int copy_scales;                // pre-quantised input: copy x_scales rows too
    QuantMode qm;                   // fused quantisation: scale format
    int64_t ntok;                   // R * T
    uint32_t* err;
};

// Destination rows of token g in ascending rank order into s_row / s_dst (overflowing
// rows flagged and dropped), then the per-row metadata: recv_src_idx, and recv_topk_idx /
// recv_topk_weights when the routing is given. Returns the number of destinations.
__device__ __forceinline__ int token_rows_and_meta(const DispatchArgs& a, int64_t g, int t, int lane,
                                                   int64_t* s_row, int* s_dst) {
    // Every metadata load of the token first (one memory round trip): send_head entries
    // (lanes d and d + 32), and the expert ids and weights (lanes < k).
    const int h0 = lane < a.R ? a.send_head[g * a.R + lane] : -1;
    const int h1 = lane + 32 < a.R ? a.send_head[g * a.R + lane + 32] : -1;
    int64_t e = -1;
    float wgt = 0.0f;
    if (a.topk_idx != nullptr && lane < a.k) {
        e = a.topk_idx[g * a.k + lane];
        if (a.topk_weights != nullptr) wgt = a.topk_weights[g * a.k + lane];
    }
    int nd = 0;
    for (int d0 = 0; d0 < a.R; d0 += 32) {
        const int d = d0 + lane;
        int64_t row = -1;
        if (d < a.R) {
            const int h = d0 == 0 ? h0 : h1;
            if (h >= 0) {
                row = a.off.v[d] + h;
                if (row >= a.off.v[d + 1]) {
                    raise_flag(a.err, EP_DEVERR_RECV_OVERFLOW);
                    row = -1;
                }
            }
        }
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, row >= 0);
        if (row >= 0) {
            const int p = nd + __popc(bal & lanemask_lt());
            s_row[p] = row;
            s_dst[p] = d;
        }
        nd += __popc(bal);
    }
    __syncwarp();

    if (a.recv_src_idx != nullptr)
        for (int p = lane; p < nd; p += 32) a.recv_src_idx[s_row[p]] = t;
    if (a.topk_idx != nullptr && lane < a.k) {
        for (int p = 0; p < nd; ++p) {
            const int64_t row = s_row[p];
            const int d = s_dst[p];
            const bool local = e >= 0 && e / a.E_loc == d;
            a.recv_topk_idx[row * a.k + lane] = local ? e - (int64_t)d * a.E_loc : -1;
            if (a.recv_topk_weights != nullptr)
                a.recv_topk_weights[row * a.k + lane] = local ? wgt : 0.0f;
        }
    }
    return nd;
}

// Pre-quantised input: the token's scales go to every destination row unchanged.
__device__ __forceinline__ void copy_scale_rows(const DispatchArgs& a, int64_t g, const int64_t* s_row,
                                                int nd, int lane) {
    const int G = a.H >> 7;
    const float* ss = a.x_scales + g * G;
    float* rs = reinterpret_cast<float*>(a.recv_x_scales);
    for (int p = 0; p < nd; ++p)
        for (int i = lane; i < G; i += 32) rs[s_row[p] * G + i] = ss[i];
}

template <int MODE, int U, bool V32 = false, int MIN_BLOCKS = 3>
__global__ void __launch_bounds__(kThreads, MIN_BLOCKS) dispatch_kernel(DispatchArgs a) {
    __shared__ int64_t s_row[kWarps][EP_MAX_RANKS];
    __shared__ int s_dst[kWarps][EP_MAX_RANKS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t out_row_bytes = (int64_t)a.H * (MODE == kCopy ? a.in_elem : 1);
    pdl_wait();

    for (int64_t g = (int64_t)blockIdx.x * kWarps + warp; g < a.ntok; g += nw) {
        const int t = (int)(g % a.T);
        const char* src = a.x + g * (int64_t)a.H * a.in_elem;
        // Quantising: the row's first batch does not depend on the metadata, so its load
        // shares the metadata's memory round trip.
        uint4 qa[U], qb[U];
        u32x8 qp[2];
        if (MODE == kQuant) quant_load<U, V32>(src, a.H >> 4, 0, lane, 32, qa, qb);
        if (MODE == kQuantPair) pair_load(src, a.H >> 5, lane, qp);

        const int nd = token_rows_and_meta(a, g, t, lane, s_row[warp], s_dst[warp]);

        // Payload.
        if (MODE == kCopy) {
            scatter_copy_row<U>(src, a.recv_x, s_row[warp], nd, out_row_bytes, lane, 32);
            if (a.copy_scales) copy_scale_rows(a, g, s_row[warp], nd, lane);
        } else if (MODE == kQuantPair) {
            scatter_quant_pairs_loaded(src, reinterpret_cast<uint8_t*>(a.recv_x), a.recv_x_scales,
                                       s_row[warp], nd, a.H, a.qm, lane, qp);
        } else {
            scatter_quant_row_loaded<U, V32>(src, reinterpret_cast<uint8_t*>(a.recv_x), a.recv_x_scales,
                                             s_row[warp], nd, a.H, a.qm, lane, 32, 0, qa, qb);
        }
        __syncwarp();
    }
    pdl_trigger();
}

// Copy modes with bulk copies (tma_row_load / tma_row_store): one warp per source token;
// while lane 0's row load is in flight the lanes compute the destination rows and write the
// metadata. The copy engine moves the payload, so the SM issues a few instructions per row
// instead of one per 16 bytes per destination, and a warp's next row can load while its
// earlier stores drain.
__global__ void __launch_bounds__(kTmaWarps * 32) dispatch_tma_kernel(DispatchArgs a) {
    extern __shared__ __align__(128) unsigned char rowbuf[];
    __shared__ int64_t s_row[kTmaWarps][EP_MAX_RANKS];
    __shared__ int s_dst[kTmaWarps][EP_MAX_RANKS];
    __shared__ __align__(8) uint64_t s_bar[kTmaWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t row_bytes = (uint32_t)a.H * (uint32_t)a.in_elem;
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
        const int nd = token_rows_and_meta(a, g, t, lane, s_row[warp], s_dst[warp]);
        if (a.copy_scales) copy_scale_rows(a, g, s_row[warp], nd, lane);
        if (lane == 0 && live)
            live = tma_row_store(buf, a.recv_x, s_row[warp], nd, row_bytes, &s_bar[warp], parity, a.err);
        __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
    pdl_trigger();
}

template <int MODE, int U, bool V32 = false, int MIN_BLOCKS = 3>
ep_status launch_dispatch(const DispatchArgs& a, int num_sms, cudaStream_t stream) {
    if (a.ntok == 0) return EP_OK;
    int64_t blocks = (a.ntok + kWarps - 1) / kWarps;
    if (num_sms > 0) {
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_kernel<MODE, U, V32, MIN_BLOCKS>, kThreads, 0);
        if (e != cudaSuccess) return cuda_fail(e);
        const int64_t cap = (int64_t)num_sms * (per_sm > 0 ? per_sm : 1);
        if (blocks > cap) blocks = cap;
    }
    if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
    cudaError_t e = launch_pdl(dispatch_kernel<MODE, U, V32, MIN_BLOCKS>, dim3((unsigned)blocks), dim3(kThreads), 0, stream, a);
    return e == cudaSuccess ? EP_OK : cuda_fail(e);
}

// Whether the copy fits the bulk-copy kernel: kTmaWarps rows of the token in shared memory.
bool tma_copy_fits(const DispatchArgs& a) {
    return (int64_t)kTmaWarps * a.H * a.in_elem <= kTmaSmemMax;
}

ep_status launch_dispatch_tma(const DispatchArgs& a, int num_sms, cudaStream_t stream) {
    if (a.ntok == 0) return EP_OK;
    const size_t smem = (size_t)kTmaWarps * (size_t)a.H * (size_t)a.in_elem;
    // Opt in to more than 48 KB of dynamic shared memory (per device, once is enough but
    // the call is cheap and enqueues nothing).
    cudaError_t e = cudaFuncSetAttribute(dispatch_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTmaSmemMax);
    if (e != cudaSuccess) return cuda_fail(e);
    int64_t blocks = (a.ntok + kTmaWarps - 1) / kTmaWarps;
    if (num_sms > 0) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_tma_kernel, kTmaWarps * 32, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        const int64_t cap = (int64_t)num_sms * (per_sm > 0 ? per_sm : 1);
        if (blocks > cap) blocks = cap;
    }
    if (blocks > 0x7FFFFFFF) blocks = 0x7FFFFFFF;
    e = launch_pdl(dispatch_tma_kernel, dim3((unsigned)blocks), dim3(kTmaWarps * 32), smem, stream, a);
    return e == cudaSuccess ? EP_OK : cuda_fail(e);
}

}  // namespace
}  // namespace ep

extern "C" ep_status ep_dispatch(const ep_shape* sh, const void* x, ep_dtype x_dtype,
                                 const float* x_scales, ep_dtype recv_dtype,
                                 const int64_t* topk_idx, const float* topk_weights,
                                 const ep_handle* handle, ep_recv* out, const ep_launch* launch) {
    using namespace ep;
    ep_status st = check_shape(sh);
    if (st != EP_OK) return st;
    if (handle == nullptr || out == nullptr || launch == nullptr) return EP_ERR_INVALID_ARG;
    const int64_t ntok = (int64_t)sh->num_ranks * sh->num_tokens;
    DispatchArgs a{};
    if ((st = load_row_offsets(out->row_offset, sh->num_ranks, &a.off)) != EP_OK) return st;
    // Receive buffers may be NULL when the regions hold no row at all (nothing is
    // written then; tokens that had a destination raise EP_DEVERR_RECV_OVERFLOW).
    const bool rows = a.off.v[sh->num_ranks] > a.off.v[0];
    if (ntok > 0 && handle->send_head == nullptr) return EP_ERR_INVALID_ARG;
    if (ntok > 0 && x == nullptr) return EP_ERR_INVALID_ARG;
    if (rows && out->recv_x == nullptr) return EP_ERR_INVALID_ARG;
    if (x_dtype == EP_FP8_E4M3 && recv_dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
    if (x_dtype != EP_BF16 && x_dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
    if (recv_dtype != EP_BF16 && recv_dtype != EP_FP8_E4M3) return EP_ERR_INVALID_ARG;
    if (recv_dtype == EP_FP8_E4M3 && rows && out->recv_x_scales == nullptr) return EP_ERR_INVALID_ARG;
    if (x_dtype == EP_FP8_E4M3 && ntok > 0 && x_scales == nullptr) return EP_ERR_INVALID_ARG;
    // Handle reuse passes no topk (the pages assert this); topk outputs then cannot be
    // produced. A first dispatch passes topk_idx and gets recv_topk_idx.
    // (With no token there is nothing to check: empty arrays may come as NULL.)
    if (ntok > 0 && topk_idx == nullptr && (topk_weights != nullptr || out->recv_topk_idx != nullptr ||
                                            out->recv_topk_weights != nullptr))
        return EP_ERR_INVALID_ARG;
    if (ntok > 0 && topk_idx != nullptr && rows && out->recv_topk_idx == nullptr) return EP_ERR_INVALID_ARG;
    if (ntok > 0 && topk_weights == nullptr && out->recv_topk_weights != nullptr) return EP_ERR_INVALID_ARG;
    // 16-byte vector access of rows.
    if (((uintptr_t)x & 15) != 0 || ((uintptr_t)out->recv_x & 15) != 0) return EP_ERR_INVALID_ARG;
    // Scale formats other than per-group fp32 apply to a fused quantisation only.
    const int fmt = out->fp8.scale_format;
    if (fmt < EP_FP8_SCALE_FP32 || fmt > EP_FP8_SCALE_TENSOR) return EP_ERR_INVALID_ARG;
    const bool fused = x_dtype == EP_BF16 && recv_dtype == EP_FP8_E4M3;
    if (fmt != EP_FP8_SCALE_FP32 && !fused) return EP_ERR_INVALID_ARG;
    if (fmt == EP_FP8_SCALE_TENSOR &&
        !(out->fp8.tensor_scale > 0.0f && out->fp8.tensor_scale <= 3.4028234e38f))
        return EP_ERR_INVALID_ARG;

    a.x = reinterpret_cast<const char*>(x);
    a.x_scales = x_scales;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.send_head = handle->send_head;
    a.recv_x = reinterpret_cast<char*>(out->recv_x);
    a.recv_x_scales = out->recv_x_scales;
    a.recv_topk_idx = out->recv_topk_idx;
    a.recv_topk_weights = out->recv_topk_weights;
    a.recv_src_idx = out->recv_src_idx;
    a.R = sh->num_ranks;
    a.T = sh->num_tokens;
    a.H = sh->hidden;
    a.k = sh->num_topk;
    a.E_loc = sh->num_experts / sh->num_ranks;
    a.in_elem = x_dtype == EP_BF16 ? 2 : 1;
    a.copy_scales = x_dtype == EP_FP8_E4M3 ? 1 : 0;
    a.qm.mode = fmt;
    a.qm.tscale = out->fp8.tensor_scale;
    a.qm.tinv = fmt == EP_FP8_SCALE_TENSOR ? 1.0f / out->fp8.tensor_scale : 0.0f;
    a.ntok = ntok;
    a.err = launch->error_flags;

    if ((st = begin_call(launch)) != EP_OK) return st;
    // Fused e4m3 with 32-byte loads. Short rows (a lane's one unit per row) and tokens with
    // at most two destinations trade load registers for resident warps (A/B on GB300, top-8
    // unless noted, fraction of the copy bandwidth: H = 1024 0.76 -> 0.90, H = 512 0.51 ->
    // 0.68; top-2 with H = 4096 0.945 -> 0.976). Rows with more destinations go by pairs of
    // units (one 32-byte store per destination and two shuffles per group instead of two
    // 16-byte stores and three: group_limited 0.980 -> 0.997, uniform top-8 0.934 -> 0.958)
    // when the receive rows are 32-byte aligned, else by units at three blocks per SM.
    const bool fp8_32 = x_dtype == EP_BF16 && recv_dtype == EP_FP8_E4M3 && ((uintptr_t)x & 31) == 0;
    if (fp8_32 && a.H <= 1024)
        st = launch_dispatch<kQuant, 1, true, 5>(a, sh->num_sms, launch->stream);
    else if (fp8_32 && (a.k <= 2 || a.R <= 2))
        st = launch_dispatch<kQuant, 2, true, 4>(a, sh->num_sms, launch->stream);
    else if (fp8_32 && ((uintptr_t)out->recv_x & 31) == 0)
        st = launch_dispatch<kQuantPair, 1, true>(a, sh->num_sms, launch->stream);
    else if (fp8_32)
        st = launch_dispatch<kQuant, 2, true>(a, sh->num_sms, launch->stream);
    else if (x_dtype == EP_BF16 && recv_dtype == EP_FP8_E4M3)
        st = launch_dispatch<kQuant, 2>(a, sh->num_sms, launch->stream);
    else if (tma_copy_fits(a))
        st = launch_dispatch_tma(a, sh->num_sms, launch->stream);
    else
        st = launch_dispatch<kCopy, 8>(a, sh->num_sms, launch->stream);
    if (st != EP_OK) return st;
    return end_call(launch);
}
