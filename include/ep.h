/*
 * ep.h -- C ABI of libep: MoE expert-parallel layout / dispatch / combine on one GPU,
 * with the R expert-parallel ranks made virtual (partitions of one device's memory).
 *
 * Sources (cited by key below):
 *   [README]  "DeepEP" -- README of the EnflameTechnology/DeepEP port: normal-kernel
 *             example (get_dispatch_layout, dispatch, combine, dispatch_backward,
 *             combine_backward), low-latency example (low_latency_dispatch,
 *             low_latency_combine), and the feature notes (FP8 per-group scales,
 *             int32 low-latency counts, clean_low_latency_buffer).
 *   [OVERLAP] "How DeepEP Achieves Communication-Computation Overlapping with
 *             EventOverlap": previous_event / async_finish / current_stream_wait.
 *   [HOOK]    "How DeepEP Enables Hook-Based Overlapping Without SM Occupation":
 *             launch-stream choice, send / receive phase split.
 *   [REUSE]   "How DeepEP Optimizes Handle Reuse for Repeated Dispatches": handle
 *             contents, the reuse fast path and its contract.
 *
 * Notation: R = num_ranks, T = num_tokens (per source rank), H = hidden,
 * E = num_experts, E_loc = E / R, k = num_topk, C = num_channels,
 * Nmax = num_max_dispatch_tokens_per_rank. Expert e lives on rank e / E_loc.
 * Every multi-rank tensor is one allocation with a leading [R] axis (source rank s
 * first unless stated). bf16 = IEEE binary32 truncated to 16 bits; e4m3 = OCP FP8
 * E4M3 (max finite 448).
 *
 * General rules for every call:
 *   - All pointers marked "dev" are device pointers owned by the caller; the library
 *     never allocates, frees or retains memory, and keeps no state between calls
 *     other than per-device caches (the SM count, a kernel's shared-memory limit set
 *     once, the static-scratch array's address per context) and a launch counter.
 *   - Calls are asynchronous on launch->stream and never synchronise the host,
 *     except the functions whose name ends in _sync.
 *   - Argument errors are detected on the host before anything is enqueued and
 *     return EP_ERR_INVALID_ARG (or EP_ERR_UNSUPPORTED for shapes beyond the limits
 *     below). A failed launch returns EP_ERR_CUDA.
 *   - Problems only visible on the device (a topk_idx entry outside [-1, E), a row
 *     beyond its receive region, a low-latency slot beyond Nmax) skip the offending
 *     write and set a bit of *launch->error_flags (if non-NULL) with atomicOr. The
 *     kernels never trap, never spin and never wait on other blocks.
 *   - Limits: 1 <= R <= 64; E % R == 0; 1 <= k <= 32; H % 128 == 0 and H >= 128;
 *     T >= 0; C >= 1; E <= 8192.
 */
#ifndef COMBINE_LAYOUT_02_EP_H
#define COMBINE_LAYOUT_02_EP_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every function below is exported from libep.so (the library is built with hidden
 * visibility for everything else). */
#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

#define EP_MAX_RANKS 64
#define EP_MAX_TOPK 32
#define EP_MAX_EXPERTS 8192
#define EP_FP8_GROUP 128
#define EP_EXPERT_MAJOR_MAX_EXPERTS 4096

typedef int32_t ep_status;
#define EP_OK 0
#define EP_ERR_INVALID_ARG 1
#define EP_ERR_CUDA 2
#define EP_ERR_UNSUPPORTED 3

/* Bits of the device error word. */
#define EP_DEVERR_BAD_EXPERT 1u    /* a topk_idx entry outside [-1, E) was skipped */
#define EP_DEVERR_RECV_OVERFLOW 2u /* a row fell outside its receive region, skipped */
#define EP_DEVERR_SLOT_OVERFLOW 4u /* a low-latency slot index reached Nmax, skipped */
#define EP_DEVERR_TIMEOUT 8u       /* a bounded device wait gave up; the affected rows were skipped */

typedef enum ep_dtype { EP_BF16 = 0, EP_FP8_E4M3 = 1 } ep_dtype;
typedef enum ep_combine_mode { EP_COMBINE_SUM = 0, EP_COMBINE_WEIGHTED = 1 } ep_combine_mode;
typedef enum ep_phase { EP_PHASE_SEND = 1, EP_PHASE_RECV = 2, EP_PHASE_BOTH = 3 } ep_phase;

/* Scale format of a fused FP8 quantisation ([README] feature notes: FP8 dispatch with
 * per-group scales; round_scale; use_ue8m0, also for the low-latency kernels; a single
 * per-tensor scale fp8_quant_scale). Groups are 128 channels; amax' = max(amax, 1e-4).
 *   EP_FP8_SCALE_FP32   scale = amax'/448 (fp32), q = e4m3(x * (448/amax'))  [default]
 *   EP_FP8_SCALE_POW2   scale = 2^ceil(log2(amax'/448)) (fp32), q = e4m3(x / scale)
 *   EP_FP8_SCALE_UE8M0  as POW2, but each scale is stored as one byte, its biased
 *                       exponent (scale = 2^(byte - 127)); recv_x_scales is uint8
 *   EP_FP8_SCALE_TENSOR every group uses the caller's tensor_scale s (> 0, finite):
 *                       q = e4m3(x * (1/s)); s is written to every scale slot
 * q is rounded to nearest even and saturated to +-448 (OCP E4M3). */
typedef enum ep_fp8_scale {
    EP_FP8_SCALE_FP32 = 0,
    EP_FP8_SCALE_POW2 = 1,
    EP_FP8_SCALE_UE8M0 = 2,
    EP_FP8_SCALE_TENSOR = 3
} ep_fp8_scale;

typedef struct ep_fp8_options {
    int32_t scale_format;   /* ep_fp8_scale; 0 (zero-initialised) = EP_FP8_SCALE_FP32 */
    float tensor_scale;     /* EP_FP8_SCALE_TENSOR only */
} ep_fp8_options;

/* Problem shape. num_sms caps the grid of the copy kernels (0 = every SM of the
 * device); it plays the role of Buffer.set_num_sms in [README]. */
typedef struct ep_shape {
    int32_t num_ranks;
    int32_t num_tokens;
    int32_t hidden;
    int32_t num_experts;
    int32_t num_topk;
    int32_t num_channels;
    int32_t num_max_dispatch_tokens_per_rank;
    int32_t num_sms;
} ep_shape;

/* Stream and ordering of one call ([OVERLAP] "Propagation Through EP Operations";
 * [HOOK] "Compute Stream vs. Communication Stream").
 *   stream       -- every kernel of the call is enqueued here; the caller picks the
 *                   compute or a communication stream (the pages' launch_stream).
 *   wait_event   -- nullable; the stream waits on it before the first kernel
 *                   (previous_event).
 *   record_event -- nullable; recorded on the stream after the last kernel
 *                   (async_finish: the caller's current_stream_wait is
 *                   cudaStreamWaitEvent on it).
 *   error_flags  -- nullable dev uint32; device-detected problems are OR-ed in. */
typedef struct ep_launch {
    cudaStream_t stream;
    cudaEvent_t wait_event;
    cudaEvent_t record_event;
    uint32_t* error_flags;
} ep_launch;

/* Outputs of get_dispatch_layout ([README] normal-kernel example). All dev.
 *   num_tokens_per_rank      [R][R] int32: [s][d] = tokens of s that go to rank d
 *   num_tokens_per_rdma_rank must be NULL (there is one node, no RDMA domain)
 *   num_tokens_per_expert    [R][E] int32: [s][e] = valid entries of s equal to e
 *   is_token_in_rank         [R][T][R] uint8: 1 if some valid entry of the token lives
 *                            on rank d (a token counts once per rank); nullable when
 *                            the handle's copy is enough. */
typedef struct ep_layout {
    int32_t* num_tokens_per_rank;
    int32_t* num_tokens_per_rdma_rank;
    int32_t* num_tokens_per_expert;
    uint8_t* is_token_in_rank;
} ep_layout;

/* The dispatch handle ([REUSE] "What the Handle Contains"). All dev, caller-owned.
 *   rank_prefix_matrix         [R][R] int32: [s][d] = sum over s' <= s of
 *                              num_tokens_per_rank[s'][d] (inclusive; row R-1 holds
 *                              N_d, the rows rank d receives)
 *   channel_prefix_matrix      [R][R][C] int32: [s][d][c] = tokens of s in channels
 *                              <= c that go to d (inclusive; channel of token t is
 *                              t / ceil(T / C))
 *   recv_channel_prefix_matrix [R][R][C] int32: [d][s][c] = first row, in d's region,
 *                              of source s's channel c
 *   recv_src_idx               [rows] int32: token index (within its source rank) of
 *                              each received row; written by ep_dispatch
 *   is_token_in_rank           [R][T][R] uint8 (as in ep_layout)
 *   send_head                  [R][T][R] int32: row of (s, t) in d's region, or -1;
 *                              rows of d are ordered by (source rank, token)
 *   num_recv_tokens_per_expert [R][E_loc] int32: rows rank d receives per local
 *                              expert (the pages' num_recv_tokens_per_expert_list)
 * Optional expert-major placement (both NULL to skip; E <= EP_EXPERT_MAJOR_MAX_EXPERTS;
 * reading of [README] low-latency example: received rows in a "specific format" for a
 * grouped GEMM, here for the normal kernels): rank d's region holds one row per valid
 * (token, k) entry whose expert lives on d, grouped by local expert, then source rank,
 * then token. Experts within one token must be distinct for this placement.
 *   expert_rows                [R][T][k] int32: row of entry (s, t, j) in its
 *                              destination's region, -1 if masked
 *   expert_prefix              [R][E_loc + 1] int32: first row of each local expert;
 *                              [d][E_loc] = rows rank d receives (sum of its entries) */
typedef struct ep_handle {
    int32_t* rank_prefix_matrix;
    int32_t* channel_prefix_matrix;
    int32_t* recv_channel_prefix_matrix;
    int32_t* recv_src_idx;
    uint8_t* is_token_in_rank;
    int32_t* send_head;
    int32_t* num_recv_tokens_per_expert;
    int32_t* expert_rows;
    int32_t* expert_prefix;
} ep_handle;

/* Receive buffers of a normal dispatch. Destination d's rows are
 * [row_offset[d], row_offset[d+1]) of each array below; row_offset is a HOST array of
 * R+1 non-decreasing int64 (worst case: row_offset[d] = d*R*T needs no host sync;
 * exact sizes need ep_read_recv_counts_sync first -- the pages' implicit CPU wait).
 *   recv_x            dev [rows][H] bf16 or e4m3 (per recv_dtype)
 *   recv_x_scales     dev [rows][H/128] fp32, or uint8 with EP_FP8_SCALE_UE8M0 (e4m3
 *                     only; dequantise as q * scale)
 *   recv_topk_idx     dev [rows][k] int64: local expert id (e - d*E_loc) if the entry's
 *                     expert lives on d, else -1. Written only when topk_idx is given.
 *   recv_topk_weights dev [rows][k] fp32: the weight if local, else 0. Written only
 *                     when topk_idx and topk_weights are given.
 *   recv_src_idx      dev [rows] int32 (nullable): token index of each row.
 *   fp8               scale format of a fused quantisation (bf16 x, e4m3 receive);
 *                     must be EP_FP8_SCALE_FP32 for other dtype combinations.
 * When the regions hold no row at all (row_offset[R] == row_offset[0]) nothing is
 * written and the row arrays may be NULL; the same holds for y and recv_topk_weights
 * of a combine over empty regions. */
typedef struct ep_recv {
    void* recv_x;
    void* recv_x_scales;
    int64_t* recv_topk_idx;
    float* recv_topk_weights;
    int32_t* recv_src_idx;
    const int64_t* row_offset;
    ep_fp8_options fp8;
} ep_recv;

/* Placement of the low-latency receive rows inside each expert's R*Nmax slots.
 *   EP_LL_LAYOUT_SLOTS   source s owns slots [s*Nmax, (s+1)*Nmax), filled in token
 *                        order (gaps after each source's count) [default]
 *   EP_LL_LAYOUT_PACKED  no gaps: the expert's rows are 0 .. recv_expert_count-1 in
 *                        (source, token) order, source s starting at the sum of the
 *                        counts of sources s' < s, so a grouped GEMM reads one
 *                        contiguous block per expert.
 * Either layout's send phase is two kernels: a per-source rank kernel (the in-source
 * rank of every entry, in entry order, and the per-expert counts; linear in T*k), then
 * the rows. */
typedef enum ep_ll_layout { EP_LL_LAYOUT_SLOTS = 0, EP_LL_LAYOUT_PACKED = 1 } ep_ll_layout;

/* Low-latency buffers and handle ([README] low-latency example; [HOOK]). All dev.
 * Reading of the pages' "specific format for a grouped GEMM": rank d holds, per local
 * expert el, R*Nmax slots, placed as `layout` says (see ep_ll_layout).
 *   recv_x            [R][E_loc][R*Nmax][H] e4m3 (use_fp8) or bf16
 *   recv_x_scales     [R][E_loc][R*Nmax][H/128] fp32, or uint8 with
 *                     EP_FP8_SCALE_UE8M0 (use_fp8 only)
 *   src_info          [R][E_loc][R*Nmax] int32: token index of each filled slot
 *   slot              [R][T][k] int32: slot of entry (s, t, j), -1 if masked/skipped
 *   send_count        [R][E_loc][R] int32: per (d, el, s) count signal, written by
 *                     the send phase and read by the receive phase
 *   recv_expert_count [R][E_loc] int32 (int32 as in the port)
 *   layout_range      [R][E_loc][R][2] int32: (first slot, count) per source
 *   fp8               scale format when use_fp8 (see ep_fp8_scale)
 *   layout            ep_ll_layout (0 = EP_LL_LAYOUT_SLOTS); the combine reads the
 *                     slot array, so it serves both layouts unchanged
 * Slots beyond each count are left unwritten (stale data of earlier calls). */
typedef struct ep_ll_buffer {
    void* recv_x;
    void* recv_x_scales;
    int32_t* src_info;
    int32_t* slot;
    int32_t* send_count;
    int32_t* recv_expert_count;
    int32_t* layout_range;
    ep_fp8_options fp8;
    int32_t layout;
} ep_ll_buffer;

/* ---------------------------------------------------------------- layout */

/* Bytes of dev scratch ep_get_layout needs (per-channel partial counts). */
EP_API size_t ep_layout_workspace_size(const ep_shape* shape);

/* get_dispatch_layout + the handle's prefix matrices ([README] normal-kernel example:
 * "Calculate layout before actual dispatch"; [REUSE] "Handle Creation"; the pages'
 * host-side prefix sums are done on the device here).
 *   topk_idx  dev [R][T][k] int64, -1 = masked.
 *   layout    outputs as described at ep_layout (layout->num_tokens_per_rdma_rank must
 *             be NULL; any other field may be NULL to skip it).
 *   handle    every field except recv_src_idx is written (recv_src_idx is ignored).
 *   workspace dev, >= ep_layout_workspace_size bytes, 16-byte aligned; contents need
 *             no initialisation and are overwritten.
 * Two kernels (three with the expert-major placement), no host synchronisation. Bad
 * entries: EP_DEVERR_BAD_EXPERT. */
EP_API ep_status ep_get_layout(const ep_shape* shape, const int64_t* topk_idx, ep_layout* layout,
                        ep_handle* handle, void* workspace, size_t workspace_bytes,
                        const ep_launch* launch);

/* Size of the fixed device scratch array used by ep_get_layout_static_scratch. */
#define EP_LAYOUT_STATIC_SCRATCH_BYTES (256 * 1024)

/* ep_get_layout without a workspace argument, for callers that cannot allocate device
 * memory (for example a plugin whose host framework owns all device memory through its
 * own pool, or a latency-critical path where cudaMalloc / cudaFree would synchronise
 * the device). The pages have no counterpart: it exists only because the layout
 * kernels need scratch. Same outputs, status codes and ordering as ep_get_layout.
 *   - The scratch is a file-scope device array of EP_LAYOUT_STATIC_SCRATCH_BYTES bytes
 *     inside libep.so; every GPU that loads the library holds it until the process
 *     exits. Shapes whose ep_layout_workspace_size exceeds it return
 *     EP_ERR_UNSUPPORTED before anything is enqueued (R=8, C=12, E=256 needs ~97 KiB).
 *   - The first call in a CUDA context (the first on a device, with that device
 *     current, and again the first after cudaDeviceReset, when the library's device
 *     code is loaded anew) looks up the array's device address; make that first call
 *     before any stream capture. A device reset makes an address cached earlier
 *     invalid, which is why the cache is keyed by the context.
 *   - The call itself allocates nothing and frees nothing.
 *   - All calls on a device share the one array. Calls whose kernels may overlap on
 *     the GPU (different streams without ordering between them) race on it and give
 *     wrong results; order them, or use ep_get_layout with separate workspaces.
 *     Stale contents from an earlier call are harmless: every word read is first
 *     written by the same call. */
EP_API ep_status ep_get_layout_static_scratch(const ep_shape* shape, const int64_t* topk_idx,
                                              ep_layout* layout, ep_handle* handle,
                                              const ep_launch* launch);

/* ---------------------------------------------------------------- dispatch */

/* dispatch ([README] normal-kernel example, dispatch_forward / combine_backward;
 * [REUSE] "Fast Path Dispatch with Handle Reuse").
 *   x            dev [R][T][H]: bf16 (x_dtype = EP_BF16) or pre-quantised e4m3
 *                (x_dtype = EP_FP8_E4M3, with x_scales dev [R][T][H/128] fp32: the
 *                pages' (fp8, scales) tuple, copied byte for byte).
 *   recv_dtype   EP_BF16 (copy) or EP_FP8_E4M3: with bf16 x, quantise once per source
 *                token, per 128-channel group: amax' = max(amax, 1e-4),
 *                scale = amax'/448, q = e4m3_rn_satfinite(x * (448/amax')) -- and send
 *                the same bytes to every destination.
 *   topk_idx,    dev [R][T][k] int64 / fp32. Given on a first dispatch to produce
 *   topk_weights recv_topk_idx / recv_topk_weights. Handle reuse: both NULL (the pages
 *                assert that no new topk is passed with a handle); then
 *                out->recv_topk_idx / recv_topk_weights must be NULL too.
 *   handle       from ep_get_layout for the same topk_idx (reusing it with a changed
 *                routing is undefined behaviour: the contract in [REUSE]
 *                "Performance Contract and Constraints"; it is not detected).
 *   out          receive buffers (see ep_recv); out->recv_src_idx may be the handle's.
 * Copies (bf16, or pre-quantised e4m3) move each row with bulk copies (one load into shared
 * memory, one store per destination) when 4 rows fit in 200 KB of shared memory, i.e.
 * H * element size <= 50 KB; wider rows use 16-byte vector copies. A row load that has not
 * landed after 1 s (twice) sets EP_DEVERR_TIMEOUT and the rows of that warp are skipped.
 * Overflowing rows: EP_DEVERR_RECV_OVERFLOW. */
EP_API ep_status ep_dispatch(const ep_shape* shape, const void* x, ep_dtype x_dtype,
                      const float* x_scales, ep_dtype recv_dtype, const int64_t* topk_idx,
                      const float* topk_weights, const ep_handle* handle, ep_recv* out,
                      const ep_launch* launch);

/* ---------------------------------------------------------------- combine */

/* combine ([README] combine_forward and dispatch_backward; [REUSE] "Combining with
 * Handle Reuse"). Reduces rows back into token order:
 *   EP_COMBINE_SUM:      out[s][t] = sum over d with send_head >= 0 of y_d[row]
 *                        (the pages' combine(x, handle)).
 *   EP_COMBINE_WEIGHTED: out[s][t] = sum_d c_d * y_d[row], c_d = sum of the token's
 *                        topk_weights over valid entries whose expert lives on d (the
 *                        weighted top-k reduce).
 * Accumulation is fp32 in registers, one bf16 round-to-nearest-even store.
 *   y            dev [rows][H] bf16, rows in the dispatch's row order; 16-byte aligned
 *                (32-byte aligned y is read with 32-byte loads, otherwise 16-byte ones)
 *   y_row_offset HOST [R+1] int64, the same regions as the dispatch's row_offset
 *   topk_idx, topk_weights  dev [R][T][k]; required for WEIGHTED, else ignored
 *   recv_topk_weights       dev [rows][k] fp32, nullable: when given,
 *                combined_topk_weights[s][t][j] = sum_d recv_topk_weights_d[row][j]
 *                (dispatch_backward's reduced weight gradient)
 *   out          dev [R][T][H] bf16; a token sent nowhere gets +0
 *   combined_topk_weights dev [R][T][k] fp32, nullable */
EP_API ep_status ep_combine(const ep_shape* shape, const void* y, const int64_t* y_row_offset,
                     const ep_handle* handle, ep_combine_mode mode, const int64_t* topk_idx,
                     const float* topk_weights, const float* recv_topk_weights, void* out,
                     float* combined_topk_weights, const ep_launch* launch);

/* ---------------------------------------------------------------- expert-major layout */

/* Dispatch into the expert-major packed layout (the handle's expert_rows from
 * ep_get_layout; see ep_handle): one row per valid entry (s, t, j), written to
 * recv_x[row_offset[d] + expert_rows[s][t][j]] where d owns the entry's expert. The row
 * is bf16 (recv_dtype EP_BF16) or quantised once per token to e4m3 with out->fp8's
 * scale format. Rows of local expert el on d start at expert_prefix[d][el]; size d's
 * region with expert_prefix[d][E_loc] rows (after ep_read_recv_counts_sync-style read
 * back) or with the worst case R*T*min(k, E_loc).
 *   x             dev [R][T][H] bf16
 *   topk_idx      dev [R][T][k] int64 (required), topk_weights dev [R][T][k] fp32 nullable
 *   out           recv_x, recv_x_scales (e4m3), recv_src_idx [rows] (nullable: token
 *                 index of each row), recv_topk_weights [rows] (nullable: the entry's
 *                 weight, one per row), row_offset (host [R+1]); recv_topk_idx must be
 *                 NULL (each row is one entry).
 * bf16 rows up to 50 KB move with bulk copies as in ep_dispatch (EP_DEVERR_TIMEOUT if a row
 * load does not land in time). Overflowing rows: EP_DEVERR_RECV_OVERFLOW. */
EP_API ep_status ep_dispatch_expert_major(const ep_shape* shape, const void* x, ep_dtype recv_dtype,
                                          const int64_t* topk_idx, const float* topk_weights,
                                          const ep_handle* handle, ep_recv* out,
                                          const ep_launch* launch);

/* Combine from the expert-major layout: out[s][t] = sum over valid j (ascending) of
 * c_j * y[y_row_offset[d] + expert_rows[s][t][j]], c_j = topk_weights[s][t][j]
 * (EP_COMBINE_WEIGHTED) or 1 (EP_COMBINE_SUM); fp32 accumulation, one bf16 store.
 *   y   dev [rows][H] bf16 (the grouped GEMM's output in the dispatch's row order)
 *   out dev [R][T][H] bf16; a token with no valid entry gets +0 */
EP_API ep_status ep_combine_expert_major(const ep_shape* shape, const void* y,
                                         const int64_t* y_row_offset, const ep_handle* handle,
                                         ep_combine_mode mode, const int64_t* topk_idx,
                                         const float* topk_weights, void* out,
                                         const ep_launch* launch);

/* ---------------------------------------------------------------- low latency */

/* low_latency_dispatch ([README] low-latency example; [HOOK] "Two-Phase Kernel
 * Architecture"). phase = EP_PHASE_SEND writes the rows (fused e4m3 quantisation when
 * use_fp8), src_info, slot and the send_count signals; EP_PHASE_RECV turns the
 * signals into recv_expert_count and layout_range; EP_PHASE_BOTH does both. A hook
 * is the caller issuing the RECV call later (there is no stored closure in a C ABI).
 *   x        dev [R][T][H] bf16; T <= Nmax is required
 *   topk_idx dev [R][T][k] int64 (-1 masked); a repeated expert within a token takes
 *            one slot per entry, in entry order
 *   buf      see ep_ll_buffer (recv_x_scales required iff use_fp8)
 * Slot overflow: EP_DEVERR_SLOT_OVERFLOW; bad experts: EP_DEVERR_BAD_EXPERT. */
EP_API ep_status ep_ll_dispatch(const ep_shape* shape, const void* x, const int64_t* topk_idx,
                         int use_fp8, ep_phase phase, ep_ll_buffer* buf,
                         const ep_launch* launch);

/* low_latency_combine ([README] low-latency example): the weighted top-k reduction
 * out[s][t] = sum over valid j of topk_weights[s][t][j] * y[d][el][slot[s][t][j]],
 * fp32 accumulation, bf16 store. Reading of the phase split: in one device memory the
 * return transfer is nothing, so EP_PHASE_SEND only orders/records events and
 * EP_PHASE_RECV (or BOTH) runs the reduction.
 *   y       dev [R][E_loc][R*Nmax][H] bf16, the expert outputs in the slot layout
 *   handle  the ep_ll_buffer of the matching ep_ll_dispatch (its slot array is used)
 *   out     dev [R][T][H] bf16; a fully masked token gets +0 */
EP_API ep_status ep_ll_combine(const ep_shape* shape, const void* y, const int64_t* topk_idx,
                        const float* topk_weights, const ep_ll_buffer* handle,
                        ep_phase phase, void* out, const ep_launch* launch);

/* clean_low_latency_buffer ([README] feature notes): zeroes send_count,
 * recv_expert_count and layout_range. Optional here (the send phase rewrites every
 * signal), kept for API parity. */
EP_API ep_status ep_clean_ll_buffer(const ep_shape* shape, ep_ll_buffer* buf, const ep_launch* launch);

/* ---------------------------------------------------------------- helpers */

/* Buffer sizes for one shape, in bytes unless named rows: the caller-owned counterpart of
 * the pages' buffer size hints ([README] normal-kernel example: Buffer sizing with
 * get_dispatch_config / get_combine_config and the NVL / RDMA size hints; low-latency
 * example: get_low_latency_rdma_size_hint). Worst cases need no host synchronisation:
 *   recv_rows          R*R*T: every token of every source reaching every destination
 *                      (row_offset[d] = d*R*T); recv_* sizes are for that many rows
 *   expert_major_rows  R*R*T*min(k, E_loc): one row per entry, at most min(k, E_loc)
 *                      entries of a token per destination
 *   ll_*               the low-latency buffer of ep_ll_buffer (R*E_loc*R*Nmax slots)
 *   layout_workspace   ep_layout_workspace_size
 * recv_dtype selects the row element (2 bytes bf16, 1 byte e4m3); scale sizes are 0 for
 * bf16, 1 byte per group with EP_FP8_SCALE_UE8M0, else 4. Returns EP_ERR_UNSUPPORTED if a
 * size does not fit in 64 bits. Host only; launches nothing. */
typedef struct ep_size_hint {
    int64_t recv_rows;
    uint64_t recv_x_bytes;
    uint64_t recv_x_scales_bytes;
    uint64_t recv_topk_idx_bytes;
    uint64_t recv_topk_weights_bytes;
    uint64_t recv_src_idx_bytes;
    int64_t expert_major_rows;
    uint64_t expert_major_x_bytes;
    uint64_t ll_slots;
    uint64_t ll_recv_x_bytes;
    uint64_t ll_recv_x_scales_bytes;
    uint64_t ll_src_info_bytes;
    uint64_t ll_slot_bytes;
    uint64_t ll_send_count_bytes;
    uint64_t ll_recv_expert_count_bytes;
    uint64_t ll_layout_range_bytes;
    uint64_t layout_workspace_bytes;
} ep_size_hint;

EP_API ep_status ep_buffer_size_hint(const ep_shape* shape, ep_dtype recv_dtype,
                                     int32_t fp8_scale_format, ep_size_hint* out);

/* The pages' implicit CPU wait for the received count ([README] note after
 * combine_backward): copies rank_prefix_matrix[R-1][*] (N_d per destination) into
 * host_counts[R] and synchronises `stream`. */
EP_API ep_status ep_read_recv_counts_sync(const ep_shape* shape, const ep_handle* handle,
                                   int32_t* host_counts, cudaStream_t stream);

/* Copies the device error word to *host_flags and synchronises `stream`. */
EP_API ep_status ep_read_error_flags_sync(const uint32_t* error_flags, uint32_t* host_flags,
                                   cudaStream_t stream);

/* Diagnostic of the bounded device waits (the pages have no counterpart; the bulk-copy
 * dispatch kernels wait on shared-memory barriers for their row loads, at most 1 s per
 * wait). Launches one thread that arms a barrier for 32 bytes but bulk-copies only 16 bytes
 * from src16, so the phase never completes: its wait must give up after timeout_ms (1 to
 * 10000) and OR EP_DEVERR_TIMEOUT into launch->error_flags (required), writing the time the
 * wait took to *elapsed_us (device, nullable). Nothing faults or hangs, and the context stays
 * usable.
 *   src16  dev, 16-byte aligned, at least 16 readable bytes (only read) */
EP_API ep_status ep_selftest_wait_timeout(const void* src16, int32_t timeout_ms, uint32_t* elapsed_us,
                                          const ep_launch* launch);

/* Static description of a status code. */
EP_API const char* ep_status_string(ep_status status);

/* Last CUDA error string seen by the library on this thread ("" if none). */
EP_API const char* ep_last_cuda_error(void);

/* Number of kernels this library has launched in this process. */
EP_API uint64_t ep_kernel_launch_count(void);

/* Library ABI version (major * 100 + minor). */
EP_API int32_t ep_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* COMBINE_LAYOUT_02_EP_H */
