// ep_internal.cuh -- helpers shared by the libep translation units (device memory
// access with cache hints, bf16 / e4m3 packing, host-side validation, event
// ordering and launch accounting). Internal: not part of the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/ep.h"

namespace ep {

// ------------------------------------------------------------------ device helpers

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    // Read-only, streaming: each source byte is read once, keep it out of L1.
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

struct u32x8 {
    uint32_t r[8];
};

// 32-byte load (sm_100+ ld .v8.b32); the address must be 32-byte aligned.
__device__ __forceinline__ u32x8 ld_stream_v8(const void* p) {
    u32x8 v;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v.r[0]), "=r"(v.r[1]), "=r"(v.r[2]), "=r"(v.r[3]), "=r"(v.r[4]),
                   "=r"(v.r[5]), "=r"(v.r[6]), "=r"(v.r[7])
                 : "l"(p));
    return v;
}

// 32-byte store (sm_100+ st .v8.b32); the address must be 32-byte aligned.
__device__ __forceinline__ void st_v8(void* p, const u32x8& v) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v.r[0]),
                 "r"(v.r[1]), "r"(v.r[2]), "r"(v.r[3]), "r"(v.r[4]), "r"(v.r[5]), "r"(v.r[6]),
                 "r"(v.r[7])
                 : "memory");
}

__device__ __forceinline__ void st_stream_v4(void* p, const uint4& v) {
    // Streaming store (evict-first): the written rows are far larger than L2.
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// bf16 pair packed in a 32-bit word -> two fp32 (exact widening: bf16 is the high
// half of a binary32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> packed bf16 pair, round to nearest even (CUDA's documented conversion).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Two fp32 -> packed e4m3 pair (lo in the low byte), round to nearest even,
// saturating to +-448 (CUDA's documented fp8 conversion, __NV_SATFINITE).
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
    __nv_fp8x2_storage_t s = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(s);
}

__device__ __forceinline__ void raise_flag(uint32_t* flags, uint32_t bit) {
    if (flags != nullptr) atomicOr(flags, bit);
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Programmatic dependent launch. A kernel launched early (while the previous kernel of
// the stream still runs) must call pdl_wait() before it reads anything the previous
// kernel may write and before its first global store, so it overlaps only the previous
// kernel's tail. Kernels that may follow arbitrary caller work wait before their first
// global access. The one exception is a kernel that only ever follows a kernel of this
// library which itself returned from pdl_wait() before its pdl_trigger(): everything
// ordered before that earlier kernel is then complete, so the later kernel may read
// the call's inputs before its own wait (the low-latency send kernel does this after the
// send phase's rank kernel). pdl_trigger() lets the next kernel of the stream start
// launching. Both are no-ops for kernels launched without the
// programmatic-serialization attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ bulk copies (TMA)
// One-dimensional bulk copies between global and shared memory executed by the
// tensor-memory-accelerator copy engine (cp.async.bulk), completed through an mbarrier
// (loads) or a bulk group (stores). Addresses and sizes must be multiples of 16 bytes.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
    // Make the initialised barrier visible to the bulk-copy (async) proxy.
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arms the barrier for one phase that completes when `bytes` have arrived.
__device__ __forceinline__ void mbar_expect_bytes(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the barrier phase with parity `parity`, giving up once `timeout_ns` of the
// GPU's global timer have passed. Returns whether the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = global_ns();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
            "selp.u32 %0, 1, 0, p; }"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if (global_ns() - t0 > timeout_ns) return false;
    }
}

// global -> shared, completing `bytes` on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// shared -> global, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The issuing thread's committed stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_smem_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// The issuing thread's committed stores are complete (written to global memory).
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's earlier async-proxy shared-memory traffic before later bulk copies.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Destination-row regions passed by value (host array copied into kernel params).
struct RowOffsets {
    int64_t v[EP_MAX_RANKS + 1];
};

// ------------------------------------------------------------------ host helpers

// Validates the shape (limits stated in ep.h). Returns EP_OK or an error status.
ep_status check_shape(const ep_shape* sh);

// Number of SMs of the current device (cached per device).
int sm_count();

// Makes launch->stream wait on launch->wait_event (if any).
ep_status begin_call(const ep_launch* launch);

// Checks the launch error state, then records launch->record_event (if any).
ep_status end_call(const ep_launch* launch);

// Records a CUDA error for ep_last_cuda_error and returns EP_ERR_CUDA.
ep_status cuda_fail(cudaError_t e);

// Adds n to the process-wide kernel launch counter.
void count_launches(uint64_t n);

// Fills a RowOffsets from a host array of R+1 entries; checks monotonicity.
ep_status load_row_offsets(const int64_t* host, int R, RowOffsets* out);

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Launches `kernel` on `stream` with programmatic stream serialization allowed (see
// pdl_wait / pdl_trigger) and counts the launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace ep
