// rowops.cuh -- the three row movements of the hot path, written once and used by
// both the normal (one warp per token) and the low-latency (one block per token)
// kernels:
//   scatter_copy_row   one source row -> nd destination rows (bytes copied)
//   scatter_quant_row  one bf16 source row -> e4m3 row + per-128-channel fp32 scales,
//                      quantised once, stored to nd destination rows (per unit of 16
//                      channels, or per pair of units with 32-byte stores)
//   gather_reduce_row  nd bf16 rows * coefficients -> one bf16 row, fp32 accumulation
// Work is split in 16-byte units: thread `first` handles units first, first+stride, ...
// Each source byte is loaded once (ld.global.nc, no L1 allocation) and every
// destination byte stored once with 16-byte vector stores; loads of an unrolled batch
// are all issued before their data is used, to keep enough bytes in flight.
#pragma once

#include "ep_internal.cuh"

namespace ep {

template <int U, bool kStreamStore = false>
__device__ __forceinline__ void scatter_copy_row(const char* __restrict__ src,
                                                 char* __restrict__ dst_base,
                                                 const int64_t* rows, int nd, int64_t row_bytes,
                                                 int first, int stride) {
    const int units = (int)(row_bytes >> 4);
    for (int u0 = 0; u0 < units; u0 += stride * U) {
        uint4 v[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int u = u0 + i * stride + first;
            if (u < units) v[i] = ld_stream_v4(src + (int64_t)u * 16);
        }
        for (int p = 0; p < nd; ++p) {
            char* dst = dst_base + rows[p] * row_bytes;
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const int u = u0 + i * stride + first;
                if (u < units) {
                    if (kStreamStore) st_stream_v4(dst + (int64_t)u * 16, v[i]);
                    else st_v4(dst + (int64_t)u * 16, v[i]);
                }
            }
        }
    }
}

// Row moves with bulk copies (one warp per token, lane 0 issues everything): the row is
// loaded into the warp's shared-memory buffer with one bulk copy and stored to each
// destination row with one bulk copy. Blocks of kTmaWarps warps, one row buffer each.
constexpr int kTmaWarps = 4;
constexpr uint64_t kTmaWaitNs = 1000000000ull;   // bound on one mbarrier wait: 1 s
constexpr int kTmaSmemMax = 200 * 1024;    // dynamic shared memory a block may use

// Lane 0: starts loading `bytes` from src into buf once the warp's earlier stores have
// finished reading buf.
__device__ __forceinline__ void tma_row_load(unsigned char* buf, const char* src, uint32_t bytes,
                                             uint64_t* bar) {
    bulk_wait_smem_read();
    mbar_expect_bytes(bar, bytes);
    bulk_load(buf, src, bytes, bar);
}

// Lane 0: waits (at most 1 s, twice) for the row started by tma_row_load, then stores it to
// rows[0..nd) of dst_base and commits the stores. A load that does not land raises
// EP_DEVERR_TIMEOUT; returns false if it never landed (the caller then stops using buf).
__device__ __forceinline__ bool tma_row_store(const unsigned char* buf, char* dst_base,
                                              const int64_t* rows, int nd, uint32_t bytes,
                                              uint64_t* bar, uint32_t& parity, uint32_t* err) {
    if (!mbar_wait_bounded(bar, parity, kTmaWaitNs)) {
        raise_flag(err, EP_DEVERR_TIMEOUT);
        if (!mbar_wait_bounded(bar, parity, kTmaWaitNs)) return false;
    }
    parity ^= 1u;
    fence_async_smem();
    for (int p = 0; p < nd; ++p) bulk_store(dst_base + rows[p] * (int64_t)bytes, buf, bytes);
    bulk_commit();
    return true;
}

// FP8 e4m3 quantisation, one scale per 128 channels ("DeepEP" README feature notes:
// FP8 dispatch with per-group scales; round_scale; use_ue8m0; fp8_quant_scale). Unit =
// 16 channels (32 bytes of bf16 in, 16 bytes of e4m3 out); 8 consecutive units (8
// consecutive lanes) form one group, so the group amax is a 3-step xor-shuffle. Every
// lane of a warp must call quant_unit together (the shuffles use the full mask).
//   amax' = max(amax, 1e-4); s0 = amax' / 448 (IEEE division);
//   FP32:   scale = s0, inv = 448 / amax' (IEEE division)
//   POW2 / UE8M0: scale = 2^ceil(log2(s0)) from the exponent bits, inv = 1 / scale (exact)
//   TENSOR: scale and inv given by the caller (inv = 1/s, IEEE division on the host)
//   q = e4m3_rn_satfinite(x * inv).
struct QuantMode {
    int mode;          // ep_fp8_scale
    float tscale;      // EP_FP8_SCALE_TENSOR
    float tinv;        // 1 / tscale
};

// The group scale, its inverse and (power-of-two modes) biased exponent byte from the
// group amax; the per-tensor mode takes the caller's scale and ignores amax.
__device__ __forceinline__ void quant_scale(float amax, const QuantMode& qm, float& scale, float& inv,
                                            uint32_t& scale_byte) {
    scale_byte = 0;
    if (qm.mode == EP_FP8_SCALE_TENSOR) {
        scale = qm.tscale;
        inv = qm.tinv;
        return;
    }
    const float am = fmaxf(amax, 1e-4f);
    if (qm.mode == EP_FP8_SCALE_FP32) {
        scale = __fdiv_rn(am, 448.0f);
        inv = __fdiv_rn(448.0f, am);
    } else {
        // s0 >= 1e-4/448 and <= bf16 max/448, so it is a normal number and the rounded-up
        // power of two and its reciprocal are normal too.
        const uint32_t bits = __float_as_uint(__fdiv_rn(am, 448.0f));
        const uint32_t e = ((bits >> 23) & 0xFFu) + ((bits & 0x7FFFFFu) != 0u ? 1u : 0u);
        scale = __uint_as_float(e << 23);
        inv = __uint_as_float((254u - e) << 23);
        scale_byte = e;
    }
}

// Four e4m3 values x * inv (round to nearest even, satfinite) packed in a word, the
// first in the low byte.
__device__ __forceinline__ uint32_t quant_word(const float* f, float inv) {
    const uint32_t lo = pack_e4m3x2(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv));
    const uint32_t hi = pack_e4m3x2(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv));
    return lo | (hi << 16);
}

// Quantises one unit (16 bf16 channels held in a, b) to 16 e4m3 bytes. Returns the
// group scale (fp32) and its biased exponent byte (power-of-two modes).
__device__ __forceinline__ uint4 quant_unit(const uint4& a, const uint4& b, const QuantMode& qm,
                                            float& scale, uint32_t& scale_byte) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float f[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        f[2 * j] = bf16_lo(w[j]);
        f[2 * j + 1] = bf16_hi(w[j]);
    }
    float amax = 0.0f;
    if (qm.mode != EP_FP8_SCALE_TENSOR) {
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    }
    float inv;
    quant_scale(amax, qm, scale, inv, scale_byte);
    return make_uint4(quant_word(f, inv), quant_word(f + 4, inv), quant_word(f + 8, inv),
                      quant_word(f + 12, inv));
}

// Quantises a pair of units (32 bf16 channels, two 32-byte loads in v) to 32 e4m3 bytes;
// 4 consecutive lanes hold a 128-channel group, so the group amax is a 2-step xor-shuffle.
// Every lane of a warp must call quant_pair together.
__device__ __forceinline__ u32x8 quant_pair(const u32x8 (&v)[2], const QuantMode& qm, float& scale,
                                            uint32_t& scale_byte) {
    float f[32];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            f[16 * h + 2 * j] = bf16_lo(v[h].r[j]);
            f[16 * h + 2 * j + 1] = bf16_hi(v[h].r[j]);
        }
    float amax = 0.0f;
    if (qm.mode != EP_FP8_SCALE_TENSOR) {
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(f[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    }
    float inv;
    quant_scale(amax, qm, scale, inv, scale_byte);
    u32x8 q;
#pragma unroll
    for (int j = 0; j < 8; ++j) q.r[j] = quant_word(f + 4 * j, inv);
    return q;
}

// Stores one quantised unit u (and, for the first unit of a group, its scale: fp32, or
// one byte in the UE8M0 mode) to every destination row.
__device__ __forceinline__ void store_quant_unit(uint8_t* __restrict__ q_base, void* __restrict__ s_base,
                                                 const int64_t* rows, int nd, int H, int u,
                                                 const uint4& q, float scale, uint32_t scale_byte,
                                                 int mode) {
    const int G = H >> 7;
    for (int p = 0; p < nd; ++p) {
        st_v4(q_base + rows[p] * (int64_t)H + (int64_t)u * 16, q);
        if ((u & 7) == 0) {
            if (mode == EP_FP8_SCALE_UE8M0)
                reinterpret_cast<uint8_t*>(s_base)[rows[p] * (int64_t)G + (u >> 3)] = (uint8_t)scale_byte;
            else
                reinterpret_cast<float*>(s_base)[rows[p] * (int64_t)G + (u >> 3)] = scale;
        }
    }
}

// Loads batch u0 of a row for quantisation: units u0 + i*stride + first (i < U), as two
// 16-byte halves each; zero beyond the row (those lanes still take part in the shuffles).
// V32: one 32-byte load per unit (src 32-byte aligned) instead of two 16-byte loads.
template <int U, bool V32 = false>
__device__ __forceinline__ void quant_load(const char* __restrict__ src, int units, int u0, int first,
                                           int stride, uint4 (&a)[U], uint4 (&b)[U]) {
#pragma unroll
    for (int i = 0; i < U; ++i) {
        const int u = u0 + i * stride + first;
        if (u < units && V32) {
            const u32x8 v = ld_stream_v8(src + (int64_t)u * 32);
            a[i] = make_uint4(v.r[0], v.r[1], v.r[2], v.r[3]);
            b[i] = make_uint4(v.r[4], v.r[5], v.r[6], v.r[7]);
        } else if (u < units) {
            a[i] = ld_stream_v4(src + (int64_t)u * 32);
            b[i] = ld_stream_v4(src + (int64_t)u * 32 + 16);
        } else {
            a[i] = make_uint4(0, 0, 0, 0);
            b[i] = make_uint4(0, 0, 0, 0);
        }
    }
}

// Quantises one row and stores it to every destination row, software-pipelined: (a, b)
// hold the batch at u_start, already loaded (the caller can issue that load before its
// own metadata loads), and each next batch is loaded before the current one is
// quantised and stored, so two batches per thread are in flight.
template <int U, bool V32 = false>
__device__ __forceinline__ void scatter_quant_row_loaded(const char* __restrict__ src,
                                                         uint8_t* __restrict__ q_base,
                                                         void* __restrict__ s_base,
                                                         const int64_t* rows, int nd, int H,
                                                         const QuantMode& qm, int first, int stride,
                                                         int u_start, uint4 (&a)[U], uint4 (&b)[U]) {
    const int units = H >> 4;
    for (int u0 = u_start; u0 < units; u0 += stride * U) {
        uint4 na[U], nb[U];
        quant_load<U, V32>(src, units, u0 + stride * U, first, stride, na, nb);
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int u = u0 + i * stride + first;
            float scale;
            uint32_t sbyte;
            const uint4 q = quant_unit(a[i], b[i], qm, scale, sbyte);
            if (u < units) store_quant_unit(q_base, s_base, rows, nd, H, u, q, scale, sbyte, qm.mode);
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            a[i] = na[i];
            b[i] = nb[i];
        }
    }
}

// Pair q of a row for quant_pair: 32 bf16 channels (64 bytes) as two 32-byte loads (src
// 32-byte aligned); zero past the row (those lanes still take part in the shuffles).
__device__ __forceinline__ void pair_load(const char* __restrict__ src, int pairs, int q, u32x8 (&v)[2]) {
    if (q < pairs) {
        v[0] = ld_stream_v8(src + (int64_t)q * 64);
        v[1] = ld_stream_v8(src + (int64_t)q * 64 + 32);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[0].r[j] = v[1].r[j] = 0u;
    }
}

// scatter_quant_row_loaded with pairs: one pair per lane per step, 32-byte loads and one
// 32-byte store per destination (q_base rows 32-byte aligned); `cur` holds pair `first`,
// already loaded, and each next pair is loaded before the current one is quantised.
__device__ __forceinline__ void scatter_quant_pairs_loaded(const char* __restrict__ src,
                                                           uint8_t* __restrict__ q_base,
                                                           void* __restrict__ s_base,
                                                           const int64_t* rows, int nd, int H,
                                                           const QuantMode& qm, int first,
                                                           u32x8 (&cur)[2]) {
    const int pairs = H >> 5, G = H >> 7;
    for (int q0 = 0; q0 < pairs; q0 += 32) {       // warp-uniform: quant_pair shuffles
        u32x8 nxt[2];
        pair_load(src, pairs, q0 + 32 + first, nxt);
        float scale;
        uint32_t sbyte;
        const u32x8 qv = quant_pair(cur, qm, scale, sbyte);
        const int q = q0 + first;
        if (q < pairs) {
            for (int p = 0; p < nd; ++p) {
                st_v8(q_base + rows[p] * (int64_t)H + (int64_t)q * 32, qv);
                if ((q & 3) == 0) {
                    if (qm.mode == EP_FP8_SCALE_UE8M0)
                        reinterpret_cast<uint8_t*>(s_base)[rows[p] * (int64_t)G + (q >> 2)] = (uint8_t)sbyte;
                    else
                        reinterpret_cast<float*>(s_base)[rows[p] * (int64_t)G + (q >> 2)] = scale;
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) cur[h] = nxt[h];
    }
}

template <int U>
__device__ __forceinline__ void scatter_quant_row(const char* __restrict__ src,
                                                  uint8_t* __restrict__ q_base,
                                                  void* __restrict__ s_base,
                                                  const int64_t* rows, int nd, int H,
                                                  const QuantMode& qm, int first, int stride,
                                                  int u_start = 0) {
    uint4 a[U], b[U];
    quant_load<U>(src, H >> 4, u_start, first, stride, a, b);
    scatter_quant_row_loaded<U>(src, q_base, s_base, rows, nd, H, qm, first, stride, u_start, a, b);
}

// gather_reduce_row with 32-byte loads (16 channels per unit); y rows 32-byte aligned.
template <int U, int P>
__device__ __forceinline__ void gather_reduce_row32(const char* __restrict__ y_base,
                                                    const int64_t* rows, const float* coef,
                                                    int nd, int H, char* __restrict__ out_row,
                                                    int first, int stride) {
    const int units = H >> 4;
    const int64_t row_bytes = (int64_t)H * 2;
    for (int u0 = 0; u0 < units; u0 += stride * U) {
        float acc[U][16];
#pragma unroll
        for (int i = 0; i < U; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[i][j] = 0.0f;
        for (int p0 = 0; p0 < nd; p0 += P) {
            u32x8 v[P][U];
#pragma unroll
            for (int p = 0; p < P; ++p) {
                if (p0 + p < nd) {
                    const char* src = y_base + rows[p0 + p] * row_bytes;
#pragma unroll
                    for (int i = 0; i < U; ++i) {
                        const int u = u0 + i * stride + first;
                        if (u < units) v[p][i] = ld_stream_v8(src + (int64_t)u * 32);
                    }
                }
            }
#pragma unroll
            for (int p = 0; p < P; ++p) {
                if (p0 + p < nd) {
                    const float c = coef[p0 + p];
#pragma unroll
                    for (int i = 0; i < U; ++i)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            acc[i][2 * j] = fmaf(c, bf16_lo(v[p][i].r[j]), acc[i][2 * j]);
                            acc[i][2 * j + 1] = fmaf(c, bf16_hi(v[p][i].r[j]), acc[i][2 * j + 1]);
                        }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int u = u0 + i * stride + first;
            if (u < units) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 o = make_uint4(pack_bf16x2(acc[i][8 * h + 0], acc[i][8 * h + 1]),
                                               pack_bf16x2(acc[i][8 * h + 2], acc[i][8 * h + 3]),
                                               pack_bf16x2(acc[i][8 * h + 4], acc[i][8 * h + 5]),
                                               pack_bf16x2(acc[i][8 * h + 6], acc[i][8 * h + 7]));
                    st_v4(out_row + (int64_t)u * 32 + h * 16, o);
                }
            }
        }
    }
}

// out = sum_p coef[p] * rows[p], fp32 accumulation in registers, one bf16 RNE store.
// Unit = 8 channels (16 bytes); units [u_begin, u_end) of the row. Rows are taken P at a
// time with every load of the batch (P rows x U units) issued before the first
// accumulation.
template <int U, int P = 8>
__device__ __forceinline__ void gather_reduce_row(const char* __restrict__ y_base,
                                                  const int64_t* rows, const float* coef,
                                                  int nd, int H, char* __restrict__ out_row,
                                                  int first, int stride, int u_begin = 0,
                                                  int u_end = 1 << 30) {
    const int units = min(H >> 3, u_end);
    const int64_t row_bytes = (int64_t)H * 2;
    for (int u0 = u_begin; u0 < units; u0 += stride * U) {
        float acc[U][8];
#pragma unroll
        for (int i = 0; i < U; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
        for (int p0 = 0; p0 < nd; p0 += P) {
            uint4 v[P][U];
#pragma unroll
            for (int p = 0; p < P; ++p) {
                if (p0 + p < nd) {
                    const char* src = y_base + rows[p0 + p] * row_bytes;
#pragma unroll
                    for (int i = 0; i < U; ++i) {
                        const int u = u0 + i * stride + first;
                        if (u < units) v[p][i] = ld_stream_v4(src + (int64_t)u * 16);
                    }
                }
            }
#pragma unroll
            for (int p = 0; p < P; ++p) {
                if (p0 + p < nd) {
                    const float c = coef[p0 + p];
#pragma unroll
                    for (int i = 0; i < U; ++i) {
                        const uint32_t w[4] = {v[p][i].x, v[p][i].y, v[p][i].z, v[p][i].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            acc[i][2 * j] = fmaf(c, bf16_lo(w[j]), acc[i][2 * j]);
                            acc[i][2 * j + 1] = fmaf(c, bf16_hi(w[j]), acc[i][2 * j + 1]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int u = u0 + i * stride + first;
            if (u < units) {
                const uint4 o = make_uint4(pack_bf16x2(acc[i][0], acc[i][1]), pack_bf16x2(acc[i][2], acc[i][3]),
                                           pack_bf16x2(acc[i][4], acc[i][5]), pack_bf16x2(acc[i][6], acc[i][7]));
                st_v4(out_row + (int64_t)u * 16, o);
            }
        }
    }
}

}  // namespace ep
