// layout.cu -- get_dispatch_layout and the handle's prefix matrices on the device.
//
// [README]  "DeepEP" README (EnflameTechnology/DeepEP), normal-kernel example:
//           get_dispatch_layout(topk_idx, num_experts, ...) -> num_tokens_per_rank,
//           num_tokens_per_rdma_rank, num_tokens_per_expert, is_token_in_rank.
// [REUSE]   "How DeepEP Optimizes Handle Reuse for Repeated Dispatches", "What the
//           Handle Contains": rank_prefix_matrix, channel_prefix_matrix,
//           recv_channel_prefix_matrix, recv_src_idx, is_token_in_rank, send_head.
//
// Two kernels, one block per (channel c, source rank s); no atomics on global memory,
// no inter-block waiting, so every result is deterministic:
//   layout_count_kernel  -- per block: expert histogram (shared-memory atomics),
//       is_token_in_rank bytes, per-destination counts of the channel (warp ballot +
//       popc). Partial counts go to the caller's workspace.
//   layout_prefix_kernel -- per block: the prefix entries of its (s, c) from the
//       partial counts (warp reductions), the expert totals, and send_head for its
//       tokens by a block-wide exclusive scan of the rank bits (ballot + popc within a
//       warp, shared-memory scan across warps). With the expert-major placement the
//       same launch has extra blocks that scan the expert columns (and give the expert
//       totals), so the placement kernel follows it directly.
// Rows of destination d are ordered by (source rank, token), so
//   send_head[s][t][d] = recv_channel_prefix_matrix[d][s][c(t)]
//                        + #{t' < t in the same channel with is_token_in_rank}.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
static_assert(EP_MAX_RANKS % kWarps == 0, "destinations split evenly over warps");

struct LayoutArgs {
    const int64_t* topk_idx;
    int R, T, E, k, C, E_loc, tpc;
    int32_t* num_tokens_per_rank;         // [R][R] nullable
    int32_t* num_tokens_per_expert;       // [R][E] nullable
    uint8_t* in_rank;                     // [R][T][R] (handle)
    uint8_t* in_rank_extra;               // [R][T][R] nullable second copy (layout)
    int32_t* rank_prefix;                 // [R][R]
    int32_t* channel_prefix;              // [R][R][C]
    int32_t* recv_channel_prefix;         // [R][R][C]
    int32_t* send_head;                   // [R][T][R]
    int32_t* num_recv_per_expert;         // [R][E_loc] == [E]
    int32_t* ws_cnt;                      // [R][R][C]: (s*R + d)*C + c
    int32_t* ws_expert;                   // [R][C][E]: (s*C + c)*E + e
    int32_t* expert_rows;                 // [R][T][k] nullable: expert-major placement
    int32_t* expert_prefix;               // [R][E_loc + 1]
    int32_t* ws_etot;                     // [E] expert totals (workspace)
    int ew;                               // bitmask words per expert (expert-major ranks)
    int scan_rows;                        // grid rows of expert column-scan blocks (0: none)
    int el_shift;                         // log2(E_loc) when E_loc is a power of two, else -1
    int vec_ids;                          // topk rows load as 16-byte pairs (k even, aligned)
    int vec_head;                         // send_head rows store as 16-byte quads (R % 4 == 0)
    uint32_t* err;
};

__device__ __forceinline__ void write_rank_bytes(uint8_t* p, uint64_t mask, int R) {
    if ((R & 7) == 0) {
        for (int d8 = 0; d8 < R; d8 += 8) {
            uint64_t w = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) w |= ((mask >> (d8 + i)) & 1ull) << (8 * i);
            *reinterpret_cast<uint64_t*>(p + d8) = w;
        }
    } else {
        for (int d = 0; d < R; ++d) p[d] = (uint8_t)((mask >> d) & 1ull);
    }
}

__device__ __forceinline__ uint64_t read_rank_bytes(const uint8_t* p, int R) {
    uint64_t mask = 0;
    if ((R & 7) == 0) {
        for (int d8 = 0; d8 < R; d8 += 8) {
            uint64_t w = *reinterpret_cast<const uint64_t*>(p + d8);
#pragma unroll
            for (int i = 0; i < 8; ++i) mask |= ((w >> (8 * i)) & 1ull) << (d8 + i);
        }
    } else {
        for (int d = 0; d < R; ++d) mask |= (uint64_t)(p[d] & 1) << d;
    }
    return mask;
}

__global__ void __launch_bounds__(kThreads) layout_count_kernel(LayoutArgs a) {
    extern __shared__ int smem[];
    int* hist = smem;          // [E]
    int* cnt = smem + a.E;     // [R]
    const int c = blockIdx.x, s = blockIdx.y, lane = threadIdx.x & 31;
    pdl_trigger();   // tiny kernel: let the prefix kernel launch right away
    for (int i = threadIdx.x; i < a.E; i += kThreads) hist[i] = 0;
    for (int i = threadIdx.x; i < a.R; i += kThreads) cnt[i] = 0;
    pdl_wait();
    __syncthreads();

    const int t0 = min(c * a.tpc, a.T), t1 = min(t0 + a.tpc, a.T);
    for (int base = t0; base < t1; base += kThreads) {   // block-uniform trip count
        const int t = base + threadIdx.x;
        uint64_t mask = 0;
        if (t < t1) {
            const int64_t* row = a.topk_idx + ((int64_t)s * a.T + t) * a.k;
            for (int j0 = 0; j0 < a.k; j0 += 8) {
                // Issue the token's loads together (as 16-byte pairs when k is even), then
                // use them.
                int64_t e[8];
                if (a.vec_ids) {
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        if (j0 + i < a.k) {
                            const longlong2 v = __ldg(reinterpret_cast<const longlong2*>(row + j0 + i));
                            e[i] = v.x;
                            e[i + 1] = v.y;
                        } else {
                            e[i] = e[i + 1] = -1;
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) e[i] = (j0 + i < a.k) ? __ldg(row + j0 + i) : -1;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (e[i] == -1) continue;
                    if (e[i] < 0 || e[i] >= a.E) {
                        raise_flag(a.err, EP_DEVERR_BAD_EXPERT);
                        continue;
                    }
                    atomicAdd(&hist[(int)e[i]], 1);
                    const int d = a.el_shift >= 0 ? (int)e[i] >> a.el_shift : (int)e[i] / a.E_loc;
                    mask |= 1ull << d;
                }
            }
            const int64_t off = ((int64_t)s * a.T + t) * a.R;
            write_rank_bytes(a.in_rank + off, mask, a.R);
            if (a.in_rank_extra != nullptr) write_rank_bytes(a.in_rank_extra + off, mask, a.R);
        }
        for (int d = 0; d < a.R; ++d) {
            const unsigned b = __ballot_sync(0xFFFFFFFFu, (mask >> d) & 1ull);
            if (lane == 0 && b != 0) atomicAdd(&cnt[d], __popc(b));
        }
    }
    __syncthreads();
    for (int d = threadIdx.x; d < a.R; d += kThreads)
        a.ws_cnt[((int64_t)s * a.R + d) * a.C + c] = cnt[d];
    int32_t* we = a.ws_expert + ((int64_t)s * a.C + c) * a.E;
    for (int e = threadIdx.x; e < a.E; e += kThreads) we[e] = hist[e];
}

// Expert-major placement, first step (blocks of the prefix launch with blockIdx.y >= R):
// one warp per expert e scans its counts over (source, channel) pairs in lexicographic
// order, in place in the workspace (exclusive prefix), and writes its total (ws_etot[e],
// which is also num_recv_tokens_per_expert) and its per-source sums
// (num_tokens_per_expert[s][e], accumulated per warp in shared memory). Up to four
// 32-value chunks are loaded before any is scanned, so most columns cost one round trip.
// These blocks are the only readers of the expert counts in this launch, which is why
// the prefix blocks leave the expert totals to them.
__device__ __forceinline__ void expert_column_scan(const LayoutArgs& a, int sb, int (*acc)[EP_MAX_RANKS]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = sb * kWarps + warp;
    const int n = a.R * a.C;
    if (e >= a.E) return;                         // warp-uniform; no block barrier follows
    for (int sp = lane; sp < a.R; sp += 32) acc[warp][sp] = 0;
    __syncwarp();
    int carry = 0;
    for (int i0 = 0; i0 < n; i0 += 128) {
        int v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = i0 + q * 32 + lane;
            v[q] = i < n ? a.ws_expert[(int64_t)i * a.E + e] : 0;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = i0 + q * 32 + lane;
            int incl = v[q];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            if (i < n) {
                a.ws_expert[(int64_t)i * a.E + e] = carry + incl - v[q];
                if (v[q] != 0) atomicAdd(&acc[warp][i / a.C], v[q]);
            }
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
    }
    __syncwarp();
    if (a.num_tokens_per_expert != nullptr)
        for (int sp = lane; sp < a.R; sp += 32) a.num_tokens_per_expert[(int64_t)sp * a.E + e] = acc[warp][sp];
    if (lane == 0) {
        a.ws_etot[e] = carry;
        a.num_recv_per_expert[e] = carry;
    }
}

__global__ void __launch_bounds__(kThreads) layout_prefix_kernel(LayoutArgs a) {
    constexpr int kDPerWarp = EP_MAX_RANKS / kWarps;   // destinations per warp, at most
    __shared__ int s_base[EP_MAX_RANKS];
    __shared__ int s_warp_tot[kWarps][EP_MAX_RANKS];
    __shared__ int s_warp_off[kWarps][EP_MAX_RANKS];
    const int c = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = a.R, C = a.C, E = a.E;
    const int nblocks = R * C, b = s * C + c;
    const int t0 = min(c * a.tpc, a.T), t1 = min(t0 + a.tpc, a.T);
    pdl_trigger();
    pdl_wait();
    if (s >= R) {                                 // expert column-scan block
        expert_column_scan(a, (s - R) * C + c, s_warp_tot);
        return;
    }
    const bool totals = a.scan_rows == 0;         // else the scan blocks write them

    // ---- Loads. Everything the block reads first is loaded before any store or
    // barrier, so the loads share one memory round trip.
    // Rank bits of this thread's token in the first tile.
    const int t_first = t0 + threadIdx.x;
    uint64_t mask = (t_first < t1) ? read_rank_bytes(a.in_rank + ((int64_t)s * a.T + t_first) * R, R) : 0ull;
    // (1) Per destination d (warp-owned): A = tokens of earlier sources, B = tokens of
    // earlier channels of s, own = this channel, F = all channels of s.
    int A[kDPerWarp], B[kDPerWarp], own[kDPerWarp], F[kDPerWarp];
#pragma unroll
    for (int q = 0; q < kDPerWarp; ++q) {
        A[q] = B[q] = own[q] = F[q] = 0;
        const int d = warp + q * kWarps;
        if (d < R) {
#pragma unroll 4
            for (int i = lane; i < s * C; i += 32) {
                const int sp = i / C, cp = i - sp * C;
                A[q] += a.ws_cnt[((int64_t)sp * R + d) * C + cp];
            }
            for (int cp = lane; cp < C; cp += 32) {
                const int v = a.ws_cnt[((int64_t)s * R + d) * C + cp];
                F[q] += v;
                if (cp < c) B[q] += v;
                if (cp == c) own[q] += v;
            }
        }
    }
    // (2) Per-source expert totals: one (source, expert) pair per thread of the grid.
    const int p2 = b * kThreads + threadIdx.x;
    int sum2 = 0;
    if (totals && a.num_tokens_per_expert != nullptr && p2 < R * E) {
        const int sp = p2 / E, e = p2 - sp * E;
        const int32_t* col = a.ws_expert + (int64_t)sp * C * E + e;
        for (int c0 = 0; c0 < C; c0 += 16) {   // 16 loads in flight before the first add
            int v[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = c0 + q < C ? col[(int64_t)(c0 + q) * E] : 0;
#pragma unroll
            for (int q = 0; q < 16; ++q) sum2 += v[q];
        }
    }
    // (3) Per-expert receive totals: one expert per warp of the grid.
    const int e3 = totals ? b * kWarps + warp : E;
    int sum3 = 0;
    if (e3 < E) {
        for (int i0 = 0; i0 < R * C; i0 += 32 * 8) {   // 8 loads per lane in flight
            int v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int i = i0 + q * 32 + lane;
                v[q] = i < R * C ? a.ws_expert[(int64_t)i * E + e3] : 0;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) sum3 += v[q];
        }
    }

    // ---- Reductions and stores.
#pragma unroll
    for (int q = 0; q < kDPerWarp; ++q) {
        const int d = warp + q * kWarps;
        if (d < R) {
            const int Aq = warp_sum(A[q]), Bq = warp_sum(B[q]), oq = warp_sum(own[q]), Fq = warp_sum(F[q]);
            if (lane == 0) {
                s_base[d] = Aq + Bq;
                a.recv_channel_prefix[((int64_t)d * R + s) * C + c] = Aq + Bq;
                a.channel_prefix[((int64_t)s * R + d) * C + c] = Bq + oq;
                if (c == 0) {
                    a.rank_prefix[s * R + d] = Aq + Fq;
                    if (a.num_tokens_per_rank != nullptr) a.num_tokens_per_rank[s * R + d] = Fq;
                }
            }
        }
    }
    if (totals && a.num_tokens_per_expert != nullptr) {
        if (p2 < R * E) a.num_tokens_per_expert[p2] = sum2;
        // Grids smaller than R*E threads take the remaining pairs in further passes.
        for (int p = p2 + nblocks * kThreads; p < R * E; p += nblocks * kThreads) {
            const int sp = p / E, e = p - sp * E;
            int sum = 0;
#pragma unroll 4
            for (int cp = 0; cp < C; ++cp) sum += a.ws_expert[((int64_t)sp * C + cp) * E + e];
            a.num_tokens_per_expert[p] = sum;
        }
    }
    if (e3 < E) {
        sum3 = warp_sum(sum3);
        if (lane == 0) a.num_recv_per_expert[e3] = sum3;
        for (int e = e3 + nblocks * kWarps; e < E; e += nblocks * kWarps) {
            int sum = 0;
#pragma unroll 4
            for (int i = lane; i < R * C; i += 32) sum += a.ws_expert[(int64_t)i * E + e];
            sum = warp_sum(sum);
            if (lane == 0) a.num_recv_per_expert[e] = sum;
        }
    }
    __syncthreads();

    // ---- send_head for the tokens of channel c of source s (block-wide scan).
    for (int tile = t0; tile < t1; tile += kThreads) {   // block-uniform trip count
        const int t = tile + threadIdx.x;
        if (tile != t0)
            mask = (t < t1) ? read_rank_bytes(a.in_rank + ((int64_t)s * a.T + t) * R, R) : 0ull;
        for (int d = 0; d < R; ++d) {
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, (mask >> d) & 1ull);
            if (lane == 0) s_warp_tot[warp][d] = __popc(bal);
        }
        __syncthreads();
        // Offsets of the warps per destination: one warp per destination scans the
        // kWarps (16) warp totals with shuffles.
        for (int d = warp; d < R; d += kWarps) {
            const int v = lane < kWarps ? s_warp_tot[lane][d] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < kWarps; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            const int run = s_base[d];
            if (lane < kWarps) s_warp_off[lane][d] = run + incl - v;
            __syncwarp();
            if (lane == kWarps - 1) s_base[d] = run + incl;
        }
        __syncthreads();
        const uint32_t lt = lanemask_lt();
        int32_t* out = a.send_head + ((int64_t)s * a.T + t) * R;
        if (a.vec_head) {
            // Four destinations per 16-byte store.
            for (int d0 = 0; d0 < R; d0 += 4) {
                int v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int d = d0 + q;
                    const bool in = (mask >> d) & 1ull;
                    const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
                    v[q] = in ? s_warp_off[warp][d] + __popc(bal & lt) : -1;
                }
                if (t < t1) *reinterpret_cast<int4*>(out + d0) = make_int4(v[0], v[1], v[2], v[3]);
            }
        } else {
            for (int d = 0; d < R; ++d) {
                const bool in = (mask >> d) & 1ull;
                const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
                if (t < t1) out[d] = in ? s_warp_off[warp][d] + __popc(bal & lt) : -1;
            }
        }
        __syncthreads();
    }
}

// ---- Expert-major placement (optional): rows of destination d grouped by local expert,
// then source rank, then token. The column-scan blocks of the prefix launch (above)
// turn the per-(source, channel) expert counts into column prefixes; then:

// One block per (channel c, source s). Each entry's row = the expert's prefix on its
// destination + the count of that expert in earlier (source, channel) pairs + the count
// of earlier tokens of the channel with the same expert. The last term comes from
// shared-memory bitmasks over sub-tiles of 32*ew tokens (one bit per token and expert,
// set with atomicOr, then popc), so the result does not depend on thread timing.
__global__ void __launch_bounds__(kThreads) layout_expert_rows_kernel(LayoutArgs a) {
    extern __shared__ uint32_t esm[];
    int* running = reinterpret_cast<int*>(esm);   // [E]
    uint32_t* mask = esm + a.E;                    // [E][ew | 1]: odd stride, no bank conflicts
    const int c = blockIdx.x, s = blockIdx.y, W = a.ew, WS = a.ew | 1, sub = 32 * a.ew;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    const int t0 = min(c * a.tpc, a.T), t1 = min(t0 + a.tpc, a.T);
    const int lt = threadIdx.x;
    // Loads that do not depend on one another go out together, before any barrier: the
    // first tile's ids (k <= 8: kept in registers for both passes over the tile) and this
    // block's column prefixes (E <= threads per block).
    const bool keep_ids = a.k <= 8;
    int64_t ev0[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ev0[i] = -1;
    if (keep_ids && lt < sub && t0 + lt < t1) {
        const int64_t* row = a.topk_idx + ((int64_t)s * a.T + t0 + lt) * a.k;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < a.k) ev0[i] = __ldg(row + i);
    }
    const int col = (a.E <= kThreads && lt < a.E) ? a.ws_expert[((int64_t)s * a.C + c) * a.E + lt] : 0;
    // Per destination d (one warp each): exclusive prefix of the expert totals over its
    // local experts -> running[e]; block (0, 0) also writes expert_prefix.
    for (int d = warp; d < a.R; d += kWarps) {
        int carry = 0;
        for (int el0 = 0; el0 < a.E_loc; el0 += 32) {
            const int el = el0 + lane;
            const int v = el < a.E_loc ? a.ws_etot[d * a.E_loc + el] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            if (el < a.E_loc) {
                running[d * a.E_loc + el] = carry + incl - v;
                if (c == 0 && s == 0) a.expert_prefix[(int64_t)d * (a.E_loc + 1) + el] = carry + incl - v;
            }
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (c == 0 && s == 0 && lane == 0) a.expert_prefix[(int64_t)d * (a.E_loc + 1) + a.E_loc] = carry;
    }
    __syncthreads();
    if (a.E <= kThreads) {
        if (lt < a.E) running[lt] += col;
    } else {
        for (int e = threadIdx.x; e < a.E; e += kThreads)
            running[e] += a.ws_expert[((int64_t)s * a.C + c) * a.E + e];
    }
    for (int base = t0; base < t1; base += sub) {   // block-uniform trip count
        for (int i = threadIdx.x; i < a.E * WS; i += kThreads) mask[i] = 0u;
        __syncthreads();
        const int t = base + lt;
        const bool mine = lt < sub && t < t1;
        const int64_t* row = a.topk_idx + ((int64_t)s * a.T + t) * a.k;
        // The token's ids are loaded in batches of 8 before any shared-memory atomic.
        const bool first = keep_ids && base == t0;
        for (int j0 = 0; j0 < a.k; j0 += 8) {
            int64_t ev[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                ev[i] = first ? ev0[i] : ((mine && j0 + i < a.k) ? __ldg(row + j0 + i) : -1);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (ev[i] >= 0 && ev[i] < a.E) atomicOr(&mask[ev[i] * WS + (lt >> 5)], 1u << (lt & 31));
        }
        __syncthreads();
        for (int j0 = 0; j0 < a.k; j0 += 8) {
            int64_t ev[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                ev[i] = first ? ev0[i] : ((mine && j0 + i < a.k) ? __ldg(row + j0 + i) : -1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (!mine || j0 + i >= a.k) continue;
                const int64_t e = ev[i];
                int r = -1;
                if (e >= 0 && e < a.E) {
                    const uint32_t* m = mask + e * WS;
                    r = running[e];
                    for (int w = 0; w < (lt >> 5); ++w) r += __popc(m[w]);
                    r += __popc(m[lt >> 5] & ((1u << (lt & 31)) - 1u));
                }
                a.expert_rows[((int64_t)s * a.T + t) * a.k + j0 + i] = r;
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < a.E; e += kThreads) {
            int add = 0;
            for (int w = 0; w < W; ++w) add += __popc(mask[e * WS + w]);
            running[e] += add;
        }
        __syncthreads();
    }
}

size_t ws_cnt_bytes(const ep_shape* sh) {
    const size_t n = (size_t)sh->num_ranks * sh->num_ranks * sh->num_channels * sizeof(int32_t);
    return (n + 255) & ~(size_t)255;
}

}  // namespace
}  // namespace ep

extern "C" {

size_t ep_layout_workspace_size(const ep_shape* sh) {
    if (ep::check_shape(sh) != EP_OK) return 0;
    return ep::ws_cnt_bytes(sh) +
           (size_t)sh->num_ranks * sh->num_channels * sh->num_experts * sizeof(int32_t) +
           (size_t)sh->num_experts * sizeof(int32_t);
}

ep_status ep_get_layout(const ep_shape* sh, const int64_t* topk_idx, ep_layout* layout,
                        ep_handle* handle, void* workspace, size_t workspace_bytes,
                        const ep_launch* launch) {
    using namespace ep;
    ep_status st = check_shape(sh);
    if (st != EP_OK) return st;
    if (handle == nullptr || launch == nullptr) return EP_ERR_INVALID_ARG;
    if (handle->rank_prefix_matrix == nullptr || handle->channel_prefix_matrix == nullptr ||
        handle->recv_channel_prefix_matrix == nullptr || handle->num_recv_tokens_per_expert == nullptr)
        return EP_ERR_INVALID_ARG;
    // Per-token arrays are empty (and may be NULL) when there are no tokens.
    if (sh->num_tokens > 0 && (handle->is_token_in_rank == nullptr || handle->send_head == nullptr))
        return EP_ERR_INVALID_ARG;
    if (layout != nullptr && layout->num_tokens_per_rdma_rank != nullptr) return EP_ERR_INVALID_ARG;
    // Expert-major placement is optional: both outputs or neither.
    const bool expert = handle->expert_rows != nullptr || handle->expert_prefix != nullptr;
    if (expert && (handle->expert_prefix == nullptr || (sh->num_tokens > 0 && handle->expert_rows == nullptr)))
        return EP_ERR_INVALID_ARG;
    if (expert && sh->num_experts > EP_EXPERT_MAJOR_MAX_EXPERTS) return EP_ERR_UNSUPPORTED;
    if (sh->num_tokens > 0 && topk_idx == nullptr) return EP_ERR_INVALID_ARG;
    const size_t need = ep_layout_workspace_size(sh);
    if (workspace == nullptr || workspace_bytes < need || ((uintptr_t)workspace & 15) != 0)
        return EP_ERR_INVALID_ARG;
    if ((sh->num_ranks & 7) == 0) {
        // 8-byte vector access of is_token_in_rank rows needs 8-byte alignment.
        if (((uintptr_t)handle->is_token_in_rank & 7) != 0) return EP_ERR_INVALID_ARG;
        if (layout != nullptr && layout->is_token_in_rank != nullptr &&
            ((uintptr_t)layout->is_token_in_rank & 7) != 0)
            return EP_ERR_INVALID_ARG;
    }

    LayoutArgs a{};
    a.topk_idx = topk_idx;
    a.R = sh->num_ranks;
    a.T = sh->num_tokens;
    a.E = sh->num_experts;
    a.k = sh->num_topk;
    a.C = sh->num_channels;
    a.E_loc = a.E / a.R;
    a.tpc = a.T > 0 ? ceil_div(a.T, a.C) : 1;
    a.num_tokens_per_rank = layout ? layout->num_tokens_per_rank : nullptr;
    a.num_tokens_per_expert = layout ? layout->num_tokens_per_expert : nullptr;
    a.in_rank = handle->is_token_in_rank;
    a.in_rank_extra = (layout && layout->is_token_in_rank != handle->is_token_in_rank)
                          ? layout->is_token_in_rank
                          : nullptr;
    a.rank_prefix = handle->rank_prefix_matrix;
    a.channel_prefix = handle->channel_prefix_matrix;
    a.recv_channel_prefix = handle->recv_channel_prefix_matrix;
    a.send_head = handle->send_head;
    a.num_recv_per_expert = handle->num_recv_tokens_per_expert;
    a.ws_cnt = reinterpret_cast<int32_t*>(workspace);
    a.ws_expert = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(workspace) + ws_cnt_bytes(sh));
    a.ws_etot = a.ws_expert + (size_t)a.R * a.C * a.E;
    a.expert_rows = handle->expert_rows;
    a.expert_prefix = handle->expert_prefix;
    // Bitmask words per expert (rows padded to an odd stride): at most ~6144 + E words. A
    // sub-tile of 32 * ew tokens has one thread per token, so ew <= kWarps.
    a.ew = expert ? (a.E >= 6144 ? 1 : (6144 / a.E > kWarps ? kWarps : 6144 / a.E)) : 1;
    a.err = launch->error_flags;

    a.el_shift = (a.E_loc & (a.E_loc - 1)) == 0 ? __builtin_ctz((unsigned)a.E_loc) : -1;
    a.vec_ids = (a.k % 2 == 0 && ((uintptr_t)topk_idx & 15) == 0) ? 1 : 0;
    a.vec_head = (a.R % 4 == 0 && ((uintptr_t)handle->send_head & 15) == 0) ? 1 : 0;
    // Expert-major placement: enough extra grid rows of the prefix launch for one warp
    // per expert.
    a.scan_rows = expert ? ceil_div(ceil_div(a.E, kWarps), a.C) : 0;

    if ((st = begin_call(launch)) != EP_OK) return st;
    const dim3 grid(a.C, a.R);
    const size_t smem = sizeof(int) * (size_t)(a.E + a.R);
    cudaError_t e = launch_pdl(layout_count_kernel, grid, dim3(kThreads), smem, launch->stream, a);
    if (e == cudaSuccess)
        e = launch_pdl(layout_prefix_kernel, dim3(a.C, a.R + a.scan_rows), dim3(kThreads), 0, launch->stream, a);
    if (e == cudaSuccess && expert)
        e = launch_pdl(layout_expert_rows_kernel, grid, dim3(kThreads),
                       sizeof(uint32_t) * (size_t)a.E * (1 + (size_t)(a.ew | 1)), launch->stream, a);
    if (e != cudaSuccess) return cuda_fail(e);
    return end_call(launch);
}

}  // extern "C"
