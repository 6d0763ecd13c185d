/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for MoE expert-parallel
 * layout / dispatch / combine with R virtual ranks.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file. The product (the CUDA library) never calls it,
 * and the two share no code, header, table or constant.
 *
 * Every result is written as the plain definition: explicit loops in natural index
 * order, no blocking, no fusion, no reordering. Build with -O2 -ffp-contract=off and
 * no fast-math so that every float operation is one IEEE-754 round-to-nearest-even
 * operation.
 *
 * Citations name the source pages:
 *   [README]  "DeepEP" -- README of the EnflameTechnology/DeepEP port (normal-kernel
 *             example with get_dispatch_layout / dispatch / combine and their
 *             backward functions; low-latency example; feature notes on FP8).
 *   [REUSE]   "How DeepEP Optimizes Handle Reuse for Repeated Dispatches".
 *   [HOOK]    "How DeepEP Enables Hook-Based Overlapping Without SM Occupation".
 * The pages name the tensors but give no formula for them; where a definition is a
 * reading of the names and signatures, the comment says "reading".
 *
 * Conventions shared with the tests (not with the GPU code):
 *   R ranks, T tokens per source rank, H hidden, E experts, E_loc = E / R, k top-k,
 *   C channels per source rank. Expert e lives on rank e / E_loc. bf16 values are
 *   passed as uint16 bit patterns; e4m3 values as uint8 bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* bf16 is binary32 with the low 16 fraction bits removed, so widening is exact. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t float_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/*
 * Round a double to the nearest bf16 value, ties to even (IEEE-754 roundTiesToEven).
 * Method: scale |v| so that the bf16 grid around it becomes the integers, round with
 * nearbyint (default rounding mode = to nearest, ties to even), scale back. bf16 has
 * 8 significant bits, exponent range like binary32: normal spacing 2^(p-7) for a value
 * in [2^p, 2^(p+1)), subnormal spacing 2^-133, overflow threshold 2^128.
 */
static uint16_t double_to_bf16_rne(double v)
{
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);            /* a = m * 2^e, 0.5 <= m < 1: leading bit 2^(e-1) */
    int q = (e - 1) - 7;           /* exponent of the last kept fraction bit */
    if (q < -133) q = -133;
    double r = nearbyint(ldexp(a, -q));
    double res = ldexp(r, q);
    if (res >= 0x1p128) return (uint16_t)(sign | 0x7F80);
    float f = (float)res;          /* exact: res is a bf16 value */
    return (uint16_t)(sign | (float_bits(f) >> 16));
}

/*
 * OCP 8-bit floating point, E4M3 variant: 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits; no infinities; S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8.
 * Normal: (1 + M/8) * 2^(E-7); subnormal (E == 0): (M/8) * 2^-6.
 */
static double e4m3_bits_to_double(uint8_t b)
{
    int s = b >> 7, E = (b >> 3) & 15, M = b & 7;
    double v;
    if (E == 15 && M == 7) return NAN;
    if (E == 0) v = ldexp((double)M, -9);
    else v = ldexp((double)(8 + M), E - 10);
    return s ? -v : v;
}

/*
 * fp32 -> e4m3, round to nearest even, saturating to +-448 (the "satfinite" mode):
 * the grid around |v| in [2^p, 2^(p+1)) has spacing 2^(p-3), subnormal spacing 2^-9.
 * NaN maps to 0x7F. The sign is kept, so a negative value that rounds to zero gives
 * 0x80.
 */
static uint8_t float_to_e4m3_rne_sat(float v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    double res;
    if (!(a < 448.0)) {
        res = 448.0;
    } else if (a == 0.0) {
        return sign;
    } else {
        int e;
        (void)frexp(a, &e);
        int q = (e - 1) - 3;
        if (q < -9) q = -9;
        res = ldexp(nearbyint(ldexp(a, -q)), q);
        if (res > 448.0) res = 448.0;
    }
    if (res == 0.0) return sign;
    int e2;
    (void)frexp(res, &e2);
    int p = e2 - 1;                              /* res in [2^p, 2^(p+1)) */
    int E, M;
    if (p < -6) { E = 0; M = (int)ldexp(res, 9); }
    else { E = p + 7; M = (int)ldexp(res, 3 - p) - 8; }
    return (uint8_t)(sign | (E << 3) | M);
}

EXPORT void oracle_bf16_from_double(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; i++) out[i] = double_to_bf16_rne(v[i]);
}

EXPORT void oracle_e4m3_encode(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; i++) out[i] = float_to_e4m3_rne_sat(v[i]);
}

EXPORT void oracle_e4m3_decode(const uint8_t* b, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; i++) out[i] = e4m3_bits_to_double(b[i]);
}

/* ------------------------------------------------------------------------- */
/* FP8 quantisation of one token row                                         */
/* ------------------------------------------------------------------------- */

/*
 * [README] feature notes: FP8 dispatch with per-group scales, and the two scale modes
 * round_scale (power-of-two scales) and use_ue8m0 (UE8M0 scale format), and a single
 * per-tensor scale fp8_quant_scale. Group = 128 channels. Per group g:
 *   amax = max |x|; amax' = max(amax, 1e-4) (floor for all-zero groups, a choice of
 *   this project); s0 = amax' / 448 (one IEEE fp32 division).
 *   mode 0 (fp32 scale):      scale = s0,                      inv = 448 / amax'
 *   mode 1 (power of two):    scale = 2^ceil(log2(s0)),        inv = 1 / scale (exact)
 *   mode 2 (UE8M0):           as mode 1; the scale is stored as the byte log2(scale) + 127
 *   mode 3 (per tensor):      scale = the caller's s for every group, inv = 1 / s (fp32)
 *   q = e4m3(x * inv), one fp32 multiply, round to nearest even, saturating.
 * Readings: "scale" is the dequantisation factor (x ~= value(q) * scale); rounding the
 * scale up to a power of two keeps |x * inv| <= 448; UE8M0 = unsigned 8-bit exponent
 * with bias 127, no mantissa; a per-tensor scale is written to every group's slot so the
 * receive format does not change.
 * Scales go to scales_f32[g] (modes 0, 1, 3) or scales_u8[g] (mode 2).
 */
static float pow2_ceil(float v)
{
    int e;
    double m = frexp((double)v, &e);     /* v = m * 2^e, 0.5 <= m < 1 */
    return (float)ldexp(1.0, m == 0.5 ? e - 1 : e);
}

EXPORT void oracle_quantize_row_mode(const uint16_t* xrow, int H, int mode, float tensor_scale,
                                     uint8_t* q, float* scales_f32, uint8_t* scales_u8)
{
    for (int g = 0; g < H / 128; g++) {
        float amax = 0.0f;
        for (int i = 0; i < 128; i++) {
            float a = fabsf(bf16_bits_to_float(xrow[g * 128 + i]));
            if (a > amax) amax = a;
        }
        float am = amax > 1e-4f ? amax : 1e-4f;
        float scale, inv;
        if (mode == 0) {
            scale = am / 448.0f;
            inv = 448.0f / am;
        } else if (mode == 1 || mode == 2) {
            scale = pow2_ceil(am / 448.0f);
            inv = (float)(1.0 / (double)scale);          /* exact: scale is 2^n */
        } else {
            scale = tensor_scale;
            inv = 1.0f / tensor_scale;
        }
        for (int i = 0; i < 128; i++) {
            float v = bf16_bits_to_float(xrow[g * 128 + i]) * inv;
            q[g * 128 + i] = float_to_e4m3_rne_sat(v);
        }
        if (mode == 2) {
            int e;
            (void)frexp((double)scale, &e);              /* scale = 2^(e-1) */
            scales_u8[g] = (uint8_t)(e - 1 + 127);
        } else {
            scales_f32[g] = scale;
        }
    }
}

EXPORT void oracle_quantize_row(const uint16_t* xrow, int H, uint8_t* q, float* scales)
{
    oracle_quantize_row_mode(xrow, H, 0, 0.0f, q, scales, NULL);
}

/* ------------------------------------------------------------------------- */
/* Layout                                                                    */
/* ------------------------------------------------------------------------- */

/*
 * [README] normal-kernel example, get_dispatch_layout: topk_idx -> num_tokens_per_rank,
 * num_tokens_per_expert, is_token_in_rank. [REUSE] "What the Handle Contains": the
 * handle holds rank_prefix_matrix, channel_prefix_matrix, recv_channel_prefix_matrix,
 * recv_src_idx, is_token_in_rank, send_head.
 *
 * Definitions (readings of the names; the pages give no formula):
 *   num_tokens_per_expert[s][e] = #{(t, j): topk_idx[s][t][j] == e}
 *   is_token_in_rank[s][t][d]   = 1 if some valid entry of token t has e / E_loc == d
 *                                  (a token counts once per rank)
 *   num_tokens_per_rank[s][d]   = sum_t is_token_in_rank[s][t][d]
 *   channel of token t          = t / ceil(T / C)
 *   channel_prefix_matrix[s][d][c]      = inclusive prefix over channels of the
 *                                         per-channel token counts
 *   rank_prefix_matrix[s][d]            = inclusive prefix over source ranks of
 *                                         num_tokens_per_rank
 *   recv_channel_prefix_matrix[d][s][c] = first row, in d's receive region, of source
 *                                         s's channel c
 *   send_head[s][t][d]          = row of (s, t) in d's region (rows ordered by source
 *                                  rank, then token), or -1
 *   num_recv_tokens_per_expert[d][j]    = sum_s num_tokens_per_expert[s][d*E_loc + j]
 * Entries equal to -1 are masked. Other entries outside [0, E) are counted as errors
 * and skipped. Returns the number of such entries.
 */
EXPORT int64_t oracle_layout(int R, int T, int E, int k, int C, const int64_t* topk_idx,
                             int32_t* num_tokens_per_rank,        /* [R][R] */
                             int32_t* num_tokens_per_expert,      /* [R][E] */
                             uint8_t* is_token_in_rank,           /* [R][T][R] */
                             int32_t* rank_prefix_matrix,         /* [R][R] */
                             int32_t* channel_prefix_matrix,      /* [R][R][C] */
                             int32_t* recv_channel_prefix_matrix, /* [R][R][C] */
                             int32_t* send_head,                  /* [R][T][R] */
                             int32_t* num_recv_tokens_per_expert) /* [R][E/R] */
{
    const int E_loc = E / R;
    const int tpc = (T + C - 1) / C;
    int64_t bad = 0;
    int32_t* cnt = (int32_t*)calloc((size_t)R * R * C, sizeof(int32_t));

    memset(num_tokens_per_rank, 0, sizeof(int32_t) * R * R);
    memset(num_tokens_per_expert, 0, sizeof(int32_t) * R * E);
    memset(is_token_in_rank, 0, (size_t)R * T * R);

    for (int s = 0; s < R; s++)
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                int64_t e = topk_idx[((int64_t)s * T + t) * k + j];
                if (e == -1) continue;
                if (e < 0 || e >= E) { bad++; continue; }
                num_tokens_per_expert[s * E + e] += 1;
                is_token_in_rank[((int64_t)s * T + t) * R + e / E_loc] = 1;
            }

    for (int s = 0; s < R; s++)
        for (int t = 0; t < T; t++)
            for (int d = 0; d < R; d++)
                if (is_token_in_rank[((int64_t)s * T + t) * R + d]) {
                    num_tokens_per_rank[s * R + d] += 1;
                    cnt[(s * R + d) * C + t / tpc] += 1;
                }

    for (int s = 0; s < R; s++)
        for (int d = 0; d < R; d++) {
            int32_t run = 0;
            for (int c = 0; c < C; c++) {
                run += cnt[(s * R + d) * C + c];
                channel_prefix_matrix[(s * R + d) * C + c] = run;
            }
        }

    for (int d = 0; d < R; d++) {
        int32_t run = 0;
        for (int s = 0; s < R; s++) {
            run += num_tokens_per_rank[s * R + d];
            rank_prefix_matrix[s * R + d] = run;
        }
    }

    for (int d = 0; d < R; d++)
        for (int s = 0; s < R; s++)
            for (int c = 0; c < C; c++) {
                int32_t base = s > 0 ? rank_prefix_matrix[(s - 1) * R + d] : 0;
                int32_t within = c > 0 ? channel_prefix_matrix[(s * R + d) * C + c - 1] : 0;
                recv_channel_prefix_matrix[(d * R + s) * C + c] = base + within;
            }

    for (int s = 0; s < R; s++)
        for (int d = 0; d < R; d++) {
            int32_t row = s > 0 ? rank_prefix_matrix[(s - 1) * R + d] : 0;
            for (int t = 0; t < T; t++) {
                int64_t i = ((int64_t)s * T + t) * R + d;
                send_head[i] = is_token_in_rank[i] ? row++ : -1;
            }
        }

    for (int d = 0; d < R; d++)
        for (int j = 0; j < E_loc; j++) {
            int32_t sum = 0;
            for (int s = 0; s < R; s++) sum += num_tokens_per_expert[s * E + d * E_loc + j];
            num_recv_tokens_per_expert[d * E_loc + j] = sum;
        }

    free(cnt);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Dispatch                                                                  */
/* ------------------------------------------------------------------------- */

/*
 * [README] normal-kernel example, dispatch; [REUSE] "Fast Path Dispatch with Handle
 * Reuse". Each token row is sent once to every rank it is in. Destination d's rows
 * live at [row_offset[d], row_offset[d+1]) of one receive allocation; the token's row
 * in that region is send_head[s][t][d].
 *
 * x_kind: 0 = bf16 rows copied as bf16 (elem 2 bytes);
 *         1 = bf16 rows quantised to e4m3 with per-128-channel scales;
 *         2 = pre-quantised e4m3 rows (x_scales [R][T][H/128]) copied byte for byte.
 * scale_mode / tensor_scale: the quantisation mode of x_kind 1 (see above); in mode 2
 * recv_x_scales holds one byte per group, otherwise one fp32 per group.
 * recv_topk_idx[row][j] = e - d*E_loc if e lives on d, else -1 (reading);
 * recv_topk_weights[row][j] = w if e lives on d, else 0 (reading);
 * recv_src_idx[row] = t. topk_idx == NULL (handle reuse) leaves the topk outputs alone.
 * Returns the number of rows that fell outside their region (skipped).
 */
EXPORT int64_t oracle_dispatch(int R, int T, int H, int E, int k, int x_kind,
                               int scale_mode, float tensor_scale,
                               const void* x, const float* x_scales,
                               const int64_t* topk_idx, const float* topk_weights,
                               const int32_t* send_head, const int64_t* row_offset,
                               void* recv_x, void* recv_x_scales,
                               int64_t* recv_topk_idx, float* recv_topk_weights,
                               int32_t* recv_src_idx)
{
    const int E_loc = E / R;
    const int G = H / 128;
    const size_t out_elem = (x_kind == 0) ? 2 : 1;
    int64_t bad = 0;
    const size_t scale_elem = (x_kind == 1 && scale_mode == 2) ? 1 : 4;
    uint8_t* qrow = (uint8_t*)malloc((size_t)H + 1);
    float* srow = (float*)malloc(sizeof(float) * (size_t)(G + 1));
    uint8_t* brow = (uint8_t*)malloc((size_t)G + 1);

    for (int s = 0; s < R; s++)
        for (int t = 0; t < T; t++) {
            const int64_t tok = (int64_t)s * T + t;
            const void* src_row;
            const void* src_scales = NULL;
            if (x_kind == 0) {
                src_row = (const uint16_t*)x + tok * H;
            } else if (x_kind == 1) {
                oracle_quantize_row_mode((const uint16_t*)x + tok * H, H, scale_mode, tensor_scale,
                                         qrow, srow, brow);
                src_row = qrow;
                src_scales = scale_mode == 2 ? (const void*)brow : (const void*)srow;
            } else {
                src_row = (const uint8_t*)x + tok * H;
                src_scales = x_scales + tok * G;
            }
            for (int d = 0; d < R; d++) {
                int32_t h = send_head[tok * R + d];
                if (h < 0) continue;
                int64_t row = row_offset[d] + h;
                if (row >= row_offset[d + 1]) { bad++; continue; }
                memcpy((uint8_t*)recv_x + (size_t)row * H * out_elem, src_row, (size_t)H * out_elem);
                if (x_kind != 0)
                    memcpy((uint8_t*)recv_x_scales + (size_t)row * G * scale_elem, src_scales,
                           scale_elem * (size_t)G);
                if (recv_src_idx) recv_src_idx[row] = t;
                if (topk_idx) {
                    for (int j = 0; j < k; j++) {
                        int64_t e = topk_idx[tok * k + j];
                        int local = (e >= 0 && e < E && e / E_loc == d);
                        if (recv_topk_idx) recv_topk_idx[row * k + j] = local ? e - (int64_t)d * E_loc : -1;
                        if (recv_topk_weights)
                            recv_topk_weights[row * k + j] = local ? topk_weights[tok * k + j] : 0.0f;
                    }
                }
            }
        }
    free(qrow);
    free(srow);
    free(brow);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Combine                                                                   */
/* ------------------------------------------------------------------------- */

/*
 * [README] normal-kernel example, combine_forward / dispatch_backward; [REUSE]
 * "Combining with Handle Reuse". Rows come back from every rank the token was sent to
 * and are reduced into token order:
 *   mode 0 (SUM, the pages' combine(x, handle)):  out = sum_d y_d[row]
 *   mode 1 (WEIGHTED, the weighted top-k reduce):  out = sum_d c_d * y_d[row],
 *          c_d = sum of topk_weights[s][t][j] over valid j with e_j / E_loc == d
 * The sum is accumulated in binary64 (the bf16 inputs and fp32 weights are exact
 * there) and rounded once to bf16, ties to even. Optional combined_topk_weights[s][t][j] = sum_d recv_topk_weights_d[row][j]
 * (binary64 sum, rounded once to fp32) -- the reduction of the weights gradient in
 * dispatch_backward.
 * Returns the number of rows that fell outside their region (skipped).
 */
EXPORT int64_t oracle_combine(int R, int T, int H, int E, int k, int mode,
                              const uint16_t* y, const int64_t* row_offset,
                              const int32_t* send_head,
                              const int64_t* topk_idx, const float* topk_weights,
                              const float* recv_topk_weights,
                              uint16_t* out, float* combined_topk_weights)
{
    const int E_loc = E / R;
    int64_t bad = 0;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(H + 1));
    double* wacc = (double*)malloc(sizeof(double) * (size_t)(k + 1));

    for (int s = 0; s < R; s++)
        for (int t = 0; t < T; t++) {
            const int64_t tok = (int64_t)s * T + t;
            for (int h = 0; h < H; h++) acc[h] = 0.0;
            for (int j = 0; j < k; j++) wacc[j] = 0.0;
            for (int d = 0; d < R; d++) {
                int32_t hd = send_head[tok * R + d];
                if (hd < 0) continue;
                int64_t row = row_offset[d] + hd;
                if (row >= row_offset[d + 1]) { bad++; continue; }
                double c = 1.0;
                if (mode == 1) {
                    c = 0.0;
                    for (int j = 0; j < k; j++) {
                        int64_t e = topk_idx[tok * k + j];
                        if (e >= 0 && e < E && e / E_loc == d) c += (double)topk_weights[tok * k + j];
                    }
                }
                for (int h = 0; h < H; h++)
                    acc[h] += c * (double)bf16_bits_to_float(y[(size_t)row * H + h]);
                if (recv_topk_weights)
                    for (int j = 0; j < k; j++) wacc[j] += (double)recv_topk_weights[row * k + j];
            }
            for (int h = 0; h < H; h++) out[(size_t)tok * H + h] = double_to_bf16_rne(acc[h]);
            if (combined_topk_weights)
                for (int j = 0; j < k; j++) combined_topk_weights[tok * k + j] = (float)wacc[j];
        }
    free(acc);
    free(wacc);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Low-latency dispatch / combine                                            */
/* ------------------------------------------------------------------------- */

/*
 * [README] low-latency example, low_latency_dispatch; [HOOK] "Two-Phase Kernel
 * Architecture". Reading of the "specific format": rank d holds, for each local expert
 * el, R*nmax fixed slots; source s owns slots [s*nmax, (s+1)*nmax). Within a source's
 * sub-slot, tokens are kept in token order: the j-th entry of token t that picks
 * expert e lands at pos = s*nmax + #{t' < t of source s that picked e}.
 *
 * Outputs: recv_x[d][el][pos] (bf16 copy, or e4m3 + per-128-channel scales when
 * use_fp8, quantised with scale_mode / tensor_scale as in oracle_quantize_row_mode;
 * the port notes the UE8M0 format for these kernels), src_info[d][el][pos] = t, slot[s][t][j] = pos (-1 when masked),
 * recv_expert_count[d][el] = sum_s count, layout_range[d][el][s] = (s*nmax, count).
 * Counts are int32 (the port returns int32 counts and handles).
 *
 * packed != 0: the same rows without gaps between the source sub-slots (the packed
 * variant of the "specific format" for a grouped GEMM): expert e's rows are numbered
 * 0, 1, 2, ... over all sources in (s, t) order, so source s starts at the sum of the
 * counts of sources s' < s; layout_range[d][el][s] = (that start, count). The per-source
 * capacity check (count <= nmax) is the same in both layouts.
 * Returns the number of entries skipped (outside [0, E), or beyond nmax).
 */
EXPORT int64_t oracle_ll_dispatch(int R, int T, int H, int E, int k, int nmax, int use_fp8,
                                  int packed, int scale_mode, float tensor_scale,
                                  const uint16_t* x, const int64_t* topk_idx,
                                  void* recv_x, void* recv_x_scales, int32_t* src_info,
                                  int32_t* slot, int32_t* recv_expert_count,
                                  int32_t* layout_range)
{
    const int E_loc = E / R;
    const int G = H / 128;
    const int64_t slots = (int64_t)R * nmax;
    const size_t out_elem = use_fp8 ? 1 : 2;
    const size_t scale_elem = scale_mode == 2 ? 1 : 4;
    int64_t bad = 0;
    int32_t* run = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t* next_row = (int32_t*)calloc((size_t)(E + 1), sizeof(int32_t));  /* packed */
    uint8_t* qrow = (uint8_t*)malloc((size_t)H + 1);
    float* srow = (float*)malloc(sizeof(float) * (size_t)(G + 1));
    uint8_t* brow = (uint8_t*)malloc((size_t)G + 1);

    memset(recv_expert_count, 0, sizeof(int32_t) * (size_t)E);
    for (int s = 0; s < R; s++) {
        for (int e = 0; e < E; e++) run[e] = 0;
        for (int e = 0; e < E; e++) {      /* where source s starts in each expert region */
            int d = e / E_loc, el = e % E_loc;
            layout_range[(((int64_t)d * E_loc + el) * R + s) * 2] = packed ? next_row[e] : s * nmax;
        }
        for (int t = 0; t < T; t++) {
            const int64_t tok = (int64_t)s * T + t;
            const uint16_t* xrow = x + tok * H;
            if (use_fp8) oracle_quantize_row_mode(xrow, H, scale_mode, tensor_scale, qrow, srow, brow);
            for (int j = 0; j < k; j++) {
                int64_t e = topk_idx[tok * k + j];
                slot[tok * k + j] = -1;
                if (e == -1) continue;
                if (e < 0 || e >= E || run[e] >= nmax) { bad++; continue; }
                int d = (int)(e / E_loc), el = (int)(e % E_loc);
                int32_t pos = packed ? next_row[e] : s * nmax + run[e];
                run[e] += 1;
                next_row[e] += 1;
                int64_t dst = ((int64_t)d * E_loc + el) * slots + pos;
                if (use_fp8) {
                    memcpy((uint8_t*)recv_x + (size_t)dst * H, qrow, (size_t)H);
                    memcpy((uint8_t*)recv_x_scales + (size_t)dst * G * scale_elem,
                           scale_mode == 2 ? (const void*)brow : (const void*)srow, scale_elem * (size_t)G);
                } else {
                    memcpy((uint8_t*)recv_x + (size_t)dst * H * out_elem, xrow, (size_t)H * out_elem);
                }
                src_info[dst] = t;
                slot[tok * k + j] = pos;
            }
        }
        for (int e = 0; e < E; e++) {
            int d = e / E_loc, el = e % E_loc;
            int64_t lr = (((int64_t)d * E_loc + el) * R + s) * 2;
            layout_range[lr + 1] = run[e];
            recv_expert_count[d * E_loc + el] += run[e];
        }
    }
    free(run);
    free(next_row);
    free(qrow);
    free(srow);
    free(brow);
    return bad;
}

/*
 * [README] low-latency example, low_latency_combine: the weighted top-k reduction
 * out[s][t] = sum over valid j (ascending) of topk_weights[s][t][j] * y[d][el][slot],
 * with y in the dispatch's slot layout [R][E_loc][R*nmax][H] (bf16). Binary64 sum,
 * rounded once to bf16. A token whose entries are all masked gives +0.
 */
EXPORT void oracle_ll_combine(int R, int T, int H, int E, int k, int nmax,
                              const uint16_t* y, const int64_t* topk_idx,
                              const float* topk_weights, const int32_t* slot, uint16_t* out)
{
    const int E_loc = E / R;
    const int64_t slots = (int64_t)R * nmax;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(H + 1));
    for (int s = 0; s < R; s++)
        for (int t = 0; t < T; t++) {
            const int64_t tok = (int64_t)s * T + t;
            for (int h = 0; h < H; h++) acc[h] = 0.0;
            for (int j = 0; j < k; j++) {
                int64_t e = topk_idx[tok * k + j];
                int32_t pos = slot[tok * k + j];
                if (e < 0 || e >= E || pos < 0) continue;
                int d = (int)(e / E_loc), el = (int)(e % E_loc);
                const uint16_t* yrow = y + ((((int64_t)d * E_loc + el) * slots) + pos) * H;
                double w = (double)topk_weights[tok * k + j];
                for (int h = 0; h < H; h++) acc[h] += w * (double)bf16_bits_to_float(yrow[h]);
            }
            for (int h = 0; h < H; h++) out[(size_t)tok * H + h] = double_to_bf16_rne(acc[h]);
        }
    free(acc);
}

/* ------------------------------------------------------------------------- */
/* Expert-major packed receive layout                                        */
/* ------------------------------------------------------------------------- */

/*
 * [README] low-latency example: the receive buffers come in a "specific format" for a
 * grouped GEMM; for the normal kernels the same packing is the expert-major layout.
 * Reading: destination d's region holds one row per valid entry (s, t, j) whose expert e
 * lives on d, grouped by local expert el = e - d*E_loc (ascending), then by source rank,
 * then by entry order (t, j):
 *   expert_prefix[d][el]  = sum over el' < el of num_recv_tokens_per_expert[d][el']
 *                           (expert_prefix[d][E_loc] = the region's row count)
 *   expert_rows[s][t][j]  = expert_prefix[d][el] + sum over s' < s of
 *                           num_tokens_per_expert[s'][e] + #{(t', j') < (t, j) of s with
 *                           expert e}, or -1 for masked / invalid entries.
 * Returns the number of entries outside [-1, E).
 */
EXPORT int64_t oracle_expert_layout(int R, int T, int E, int k, const int64_t* topk_idx,
                                    int32_t* expert_rows, int32_t* expert_prefix)
{
    const int E_loc = E / R;
    int64_t bad = 0;
    int32_t* cnt = (int32_t*)calloc((size_t)R * E + 1, sizeof(int32_t));    /* [s][e] */
    int32_t* run = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
    int32_t* base = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));

    for (int s = 0; s < R; s++)
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                int64_t e = topk_idx[((int64_t)s * T + t) * k + j];
                if (e == -1) continue;
                if (e < 0 || e >= E) { bad++; continue; }
                cnt[s * E + e] += 1;
            }
    for (int d = 0; d < R; d++) {
        int32_t acc = 0;
        for (int el = 0; el < E_loc; el++) {
            expert_prefix[d * (E_loc + 1) + el] = acc;
            for (int s = 0; s < R; s++) acc += cnt[s * E + d * E_loc + el];
        }
        expert_prefix[d * (E_loc + 1) + E_loc] = acc;
    }
    for (int s = 0; s < R; s++) {
        for (int e = 0; e < E; e++) {
            int d = e / E_loc, el = e % E_loc;
            int32_t b = expert_prefix[d * (E_loc + 1) + el];
            for (int sp = 0; sp < s; sp++) b += cnt[sp * E + e];
            base[e] = b;
            run[e] = 0;
        }
        for (int t = 0; t < T; t++)
            for (int j = 0; j < k; j++) {
                int64_t i = ((int64_t)s * T + t) * k + j;
                int64_t e = topk_idx[i];
                if (e < 0 || e >= E) { expert_rows[i] = -1; continue; }
                expert_rows[i] = base[e] + run[e]++;
            }
    }
    free(cnt);
    free(run);
    free(base);
    return bad;
}

/*
 * Expert-major dispatch: every valid entry (s, t, j) with expert e on rank d writes the
 * token's row to recv_x[row_offset[d] + expert_rows[s][t][j]] (bf16 copy, or e4m3 with
 * per-128-channel scales quantised once per token as in oracle_quantize_row_mode), and
 * recv_src_idx[row] = t, recv_weights[row] = topk_weights[s][t][j] (one weight per row).
 * Returns the number of rows outside their region.
 */
EXPORT int64_t oracle_dispatch_expert_major(int R, int T, int H, int E, int k, int quantize,
                                            int scale_mode, float tensor_scale,
                                            const uint16_t* x, const int64_t* topk_idx,
                                            const float* topk_weights, const int32_t* expert_rows,
                                            const int64_t* row_offset, void* recv_x,
                                            void* recv_x_scales, int32_t* recv_src_idx,
                                            float* recv_weights)
{
    const int E_loc = E / R;
    const int G = H / 128;
    const size_t scale_elem = scale_mode == 2 ? 1 : 4;
    int64_t bad = 0;
    uint8_t* qrow = (uint8_t*)malloc((size_t)H + 1);
    float* srow = (float*)malloc(sizeof(float) * (size_t)(G + 1));
    uint8_t* brow = (uint8_t*)malloc((size_t)G + 1);
    for (int s = 0; s < R; s++)
        for (int t = 0; t < T; t++) {
            const int64_t tok = (int64_t)s * T + t;
            const uint16_t* xrow = x + tok * H;
            if (quantize) oracle_quantize_row_mode(xrow, H, scale_mode, tensor_scale, qrow, srow, brow);
            for (int j = 0; j < k; j++) {
                int64_t e = topk_idx[tok * k + j];
                int32_t r = expert_rows[tok * k + j];
                if (e < 0 || e >= E || r < 0) continue;
                int d = (int)(e / E_loc);
                int64_t row = row_offset[d] + r;
                if (row >= row_offset[d + 1]) { bad++; continue; }
                if (quantize) {
                    memcpy((uint8_t*)recv_x + (size_t)row * H, qrow, (size_t)H);
                    memcpy((uint8_t*)recv_x_scales + (size_t)row * G * scale_elem,
                           scale_mode == 2 ? (const void*)brow : (const void*)srow, scale_elem * (size_t)G);
                } else {
                    memcpy((uint16_t*)recv_x + (size_t)row * H, xrow, sizeof(uint16_t) * (size_t)H);
                }
                if (recv_src_idx) recv_src_idx[row] = t;
                if (recv_weights) recv_weights[row] = topk_weights[tok * k + j];
            }
        }
    free(qrow);
    free(srow);
    free(brow);
    return bad;
}

/*
 * Expert-major combine: out[s][t] = sum over valid j (ascending) of
 * c_j * y[row_offset[d] + expert_rows[s][t][j]], c_j = topk_weights[s][t][j] (weighted)
 * or 1 (sum); binary64 accumulation, one bf16 rounding. A token with no valid entry
 * gives +0.
 */
EXPORT void oracle_combine_expert_major(int R, int T, int H, int E, int k, int weighted,
                                        const uint16_t* y, const int64_t* row_offset,
                                        const int64_t* topk_idx, const float* topk_weights,
                                        const int32_t* expert_rows, uint16_t* out)
{
    const int E_loc = E / R;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(H + 1));
    for (int s = 0; s < R; s++)
        for (int t = 0; t < T; t++) {
            const int64_t tok = (int64_t)s * T + t;
            for (int h = 0; h < H; h++) acc[h] = 0.0;
            for (int j = 0; j < k; j++) {
                int64_t e = topk_idx[tok * k + j];
                int32_t r = expert_rows[tok * k + j];
                if (e < 0 || e >= E || r < 0) continue;
                int d = (int)(e / E_loc);
                int64_t row = row_offset[d] + r;
                if (row >= row_offset[d + 1]) continue;
                double c = weighted ? (double)topk_weights[tok * k + j] : 1.0;
                for (int h = 0; h < H; h++) acc[h] += c * (double)bf16_bits_to_float(y[(size_t)row * H + h]);
            }
            for (int h = 0; h < H; h++) out[(size_t)tok * H + h] = double_to_bf16_rne(acc[h]);
        }
    free(acc);
}
