/*
 * Reference (oracle) implementation of the expanded-layout MoE prefill layer.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the package smoke entry and
 * the benchmark's CPU-baseline leg, never by the product path. Plain C11,
 * single-threaded, double precision wherever the method leaves the precision
 * open; fp32 exactly where the kernel's decision is taken in fp32 (the
 * quantiser's scale and the value it rounds), so that both sides decide each
 * fp8 code in the same precision. Built with -ffp-contract=off so that no
 * multiply-add is fused on either host architecture.
 *
 * Source pages and readings are listed in moe_oracle.h.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Codecs                                                                    */
/* ------------------------------------------------------------------------ */

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 is subnormal; the all-ones
 * exponent with all-ones mantissa is NaN; there is no infinity, so the
 * largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t code) {
    int sign = code >> 7;
    int ex = (code >> 3) & 0xF;
    int man = code & 0x7;
    double v;
    if (ex == 0xF && man == 0x7) return NAN;
    if (ex == 0)
        v = ldexp((double)man, -9);              /* (man/8) * 2^(1-7) */
    else
        v = ldexp((double)(8 + man), ex - 10);   /* (1 + man/8) * 2^(ex-7) */
    return sign ? -v : v;
}

/* Nearest representable multiple of the local quantum, ties to even. */
static double round_to_quantum(double a, int min_normal_exp, int mant_bits) {
    int e;
    double q;
    if (a == 0.0) return 0.0;
    frexp(a, &e);                       /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                             /* floor(log2(a)) */
    if (e < min_normal_exp) e = min_normal_exp;
    q = ldexp(1.0, e - mant_bits);
    return rint(a / q) * q;             /* rint: round half to even */
}

uint8_t orc_e4m3_encode(float vf) {
    double v = (double)vf;
    double a, r;
    uint8_t code;
    int neg = signbit(v) ? 1 : 0;
    if (isnan(v)) return neg ? 0xFF : 0x7F;
    a = fabs(v);
    r = round_to_quantum(a, -6, 3);     /* normals from 2^-6, 3 mantissa bits */
    if (r > 448.0) r = 448.0;           /* saturate to the largest finite value */
    /* The code whose value is r. */
    for (code = 0; code < 0x7F; ++code)
        if (orc_e4m3_decode(code) == r) break;
    return (uint8_t)(neg ? (code | 0x80) : code);
}

/* bfloat16: the upper half of an IEEE binary32; 8 exponent bits, 7 stored
 * mantissa bits, normals down to 2^-126, subnormal quantum 2^-133. */
uint16_t orc_bf16_encode(double v) {
    float f;
    uint32_t bits;
    double a, r;
    int neg = signbit(v) ? 1 : 0;
    if (isnan(v)) return 0x7FC0;
    a = fabs(v);
    r = round_to_quantum(a, -126, 7);
    if (r >= ldexp(1.0, 128)) {
        bits = 0x7F800000u;              /* rounds past the largest finite: inf */
    } else {
        f = (float)r;                   /* exact: r is a bf16 value */
        memcpy(&bits, &f, 4);
    }
    return (uint16_t)((bits >> 16) | (neg ? 0x8000u : 0u));
}

double orc_bf16_decode(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* fp32 scale -> ue8m0 exponent byte, as _cast_to_e8m0_with_rounding_up in
 * deep_gemm.py defines it: take the biased exponent field; add one when the
 * mantissa is non-zero, unless the exponent is already 0xFE, or the value is
 * subnormal with a mantissa of at most 0x400000. */
uint8_t orc_ue8m0_encode(float s) {
    uint32_t bits;
    uint32_t ex, man;
    int round_up;
    memcpy(&bits, &s, 4);
    ex = (bits >> 23) & 0xFFu;
    man = bits & 0x7FFFFFu;
    round_up = (man > 0) && (ex != 0xFE) && !(ex == 0 && man <= 0x400000u);
    if (round_up) ex += 1;
    return (uint8_t)ex;
}

float orc_ue8m0_decode(uint8_t byte) {
    return (float)ldexp(1.0, (int)byte - 127);
}

void orc_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}
void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}
void orc_bf16_encode_array(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_encode(v[i]);
}
void orc_ue8m0_encode_array(const float* s, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_ue8m0_encode(s[i]);
}

/* ------------------------------------------------------------------------ */
/* Capacity: _get_compact_all_tokens in deep_gemm.py. Each non-empty expert  */
/* can waste at most align-1 padding rows, so the padded total over every    */
/* routing of A assignments is bounded by align*(ne + (A-ne)/align) with ne  */
/* = min(A, E).                                                               */
/* ------------------------------------------------------------------------ */
int64_t orc_expanded_capacity(int64_t A, int64_t E, int64_t align) {
    int64_t ne = A < E ? A : E;
    if (A < 0 || E <= 0 || align <= 0) return -1;
    return align * (ne + (A - ne) / align);
}

static int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

/* ------------------------------------------------------------------------ */
/* Layout                                                                    */
/*                                                                           */
/* The per-expert prefix follows the corrected definition in the review of  */
/* SGLang PR 37261: psum[e] = align(psum[e-1]) + count_e, inclusive, with    */
/* only the earlier experts aligned; expert e's rows start at                */
/* align(psum[e-1]) and its aligned segment ends at align(psum[e]); the      */
/* buffer's rows past align(psum[E-1]) keep the label -1 so the grouped GEMM */
/* skips them (pre_permute_deepep_v2_to_deep_gemm fills m_indices with -1     */
/* and labels only the aligned segments). Pairs count only for rows below    */
/* the valid-row prefix, and a -1 id is no pair (the PaddedStandard contract */
/* in vLLM PR 54109). Inside a segment, pairs are placed in ascending        */
/* (token, k) order: the pages leave this order open.                        */
/* ------------------------------------------------------------------------ */
int orc_layout(const int32_t* topk_ids, int64_t T, int K, int E, int align,
               int64_t n_valid, int64_t M_cap, int block_m,
               int32_t* psum, int32_t* start, int32_t* total,
               int32_t* m_indices, int32_t* src2dst, int32_t* tile_prefix) {
    int rc = ORC_OK;
    int64_t* count;
    int64_t* next;
    int64_t prev, tot;
    if (!topk_ids || !psum || !start || !total || !m_indices || !src2dst || !tile_prefix)
        return ORC_ERR_ARG;
    if (T < 0 || K <= 0 || E <= 0 || align <= 0 || block_m <= 0 || n_valid < 0 ||
        n_valid > T || M_cap < 0)
        return ORC_ERR_ARG;
    count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    next = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    if (!count || !next) { free(count); free(next); return ORC_ERR_ARG; }

    /* Histogram of the valid (token, expert) pairs. */
    for (int64_t t = 0; t < n_valid; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t id = topk_ids[t * K + k];
            if (id < 0) continue;
            if (id >= E) { rc = ORC_ERR_BAD_ID; continue; }
            count[id] += 1;
        }

    /* Aligned prefix. */
    prev = 0;
    for (int e = 0; e < E; ++e) {
        start[e] = (int32_t)align_up(prev, align);
        psum[e] = (int32_t)(start[e] + count[e]);
        prev = psum[e];
    }
    tot = align_up(prev, align);
    *total = (int32_t)tot;

    /* Per-expert 128-row tile prefix (tiles of the aligned segments). */
    tile_prefix[0] = 0;
    for (int e = 0; e < E; ++e) {
        int64_t seg = align_up(psum[e], align) - start[e];
        tile_prefix[e + 1] = (int32_t)(tile_prefix[e] + (seg + block_m - 1) / block_m);
    }

    if (tot > M_cap) {
        free(count); free(next);
        return ORC_ERR_CAPACITY;
    }

    /* Row labels. */
    for (int e = 0; e < E; ++e)
        for (int64_t r = start[e]; r < align_up(psum[e], align); ++r) m_indices[r] = e;
    for (int64_t r = tot; r < M_cap; ++r) m_indices[r] = -1;

    /* Destination row of each pair: a counting sort, stable in (t, k). */
    for (int e = 0; e < E; ++e) next[e] = start[e];
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t id = topk_ids[t * K + k];
            if (t >= n_valid || id < 0 || id >= E) {
                src2dst[t * K + k] = -1;
                continue;
            }
            src2dst[t * K + k] = (int32_t)next[id];
            next[id] += 1;
        }
    free(count);
    free(next);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Expand-scatter: one row per valid (token, expert) pair, grouped by expert */
/* ("per-(token, expert) rows grouped by expert", the do_expand=True section */
/* of SGLang PR 37261). The pair's row gets the token's fp8 bytes, its scale */
/* row, and its top-k weight. The alignment gaps [psum[e], align(psum[e]))   */
/* are zeroed: bytes, scales and weight ("those gaps are zeroed", vLLM PR    */
/* 54109 Motivation; packed ue8m0 scales need zero lanes, deep_gemm.py).     */
/* ------------------------------------------------------------------------ */
int orc_scatter(const uint8_t* x, const void* x_scale, int scale_layout, int64_t ld_xs,
                const float* topk_w, const int32_t* src2dst,
                const int32_t* psum, const int32_t* start, int64_t n_valid,
                int64_t T, int H, int K, int E, int align,
                uint8_t* xe, void* xe_scale, int64_t ld_xes, float* row_w) {
    int G = H / 128;
    int W = (G + 3) / 4;
    (void)start;
    if (!x || !x_scale || !topk_w || !src2dst || !psum || !xe || !xe_scale || !row_w)
        return ORC_ERR_ARG;
    if (H % 128 != 0 || n_valid > T || align <= 0) return ORC_ERR_ARG;
    for (int64_t t = 0; t < n_valid; ++t)
        for (int k = 0; k < K; ++k) {
            int64_t r = src2dst[t * K + k];
            if (r < 0) continue;
            memcpy(xe + r * H, x + t * H, (size_t)H);
            if (scale_layout == ORC_SCALE_F32) {
                const float* s = (const float*)x_scale;
                float* d = (float*)xe_scale;
                for (int g = 0; g < G; ++g) d[r * ld_xes + g] = s[t * ld_xs + g];
            } else {
                const int32_t* s = (const int32_t*)x_scale;
                int32_t* d = (int32_t*)xe_scale;
                for (int j = 0; j < W; ++j) d[j * ld_xes + r] = s[j * ld_xs + t];
            }
            row_w[r] = topk_w[t * K + k];
        }
    for (int e = 0; e < E; ++e)
        for (int64_t r = psum[e]; r < align_up(psum[e], align); ++r) {
            memset(xe + r * H, 0, (size_t)H);
            if (scale_layout == ORC_SCALE_F32) {
                float* d = (float*)xe_scale;
                for (int g = 0; g < G; ++g) d[r * ld_xes + g] = 0.0f;
            } else {
                int32_t* d = (int32_t*)xe_scale;
                for (int j = 0; j < W; ++j) d[j * ld_xes + r] = 0;
            }
            row_w[r] = 0.0f;
        }
    return ORC_OK;
}

/* Scale of 128-group g of row `row` in either layout, as a real number. */
static double act_scale(const void* s, int layout, int64_t ld, int64_t row, int g) {
    if (layout == ORC_SCALE_F32) return (double)((const float*)s)[row * ld + g];
    {
        uint32_t word = (uint32_t)((const int32_t*)s)[(int64_t)(g / 4) * ld + row];
        uint8_t byte = (uint8_t)((word >> (8 * (g % 4))) & 0xFFu);
        return (double)orc_ue8m0_decode(byte);
    }
}

/* Scale of the 128x128 weight block (nb, kb) of expert e. */
static double weight_scale(const void* s, int layout, int e, int NB, int KB, int nb, int kb) {
    int64_t i = ((int64_t)e * NB + nb) * KB + kb;
    if (layout == ORC_SCALE_F32) return (double)((const float*)s)[i];
    return (double)orc_ue8m0_decode(((const uint8_t*)s)[i]);
}

/* ------------------------------------------------------------------------ */
/* Block-scaled grouped GEMM (grouped_gemm_nt_f8f8bf16_contig in            */
/* _run_contiguous_gemm): row r of the expanded activations times expert    */
/* m_indices[r]'s weight, transposed ("nt"), bf16 out. Dequantisation is     */
/* value = code * scale; activations carry one scale per 1x128 group and    */
/* weights one per 128x128 block, so                                         */
/*   out[r, n] = sum_kb s_a[r, kb] * s_w[e, n/128, kb]                        */
/*               * sum_{k in block kb} dec(a[r, k]) * dec(w[e, n, k]).        */
/* The inner sum of 128 products of fp8 values is exact in double (each     */
/* product has at most 8 significant bits and the sum spans under 45 bits). */
/* ------------------------------------------------------------------------ */
int orc_gemm_rows(const uint8_t* A, int64_t lda, const void* A_scale, int scale_layout,
                  int64_t ld_as, const int64_t* rows, const int32_t* experts, int64_t n,
                  const uint8_t* W, const void* W_scale, int E, int N, int Kd,
                  uint16_t* out, double* out_f64) {
    int KB = Kd / 128, NB = N / 128;
    double* a = NULL;
    double lut[256];
    if (!A || !A_scale || !rows || !experts || !W || !W_scale || !out) return ORC_ERR_ARG;
    if (Kd % 128 != 0 || N % 128 != 0) return ORC_ERR_ARG;
    for (int c = 0; c < 256; ++c) lut[c] = orc_e4m3_decode((uint8_t)c);
    a = (double*)malloc(sizeof(double) * (size_t)Kd);
    if (!a) return ORC_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) {
        int64_t r = rows[i];
        int e = experts[i];
        if (e < 0 || e >= E) {
            for (int c = 0; c < N; ++c) {
                out[i * N + c] = 0;
                if (out_f64) out_f64[i * N + c] = 0.0;
            }
            continue;
        }
        for (int k = 0; k < Kd; ++k) a[k] = lut[A[r * lda + k]];
        for (int c = 0; c < N; ++c) {
            const uint8_t* w = W + ((int64_t)e * N + c) * Kd;
            double acc = 0.0;
            for (int kb = 0; kb < KB; ++kb) {
                double part = 0.0;
                double sa = act_scale(A_scale, scale_layout, ld_as, r, kb);
                double sw = weight_scale(W_scale, scale_layout, e, NB, KB, c / 128, kb);
                for (int k = kb * 128; k < kb * 128 + 128; ++k) part += a[k] * lut[w[k]];
                acc += (sa * sw) * part;
            }
            out[i * N + c] = orc_bf16_encode(acc);
            if (out_f64) out_f64[i * N + c] = acc;
        }
    }
    free(a);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* silu(g)*u, then per-token-group fp8 quantisation of down_proj's input    */
/* (_run_contiguous_gemm's default branch: silu_and_mul into a bf16 tensor, */
/* then per-token-group quant with group 128). Gate is the first I columns, */
/* up the last I. Per group: amax = max(max|h|, 1e-10), stored scale         */
/* s = amax/448, codes h * (448/amax) rounded to e4m3 (the quantiser formula */
/* of _situ_mul_quant_contig_kernel). With fp32 scales the row's top-k weight */
/* is folded into the stored scale, s*w (SGLang PR 37261, Modifications /    */
/* Core: dequant is q*scale and down_proj is linear, so the per-row factor  */
/* moves into the scale). With ue8m0 scales s is rounded up to a power of   */
/* two and stored as its exponent byte; the weight is applied to the output */
/* rows instead, because a power-of-two scale cannot absorb it.             */
/* ------------------------------------------------------------------------ */
int orc_act_quant_rows(const uint16_t* gu, int64_t n, int I, const float* row_w,
                       int scale_layout, uint8_t* di, void* di_scale, int64_t ld_ds) {
    int G = I / 128;
    float* h;
    if (!gu || !di || !di_scale || I % 128 != 0) return ORC_ERR_ARG;
    h = (float*)malloc(sizeof(float) * (size_t)I);
    if (!h) return ORC_ERR_ARG;
    if (scale_layout == ORC_SCALE_UE8M0) {
        int32_t* d = (int32_t*)di_scale;
        for (int64_t i = 0; i < n; ++i)
            for (int j = 0; j < (G + 3) / 4; ++j) d[j * ld_ds + i] = 0;
    }
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t* row = gu + i * 2 * (int64_t)I;
        for (int j = 0; j < I; ++j) {
            double g = orc_bf16_decode(row[j]);
            double u = orc_bf16_decode(row[I + j]);
            double silu = g / (1.0 + exp(-g));
            h[j] = (float)orc_bf16_decode(orc_bf16_encode(silu * u));
        }
        for (int gi = 0; gi < G; ++gi) {
            float amax = 0.0f;
            float s;
            for (int j = gi * 128; j < gi * 128 + 128; ++j) {
                float m = fabsf(h[j]);
                if (m > amax) amax = m;
            }
            if (amax < 1e-10f) amax = 1e-10f;
            s = amax / 448.0f;
            if (scale_layout == ORC_SCALE_F32) {
                float w = row_w ? row_w[i] : 1.0f;
                float stored = s * w;
                float inv = 448.0f / amax;      /* codes are h * (448 / amax) */
                for (int j = gi * 128; j < gi * 128 + 128; ++j) {
                    float v = h[j] * inv;
                    di[i * I + j] = orc_e4m3_encode(v);
                }
                ((float*)di_scale)[i * ld_ds + gi] = stored;
            } else {
                uint8_t b = orc_ue8m0_encode(s);
                float sd = orc_ue8m0_decode(b);
                int32_t* d = (int32_t*)di_scale;
                for (int j = gi * 128; j < gi * 128 + 128; ++j) {
                    float v = h[j] / sd;
                    di[i * I + j] = orc_e4m3_encode(v);
                }
                d[(int64_t)(gi / 4) * ld_ds + i] =
                    (int32_t)((uint32_t)d[(int64_t)(gi / 4) * ld_ds + i] |
                              ((uint32_t)b << (8 * (gi % 4))));
            }
        }
    }
    free(h);
    return ORC_OK;
}

/* ue8m0 path: down_output rows times their top-k weight before combine
 * (SGLang PR 37261, Modifications/Core: "weights down_output with
 * scale_expanded_rows_"). One rounding to bf16 of the fp32-weighted value. */
int orc_weight_rows(uint16_t* down, int64_t n, int H, const float* row_w) {
    if (!down || !row_w) return ORC_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        for (int c = 0; c < H; ++c)
            down[i * H + c] = orc_bf16_encode(orc_bf16_decode(down[i * H + c]) * (double)row_w[i]);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Combine: y[t] = sum over the token's pairs of its expert-output row      */
/* (ep_gather / the expand-mode combine's un-expand and reduction). A pair  */
/* with src2dst = -1 adds nothing; a token with no pair gives zeros; rows   */
/* t >= n_valid are neither read nor written (vLLM PR 54109: inactive rows  */
/* are skipped or safely discarded). Optional per-row weights for callers   */
/* that did not fold them earlier.                                          */
/* ------------------------------------------------------------------------ */
int orc_combine(const uint16_t* down, const int32_t* src2dst, const float* row_w,
                int64_t n_valid, int64_t T, int H, int K, uint16_t* y) {
    double* acc;
    if (!down || !src2dst || !y || n_valid > T) return ORC_ERR_ARG;
    acc = (double*)malloc(sizeof(double) * (size_t)H);
    if (!acc) return ORC_ERR_ARG;
    for (int64_t t = 0; t < n_valid; ++t) {
        for (int c = 0; c < H; ++c) acc[c] = 0.0;
        for (int k = 0; k < K; ++k) {
            int64_t r = src2dst[t * K + k];
            double w;
            if (r < 0) continue;
            w = row_w ? (double)row_w[r] : 1.0;
            for (int c = 0; c < H; ++c) acc[c] += orc_bf16_decode(down[r * H + c]) * w;
        }
        for (int c = 0; c < H; ++c) y[t * H + c] = orc_bf16_encode(acc[c]);
    }
    free(acc);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* One token through the layer with no expansion at all: for each of its    */
/* top-k experts, gate_up GEMM, activation + quantisation (weight folded or */
/* not, as above), down GEMM (and, on the ue8m0 path, the output weighting), */
/* then the sum over k in k order. Rows are independent, so this must equal */
/* the expanded path bit for bit.                                            */
/* ------------------------------------------------------------------------ */
int orc_token_forward(const uint8_t* x, const void* x_scale, int scale_layout, int64_t ld_xs,
                      int64_t t, const int32_t* ids, const float* w, int K,
                      const uint8_t* W13, const void* S13, const uint8_t* W2, const void* S2,
                      int E, int H, int I, uint16_t* y_row) {
    int GI = I / 128;
    uint16_t* gu = (uint16_t*)malloc(sizeof(uint16_t) * 2 * (size_t)I);
    uint8_t* di = (uint8_t*)malloc((size_t)I);
    float di_sf[64];
    int32_t di_su[16];
    uint16_t* down = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
    double* acc = (double*)calloc((size_t)H, sizeof(double));
    int rc = ORC_OK;
    if (!gu || !di || !down || !acc || GI > 64) { rc = ORC_ERR_ARG; goto done; }
    for (int k = 0; k < K; ++k) {
        int32_t e = ids[k];
        int64_t row = t, zero = 0;
        if (e < 0 || e >= E) continue;
        rc = orc_gemm_rows(x, H, x_scale, scale_layout, ld_xs, &row, &e, 1,
                           W13, S13, E, 2 * I, H, gu, NULL);
        if (rc) goto done;
        if (scale_layout == ORC_SCALE_F32) {
            rc = orc_act_quant_rows(gu, 1, I, &w[k], ORC_SCALE_F32, di, di_sf, GI);
            if (rc) goto done;
            rc = orc_gemm_rows(di, I, di_sf, ORC_SCALE_F32, GI, &zero, &e, 1,
                               W2, S2, E, H, I, down, NULL);
        } else {
            rc = orc_act_quant_rows(gu, 1, I, NULL, ORC_SCALE_UE8M0, di, di_su, 1);
            if (rc) goto done;
            rc = orc_gemm_rows(di, I, di_su, ORC_SCALE_UE8M0, 1, &zero, &e, 1,
                               W2, S2, E, H, I, down, NULL);
            if (rc) goto done;
            rc = orc_weight_rows(down, 1, H, &w[k]);
        }
        if (rc) goto done;
        for (int c = 0; c < H; ++c) acc[c] += orc_bf16_decode(down[c]);
    }
    for (int c = 0; c < H; ++c) y_row[c] = orc_bf16_encode(acc[c]);
done:
    free(gu); free(di); free(down); free(acc);
    return rc;
}
