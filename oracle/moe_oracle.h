/*
 * Reference (oracle) implementation of the expanded-layout MoE prefill layer.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded CPU
 * restatement of what the layer computes, written from the method's
 * description and used to check the CUDA library. Only the test suite, the
 * package's smoke entry and the benchmark's CPU-baseline leg may load it; the
 * product path never calls it. It shares no code, header, table or constant
 * with the CUDA library.
 *
 * Sources (page title, then the part of it followed):
 *   [SGL-37261] SGLang PR 37261, "feat(deepep_v2): expanded (do_expand=True)
 *               prefill dispatch for DeepEP-V2": Modifications/Core, the
 *               SGLANG_DEEPEP_V2_PREFILL_DO_EXPAND section, and the review
 *               thread's correction of the psum definition.
 *   [VLLM-54109] vLLM PR 54109, "PaddedStandard activation format":
 *               Motivation and Design (the padded-row contract).
 *   [DG-RUNNER] SGLang moe_runner/deep_gemm.py: _run_contiguous_gemm,
 *               _cast_to_e8m0_with_rounding_up, _get_compact_all_tokens,
 *               pre_permute_deepep_v2_to_deep_gemm,
 *               post_permute_deep_gemm_to_deepep_v2, _situ_mul_quant_contig_kernel
 *               (its quantisation formula).
 *
 * Parity unpinned (readings, covered by tolerance rather than by a pin):
 *   - order of pairs inside one expert's segment (ascending token, then k);
 *   - codes as h*(448/amax) (the pages' formula) rather than h/s;
 *   - the bf16 rounding of silu(g)*u before quantisation;
 *   - the ue8m0 output weighting in fp32 with one bf16 rounding.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Scale layouts (the oracle's own numbering). */
#define ORC_SCALE_F32   0   /* fp32 [rows, ld] row-major, one value per 128-group */
#define ORC_SCALE_UE8M0 1   /* int32 [ceil(G/4), ld] column-major, 4 exponent bytes per word */

/* Return codes. */
#define ORC_OK            0
#define ORC_ERR_ARG      -1
#define ORC_ERR_CAPACITY -2  /* aligned total exceeds the buffer capacity */
#define ORC_ERR_BAD_ID   -3  /* an id >= E in a valid row (the pair is skipped) */

/* ---- codecs ---------------------------------------------------------- */
double   orc_e4m3_decode(uint8_t code);
uint8_t  orc_e4m3_encode(float v);             /* round-to-nearest-even, saturating */
uint16_t orc_bf16_encode(double v);            /* round-to-nearest-even */
double   orc_bf16_decode(uint16_t bits);
uint8_t  orc_ue8m0_encode(float s);            /* exponent byte, rounded up */
float    orc_ue8m0_decode(uint8_t byte);       /* 2^(byte-127) */

void orc_e4m3_decode_array(const uint8_t* c, int64_t n, double* out);
void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out);
void orc_bf16_encode_array(const double* v, int64_t n, uint16_t* out);
void orc_ue8m0_encode_array(const float* s, int64_t n, uint8_t* out);

/* ---- host capacity bound -------------------------------------------- */
int64_t orc_expanded_capacity(int64_t num_assignments, int64_t E, int64_t align);

/* ---- layout ----------------------------------------------------------- */
int orc_layout(const int32_t* topk_ids, int64_t T, int K, int E, int align,
               int64_t n_valid, int64_t M_cap, int block_m,
               int32_t* psum, int32_t* start, int32_t* total,
               int32_t* m_indices, int32_t* src2dst, int32_t* tile_prefix);

/* ---- expand-scatter ---------------------------------------------------- */
int orc_scatter(const uint8_t* x, const void* x_scale, int scale_layout, int64_t ld_xs,
                const float* topk_w, const int32_t* src2dst,
                const int32_t* psum, const int32_t* start, int64_t n_valid,
                int64_t T, int H, int K, int E, int align,
                uint8_t* xe, void* xe_scale, int64_t ld_xes, float* row_w);

/* ---- block-scaled grouped GEMM on a list of rows ------------------------ */
int orc_gemm_rows(const uint8_t* A, int64_t lda, const void* A_scale, int scale_layout,
                  int64_t ld_as, const int64_t* rows, const int32_t* experts, int64_t n,
                  const uint8_t* W, const void* W_scale, int E, int N, int Kd,
                  uint16_t* out, double* out_f64);

/* ---- silu(g)*u + per-128-group fp8 quantisation (+ weight fold) -------- */
int orc_act_quant_rows(const uint16_t* gu, int64_t n, int I, const float* row_w,
                       int scale_layout, uint8_t* di, void* di_scale, int64_t ld_ds);

/* ---- ue8m0 path: weight expanded output rows --------------------------- */
int orc_weight_rows(uint16_t* down, int64_t n, int H, const float* row_w);

/* ---- combine ----------------------------------------------------------- */
int orc_combine(const uint16_t* down, const int32_t* src2dst, const float* row_w,
                int64_t n_valid, int64_t T, int H, int K, uint16_t* y);

/* ---- one token through the layer, without any expansion ---------------- */
int orc_token_forward(const uint8_t* x, const void* x_scale, int scale_layout, int64_t ld_xs,
                      int64_t t, const int32_t* ids, const float* w, int K,
                      const uint8_t* W13, const void* S13, const uint8_t* W2, const void* S2,
                      int E, int H, int I, uint16_t* y_row);

#ifdef __cplusplus
}
#endif
#endif
