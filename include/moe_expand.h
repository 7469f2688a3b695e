/*
 * moe_expand.h - C ABI of libmoe_expand.so, the expanded-layout MoE prefill
 * layer for NVIDIA GB300 (sm_103a).
 *
 * The layer (SGLang PR 37261, "feat(deepep_v2): expanded (do_expand=True)
 * prefill dispatch for DeepEP-V2", Modifications/Core and the
 * SGLANG_DEEPEP_V2_PREFILL_DO_EXPAND section; SGLang moe_runner/deep_gemm.py,
 * _run_contiguous_gemm) on one GPU, with no all-to-all:
 *
 *   moe_expand_layout   per-expert histogram, aligned prefix (psum), row
 *                       labels (m_indices), each pair's expanded row
 *   moe_expand_scatter  one fp8 row per (token, expert) pair, grouped by
 *                       expert, alignment gaps zeroed
 *   moe_grouped_ffn     FP8 block-scaled grouped gate_up GEMM, silu*mul +
 *                       per-128-group fp8 quant (top-k weight folded into the
 *                       fp32 scale), grouped down GEMM
 *   moe_combine         sum of each token's expert outputs back to [T, H] bf16
 *
 * Conventions for every call:
 *  - All pointers named d_* or documented as "device" point to device memory
 *    owned by the caller; the library allocates nothing and keeps no pointer
 *    after a call returns. Host-only helpers say so.
 *  - Calls are asynchronous on the given stream (NULL = legacy default
 *    stream), do no host synchronisation and never read a device value on
 *    the host: the valid-row count and the aligned total stay on the device
 *    (vLLM PR 54109, "PaddedStandard activation format", Motivation: reading
 *    the real/padding boundary on the host would break graph capture).
 *  - The return value reports host-detectable errors (bad arguments, a
 *    launch failure). Errors only the device can see (an expert id >= E in a
 *    valid row, more expanded rows than M_cap, a bounded wait that gave up)
 *    are written, first error wins, to the optional device word d_status
 *    (int32, caller zeroes it); the kernel then skips the offending work and
 *    returns instead of trapping.
 *  - Row-major fp32 scales are [rows, ld] with ld >= G; packed ue8m0 scales
 *    are int32 [ceil(G/4), ld] column-major with ld >= rows, four exponent
 *    bytes per word, group 4j in the low byte, unused bytes zero (the layout
 *    DeepGEMM's ue8m0 path reads; deep_gemm.py, pre_permute_deepep_v2_to_deep_gemm:
 *    "packed UE8M0 scales require zero padding lanes").
 *  - fp8 is OCP E4M3 stored as uint8; bf16 is stored as uint16.
 */
#ifndef MOE_EXPAND_H
#define MOE_EXPAND_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* the same type as cudaStream_t */

/* Return / status codes. */
#define MOE_OK                0
#define MOE_ERR_INVALID_ARG  -1  /* null pointer, bad shape or alignment */
#define MOE_ERR_UNSUPPORTED  -2  /* device is not sm_103 */
#define MOE_ERR_CUDA         -3  /* a CUDA call failed; see moe_last_error_string() */
#define MOE_ERR_WORKSPACE    -4  /* workspace missing or too small */
#define MOE_ERR_DEVICE_CHECK -5  /* device-detected: id >= E in a valid row, or total > M_cap */
#define MOE_ERR_TIMEOUT      -6  /* device-detected: a bounded wait gave up */

/* Scale layouts. */
#define MOE_SCALE_F32_ROWMAJOR          0
#define MOE_SCALE_UE8M0_PACKED_COLMAJOR 1

/* moe_grouped_ffn / moe_grouped_gemm / moe_act_quant flags. */
#define MOE_FOLD_WEIGHT_INTO_SCALE 1 /* fp32 path: store s*w as down_proj's input scale */
#define MOE_WEIGHT_OUTPUT_ROWS     2 /* ue8m0 path: multiply the down_proj output row by w */
#define MOE_GEMM_TILE_N128        16 /* tuning: use 128-column GEMM tiles even when N % 256 == 0 */
#define MOE_GEMM_PER_KBLOCK_PROMOTION 64 /* ue8m0 scales: promote per K block in registers instead of
                                            the tensor core's block scaling */
#define MOE_FFN_UNFUSED          128 /* moe_grouped_ffn: gate_up, act+quant and down as three launches */

/* Rows per grouped-GEMM tile; tile_prefix counts tiles of this height. */
#define MOE_BLOCK_M 128

/* Host. Upper bound on the expanded (aligned) row count over every routing
 * of T*K assignments to E experts (deep_gemm.py, _get_compact_all_tokens):
 * align * (min(A, E) + (A - min(A, E)) / align), A = T*K. Returns -1 on bad
 * arguments. Size M_cap with it. */
int64_t moe_expanded_capacity(int64_t T, int K, int E, int align);

/* Host. Bytes of device workspace moe_expand_layout needs for (T, K, E).
 * The workspace must be zero-filled once before its first use; every call
 * leaves it ready for the next call. Its first 256 bytes hold the
 * completion ticket and the cooperative launch's barrier words, at the same
 * place for every (T, K, E), so one workspace sized for the largest call
 * serves smaller ones too; then come per-(expert, 2048-pair chunk) counts
 * and offsets, rewritten by every call. Its size depends on T*K and E only;
 * unlike a workspace sized by the expanded capacity, it takes no M_cap
 * argument. */
size_t moe_workspace_size(int64_t T, int K, int E);

/*
 * Layout (SGLang PR 37261: fill_m_indices_from_psum; the review's
 * definition psum[i] = align(psum[i-1]) + count_i; pre_permute_deepep_v2_to_deep_gemm).
 *   topk_ids   device int32 [T, K]; -1 = no pair. Rows t >= *d_n_valid are
 *              never read.
 *   d_n_valid  device int32, rows [0, n_valid) are valid; NULL = all T.
 *   align      expert_alignment (> 0).
 *   M_cap      rows of the expanded buffers (m_indices length).
 * Outputs (device, written every call):
 *   psum       int32 [E]   inclusive aligned prefix: psum[e] = start[e] + count[e]
 *   start      int32 [E]   start[e] = align(psum[e-1]), start[0] = 0
 *   d_total    int32 [1]   align(psum[E-1]), a multiple of align
 *   m_indices  int32 [M_cap]  e on [start[e], align(psum[e])), -1 on [total, M_cap)
 *   src2dst    int32 [T, K]   expanded row of each valid pair, -1 otherwise;
 *                             pairs of one expert are in ascending (t, k) order
 *   tile_prefix int32 [E+1]   tile_prefix[e+1] - tile_prefix[e] =
 *                             ceil((align(psum[e]) - start[e]) / MOE_BLOCK_M)
 *   ws, ws_bytes  workspace of moe_workspace_size(T, K, E) bytes.
 * Launches: one block when T*K <= 2048. Otherwise, when a cooperative grid
 * (three 512-thread blocks per SM, fewer for very large E) holds one block
 * per 2048-pair chunk, one launch: the blocks rank their chunk's pairs,
 * publish their counts, meet at a grid-wide barrier, then each derives the
 * offsets from the whole count table and writes its chunk's rows. The
 * barrier wait is bounded; if it gives up the status word gets
 * MOE_ERR_TIMEOUT and the outputs are not valid. More chunks take two
 * launches (count and scan, then rank). All give the same outputs bit for
 * bit.
 * Device errors: MOE_ERR_DEVICE_CHECK for an id >= E in a valid row (that
 * pair is skipped) or total > M_cap (rows past M_cap are not written).
 */
int moe_expand_layout(const int32_t* topk_ids, int64_t T, int K, int E, int align,
                      const int32_t* d_n_valid, int64_t M_cap,
                      int32_t* psum, int32_t* start, int32_t* d_total,
                      int32_t* m_indices, int32_t* src2dst, int32_t* tile_prefix,
                      void* ws, size_t ws_bytes, int32_t* d_status, moe_stream_t stream);

/*
 * moe_expand_layout without a workspace argument. The pages have no
 * counterpart of this call; it exists for callers that cannot allocate
 * device memory when the layer runs - for example a serving engine that has
 * handed nearly all of HBM to its own pool up front, or a host loop that
 * must not call cudaMalloc on this path because cudaMalloc can synchronise
 * the device. Arguments and outputs are those of moe_expand_layout.
 *  - Scratch: a fixed 1 MiB array in the library's device image, held by
 *    every GPU that loads the library until the process exits. A call needs
 *    moe_workspace_size(T, K, E) bytes of it: 8*E bytes per chunk of 2048
 *    (token, expert) pairs, rounded up to 256, plus 256. So it holds at most
 *    floor((2^20 - 256) / (8*E)) chunks: 4095 chunks (8,386,560 pairs) at
 *    E = 32, 127 chunks (260,096 pairs) at E = 1024. Larger sizes are
 *    rejected with MOE_ERR_INVALID_ARG and a message, before any device work.
 *  - When all pairs fit one chunk (T*K <= 2048, a decode-sized batch) the
 *    call is the single launch moe_expand_layout also uses there; it touches
 *    no scratch, no lookup and no memset.
 *  - Otherwise the first call on a device looks up the array's device
 *    address (cudaGetSymbolAddress) with that device current, and again
 *    whenever the current CUDA context of the device has changed (after a
 *    device reset); make that first call before any stream capture.
 *  - Every call shares the one array and it keeps the last call's contents;
 *    the call clears the part that must start at zero (an asynchronous
 *    256-byte memset on the stream) and then launches what
 *    moe_expand_layout launches. Calls ordered on one stream may follow
 *    each other without a host wait. Calls that overlap on the GPU (different streams,
 *    no ordering between them) race on the array and give wrong results.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
int moe_expand_layout_noalloc(const int32_t* topk_ids, int64_t T, int K, int E, int align,
                              const int32_t* d_n_valid, int64_t M_cap,
                              int32_t* psum, int32_t* start, int32_t* d_total,
                              int32_t* m_indices, int32_t* src2dst, int32_t* tile_prefix,
                              int32_t* d_status, moe_stream_t stream);

/*
 * Layout fused into the expand-scatter (SGLang PR 37261: the layout kernels
 * and the expand copy of the do_expand=True dispatch). For two or more
 * 2048-pair chunks, when a cooperative grid of two 512-thread blocks per SM
 * holds one block per chunk: ONE launch that runs the layout as
 * moe_expand_layout does, meets at a second bounded grid-wide barrier, then
 * labels m_indices, zeroes the gaps and copies every valid token's row with
 * all its blocks. Otherwise (one chunk, or more chunks than that grid):
 * moe_expand_layout followed by moe_expand_scatter.
 * Arguments: those of moe_expand_layout (topk_ids .. tile_prefix, the same
 * workspace of moe_workspace_size bytes, zeroed before its first use) plus
 * those of moe_expand_scatter (topk_w, x, x_scale/scale_layout/ld_xs, H, xe,
 * xe_scale/ld_xes, row_w). Every output equals, bit for bit, what
 * moe_expand_layout followed by moe_expand_scatter write. Asynchronous on
 * `stream`; the workspace must not be shared with a call that can overlap
 * this one. Errors: as the two calls it replaces, plus MOE_ERR_TIMEOUT in the
 * status word if a grid-wide barrier gives up (outputs then not valid).
 */
int moe_expand_layout_scatter(const int32_t* topk_ids, const float* topk_w, const uint8_t* x,
                              const void* x_scale, int scale_layout, int64_t ld_xs, int64_t T,
                              int H, int K, int E, int align, const int32_t* d_n_valid,
                              int64_t M_cap, int32_t* psum, int32_t* start, int32_t* d_total,
                              int32_t* m_indices, int32_t* src2dst, int32_t* tile_prefix,
                              uint8_t* xe, void* xe_scale, int64_t ld_xes, float* row_w, void* ws,
                              size_t ws_bytes, int32_t* d_status, moe_stream_t stream);

/* Host. Bytes of the fixed scratch array moe_expand_layout_noalloc uses. */
size_t moe_expand_layout_noalloc_max_scratch(void);

/*
 * Expand-scatter (SGLang PR 37261, do_expand=True: per-(token, expert) rows
 * grouped by expert; the copy ep_scatter_2 made before; vLLM PR 54109:
 * alignment gaps are zeroed).
 *   x          device uint8 [T, H] fp8 rows (H % 128 == 0, H <= 16384)
 *   x_scale    device, scale_layout: fp32 [T, ld_xs] or packed ue8m0 [ceil(H/512), ld_xs]
 *   topk_w     device fp32 [T, K]
 *   src2dst, psum, start: from moe_expand_layout with the same align
 * Outputs (device): xe uint8 [M_cap, H], xe_scale in the same layout family
 * with leading dimension ld_xes, row_w fp32 [M_cap] (the pair's top-k
 * weight). Row src2dst[t,k] = token t's bytes, scales and weight; rows
 * [psum[e], align(psum[e])) are zero. Rows >= total are not written.
 */
int moe_expand_scatter(const uint8_t* x, const void* x_scale, int scale_layout, int64_t ld_xs,
                       const float* topk_w, const int32_t* src2dst,
                       const int32_t* psum, const int32_t* start, const int32_t* d_n_valid,
                       int64_t T, int H, int K, int E, int align, int64_t M_cap,
                       uint8_t* xe, void* xe_scale, int64_t ld_xes, float* row_w,
                       int32_t* d_status, moe_stream_t stream);

/*
 * One block-scaled FP8 grouped GEMM over the expanded rows (DeepGEMM's
 * grouped_gemm_nt_f8f8bf16_contig as _run_contiguous_gemm calls it):
 *   out[r, n] = bf16( sum_kb sA[r, kb] * sW[e, n/128, kb] * sum_{k in kb} A[r,k] W[e,n,k] )
 * for r in expert e's aligned segment, r < *d_total; other rows untouched.
 *   A        device uint8 [M_cap, Kd], K-major, 16-byte aligned
 *   A_scale  device, scale_layout, leading dimension ld_as
 *   W        device uint8 [E, N, Kd] K-major ("nt"); W_scale fp32 [E, N/128, Kd/128]
 *            (scale_layout F32) or uint8 ue8m0 bytes (scale_layout UE8M0)
 *   start, tile_prefix, d_total: from moe_expand_layout. The GEMM takes the
 *            segment starts and the per-expert 128-row tile prefix, not the
 *            per-row m_indices labels: a persistent CTA turns a linear tile
 *            id into (expert, m block) by a binary search over E+1 prefix
 *            entries kept in shared memory, and the tile count comes from
 *            the prefix's last entry, which a per-row label array cannot
 *            give without a scan. m_indices stays a layout output for
 *            callers whose GEMM reads per-row labels (DeepGEMM's contiguous
 *            layout); nothing in this library reads it.
 *   row_w    device fp32 [M_cap], read only with MOE_WEIGHT_OUTPUT_ROWS
 *   out      device bf16 [M_cap, N]
 * With MOE_WEIGHT_OUTPUT_ROWS the sum is multiplied by row_w[r] before the
 * bf16 rounding. With ue8m0 scales and N % 256 == 0 the scales are applied
 * by the tensor core (kind::mxf8f6f4 block scaling, one accumulator per
 * tile); otherwise each K block's partial sum is scaled and added in fp32
 * registers. Both equal the formula up to fp32 summation order.
 * Needs N % 128 == 0, Kd % 128 == 0, E <= 1024.
 */
int moe_grouped_gemm(const uint8_t* A, const void* A_scale, int scale_layout, int64_t ld_as,
                     const int32_t* start, const int32_t* tile_prefix, const int32_t* d_total,
                     const uint8_t* W, const void* W_scale, const float* row_w, int flags,
                     int E, int N, int Kd, int64_t M_cap, uint16_t* out,
                     int32_t* d_status, moe_stream_t stream);

/*
 * silu(g)*u and per-token-group fp8 quantisation (deep_gemm.py,
 * _run_contiguous_gemm: silu_and_mul then per_token_group_quant with group
 * 128; gate = columns [0, I), up = [I, 2I)). Per 128-group of h (h rounded to
 * bf16): amax = max(max|h|, 1e-10), s = amax/448, q = e4m3_rn_sat(h/s).
 * fp32 layout: stored scale s*row_w[r] with MOE_FOLD_WEIGHT_INTO_SCALE (the
 * fold of SGLang PR 37261), else s. ue8m0 layout: s rounded up to a power of
 * two (_cast_to_e8m0_with_rounding_up), stored as its exponent byte.
 *   gu       device bf16 [M_cap, 2I]; rows r < *d_total are processed
 *   di       device uint8 [M_cap, I]; di_scale in scale_layout with ld_ds
 */
int moe_act_quant(const uint16_t* gu, int I, const float* row_w, int flags, int scale_layout,
                  const int32_t* d_total, int64_t M_cap, uint8_t* di, void* di_scale,
                  int64_t ld_ds, int32_t* d_status, moe_stream_t stream);

/*
 * gate_up GEMM with silu(gate)*up and the fp8 quantiser of down_proj's input
 * in its epilogue: the result equals moe_grouped_gemm into a bf16 [M_cap, 2I]
 * buffer followed by moe_act_quant, bit for bit, without that buffer going
 * through memory (the fusion the pages' _situ_mul_quant_contig_kernel makes of
 * silu_and_mul and the group quant, here taken into the GEMM itself).
 *   A, A_scale, ld_as, start, tile_prefix, d_total: as moe_grouped_gemm
 *   W13      device uint8 [E, 2I, H]: gate rows [0, I), up rows [I, 2I)
 *   di       device uint8 [M_cap, I], 16-byte aligned; rows r < *d_total written
 *   di_scale packed ue8m0 int32 [ceil(I/512), ld_ds], ld_ds >= M_cap
 *   row_w    device fp32 [M_cap], read with MOE_FOLD_WEIGHT_INTO_SCALE (fp32
 *            scales only: the stored scale is s * row_w[r], as moe_act_quant)
 *   flags    MOE_FOLD_WEIGHT_INTO_SCALE, MOE_GEMM_PER_KBLOCK_PROMOTION
 * Both scale layouts: ue8m0 scales go to the tensor core's block scaling,
 * fp32 scales to the per-K-block promotion kernel; either way the epilogue
 * forms h = bf16(silu(g) u) per 128-column group and writes its codes and
 * scale. Needs I % 128 == 0, H % 128 == 0, E <= 1024.
 */
int moe_grouped_gemm_act_quant(const uint8_t* A, const void* A_scale, int scale_layout,
                               int64_t ld_as, const int32_t* start, const int32_t* tile_prefix,
                               const int32_t* d_total, const uint8_t* W13, const void* W13_scale,
                               const float* row_w, int flags, int E, int I, int H, int64_t M_cap,
                               uint8_t* di, void* di_scale, int64_t ld_ds, int32_t* d_status,
                               moe_stream_t stream);

/*
 * The expert FFN over the expanded rows: moe_grouped_gemm with W13 [E, 2I, H]
 * into gateup_ws bf16 [M_cap, 2I], moe_act_quant into down_in uint8
 * [M_cap, I] / down_in_scale (ld_dis), moe_grouped_gemm with W2 [E, H, I]
 * into down_out bf16 [M_cap, H].
 * flags: MOE_FOLD_WEIGHT_INTO_SCALE (fp32 scales) or MOE_WEIGHT_OUTPUT_ROWS
 * (ue8m0 scales; a power-of-two scale cannot absorb the weight, so the output
 * row is weighted instead), or 0 (unweighted; moe_combine may weight).
 * The first two steps run as one launch (moe_grouped_gemm_act_quant) and
 * gateup_ws is not touched (it may be NULL); MOE_FFN_UNFUSED keeps three
 * launches (gateup_ws required).
 */
int moe_grouped_ffn(const uint8_t* xe, const void* xe_scale, int64_t ld_xes, int scale_layout,
                    const int32_t* start, const int32_t* tile_prefix, const int32_t* d_total,
                    const uint8_t* w13, const void* s13, const uint8_t* w2, const void* s2,
                    const float* row_w, int flags, int E, int H, int I, int64_t M_cap,
                    uint16_t* gateup_ws, uint8_t* down_in, void* down_in_scale, int64_t ld_dis,
                    uint16_t* down_out, int32_t* d_status, moe_stream_t stream);

/*
 * Combine (the expand-mode combine's un-expand and reduction; ep_gather):
 *   y[t, :] = bf16( sum_{k: src2dst[t,k] >= 0} f32(down_out[src2dst[t,k], :]) * (row_w ? row_w[row] : 1) )
 * for t < *d_n_valid, summed in k order in fp32. A token with no pair gets
 * zeros; rows t >= n_valid are not written.
 *   down_out device bf16 [M_cap, H] (H % 8 == 0); y device bf16 [T, H].
 */
int moe_combine(const uint16_t* down_out, const int32_t* src2dst, const float* row_w,
                const int32_t* d_n_valid, int64_t T, int H, int K, uint16_t* y,
                moe_stream_t stream);

/*
 * Decode variant, before the GEMMs: expanded rows -> masked slab (SGLang PR
 * 37261: the deepep_v2 decode path's expand_to_masked_slab, feeding a masked
 * grouped GEMM with a fixed-height slab [E, max_m, H]). Expert e's first
 * masked_m[e] = min(count_e, max_m) expanded rows (count_e = psum[e] -
 * start[e]) go to slab rows e*max_m + j with their scale rows; slab rows
 * [masked_m[e], round_up(masked_m[e], 128)) below max_m are zeroed; other
 * slab rows are not touched. count_e > max_m drops the extra rows and sets
 * MOE_ERR_DEVICE_CHECK on d_status. Also writes the layout the grouped GEMMs
 * take for the slab: slab_start[e] = e*max_m, slab_tile_prefix [E+1] (128-row
 * tiles of masked_m), *slab_total = E*max_m; pass M_cap = E*max_m to them.
 *   xe, xe_scale (ld_xes), psum, start: from moe_expand_scatter / layout
 *   slab     device uint8 [E*max_m, H]; slab_scale fp32 [E*max_m, ld_ss] or
 *            packed ue8m0 int32 [ceil(H/512), ld_ss >= E*max_m]
 *   masked_m, slab_start device int32 [E]; slab_tile_prefix [E+1]; slab_total [1]
 */
int moe_expand_to_masked_slab(const uint8_t* xe, const void* xe_scale, int scale_layout,
                              int64_t ld_xes, const int32_t* psum, const int32_t* start, int E,
                              int H, int64_t max_m, uint8_t* slab, void* slab_scale, int64_t ld_ss,
                              int32_t* masked_m, int32_t* slab_start, int32_t* slab_tile_prefix,
                              int32_t* slab_total, int32_t* d_status, moe_stream_t stream);

/*
 * Decode variant, after the GEMMs: masked slab -> expanded rows (the decode
 * path's masked_slab_to_expand, which takes the top-k weights):
 *   out[start[e] + j] = bf16( f32(slab_out[e*max_m + j]) * (row_w ? row_w[start[e]+j] : 1) )
 * for j < min(count_e, max_m); every other row below *d_total is zeroed
 * (alignment gaps, dropped rows); rows >= *d_total are not written.
 *   slab_out device bf16 [E*max_m, H] (H % 8 == 0); out bf16 [M_cap, H]
 */
int moe_masked_slab_to_expand(const uint16_t* slab_out, int64_t max_m, const int32_t* psum,
                              const int32_t* start, const int32_t* d_total, const float* row_w,
                              int E, int H, int64_t M_cap, uint16_t* out, moe_stream_t stream);

/* Host. Diagnostics: when d_trace is not NULL, every later grouped-GEMM
 * launch (moe_grouped_gemm, moe_grouped_gemm_act_quant) writes 8 uint64
 * counters per CTA (grid = SM count) to d_trace: kernel cycles, producer
 * cycles waiting for a free stage, MMA cycles waiting for a free accumulator,
 * MMA cycles waiting for operand data, then (per-K-block promotion kernel)
 * one unused word, epilogue cycles in tile-end work, one unused word, or
 * (block-scaled kernel) MMA cycles waiting for
 * scales, epilogue wait, epilogue tile work; last, K blocks processed. NULL
 * turns it off. Not thread-safe with respect to concurrent launches on other
 * threads. */
int moe_gemm_set_trace(uint64_t* d_trace);

/* Diagnostics (no counterpart in the pages): runs the library's bounded
 * mbarrier waits on barriers nothing arrives at. Block 0: a single-thread
 * waiter gives up after limit_cycles (0 < limit <= 4e9; the kernels use
 * ~4e9), writes MOE_ERR_TIMEOUT to *d_status and raises its block's abort
 * flag; a second single-thread waiter and a warp in the warp-collective wait,
 * each with a 4x longer limit, leave on the flag. Block 1: a warp in the
 * warp-collective wait gives up on its own limit. d_out (device int64 [8]):
 * per waiter its result (single thread: 1 = phase completed, 0 = gave up;
 * warp: the ballot of lanes that saw completion) and the cycles it waited,
 * in that order. */
int moe_selftest_bounded_wait(int64_t limit_cycles, int32_t* d_status, int64_t* d_out,
                              moe_stream_t stream);

/* Host. Text of the last error raised on this thread (never NULL). */
const char* moe_last_error_string(void);

/* Host. 1 when `device` can run this library (compute capability 10.3). */
int moe_device_supported(int device);

#ifdef __cplusplus
}
#endif
#endif /* MOE_EXPAND_H */
