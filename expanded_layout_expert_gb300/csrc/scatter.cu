// moe_expand_scatter: one fp8 row per valid (token, expert) pair, grouped by
// expert (SGLang PR 37261, do_expand=True: "per-(token, expert) rows grouped
// by expert", the work ep_scatter_2's full-hidden copy did), with the pair's
// scale row and top-k weight; the alignment gaps of every expert segment are
// zeroed (vLLM PR 54109, Motivation: "those gaps are zeroed").
//
// Each token's row is read from HBM once and written to its K destination
// rows with 16-byte vector stores; a persistent grid walks the valid tokens
// (the valid-row count is read on the device). Gap rows are zeroed by a
// separate set of blocks placed first in the grid so they never form a tail.
#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

constexpr int kPadRowsPerBlock = 8;
constexpr int kMaxK = 32;

__global__ void scatter_kernel(const uint4* __restrict__ x, const void* __restrict__ x_scale,
                               int ue8m0, int64_t ld_xs, const float* __restrict__ topk_w,
                               const int32_t* __restrict__ src2dst, const int32_t* __restrict__ psum,
                               const int32_t* __restrict__ d_n_valid, int64_t T, int H, int K, int E,
                               int align, int64_t M_cap, uint4* __restrict__ xe,
                               void* __restrict__ xe_scale, int64_t ld_xes,
                               float* __restrict__ row_w, int pad_blocks_per_expert,
                               int token_blocks, int32_t* __restrict__ status) {
  const int tid = threadIdx.x;
  const int nvec = H / 16;
  const int G = H / 128;
  const int W = (G + 3) / 4;
  const int pad_blocks = E * pad_blocks_per_expert;

  if (static_cast<int>(blockIdx.x) < pad_blocks) {
    const int e = blockIdx.x / pad_blocks_per_expert;
    const int sub = blockIdx.x % pad_blocks_per_expert;
    const int64_t seg_end = align_up(psum[e], align);
    const int64_t r0 = static_cast<int64_t>(psum[e]) + static_cast<int64_t>(sub) * kPadRowsPerBlock;
    int64_t r1 = r0 + kPadRowsPerBlock;
    if (r1 > seg_end) r1 = seg_end;
    if (r1 > M_cap) r1 = M_cap;
    for (int64_t r = r0; r < r1; ++r) {
      for (int v = tid; v < nvec; v += blockDim.x) xe[r * nvec + v] = make_uint4(0, 0, 0, 0);
      if (!ue8m0) {
        for (int g = tid; g < G; g += blockDim.x) static_cast<float*>(xe_scale)[r * ld_xes + g] = 0.0f;
      } else {
        for (int j = tid; j < W; j += blockDim.x) static_cast<int32_t*>(xe_scale)[j * ld_xes + r] = 0;
      }
      if (tid == 0) row_w[r] = 0.0f;
    }
    return;
  }

  __shared__ int s_dst[kMaxK];
  __shared__ float s_w[kMaxK];
  int64_t nv = T;
  if (d_n_valid != nullptr) {
    nv = *d_n_valid;
    nv = nv < 0 ? 0 : (nv > T ? T : nv);
  }
  for (int64_t t = blockIdx.x - pad_blocks; t < nv; t += token_blocks) {
    __syncthreads();
    if (tid < K) {
      int r = src2dst[t * K + tid];
      if (r >= M_cap) {
        set_status(status, MOE_ERR_DEVICE_CHECK);
        r = -1;
      }
      s_dst[tid] = r;
      s_w[tid] = topk_w[t * K + tid];
    }
    __syncthreads();
    for (int v = tid; v < nvec; v += blockDim.x) {
      const uint4 val = __ldcs(x + t * nvec + v);
      for (int k = 0; k < K; ++k) {
        const int r = s_dst[k];
        if (r >= 0) xe[static_cast<int64_t>(r) * nvec + v] = val;
      }
    }
    if (!ue8m0) {
      const float* xs = static_cast<const float*>(x_scale);
      for (int g = tid; g < G; g += blockDim.x) {
        const float sv = xs[t * ld_xs + g];
        for (int k = 0; k < K; ++k) {
          const int r = s_dst[k];
          if (r >= 0) static_cast<float*>(xe_scale)[static_cast<int64_t>(r) * ld_xes + g] = sv;
        }
      }
    } else {
      const int32_t* xs = static_cast<const int32_t*>(x_scale);
      for (int j = tid; j < W; j += blockDim.x) {
        const int32_t wv = xs[j * ld_xs + t];
        for (int k = 0; k < K; ++k) {
          const int r = s_dst[k];
          if (r >= 0) static_cast<int32_t*>(xe_scale)[j * ld_xes + r] = wv;
        }
      }
    }
    if (tid < K && s_dst[tid] >= 0) row_w[s_dst[tid]] = s_w[tid];
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_expand_scatter(const uint8_t* x, const void* x_scale, int scale_layout,
                                  int64_t ld_xs, const float* topk_w, const int32_t* src2dst,
                                  const int32_t* psum, const int32_t* start,
                                  const int32_t* d_n_valid, int64_t T, int H, int K, int E,
                                  int align, int64_t M_cap, uint8_t* xe, void* xe_scale,
                                  int64_t ld_xes, float* row_w, int32_t* d_status,
                                  moe_stream_t stream) {
  (void)start;
  MOE_REQUIRE(psum && xe && xe_scale && row_w, "moe_expand_scatter: null output");
  MOE_REQUIRE(T == 0 || (x && x_scale && topk_w && src2dst), "moe_expand_scatter: null input");
  MOE_REQUIRE(T >= 0 && K > 0 && K <= moe::kMaxK && E > 0 && align > 0 && M_cap >= 0,
              "moe_expand_scatter: bad sizes");
  MOE_REQUIRE(H > 0 && H % 128 == 0 && H <= 16384, "moe_expand_scatter: H must be a multiple of 128, <= 16384");
  MOE_REQUIRE(scale_layout == MOE_SCALE_F32_ROWMAJOR || scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR,
              "moe_expand_scatter: bad scale layout");
  const int G = H / 128;
  if (scale_layout == MOE_SCALE_F32_ROWMAJOR) {
    MOE_REQUIRE(ld_xs >= G && ld_xes >= G, "moe_expand_scatter: scale leading dimension < H/128");
  } else {
    MOE_REQUIRE(ld_xs >= T && ld_xes >= M_cap, "moe_expand_scatter: packed scale leading dimension < rows");
  }
  MOE_REQUIRE(moe::aligned(x, 16) && moe::aligned(xe, 16), "moe_expand_scatter: x/xe not 16-byte aligned");
  MOE_REQUIRE_DEVICE();
  const int nvec = H / 16;
  int threads = ((nvec + 31) / 32) * 32;
  if (threads > 1024) threads = 1024;
  if (threads < 64) threads = 64;
  const int pad_per_expert = (align - 1 + moe::kPadRowsPerBlock - 1) / moe::kPadRowsPerBlock;
  int64_t token_blocks = static_cast<int64_t>(moe::device_sm_count()) * (2048 / threads);
  if (token_blocks > T) token_blocks = T;
  if (token_blocks < 1) token_blocks = 1;
  const int64_t grid = static_cast<int64_t>(E) * pad_per_expert + token_blocks;
  MOE_REQUIRE(grid < (1ll << 31), "moe_expand_scatter: grid too large");
  moe::scatter_kernel<<<static_cast<unsigned>(grid), threads, 0,
                        reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(x), x_scale, scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR,
      ld_xs, topk_w, src2dst, psum, d_n_valid, T, H, K, E, align, M_cap,
      reinterpret_cast<uint4*>(xe), xe_scale, ld_xes, row_w, pad_per_expert,
      static_cast<int>(token_blocks), d_status);
  return moe::check_launch("scatter_kernel");
}
