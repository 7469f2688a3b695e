// The decode variant's bridge between the expanded layout and a masked slab
// (SGLang PR 37261, "The deepep_v2 decode (expand + masked slab) path" and
// the pre/post permute's deepep_v2_masked branch: expand_to_masked_slab
// before the masked grouped GEMM, masked_slab_to_expand after it, the latter
// taking the top-k weights). A slab holds each expert's rows at a fixed
// height: expert e's j-th row at slab row e * max_m + j, with masked_m[e]
// rows in use.
//
//  - moe_expand_to_masked_slab copies expert e's first min(count_e, max_m)
//    expanded rows (fp8 bytes and their scale row) into its slab, zeroes the
//    rest of the last 128-row tile in use, and writes the slab's row count
//    and the start / tile prefix / total that the grouped GEMMs take, so the
//    same GEMM kernels run on the slab (tiles past masked_m are never
//    visited). Rows beyond max_m are dropped and flagged on the status word.
//  - moe_masked_slab_to_expand copies the GEMM output back to the expanded
//    rows, multiplying each by its pair's weight (bf16 once, from fp32), and
//    zeroes the expanded rows that had no slab row (alignment gaps and
//    dropped rows).
// Both are plain HBM copies: one warp per row, 16-byte vectors.
#include <cuda_bf16.h>

#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxE = 1024;

// Block 0: per-expert slab metadata (row counts, starts, 128-row tile prefix,
// total). Every block: warps walk the slab rows in use.
__global__ void __launch_bounds__(kThreads) expand_to_slab_kernel(
    const uint4* __restrict__ xe, const void* __restrict__ xe_scale, int ue8m0, int64_t ld_xes,
    const int32_t* __restrict__ psum, const int32_t* __restrict__ start, int E, int H,
    int64_t max_m, uint4* __restrict__ slab, void* __restrict__ slab_scale, int64_t ld_ss,
    int32_t* __restrict__ masked_m, int32_t* __restrict__ slab_start,
    int32_t* __restrict__ slab_tiles, int32_t* __restrict__ slab_total,
    int32_t* __restrict__ status) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (blockIdx.x == 0) {
    __shared__ int s_tiles[kMaxE];
    for (int e = tid; e < E; e += kThreads) {
      const int c = psum[e] - start[e];
      const int m = c < max_m ? c : static_cast<int>(max_m);
      if (c > max_m) set_status(status, MOE_ERR_DEVICE_CHECK);
      masked_m[e] = m;
      slab_start[e] = static_cast<int32_t>(e * max_m);
      s_tiles[e] = (m + MOE_BLOCK_M - 1) / MOE_BLOCK_M;
    }
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int e = 0; e < E; ++e) {
        slab_tiles[e] = acc;
        acc += s_tiles[e];
      }
      slab_tiles[E] = acc;
      *slab_total = static_cast<int32_t>(E * max_m);
    }
  }
  const int nvec = H / 16;
  const int G = H / 128;
  const int W = (G + 3) / 4;
  const int64_t rows = static_cast<int64_t>(E) * max_m;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * kThreads + tid) >> 5; r < rows; r += nwarps) {
    const int e = static_cast<int>(r / max_m);
    const int j = static_cast<int>(r - static_cast<int64_t>(e) * max_m);
    const int c = psum[e] - start[e];
    const int m = c < max_m ? c : static_cast<int>(max_m);
    const int used = (m + MOE_BLOCK_M - 1) / MOE_BLOCK_M * MOE_BLOCK_M;
    if (j >= used) continue;  // never read by the GEMM: left as it is
    const bool copy = j < m;
    const int64_t src = static_cast<int64_t>(start[e]) + j;
    for (int v = lane; v < nvec; v += 32)
      slab[r * nvec + v] = copy ? __ldcs(xe + src * nvec + v) : make_uint4(0, 0, 0, 0);
    if (!ue8m0) {
      const float* xs = static_cast<const float*>(xe_scale);
      float* ss = static_cast<float*>(slab_scale);
      for (int g = lane; g < G; g += 32) ss[r * ld_ss + g] = copy ? xs[src * ld_xes + g] : 0.0f;
    } else {
      const int32_t* xs = static_cast<const int32_t*>(xe_scale);
      int32_t* ss = static_cast<int32_t*>(slab_scale);
      for (int w = lane; w < W; w += 32) ss[w * ld_ss + r] = copy ? xs[w * ld_xes + src] : 0;
    }
  }
}

MOE_DEV uint32_t scale_bf16x2(uint32_t v, float w) {
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v);
  const float2 f = __bfloat1622float2(b);
  const __nv_bfloat162 o = __floats2bfloat162_rn(f.x * w, f.y * w);
  return *reinterpret_cast<const uint32_t*>(&o);
}

// One warp per expanded row r < total: the slab row times the pair's weight,
// or zero where the expert had no slab row for it.
__global__ void __launch_bounds__(kThreads) slab_to_expand_kernel(
    const uint4* __restrict__ slab_out, int64_t max_m, const int32_t* __restrict__ psum,
    const int32_t* __restrict__ start, const int32_t* __restrict__ d_total,
    const float* __restrict__ row_w, int E, int H, int64_t M_cap, uint4* __restrict__ out) {
  __shared__ int s_start[kMaxE];
  __shared__ int s_cnt[kMaxE];
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += kThreads) {
    s_start[e] = start[e];
    s_cnt[e] = psum[e] - start[e];
  }
  __syncthreads();
  int64_t total = *d_total;
  if (total > M_cap) total = M_cap;
  const int nvec = H / 8;  // 16-byte vectors of 8 bf16
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * kThreads + tid) >> 5; r < total; r += nwarps) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_start[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int j = static_cast<int>(r - s_start[e]);
    const int c = s_cnt[e];
    const int m = c < max_m ? c : static_cast<int>(max_m);
    const bool has = j < m;
    const float w = (has && row_w != nullptr) ? row_w[r] : 1.0f;
    const int64_t srow = static_cast<int64_t>(e) * max_m + j;
    for (int v = lane; v < nvec; v += 32) {
      uint4 o = make_uint4(0, 0, 0, 0);
      if (has) {
        const uint4 a = __ldcs(slab_out + srow * nvec + v);
        if (row_w != nullptr) {
          o.x = scale_bf16x2(a.x, w);
          o.y = scale_bf16x2(a.y, w);
          o.z = scale_bf16x2(a.z, w);
          o.w = scale_bf16x2(a.w, w);
        } else {
          o = a;
        }
      }
      out[r * nvec + v] = o;
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_expand_to_masked_slab(const uint8_t* xe, const void* xe_scale, int scale_layout,
                                         int64_t ld_xes, const int32_t* psum, const int32_t* start,
                                         int E, int H, int64_t max_m, uint8_t* slab,
                                         void* slab_scale, int64_t ld_ss, int32_t* masked_m,
                                         int32_t* slab_start, int32_t* slab_tile_prefix,
                                         int32_t* slab_total, int32_t* d_status,
                                         moe_stream_t stream) {
  MOE_REQUIRE(xe && xe_scale && psum && start && slab && slab_scale && masked_m && slab_start &&
                  slab_tile_prefix && slab_total,
              "moe_expand_to_masked_slab: null pointer");
  MOE_REQUIRE(E > 0 && E <= moe::kMaxE && max_m > 0 && static_cast<int64_t>(E) * max_m <= INT32_MAX,
              "moe_expand_to_masked_slab: bad sizes (E in [1, 1024], E * max_m < 2^31)");
  MOE_REQUIRE(H > 0 && H % 128 == 0, "moe_expand_to_masked_slab: H must be a multiple of 128");
  MOE_REQUIRE(scale_layout == MOE_SCALE_F32_ROWMAJOR || scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR,
              "moe_expand_to_masked_slab: bad scale layout");
  const int G = H / 128;
  if (scale_layout == MOE_SCALE_F32_ROWMAJOR) {
    MOE_REQUIRE(ld_xes >= G && ld_ss >= G, "moe_expand_to_masked_slab: scale leading dimension < H/128");
  } else {
    MOE_REQUIRE(ld_ss >= static_cast<int64_t>(E) * max_m,
                "moe_expand_to_masked_slab: packed slab scale leading dimension < E * max_m");
  }
  MOE_REQUIRE(moe::aligned(xe, 16) && moe::aligned(slab, 16),
              "moe_expand_to_masked_slab: xe/slab not 16-byte aligned");
  MOE_REQUIRE_DEVICE();
  const int64_t rows = static_cast<int64_t>(E) * max_m;
  int64_t grid = (rows + moe::kThreads / 32 - 1) / (moe::kThreads / 32);
  const int64_t cap = static_cast<int64_t>(moe::device_sm_count()) * (2048 / moe::kThreads);
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  moe::expand_to_slab_kernel<<<static_cast<unsigned>(grid), moe::kThreads, 0,
                               reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(xe), xe_scale, scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR,
      ld_xes, psum, start, E, H, max_m, reinterpret_cast<uint4*>(slab), slab_scale, ld_ss, masked_m,
      slab_start, slab_tile_prefix, slab_total, d_status);
  return moe::check_launch("expand_to_slab_kernel");
}

extern "C" int moe_masked_slab_to_expand(const uint16_t* slab_out, int64_t max_m,
                                         const int32_t* psum, const int32_t* start,
                                         const int32_t* d_total, const float* row_w, int E, int H,
                                         int64_t M_cap, uint16_t* out, moe_stream_t stream) {
  MOE_REQUIRE(slab_out && psum && start && d_total && out, "moe_masked_slab_to_expand: null pointer");
  MOE_REQUIRE(E > 0 && E <= moe::kMaxE && max_m > 0 && M_cap >= 0 && H > 0 && H % 8 == 0,
              "moe_masked_slab_to_expand: bad sizes");
  MOE_REQUIRE(moe::aligned(slab_out, 16) && moe::aligned(out, 16),
              "moe_masked_slab_to_expand: buffers not 16-byte aligned");
  MOE_REQUIRE_DEVICE();
  if (M_cap == 0) return MOE_OK;
  int64_t grid = (M_cap + moe::kThreads / 32 - 1) / (moe::kThreads / 32);
  const int64_t cap = static_cast<int64_t>(moe::device_sm_count()) * (2048 / moe::kThreads);
  if (grid > cap) grid = cap;
  moe::slab_to_expand_kernel<<<static_cast<unsigned>(grid), moe::kThreads, 0,
                               reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(slab_out), max_m, psum, start, d_total, row_w, E, H, M_cap,
      reinterpret_cast<uint4*>(out));
  return moe::check_launch("slab_to_expand_kernel");
}
