// moe_combine: y[t] = sum over the token's pairs of its expert-output row,
// in fp32, k order, then bf16 (the un-expand and reduction of the expand-mode
// combine; ep_gather in SGLang moe_runner/deep_gemm.py). Tokens whose ids are
// all -1 get zeros; rows t >= n_valid are neither read nor written (vLLM PR
// 54109, Design: kernels must skip inactive rows or make them safe to
// discard, and never trust row contents).
//
// A persistent grid of warps walks (valid token, 256-column chunk) tasks;
// each lane owns one 16-byte column vector (8 bf16) of the chunk and issues
// the K gathers for it back to back before accumulating.
#include <cuda_bf16.h>

#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

constexpr int kMaxK = 32;

MOE_DEV void acc8(float (&a)[8], const uint4& v, float w) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    a[2 * i] = __fadd_rn(a[2 * i], __fmul_rn(f.x, w));
    a[2 * i + 1] = __fadd_rn(a[2 * i + 1], __fmul_rn(f.y, w));
  }
}

constexpr int kThreads = 256;

// One warp per (token, 256-column chunk): lane k < K holds the token's k-th
// expanded row (and its weight) and broadcasts it by shuffle; each lane owns
// one 16-byte column vector of the chunk, with the K gathers of that vector
// issued back to back before they are summed. Chunking the row keeps the GPU
// busy when there are few tokens (a decode batch) as well as many.
__global__ void __launch_bounds__(kThreads) combine_kernel(
    const uint4* __restrict__ down, const int32_t* __restrict__ src2dst,
    const float* __restrict__ row_w, const int32_t* __restrict__ d_n_valid, int64_t T, int H,
    int K, uint4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int nvec = H / 8;
  const int nchunk = (nvec + 31) / 32;
  int64_t nv = T;
  if (d_n_valid != nullptr) {
    nv = *d_n_valid;
    nv = nv < 0 ? 0 : (nv > T ? T : nv);
  }
  const int64_t tasks = nv * nchunk;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t task = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
       task < tasks; task += nwarps) {
    const int64_t t = task / nchunk;
    const int v = static_cast<int>(task - t * nchunk) * 32 + lane;
    int my_r = -1;
    float my_w = 1.0f;
    if (lane < K) {
      my_r = src2dst[t * K + lane];
      if (my_r >= 0 && row_w != nullptr) my_w = row_w[my_r];
    }
    // warp-uniform from here (the shuffles need every lane); lanes past the
    // row idle
    const bool act = v < nvec;
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.0f;
    for (int k0 = 0; k0 < K; k0 += 4) {
      uint4 d[4];
      int r[4];
      float w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        r[j] = __shfl_sync(0xffffffffu, my_r, (k0 + j) & 31);
        w[j] = __shfl_sync(0xffffffffu, my_w, (k0 + j) & 31);
        if (k0 + j >= K || !act) r[j] = -1;
        d[j] = r[j] >= 0 ? __ldcs(down + static_cast<int64_t>(r[j]) * nvec + v)
                         : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (r[j] >= 0) acc8(a, d[j], w[j]);
    }
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
      ow[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    if (act) y[t * nvec + v] = o;
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_combine(const uint16_t* down_out, const int32_t* src2dst, const float* row_w,
                           const int32_t* d_n_valid, int64_t T, int H, int K, uint16_t* y,
                           moe_stream_t stream) {
  MOE_REQUIRE(T == 0 || (down_out && src2dst && y), "moe_combine: null pointer");
  MOE_REQUIRE(T >= 0 && K > 0 && K <= moe::kMaxK && H > 0 && H % 8 == 0,
              "moe_combine: bad sizes (K <= 32, H % 8 == 0)");
  MOE_REQUIRE(moe::aligned(down_out, 16) && moe::aligned(y, 16), "moe_combine: misaligned buffers");
  MOE_REQUIRE_DEVICE();
  if (T == 0) return MOE_OK;
  int64_t grid = static_cast<int64_t>(moe::device_sm_count()) * (2048 / moe::kThreads);
  const int64_t tasks = T * ((H / 8 + 31) / 32);
  const int64_t need = (tasks + (moe::kThreads / 32) - 1) / (moe::kThreads / 32);
  if (grid > need) grid = need;
  moe::combine_kernel<<<static_cast<unsigned>(grid), moe::kThreads, 0,
                        reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(down_out), src2dst, row_w, d_n_valid, T, H, K,
      reinterpret_cast<uint4*>(y));
  return moe::check_launch("combine_kernel");
}
