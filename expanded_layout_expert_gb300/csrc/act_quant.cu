// moe_act_quant: silu(gate) * up, rounded to bf16, then per-128-group fp8
// quantisation of down_proj's input, with the pair's top-k weight folded into
// the fp32 scale (SGLang moe_runner/deep_gemm.py, _run_contiguous_gemm:
// silu_and_mul then per-token-group quant, group 128; SGLang PR 37261,
// Modifications/Core: the fold; _situ_mul_quant_contig_kernel: amax clamped
// to 1e-10, scale amax/448). On the ue8m0 path the scale is rounded up to a
// power of two by the rule of _cast_to_e8m0_with_rounding_up and stored as
// its exponent byte, packed four groups per int32, column-major.
//
// One warp per (row, 4-group quad = 512 columns): each lane owns 8 columns
// in each 256-column half, so every load and store instruction of the warp
// is one contiguous, fully coalesced run. HBM-bound: 4I bytes read and
// I + scales written per row.
#include "act_quant.cuh"
#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

// 8 bf16 gate + 8 bf16 up -> 8 bf16-rounded silu(g)*u values.
MOE_DEV void silu_mul8(const uint4& g, const uint4& u, float (&h)[8]) {
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
  const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 gf = __bfloat1622float2(g2[i]);
    const float2 uf = __bfloat1622float2(u2[i]);
    h[2 * i] = silu_mul_bf16(gf.x, uf.x);
    h[2 * i + 1] = silu_mul_bf16(gf.y, uf.y);
  }
}

__global__ void __launch_bounds__(kThreads) act_quant_kernel(
    const uint16_t* __restrict__ gu, int I, const float* __restrict__ row_w, int fold, int ue8m0,
    const int32_t* __restrict__ d_total, int64_t M_cap, uint8_t* __restrict__ di,
    void* __restrict__ di_scale, int64_t ld_ds) {
  const int G = I / 128;
  const int Q = (G + 3) / 4;
  int64_t total = *d_total;
  if (total > M_cap) total = M_cap;
  if (total < 0) total = 0;
  const int64_t items = total * Q;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t it = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5; it < items;
       it += nwarps) {
    const int64_t r = it / Q;
    const int q = static_cast<int>(it % Q);
    const int c0 = q * 512 + lane * 8;  // half 0: groups 4q + lane/16
    const int c1 = c0 + 256;            // half 1: groups 4q + 2 + lane/16
    const bool a0 = c0 < I, a1 = c1 < I;
    const uint16_t* row = gu + r * 2 * I;
    float h0[8], h1[8];
    float m0 = 0.0f, m1 = 0.0f;
    if (a0) {
      silu_mul8(__ldcs(reinterpret_cast<const uint4*>(row + c0)),
                __ldcs(reinterpret_cast<const uint4*>(row + I + c0)), h0);
#pragma unroll
      for (int j = 0; j < 8; ++j) m0 = fmaxf(m0, fabsf(h0[j]));
    }
    if (a1) {
      silu_mul8(__ldcs(reinterpret_cast<const uint4*>(row + c1)),
                __ldcs(reinterpret_cast<const uint4*>(row + I + c1)), h1);
#pragma unroll
      for (int j = 0; j < 8; ++j) m1 = fmaxf(m1, fabsf(h1[j]));
    }
    // amax over the 16 lanes that share a 128-column group
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    // stored scale amax/448; codes h * (448/amax), as the pages' quantiser
    // (_situ_mul_quant_contig_kernel) computes them; ue8m0: the scale rounded
    // up to a power of two, whose inverse is exact
    float s0, s1, inv0, inv1;
    uint32_t b0, b1;
    group_scale(m0, ue8m0 != 0, s0, inv0, b0);
    group_scale(m1, ue8m0 != 0, s1, inv1, b1);
    uint8_t* out = di + r * I;
    if (a0) *reinterpret_cast<uint2*>(out + c0) = fp8x8(h0, inv0);
    if (a1) *reinterpret_cast<uint2*>(out + c1) = fp8x8(h1, inv1);

    const int half_lane = lane & 15;
    const int g0 = q * 4 + (lane >> 4);
    const int g1 = g0 + 2;
    if (!ue8m0) {
      const float w = fold ? row_w[r] : 1.0f;
      float* ds = static_cast<float*>(di_scale);
      if (half_lane == 0 && a0) ds[r * ld_ds + g0] = __fmul_rn(s0, w);
      if (half_lane == 0 && a1) ds[r * ld_ds + g1] = __fmul_rn(s1, w);
    } else {
      // groups 4q..4q+3 are (lane 0, half 0), (lane 16, half 0), (lane 0,
      // half 1), (lane 16, half 1); groups past G stay zero
      const uint32_t v0 = a0 ? b0 : 0u, v1 = a1 ? b1 : 0u;
      const uint32_t hi0 = __shfl_sync(0xffffffffu, v0, 16);
      const uint32_t hi1 = __shfl_sync(0xffffffffu, v1, 16);
      if (lane == 0) {
        const uint32_t word = v0 | (hi0 << 8) | (v1 << 16) | (hi1 << 24);
        static_cast<int32_t*>(di_scale)[q * ld_ds + r] = static_cast<int32_t>(word);
      }
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_act_quant(const uint16_t* gu, int I, const float* row_w, int flags,
                             int scale_layout, const int32_t* d_total, int64_t M_cap, uint8_t* di,
                             void* di_scale, int64_t ld_ds, int32_t* d_status,
                             moe_stream_t stream) {
  (void)d_status;
  MOE_REQUIRE(gu && d_total && di && di_scale, "moe_act_quant: null pointer");
  MOE_REQUIRE(I > 0 && I % 128 == 0 && M_cap >= 0, "moe_act_quant: I must be a multiple of 128");
  MOE_REQUIRE(scale_layout == MOE_SCALE_F32_ROWMAJOR || scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR,
              "moe_act_quant: bad scale layout");
  const bool fold = (flags & MOE_FOLD_WEIGHT_INTO_SCALE) != 0;
  MOE_REQUIRE(!fold || (row_w && scale_layout == MOE_SCALE_F32_ROWMAJOR),
              "moe_act_quant: the fold needs row_w and fp32 scales");
  if (scale_layout == MOE_SCALE_F32_ROWMAJOR) {
    MOE_REQUIRE(ld_ds >= I / 128, "moe_act_quant: scale leading dimension < I/128");
  } else {
    MOE_REQUIRE(ld_ds >= M_cap, "moe_act_quant: packed scale leading dimension < M_cap");
  }
  MOE_REQUIRE(moe::aligned(gu, 16) && moe::aligned(di, 8), "moe_act_quant: misaligned gu/di");
  MOE_REQUIRE_DEVICE();
  const int grid = moe::device_sm_count() * (2048 / moe::kThreads);
  moe::act_quant_kernel<<<grid, moe::kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      gu, I, row_w, fold ? 1 : 0, scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR, d_total, M_cap,
      di, di_scale, ld_ds);
  return moe::check_launch("act_quant_kernel");
}
