// Device arithmetic of silu(gate)*up and of the per-128-group fp8 quantiser
// (SGLang moe_runner/deep_gemm.py: silu_and_mul, per-token-group quant with
// group 128, _situ_mul_quant_contig_kernel's amax clamp and amax/448 scale,
// _cast_to_e8m0_with_rounding_up). Shared by the stand-alone act+quant
// kernel and the gate_up GEMM epilogue that fuses it, so both produce the
// same codes and scales bit for bit.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// ue8m0 exponent byte of s rounded up to a power of two.
MOE_DEV uint32_t ue8m0_round_up(float s) {
  const uint32_t bits = __float_as_uint(s);
  uint32_t ex = (bits >> 23) & 0xFFu;
  const uint32_t man = bits & 0x7FFFFFu;
  if (man != 0u && ex != 0xFEu && !(ex == 0u && man <= 0x400000u)) ex += 1u;
  return ex & 0xFFu;
}

// 2^(127-b) for an exponent byte b, as fp32 (2^-127 is the subnormal 0x00400000).
MOE_DEV float pow2_inverse(uint32_t b) {
  if (b <= 253u) return __uint_as_float((254u - b) << 23);
  return b == 254u ? __uint_as_float(0x00400000u) : __uint_as_float(0x00200000u);
}

MOE_DEV float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// bf16( silu(g) * u ) for bf16-valued g and u; silu in fast fp32 (the value
// is rounded to bf16 right after): g / (1 + e^-g).
MOE_DEV float silu_mul_bf16(float g, float u) {
  return bf16_round(__fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), u));
}

// Scale of one 128-group from its amax: stored scale s = max(amax,1e-10)/448;
// the codes are h * inv with inv = 448/amax (fp32 scales) or, for ue8m0, the
// exact inverse of s rounded up to a power of two (exponent byte in *b).
MOE_DEV void group_scale(float amax, bool ue8m0, float& s, float& inv, uint32_t& b) {
  const float m = fmaxf(amax, 1e-10f);
  s = __fdiv_rn(m, 448.0f);
  if (ue8m0) {
    b = ue8m0_round_up(s);
    inv = pow2_inverse(b);
  } else {
    b = 0u;
    inv = __fdiv_rn(448.0f, m);
  }
}

// Two values times the inverse scale -> two e4m3 codes (round to nearest
// even, saturating to +-448), low byte first.
MOE_DEV uint32_t fp8x2(float a, float b, float inv) {
  const float2 v = make_float2(__fmul_rn(a, inv), __fmul_rn(b, inv));
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// Eight values -> eight codes.
MOE_DEV uint2 fp8x8(const float* h, float inv) {
  return make_uint2(fp8x2(h[0], h[1], inv) | (fp8x2(h[2], h[3], inv) << 16),
                    fp8x2(h[4], h[5], inv) | (fp8x2(h[6], h[7], inv) << 16));
}

}  // namespace moe
