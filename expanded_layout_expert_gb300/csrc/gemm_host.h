// Host-side pieces shared by the two grouped-GEMM implementations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// TMA descriptor for a 2-D uint8 tensor [outer, inner] with a row stride of
// `stride` bytes, copied in boxes of box_outer rows x 128 bytes with 128-byte
// swizzling; rows past `outer` read as zero. Returns MOE_OK or MOE_ERR_CUDA
// (message set).
int make_tmap_k128(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t stride, uint32_t box_outer);

// Arguments of the block-scaled (ue8m0) grouped GEMM, already validated.
struct MxGemmArgs {
  const uint8_t* A;
  const uint32_t* A_scale;  // packed ue8m0, column-major words [ceil(Kd/512), ld_as]
  int64_t ld_as;
  const int32_t* start;
  const int32_t* tile_prefix;
  const int32_t* d_total;
  const uint8_t* W;
  const uint8_t* W_scale;   // ue8m0 bytes [E, N/128, Kd/128]
  const float* row_w;       // non-null: output row r is multiplied by row_w[r]
  int E, N, Kd;
  int64_t M_cap;
  uint16_t* out;
  int32_t* status;
  unsigned long long* trace;  // optional per-CTA cycle counters
  // Non-null: W is W13 [E, N = 2I, Kd] and the kernel applies silu(gate)*up
  // and the ue8m0 fp8 quantiser in its epilogue, writing down_proj's input
  // di [M_cap, I] and its packed scales (int32 words [ceil(I/512), ld_ds],
  // addressed as bytes) instead of `out`.
  uint8_t* di = nullptr;
  uint8_t* di_scale = nullptr;
  int64_t ld_ds = 0;
};

// Launches the tcgen05 block-scaled kernel (N % 256 == 0).
int launch_grouped_gemm_mx(const MxGemmArgs& a, cudaStream_t s);

}  // namespace moe
