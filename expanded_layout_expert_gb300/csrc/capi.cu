// Host-side parts of the C ABI that belong to no single kernel: error text,
// device checks, the capacity bound and the composite FFN call.
#include <cstdarg>
#include <cstring>
#include <mutex>

#include "host_util.h"

namespace moe {

namespace {
thread_local char g_err[512] = "no error";

struct DevInfo {
  int sm_count = 0;
  int supported = -1;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

DevInfo& info_for_current() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.supported < 0) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    d.sm_count = sms > 0 ? sms : 1;
    d.supported = (major == 10 && minor == 3) ? 1 : 0;
  }
  return d;
}
}  // namespace

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

int device_sm_count() { return info_for_current().sm_count; }

bool current_device_supported() { return info_for_current().supported == 1; }

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe

extern "C" {

const char* moe_last_error_string(void) { return moe::g_err; }

int moe_device_supported(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return (major == 10 && minor == 3) ? 1 : 0;
}

int64_t moe_expanded_capacity(int64_t T, int K, int E, int align) {
  if (T < 0 || K <= 0 || E <= 0 || align <= 0) return -1;
  const int64_t A = T * static_cast<int64_t>(K);
  const int64_t ne = A < E ? A : static_cast<int64_t>(E);
  return static_cast<int64_t>(align) * (ne + (A - ne) / align);
}

int moe_grouped_ffn(const uint8_t* xe, const void* xe_scale, int64_t ld_xes, int scale_layout,
                    const int32_t* start, const int32_t* tile_prefix, const int32_t* d_total,
                    const uint8_t* w13, const void* s13, const uint8_t* w2, const void* s2,
                    const float* row_w, int flags, int E, int H, int I, int64_t M_cap,
                    uint16_t* gateup_ws, uint8_t* down_in, void* down_in_scale, int64_t ld_dis,
                    uint16_t* down_out, int32_t* d_status, moe_stream_t stream) {
  MOE_REQUIRE(!((flags & MOE_FOLD_WEIGHT_INTO_SCALE) && (flags & MOE_WEIGHT_OUTPUT_ROWS)),
              "moe_grouped_ffn: choose one weighting flag");
  MOE_REQUIRE(!(flags & MOE_FOLD_WEIGHT_INTO_SCALE) || scale_layout == MOE_SCALE_F32_ROWMAJOR,
              "moe_grouped_ffn: the fold needs fp32 scales (a power-of-two scale cannot absorb a weight)");
  int rc;
  const bool fused = !(flags & MOE_FFN_UNFUSED);
  if (fused) {
    // gate_up with silu*mul and the quantiser in its epilogue: gateup_ws unused
    rc = moe_grouped_gemm_act_quant(
        xe, xe_scale, scale_layout, ld_xes, start, tile_prefix, d_total, w13, s13, row_w,
        flags & (MOE_FOLD_WEIGHT_INTO_SCALE | MOE_GEMM_PER_KBLOCK_PROMOTION), E, I, H, M_cap,
        down_in, down_in_scale, ld_dis, d_status, stream);
    if (rc != MOE_OK) return rc;
  } else {
    MOE_REQUIRE(gateup_ws, "moe_grouped_ffn: null gateup_ws");
    const int gflags = flags & MOE_GEMM_PER_KBLOCK_PROMOTION;
    rc = moe_grouped_gemm(xe, xe_scale, scale_layout, ld_xes, start, tile_prefix, d_total, w13,
                          s13, nullptr, gflags, E, 2 * I, H, M_cap, gateup_ws, d_status, stream);
    if (rc != MOE_OK) return rc;
    rc = moe_act_quant(gateup_ws, I, row_w, flags & MOE_FOLD_WEIGHT_INTO_SCALE, scale_layout,
                       d_total, M_cap, down_in, down_in_scale, ld_dis, d_status, stream);
    if (rc != MOE_OK) return rc;
  }
  return moe_grouped_gemm(down_in, down_in_scale, scale_layout, ld_dis, start, tile_prefix,
                          d_total, w2, s2, row_w,
                          flags & (MOE_WEIGHT_OUTPUT_ROWS | MOE_GEMM_PER_KBLOCK_PROMOTION), E, H, I,
                          M_cap, down_out, d_status, stream);
}

}  // extern "C"
