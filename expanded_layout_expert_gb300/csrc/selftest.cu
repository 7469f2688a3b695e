// moe_selftest_bounded_wait: exercises the bounded mbarrier waits that the
// pipeline roles of the GEMM kernels use, on barriers that nothing ever
// arrives at. Block 0: a single-thread waiter gives up after `limit_cycles`,
// records MOE_ERR_TIMEOUT and raises the block's abort flag; a second
// single-thread waiter and a whole warp in the warp-collective wait, both
// given a limit four times longer, must leave as soon as they see the flag.
// Block 1: a warp in the warp-collective wait gives up on its own limit.
// Nothing faults or traps, and the context stays usable afterwards.
#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

__global__ void wait_selftest_kernel(long long limit, int32_t* status, long long* out) {
  __shared__ uint64_t bar[3];
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&bar[i], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    if (tid == 0) {
      const long long t0 = clock64();
      const bool ok = mbar_wait(&bar[0], 0, &abort_flag, status, limit);
      out[0] = ok ? 1 : 0;
      out[1] = clock64() - t0;
    } else if (tid == 32) {
      const long long t0 = clock64();
      const bool ok = mbar_wait(&bar[1], 0, &abort_flag, status, 4 * limit);
      out[2] = ok ? 1 : 0;
      out[3] = clock64() - t0;
    } else if (warp == 2) {
      const long long t0 = clock64();
      const bool ok = mbar_wait_warp(&bar[2], 0, &abort_flag, status, 4 * limit);
      const unsigned votes = __ballot_sync(0xffffffffu, ok);  // lanes that saw success
      if (lane == 0) {
        out[4] = votes;
        out[5] = clock64() - t0;
      }
    }
  } else if (warp == 0) {
    const long long t0 = clock64();
    const bool ok = mbar_wait_warp(&bar[0], 0, &abort_flag, status, limit);
    const unsigned votes = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) {
      out[6] = votes;
      out[7] = clock64() - t0;
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_selftest_bounded_wait(int64_t limit_cycles, int32_t* d_status, int64_t* d_out,
                                         moe_stream_t stream) {
  MOE_REQUIRE(d_status && d_out, "moe_selftest_bounded_wait: null pointer");
  MOE_REQUIRE(limit_cycles > 0 && limit_cycles <= 4000000000LL,
              "moe_selftest_bounded_wait: limit must be in (0, 4e9] cycles");
  MOE_REQUIRE_DEVICE();
  moe::wait_selftest_kernel<<<2, 96, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      limit_cycles, d_status, reinterpret_cast<long long*>(d_out));
  return moe::check_launch("wait_selftest_kernel");
}
