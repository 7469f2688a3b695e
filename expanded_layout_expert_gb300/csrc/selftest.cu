// moe_selftest_bounded_wait: exercises the bounded mbarrier wait that every
// pipeline role of the GEMM kernels uses, on a barrier that nothing ever
// arrives at. The first waiter gives up after `limit_cycles`, records
// MOE_ERR_TIMEOUT and raises the block's abort flag; a second waiter, given a
// limit four times longer, must leave as soon as it sees the flag. Nothing
// faults or traps, and the context stays usable afterwards.
#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

__global__ void wait_selftest_kernel(long long limit, int32_t* status, long long* out) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
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
  moe::wait_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      limit_cycles, d_status, reinterpret_cast<long long*>(d_out));
  return moe::check_launch("wait_selftest_kernel");
}
