// Internal host helpers of libmoe_expand.so: thread-local error text,
// device capability and SM-count caches, argument checks.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>

#include "moe_expand.h"

namespace moe {

void set_error(const char* fmt, ...);
int device_sm_count();            // of the current device
bool current_device_supported();  // compute capability 10.3

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Checks the launch that was just queued. Returns MOE_OK or MOE_ERR_CUDA.
int check_launch(const char* what);

}  // namespace moe

#define MOE_REQUIRE(cond, ...)             \
  do {                                     \
    if (!(cond)) {                         \
      ::moe::set_error(__VA_ARGS__);       \
      return MOE_ERR_INVALID_ARG;          \
    }                                      \
  } while (0)

#define MOE_REQUIRE_DEVICE()                                         \
  do {                                                               \
    if (!::moe::current_device_supported()) {                        \
      ::moe::set_error("current device is not compute capability 10.3"); \
      return MOE_ERR_UNSUPPORTED;                                    \
    }                                                                \
  } while (0)
