// Internal helpers shared by the libpkv translation units (host side).
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "../../include/pkv.h"

namespace pkv {

// Records a thread-local message for pkv_last_error() and returns `code`.
int fail(int code, const char *fmt, ...);
// Clears the thread-local message and returns PKV_OK.
int ok();

// Number of SMs of the current device (cached per device; 0 if unknown).
int sm_count();

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}
inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

}  // namespace pkv

#define PKV_CUDA_CHECK(call)                                                  \
  do {                                                                        \
    cudaError_t e_ = (call);                                                  \
    if (e_ != cudaSuccess)                                                    \
      return pkv::fail(PKV_E_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)
