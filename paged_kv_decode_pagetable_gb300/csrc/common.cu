// Status reporting, device queries and the error-word read-back.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {

static thread_local char g_msg[512] = "";

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_msg[0] = '\0';
  return PKV_OK;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) ==
        cudaSuccess)
      cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace pkv

extern "C" {

const char *pkv_last_error(void) { return pkv::g_msg; }

int pkv_read_error_word(const int32_t *err_word, void *stream,
                        int32_t *host_out) {
  if (!err_word || !host_out)
    return pkv::fail(PKV_E_BAD_ARG, "pkv_read_error_word: NULL pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PKV_CUDA_CHECK(cudaMemcpyAsync(host_out, err_word, sizeof(int32_t),
                                 cudaMemcpyDeviceToHost, s));
  PKV_CUDA_CHECK(cudaStreamSynchronize(s));
  return pkv::ok();
}

}  // extern "C"
