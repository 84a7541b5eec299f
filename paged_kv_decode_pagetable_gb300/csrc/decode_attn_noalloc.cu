// paged_decode_attn_noalloc: paged_decode_attn for callers that cannot
// allocate device memory.
//
// paged_decode_attn needs a caller-provided workspace for its split partial
// results. Some callers have no way to provide one: a plain C program that
// links only this library and has no device allocator of its own, or a
// plugin inside a host framework that owns all device memory through its
// own pool and gives extensions no scratch buffer. This entry point
// takes the same arguments minus the workspace and uses a fixed scratch
// array that lives in the library's device image instead.
//
// The scratch is a file-scope __device__ array of kNoallocScratchBytes. Every
// GPU that loads the library holds that much device memory until the process
// exits. All calls share it. The split partials must be zero when a call
// starts (the array starts zeroed, and every call that completes leaves them
// zero); a call that gave up on a wait (PKV_ERR_TIMEOUT) can leave some
// behind, so every call first launches a small kernel on the caller's stream
// that clears them when the error word holds PKV_ERR_TIMEOUT and otherwise
// returns at once (no allocation; with err_word NULL nothing is checked).
// Two calls whose kernels overlap on the GPU (for instance on two streams,
// or from two threads) race on the scratch and corrupt each other's
// results: serialize them.
//
// The first call on each device looks the array's device address up with
// cudaGetSymbolAddress while that device is current, and caches it; make that
// first call before any stream capture begins. No call allocates or frees
// memory. Sizes whose partial results do not fit the scratch are rejected
// with PKV_E_BAD_ARG.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch for the current device. In host code
// the name g_noalloc_scratch is only a host-side stand-in, not a device
// address, so it is never passed to a kernel directly.
int scratch_address(void **out) {
  static std::mutex mu;
  static void *addr[kMaxDevices] = {nullptr};
  int dev = 0;
  PKV_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices)
    return pkv::fail(PKV_E_CUDA, "paged_decode_attn_noalloc: device id %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return pkv::fail(PKV_E_CUDA, "paged_decode_attn_noalloc: cudaGetSymbolAddress: %s",
                       cudaGetErrorString(e));
    addr[dev] = p;
  }
  *out = addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" {

int paged_decode_attn_noalloc(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                              const pkv_bf16 *v_cache, const int32_t *dev_table,
                              int n_slots, int max_pages_per_seq, int page_size,
                              int n_pages, const int32_t *batch_idx,
                              const int32_t *seq_lens, int window, float scale,
                              int B, int Hq, int Hkv, int D, int num_splits,
                              pkv_bf16 *out, int32_t *err_word, void *stream) {
  if (num_splits < 0) return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn_noalloc: num_splits < 0");
  if (max_pages_per_seq < 1 || page_size < 1)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn_noalloc: bad size argument");
  // the parts paged_decode_attn will actually cut a row into: num_splits
  // capped at the tiles of the longest row the table can hold (the same cap
  // it applies), so a large num_splits on short rows needs little scratch
  const int parts = pkv::decode_max_parts(max_pages_per_seq, page_size, window, num_splits);
  const size_t need = paged_decode_attn_workspace(B, Hq, D, parts);
  if (need > kNoallocScratchBytes)
    return pkv::fail(PKV_E_BAD_ARG,
                     "paged_decode_attn_noalloc: %d parts x %d rows x %d heads x D=%d need "
                     "%zu bytes of scratch, more than the fixed %zu; use paged_decode_attn "
                     "with a caller workspace, or fewer splits",
                     parts, B, Hq, D, need, kNoallocScratchBytes);
  void *scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
  // the partials must be zero when a call starts; only a call that gave up
  // on a wait leaves some behind
  st = pkv::decode_scrub_after_timeout(scratch, B, Hq, D, parts, err_word,
                                       static_cast<cudaStream_t>(stream));
  if (st != PKV_OK) return st;
  return paged_decode_attn(q, k_cache, v_cache, dev_table, n_slots, max_pages_per_seq,
                           page_size, n_pages, batch_idx, seq_lens, window, scale, B, Hq, Hkv,
                           D, num_splits, scratch, kNoallocScratchBytes, out, err_word, stream);
}

}  // extern "C"
