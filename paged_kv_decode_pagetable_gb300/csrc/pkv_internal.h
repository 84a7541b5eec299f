// Internal helpers shared by the libpkv translation units (host side).
#pragma once

#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>
#include <utility>

#include "../../include/pkv.h"

namespace pkv {

// Records a thread-local message for pkv_last_error() and returns `code`.
int fail(int code, const char *fmt, ...);
// Clears the thread-local message and returns PKV_OK.
int ok();

// Number of SMs of the current device (cached per device; 0 if unknown).
int sm_count();

// Most parts paged_decode_attn cuts one (row, head) into for these arguments
// (num_splits 0 = automatic), the count its workspace is sized for with
// paged_decode_attn_workspace; 0 if the arguments are out of range.
int decode_max_parts(int max_pages_per_seq, int page_size, int window, int num_splits);
// Launches a kernel on `stream` that zeroes the split partials of a
// workspace sized by paged_decode_attn_workspace(B, Hq, D, parts) when
// *err_word reports PKV_ERR_TIMEOUT (a call that gave up on a wait can leave
// unread partials behind); it does nothing otherwise, or when there is no
// error word or no partial area.
int decode_scrub_after_timeout(void *workspace, int B, int Hq, int D, int parts,
                               const int32_t *err_word, cudaStream_t stream);

// Document-causal prefill attention on tcgen05 (prefill_tc.cu), D in {64, 128};
// arguments already validated by the public entry point.
template <int D>
int launch_prefill_tc(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                      const int32_t *docs, const int32_t *kv_num, const int32_t *kv_idx,
                      const int32_t *full_num, const int32_t *full_idx, int L, int Hq, int Hkv,
                      int window, float scale, pkv_bf16 *out, cudaStream_t s);
// The same for D in {256, 512} (prefill_tc_wide.cu).
template <int D>
int launch_prefill_wide(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                        const int32_t *docs, const int32_t *kv_num, const int32_t *kv_idx,
                        const int32_t *full_num, const int32_t *full_idx, int L, int Hq, int Hkv,
                        int window, float scale, pkv_bf16 *out, cudaStream_t s);
}  // namespace pkv

struct CUtensorMap_st;
namespace pkv {
// Tensor maps of the prefill kernels (defined in prefill_tc.cu): a 3-D map {column,
// token, head} over a [heads][L][D] bf16 tensor with [box_rows][64] boxes and
// 128-byte swizzle (tokens past L read zeros), and a 1-D map over the int32
// document ids in 64-id boxes (ids past L read zeros).
int prefill_head_map(CUtensorMap_st *tm, const void *base, int heads, int L, int D,
                     int box_rows);
int prefill_docs_map(CUtensorMap_st *tm, const int32_t *docs, int L);
// A 4-D map {64 columns, token, head, 64-column atom} over the same tensor:
// one box of {64, box_rows, box_heads, box_atoms} lands as box_atoms atoms of
// [box_heads][box_rows][64], 128-byte swizzle (tokens past L read zeros).
int prefill_atoms_map(CUtensorMap_st *tm, const void *base, int heads, int L, int D,
                      int box_rows, int box_heads, int box_atoms);

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}
inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Launches a kernel that may begin while the previous kernel of the stream
// is still running (programmatic dependent launch). Every kernel launched
// this way executes griddepcontrol.wait before it touches global memory, so
// it observes the same ordering as a plain launch; only the launch latency
// and the set-up of shared memory overlap the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pkv

#ifdef __CUDACC__
// Waits until the previous kernel of the stream has completed and its
// memory is visible (a no-op for a plain launch). Every kernel calls it
// before its first global memory access.
__device__ __forceinline__ void pkv_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel of the stream be scheduled before this one ends. It
// takes effect once every CTA of this grid has issued it (or exited), so the
// next kernel never waits for resources held by CTAs that have not started.
// Kernels that do not call it release their dependents as their CTAs exit.
// The small kernels whose CTAs leave room for the persistent attention CTAs
// (kv_append, qk_norm_rope, combine) and the attention kernel itself call it
// early; the fused prologue does not, because its CTAs fill the register
// file and would delay the attention CTAs it released.
__device__ __forceinline__ void pkv_allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

#define PKV_CUDA_CHECK(call)                                                  \
  do {                                                                        \
    cudaError_t e_ = (call);                                                  \
    if (e_ != cudaSuccess)                                                    \
      return pkv::fail(PKV_E_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)
