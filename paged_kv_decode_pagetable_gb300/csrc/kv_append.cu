// kv_append: decode scatter of one new K/V token per row into its page.
//
// Address map of "unsloth: compare main...transformers-continuous-batching-
// qwen3" · scripts/benchmarks/flex_paged_attention.py · PageTable.assign:
//   row = table[slot][pos / page_size] * page_size + pos % page_size.
//
// One thread moves 16 bytes (8 bf16). Threads of a warp cover consecutive
// 16-byte chunks of the same [row][head] vector, so loads from k/v and
// stores into the cache are both fully coalesced; the table entry is one
// broadcast load per (row). Nothing is read or written through an invalid
// index: the error word records it and the thread returns.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace {

__device__ __forceinline__ void report(int32_t *err, int bits) {
  if (err) atomicOr(err, bits);
}

// k / v element (row b, head h) starts at chunk b * row_stride + h * head_stride
// (token-major [B][Hkv][D]: row_stride = Hkv * chunks, head_stride = chunks;
// head-major [Hkv][B][D] as the pages' prefill [1, H, L, D]: row_stride =
// chunks, head_stride = B * chunks).
__global__ void kv_append_kernel(const uint4 *__restrict__ k,
                                 const uint4 *__restrict__ v,
                                 const int32_t *__restrict__ batch_idx,
                                 const int32_t *__restrict__ input_pos,
                                 const int32_t *__restrict__ table, int B,
                                 int n_slots, int max_pages, int page_size,
                                 int n_pages, uint4 *__restrict__ k_cache,
                                 uint4 *__restrict__ v_cache, int Hkv,
                                 int chunks_per_head, long long row_stride,
                                 long long head_stride, int32_t *err) {
  pkv_wait_prior_grid();
  pkv_allow_next_grid();
  // linear index over [2 (k|v)][B][Hkv][chunks_per_head]
  long long per_tensor = 1LL * B * Hkv * chunks_per_head;
  long long i = blockIdx.x * 1LL * blockDim.x + threadIdx.x;
  if (i >= 2 * per_tensor) return;
  const bool is_v = i >= per_tensor;
  long long j = is_v ? i - per_tensor : i;
  int c = static_cast<int>(j % chunks_per_head);
  long long bh = j / chunks_per_head;
  int h = static_cast<int>(bh % Hkv);
  int b = static_cast<int>(bh / Hkv);

  int slot = batch_idx ? batch_idx[b] : b;
  int pos = input_pos[b];
  // only one thread per row reports, so each bad row sets its bit once
  const bool reporter = (!is_v && h == 0 && c == 0);
  if (slot < 0 || slot >= n_slots) {
    if (reporter) report(err, PKV_ERR_SLOT);
    return;
  }
  if (pos < 0 || pos / page_size >= max_pages) {
    if (reporter) report(err, PKV_ERR_POS);
    return;
  }
  int page = table[static_cast<long long>(slot) * max_pages + pos / page_size];
  if (page < 0) {
    if (reporter) report(err, PKV_ERR_PAGE_NEG);
    return;
  }
  if (page >= n_pages) {
    if (reporter) report(err, PKV_ERR_PAGE_RANGE);
    return;
  }
  long long row = 1LL * page * page_size + pos % page_size;
  long long dst = ((1LL * h * n_pages * page_size) + row) * chunks_per_head + c;
  const long long srci = b * row_stride + h * head_stride + c;
  if (is_v)
    v_cache[dst] = v[srci];
  else
    k_cache[dst] = k[srci];
}

}  // namespace

namespace {

int launch_append(const pkv_bf16 *k, const pkv_bf16 *v, const int32_t *batch_idx,
                  const int32_t *input_pos, int B, const int32_t *dev_table, int n_slots,
                  int max_pages_per_seq, int page_size, int n_pages, pkv_bf16 *k_cache,
                  pkv_bf16 *v_cache, int Hkv, int D, bool head_major, int32_t *err_word,
                  void *stream, const char *fn) {
  if (B < 0 || Hkv < 1 || D < 8 || D % 8 || page_size < 1 || n_pages < 1 ||
      n_slots < 1 || max_pages_per_seq < 1)
    return pkv::fail(PKV_E_BAD_ARG, "%s: bad shape (D must be a multiple of 8)", fn);
  if (B == 0) return pkv::ok();
  if (!k || !v || !input_pos || !dev_table || !k_cache || !v_cache)
    return pkv::fail(PKV_E_BAD_ARG, "%s: NULL tensor", fn);
  if (!pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(k_cache) ||
      !pkv::aligned16(v_cache))
    return pkv::fail(PKV_E_BAD_ARG, "%s: tensors must be 16-byte aligned", fn);
  int chunks = D / 8;
  long long total = 2LL * B * Hkv * chunks;
  int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return pkv::fail(PKV_E_BAD_ARG, "%s: too large", fn);
  const long long row_stride = head_major ? chunks : 1LL * Hkv * chunks;
  const long long head_stride = head_major ? 1LL * B * chunks : chunks;
  PKV_CUDA_CHECK(pkv::launch_pdl(
      kv_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
      static_cast<cudaStream_t>(stream), reinterpret_cast<const uint4 *>(k),
      reinterpret_cast<const uint4 *>(v), batch_idx, input_pos, dev_table, B, n_slots,
      max_pages_per_seq, page_size, n_pages, reinterpret_cast<uint4 *>(k_cache),
      reinterpret_cast<uint4 *>(v_cache), Hkv, chunks, row_stride, head_stride, err_word));
  return pkv::ok();
}

}  // namespace

extern "C" int kv_append(const pkv_bf16 *k, const pkv_bf16 *v,
                         const int32_t *batch_idx, const int32_t *input_pos,
                         int B, const int32_t *dev_table, int n_slots,
                         int max_pages_per_seq, int page_size, int n_pages,
                         pkv_bf16 *k_cache, pkv_bf16 *v_cache, int Hkv, int D,
                         int32_t *err_word, void *stream) {
  return launch_append(k, v, batch_idx, input_pos, B, dev_table, n_slots, max_pages_per_seq,
                       page_size, n_pages, k_cache, v_cache, Hkv, D, false, err_word, stream,
                       "kv_append");
}

extern "C" int kv_append_prefill(const pkv_bf16 *k, const pkv_bf16 *v,
                                 const int32_t *batch_idx, const int32_t *input_pos, int L,
                                 const int32_t *dev_table, int n_slots,
                                 int max_pages_per_seq, int page_size, int n_pages,
                                 pkv_bf16 *k_cache, pkv_bf16 *v_cache, int Hkv, int D,
                                 int32_t *err_word, void *stream) {
  return launch_append(k, v, batch_idx, input_pos, L, dev_table, n_slots, max_pages_per_seq,
                       page_size, n_pages, k_cache, v_cache, Hkv, D, true, err_word, stream,
                       "kv_append_prefill");
}
