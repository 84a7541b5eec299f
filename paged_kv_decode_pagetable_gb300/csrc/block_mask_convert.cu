// convert_logical_block_mask: re-points a block mask's logical key-block
// indices at the paged cache ("unsloth: compare main...transformers-
// continuous-batching-qwen3" · flex_paged_attention.py ·
// PageTable.convert_logical_block_mask):
//   out[b][h][r][c] = table[slot(b)][idx[b][h][r][c]]  for c < M,  0 after.
// One thread per output element, grid-stride; an index outside the table
// row gives -1 and PKV_ERR_POS, a slot outside [0, n_slots) gives -1 and
// PKV_ERR_SLOT (reported once per batch row).
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace {

__device__ __forceinline__ void report(int32_t *err, int bits) {
  if (err) atomicOr(err, bits);
}

__global__ void convert_block_mask_kernel(const int32_t *__restrict__ table, int n_slots,
                                          int max_pages, const int32_t *__restrict__ batch_idx,
                                          long long rows_per_b, long long total_rows, int M,
                                          const int32_t *__restrict__ idx, int n_cols,
                                          int32_t *__restrict__ out, int32_t *err) {
  pkv_wait_prior_grid();
  pkv_allow_next_grid();
  const long long total = total_rows * n_cols;
  const long long stride = 1LL * gridDim.x * blockDim.x;
  for (long long e = 1LL * blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    const long long row = e / n_cols;
    const int c = static_cast<int>(e - row * n_cols);
    int v = 0;
    if (c < M) {
      const long long b = row / rows_per_b;
      const int slot = batch_idx ? batch_idx[b] : static_cast<int>(b);
      if (slot < 0 || slot >= n_slots) {
        v = -1;
        if (c == 0 && row == b * rows_per_b) report(err, PKV_ERR_SLOT);
      } else {
        const int j = idx[row * M + c];
        if (j < 0 || j >= max_pages) {
          v = -1;
          report(err, PKV_ERR_POS);
        } else {
          v = table[1LL * slot * max_pages + j];
        }
      }
    }
    out[e] = v;
  }
}

}  // namespace

extern "C" int convert_logical_block_mask(const int32_t *dev_table, int n_slots,
                                          int max_pages_per_seq, const int32_t *batch_idx,
                                          int B, int H, int rows, int max_blocks,
                                          const int32_t *kv_indices, int n_cols,
                                          int32_t *new_kv_indices, int32_t *err_word,
                                          void *stream) {
  if (B < 0 || H < 1 || rows < 0 || max_blocks < 0 || n_cols < max_blocks || n_slots < 1 ||
      max_pages_per_seq < 1)
    return pkv::fail(PKV_E_BAD_ARG, "convert_logical_block_mask: bad shape "
                                    "(n_cols must be >= max_blocks)");
  const long long total_rows = 1LL * B * H * rows;
  if (total_rows == 0 || n_cols == 0) return pkv::ok();
  if (!dev_table || !new_kv_indices || (max_blocks > 0 && !kv_indices))
    return pkv::fail(PKV_E_BAD_ARG, "convert_logical_block_mask: NULL pointer");
  const long long total = total_rows * n_cols;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  const long long cap = 8LL * pkv::sm_count();
  if (blocks > cap) blocks = cap;
  PKV_CUDA_CHECK(pkv::launch_pdl(convert_block_mask_kernel, dim3(static_cast<unsigned>(blocks)),
                                 dim3(threads), 0, static_cast<cudaStream_t>(stream), dev_table,
                                 n_slots, max_pages_per_seq, batch_idx, 1LL * H * rows,
                                 total_rows, max_blocks, kv_indices, n_cols, new_kv_indices,
                                 err_word));
  return pkv::ok();
}
