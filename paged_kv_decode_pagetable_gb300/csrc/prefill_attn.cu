// prefill_block_mask + prefill_attn: document-causal attention over packed
// prefill tokens, driven by a block mask.
//
// Semantics: "unsloth: compare main...transformers-continuous-batching-qwen3"
// · scripts/benchmarks/flex_paged_attention.py ·
// PagedKVCache.create_prefill_blockmask_no_paging, and the sliding variant
// _create_prefill_sliding_blockmask of the Gemma-4 inference script. L prompt
// tokens of several documents are packed into one row; docs[t] is the
// document of token t (in any order) and query i keeps key j iff j <= i,
// docs[j] == docs[i] and, with a window W > 0, i - j < W. The attention runs
// on the packed q, k, v themselves ("no paging"), with GQA (query head h
// reads kv head h / (Hq / Hkv)).
//
// The block mask is the tiled summary create_block_mask makes of that mask,
// at 64 query rows x 64 keys: per query block, the ascending lists of FULL key
// blocks (all 64 x 64 pairs inside L and kept: no masking needed) and PARTIAL
// ones (some pair kept). It depends only on docs and W, so one build serves
// every layer and head of a batch. prefill_block_mask_kernel: one CTA per
// query block; each thread summarises one key block's document range, the
// blocks whose range meets the query block's are tested pair by pair by a
// warp (ballots), and the flags are compacted in ascending order by ballot
// prefix counts.
//
// The attention itself is prefill_tc_kernel (prefill_tc.cu): tcgen05 MMAs
// with TMEM accumulators, fed by TMA, over the listed blocks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "pkv_internal.h"

namespace {

constexpr int kBM = 64;   // query rows of a block
constexpr int kBN = 64;   // keys of a block

// ---------------------------------------------------------------------------
// Block mask builder
// ---------------------------------------------------------------------------
constexpr int kMThreads = 128;   // key blocks summarised per pass

__global__ void __launch_bounds__(kMThreads)
    prefill_block_mask_kernel(const int32_t *__restrict__ docs, int L, int n, int window,
                              int32_t *__restrict__ kv_num, int32_t *__restrict__ kv_idx,
                              int32_t *__restrict__ full_num, int32_t *__restrict__ full_idx) {
  __shared__ int s_qd[kBM];
  __shared__ int s_cand[kMThreads];
  __shared__ uint8_t s_flag[kMThreads];
  __shared__ int s_ncand, s_qlo, s_qhi;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pkv_wait_prior_grid();
  pkv_allow_next_grid();
  const int qb = blockIdx.x, row0 = qb * kBM;
  const int nq = min(kBM, L - row0);
  if (tid < kBM) s_qd[tid] = tid < nq ? docs[row0 + tid] : 0;
  __syncthreads();
  if (warp == 0) {   // document range of the query block's rows inside L
    int lo = 2147483647, hi = -2147483647 - 1;
    for (int r = lane; r < nq; r += 32) {
      lo = min(lo, s_qd[r]);
      hi = max(hi, s_qd[r]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      s_qlo = lo;
      s_qhi = hi;
    }
  }
  // rows of this block that are inside L: lane and lane + 32
  const int qd0 = s_qd[lane], qd1 = s_qd[lane + 32];
  const int qi0 = row0 + lane, qi1 = qi0 + 32;
  const bool qv0 = lane < nq, qv1 = lane + 32 < nq;
  int kb_lo = 0;   // no key before row0 - W + 1 is kept
  if (window > 0 && row0 - window + 1 > 0) kb_lo = (row0 - window + 1) / kBN;
  int np = 0, nf = 0;   // list lengths so far (kept by warp 0)
  int32_t *prow = kv_idx + static_cast<size_t>(qb) * n;
  int32_t *frow = full_idx + static_cast<size_t>(qb) * n;
  for (int c0 = kb_lo; c0 <= qb; c0 += kMThreads) {
    if (tid == 0) s_ncand = 0;
    s_flag[tid] = 0;
    __syncthreads();   // s_qlo / s_qhi visible; s_ncand reset
    const int kb = c0 + tid;
    if (kb <= qb) {
      const int j0 = kb * kBN, nk = min(kBN, L - j0);
      int lo = 2147483647, hi = -2147483647 - 1;
      for (int r = 0; r < nk; ++r) {
        const int d = __ldg(docs + j0 + r);
        lo = min(lo, d);
        hi = max(hi, d);
      }
      if (lo <= s_qhi && s_qlo <= hi) s_cand[atomicAdd(&s_ncand, 1)] = kb;
    }
    __syncthreads();
    const int nc = s_ncand;
    for (int c = warp; c < nc; c += kMThreads / 32) {   // exact test, one warp per block
      const int kbc = s_cand[c], j0 = kbc * kBN;
      const bool kv0 = j0 + lane < L, kv1 = j0 + lane + 32 < L;
      const int kd0 = kv0 ? docs[j0 + lane] : 0, kd1 = kv1 ? docs[j0 + lane + 32] : 0;
      bool any = false, all = nq == kBM && j0 + kBN <= L;
#pragma unroll 4
      for (int t = 0; t < kBN; ++t) {
        const int kd = __shfl_sync(0xffffffffu, t < 32 ? kd0 : kd1, t & 31);
        const int j = j0 + t;
        const bool in = j < L;
        const bool k0 = qv0 && in && j <= qi0 && kd == qd0 && (window == 0 || qi0 - j < window);
        const bool k1 = qv1 && in && j <= qi1 && kd == qd1 && (window == 0 || qi1 - j < window);
        any |= k0 || k1;
        all &= k0 && k1;
      }
      any = __any_sync(0xffffffffu, any);
      all = __all_sync(0xffffffffu, all);
      if (lane == 0) s_flag[kbc - c0] = all ? 2 : (any ? 1 : 0);
    }
    __syncthreads();
    if (warp == 0) {   // ascending compaction of this pass's flags
      const unsigned lt = (1u << lane) - 1u;
#pragma unroll
      for (int g = 0; g < kMThreads / 32; ++g) {
        const int kbg = c0 + g * 32 + lane;
        const int f = kbg <= qb ? s_flag[g * 32 + lane] : 0;
        const unsigned mp = __ballot_sync(0xffffffffu, f == 1);
        const unsigned mf = __ballot_sync(0xffffffffu, f == 2);
        if (f == 1) prow[np + __popc(mp & lt)] = kbg;
        if (f == 2) frow[nf + __popc(mf & lt)] = kbg;
        np += __popc(mp);
        nf += __popc(mf);
      }
    }
    __syncthreads();   // flags and candidates are rewritten by the next pass
  }
  if (tid == 0) {
    kv_num[qb] = np;
    full_num[qb] = nf;
  }
}

}  // namespace

extern "C" int prefill_block_mask(const int32_t *docs, int L, int window,
                                  int32_t *kv_num_blocks, int32_t *kv_indices,
                                  int32_t *full_kv_num_blocks, int32_t *full_kv_indices,
                                  void *stream) {
  if (L < 0 || L > 0x7fffffff - kBM || window < 0)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_block_mask: bad L or window");
  if (L == 0) return pkv::ok();
  if (!docs || !kv_num_blocks || !kv_indices || !full_kv_num_blocks || !full_kv_indices)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_block_mask: NULL pointer");
  const int n = (L + kBM - 1) / kBM;
  PKV_CUDA_CHECK(pkv::launch_pdl(prefill_block_mask_kernel, dim3(n), dim3(kMThreads), 0,
                                 static_cast<cudaStream_t>(stream), docs, L, n, window,
                                 kv_num_blocks, kv_indices, full_kv_num_blocks,
                                 full_kv_indices));
  return pkv::ok();
}

extern "C" int prefill_attn(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                            const int32_t *docs, const int32_t *kv_num_blocks,
                            const int32_t *kv_indices, const int32_t *full_kv_num_blocks,
                            const int32_t *full_kv_indices, int L, int Hq, int Hkv, int D,
                            int window, float scale, pkv_bf16 *out, void *stream) {
  if (D != 64 && D != 128 && D != 256 && D != 512)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: D must be 64, 128, 256 or 512");
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: need Hq %% Hkv == 0");
  if (L < 0 || L > 0x7fffffff - kBM || Hq > 65535 || window < 0)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: bad size or window");
  // work items of 128 query rows, one head and (D = 512) one output half are
  // counted in 32 bits
  if (1LL * ((L + 2 * kBM - 1) / (2 * kBM)) * Hq * (D == 512 ? 2 : 1) > 0x7fffffffLL)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: L x Hq too large");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: scale must be finite and > 0");
  if (L == 0) return pkv::ok();
  if (!q || !k || !v || !docs || !out || !kv_num_blocks || !kv_indices || !full_kv_num_blocks ||
      !full_kv_indices)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: NULL pointer");
  if (!pkv::aligned16(q) || !pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(out) ||
      !pkv::aligned16(docs))
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: tensors and docs must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
#define PKV_PREFILL(FN, DD)                                                                  \
  pkv::FN<DD>(q, k, v, docs, kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices, L, \
              Hq, Hkv, window, scale, out, s)
  const int st = D == 64    ? PKV_PREFILL(launch_prefill_tc, 64)
                 : D == 128 ? PKV_PREFILL(launch_prefill_tc, 128)
                 : D == 256 ? PKV_PREFILL(launch_prefill_wide, 256)
                            : PKV_PREFILL(launch_prefill_wide, 512);
#undef PKV_PREFILL
  if (st != PKV_OK) return st;
  return pkv::ok();
}
