// qk_norm_rope: per-head RMSNorm followed by rotate-half RoPE, in place.
//
// The arithmetic (fp32, one rounding to bf16) is pkv_norm_rope_lane in
// norm_rope.cuh, shared with the fused decode step. One warp per (row, head).
// qk_norm_rope_append fuses the decode K/V scatter of "unsloth: compare
// main...transformers-continuous-batching-qwen3" · flex_paged_attention.py ·
// PageTable.assign into the same pass (write-then-attend order of the
// attention forward).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "norm_rope.cuh"
#include "pkv_internal.h"

namespace {

constexpr int kMaxPairsPerLane = 16;  // D <= 1024

__device__ __forceinline__ void norm_rope_warp(const __nv_bfloat16 *__restrict__ x,
                                               const __nv_bfloat16 *__restrict__ g, float p,
                                               float log2_theta, int rot_pairs, float eps, int D,
                                               int lane, float (&lo)[kMaxPairsPerLane],
                                               float (&hi)[kMaxPairsPerLane]) {
  pkv_norm_rope_lane<kMaxPairsPerLane>(x, g, p, log2_theta, rot_pairs, eps, D, lane, lo, hi);
}

// One warp per (row, head) over the q heads, the k heads and (when v is
// given) the v heads: q and k get norm + rotary on the leading rot_pairs
// pairs; v gets the gain-free RMSNorm.
__global__ void qk_norm_rope_kernel(__nv_bfloat16 *__restrict__ q,
                                    __nv_bfloat16 *__restrict__ k,
                                    __nv_bfloat16 *__restrict__ v,
                                    const __nv_bfloat16 *__restrict__ gq,
                                    const __nv_bfloat16 *__restrict__ gk,
                                    const int32_t *__restrict__ pos,
                                    float log2_theta, float eps, int rot_pairs, int B, int Hq,
                                    int Hkv, int D) {
  pkv_wait_prior_grid();
  pkv_allow_next_grid();
  const int warps_per_block = blockDim.x >> 5;
  const long long w = blockIdx.x * 1LL * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int H = Hq + Hkv + (v ? Hkv : 0);
  if (w >= 1LL * B * H) return;
  const int b = static_cast<int>(w / H);
  const int h = static_cast<int>(w % H);
  const int half = D >> 1;
  float lo[kMaxPairsPerLane], hi[kMaxPairsPerLane];
  __nv_bfloat16 *x;
  if (h < Hq + Hkv) {
    const bool is_q = h < Hq;
    x = is_q ? q + (1LL * b * Hq + h) * D : k + (1LL * b * Hkv + (h - Hq)) * D;
    norm_rope_warp(x, is_q ? gq : gk, static_cast<float>(pos[b]), log2_theta, rot_pairs, eps, D,
                   lane, lo, hi);
  } else {
    x = v + (1LL * b * Hkv + (h - Hq - Hkv)) * D;
    pkv_rms_norm_lane<kMaxPairsPerLane>(x, eps, D, lane, lo, hi);
  }
#pragma unroll
  for (int j = 0; j < kMaxPairsPerLane; ++j) {
    int i = lane + 32 * j;
    if (i < half) {
      x[i] = __float2bfloat16_rn(lo[j]);
      x[i + half] = __float2bfloat16_rn(hi[j]);
    }
  }
}

// qk_norm_rope followed by kv_append in one pass: query heads are rotated in
// place; a kv head's rotated k is written back to k and, with v, straight to
// its cache row (the scatter address of kv_append, same checks and error
// bits). The table entry is the only dependent load and it overlaps the
// norm/rotary arithmetic.
__global__ void qk_norm_rope_append_kernel(
    __nv_bfloat16 *__restrict__ q, __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ gq,
    const __nv_bfloat16 *__restrict__ gk, const int32_t *__restrict__ batch_idx,
    const int32_t *__restrict__ pos, float log2_theta, float eps, int B, int Hq, int Hkv,
    int D, const int32_t *__restrict__ table, int n_slots, int max_pages, int page_size,
    int n_pages, __nv_bfloat16 *__restrict__ k_cache, __nv_bfloat16 *__restrict__ v_cache,
    int32_t *__restrict__ err) {
  pkv_wait_prior_grid();
  const int warps_per_block = blockDim.x >> 5;
  const long long w = blockIdx.x * 1LL * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int H = Hq + Hkv;
  if (w >= 1LL * B * H) return;
  const int b = static_cast<int>(w / H);
  const int h = static_cast<int>(w % H);
  const bool is_q = h < Hq;
  const int half = D >> 1;
  const int pb = pos[b];
  if (is_q) {
    __nv_bfloat16 *x = q + (1LL * b * Hq + h) * D;
    float lo[kMaxPairsPerLane], hi[kMaxPairsPerLane];
    norm_rope_warp(x, gq, static_cast<float>(pb), log2_theta, D / 2, eps, D, lane, lo, hi);
#pragma unroll
    for (int j = 0; j < kMaxPairsPerLane; ++j) {
      int i = lane + 32 * j;
      if (i < half) {
        x[i] = __float2bfloat16_rn(lo[j]);
        x[i + half] = __float2bfloat16_rn(hi[j]);
      }
    }
    return;
  }
  const int hk = h - Hq;
  // scatter address (issued before the arithmetic so the table load overlaps it)
  const int slot = batch_idx ? batch_idx[b] : b;
  int bits = 0, page = -1;
  if (slot < 0 || slot >= n_slots) {
    bits = PKV_ERR_SLOT;
  } else if (pb < 0 || pb / page_size >= max_pages) {
    bits = PKV_ERR_POS;
  } else {
    page = table[static_cast<long long>(slot) * max_pages + pb / page_size];
  }
  __nv_bfloat16 *x = k + (1LL * b * Hkv + hk) * D;
  const __nv_bfloat16 *vx = v + (1LL * b * Hkv + hk) * D;
  float lo[kMaxPairsPerLane], hi[kMaxPairsPerLane];
  norm_rope_warp(x, gk, static_cast<float>(pb), log2_theta, D / 2, eps, D, lane, lo, hi);
  if (!bits) {
    if (page < 0) bits = PKV_ERR_PAGE_NEG;
    else if (page >= n_pages) bits = PKV_ERR_PAGE_RANGE;
  }
  if (bits && hk == 0 && lane == 0 && err) atomicOr(err, bits);
  const long long row = 1LL * page * page_size + pb % page_size;
  __nv_bfloat16 *kc = k_cache + ((1LL * hk * n_pages * page_size) + row) * D;
  __nv_bfloat16 *vc = v_cache + ((1LL * hk * n_pages * page_size) + row) * D;
#pragma unroll
  for (int j = 0; j < kMaxPairsPerLane; ++j) {
    int i = lane + 32 * j;
    if (i < half) {
      const __nv_bfloat16 a = __float2bfloat16_rn(lo[j]), c = __float2bfloat16_rn(hi[j]);
      x[i] = a;
      x[i + half] = c;
      if (!bits) {
        kc[i] = a;
        kc[i + half] = c;
        vc[i] = vx[i];
        vc[i + half] = vx[i + half];
      }
    }
  }
}

}  // namespace

namespace {

int launch_qkv(pkv_bf16 *q, pkv_bf16 *k, pkv_bf16 *v, const pkv_bf16 *gamma_q,
               const pkv_bf16 *gamma_k, const int32_t *pos, float theta, float eps,
               int rotary_dims, int B, int Hq, int Hkv, int D, void *stream, const char *fn) {
  if (B < 0 || Hq < 0 || Hkv < 0 || D < 2 || D % 2 || D > 64 * kMaxPairsPerLane)
    return pkv::fail(PKV_E_BAD_ARG, "%s: bad shape (D even, <= 1024)", fn);
  if (rotary_dims < 0 || rotary_dims > D || rotary_dims % 2)
    return pkv::fail(PKV_E_BAD_ARG, "%s: rotary_dims must be even and in [0, D]", fn);
  if (!(theta > 0.f)) return pkv::fail(PKV_E_BAD_ARG, "%s: theta must be > 0", fn);
  if (!(eps >= 0.f)) return pkv::fail(PKV_E_BAD_ARG, "%s: eps must be >= 0", fn);
  if (Hkv > 0 && (gamma_q == nullptr) != (gamma_k == nullptr))
    return pkv::fail(PKV_E_BAD_ARG, "%s: give both gains or neither", fn);
  const int H = Hq + Hkv + (v ? Hkv : 0);
  if (B == 0 || H == 0) return pkv::ok();
  if (!pos || (Hq && !q) || (Hkv && !k))
    return pkv::fail(PKV_E_BAD_ARG, "%s: NULL tensor", fn);
  const long long warps = 1LL * B * H;
  const int threads = 256, wpb = threads / 32;
  long long blocks = (warps + wpb - 1) / wpb;
  PKV_CUDA_CHECK(pkv::launch_pdl(
      qk_norm_rope_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
      static_cast<cudaStream_t>(stream), reinterpret_cast<__nv_bfloat16 *>(q),
      reinterpret_cast<__nv_bfloat16 *>(k), reinterpret_cast<__nv_bfloat16 *>(v),
      reinterpret_cast<const __nv_bfloat16 *>(gamma_q),
      reinterpret_cast<const __nv_bfloat16 *>(gamma_k), pos, log2f(theta), eps,
      rotary_dims / 2, B, Hq, Hkv, D));
  return pkv::ok();
}

}  // namespace

extern "C" int qk_norm_rope(pkv_bf16 *q, pkv_bf16 *k, const pkv_bf16 *gamma_q,
                            const pkv_bf16 *gamma_k, const int32_t *pos,
                            float theta, float eps, int B, int Hq, int Hkv,
                            int D, void *stream) {
  return launch_qkv(q, k, nullptr, gamma_q, gamma_k, pos, theta, eps, D, B, Hq, Hkv, D, stream,
                    "qk_norm_rope");
}

extern "C" int qkv_norm_rope(pkv_bf16 *q, pkv_bf16 *k, pkv_bf16 *v, const pkv_bf16 *gamma_q,
                             const pkv_bf16 *gamma_k, const int32_t *pos, float theta,
                             float eps, int rotary_dims, int B, int Hq, int Hkv, int D,
                             void *stream) {
  return launch_qkv(q, k, v, gamma_q, gamma_k, pos, theta, eps, rotary_dims, B, Hq, Hkv, D,
                    stream, "qkv_norm_rope");
}

extern "C" int qk_norm_rope_append(pkv_bf16 *q, pkv_bf16 *k, const pkv_bf16 *v,
                                   const pkv_bf16 *gamma_q, const pkv_bf16 *gamma_k,
                                   const int32_t *batch_idx, const int32_t *input_pos,
                                   float theta, float eps, int B, int Hq, int Hkv, int D,
                                   const int32_t *dev_table, int n_slots,
                                   int max_pages_per_seq, int page_size, int n_pages,
                                   pkv_bf16 *k_cache, pkv_bf16 *v_cache, int32_t *err_word,
                                   void *stream) {
  if (B < 0 || Hq < 0 || Hkv < 1 || D < 2 || D % 2 || D > 64 * kMaxPairsPerLane)
    return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope_append: bad shape (Hkv >= 1, D even, <= 1024)");
  if (page_size < 1 || n_pages < 1 || n_slots < 1 || max_pages_per_seq < 1)
    return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope_append: bad table geometry");
  if (!(theta > 0.f)) return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope_append: theta must be > 0");
  if (!(eps >= 0.f)) return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope_append: eps must be >= 0");
  if ((gamma_q == nullptr) != (gamma_k == nullptr))
    return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope_append: give both gains or neither");
  if (B == 0) return pkv::ok();
  if (!input_pos || (Hq && !q) || !k || !v || !dev_table || !k_cache || !v_cache)
    return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope_append: NULL tensor");
  const long long warps = 1LL * B * (Hq + Hkv);
  const int threads = 256, wpb = threads / 32;
  long long blocks = (warps + wpb - 1) / wpb;
  PKV_CUDA_CHECK(pkv::launch_pdl(
      qk_norm_rope_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
      static_cast<cudaStream_t>(stream), reinterpret_cast<__nv_bfloat16 *>(q),
      reinterpret_cast<__nv_bfloat16 *>(k), reinterpret_cast<const __nv_bfloat16 *>(v),
      reinterpret_cast<const __nv_bfloat16 *>(gamma_q),
      reinterpret_cast<const __nv_bfloat16 *>(gamma_k), batch_idx, input_pos, log2f(theta),
      eps, B, Hq, Hkv, D, dev_table, n_slots, max_pages_per_seq, page_size, n_pages,
      reinterpret_cast<__nv_bfloat16 *>(k_cache), reinterpret_cast<__nv_bfloat16 *>(v_cache),
      err_word));
  return pkv::ok();
}
