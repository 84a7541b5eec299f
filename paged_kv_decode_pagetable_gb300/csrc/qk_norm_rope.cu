// qk_norm_rope: per-head RMSNorm followed by rotate-half RoPE, in place.
//
// Order and convention from "unsloth: compare main...flex-moe-qwen3" ·
// unsloth/inference/flex_gemma4_moe.py · attention forward (q_norm / k_norm
// on the head axis, then rotary) and Rotary helpers (rotate_half =
// cat(-x2, x1); x*cos + rotate_half(x)*sin):
//   r = x * rsqrt(mean(x^2) + eps) * gamma
//   y_i = r_i cos(phi_i) - r_{i+D/2} sin(phi_i)
//   y_{i+D/2} = r_{i+D/2} cos(phi_i) + r_i sin(phi_i),  phi_i = pos*theta^(-2i/D)
//
// One warp per (row, head); lane l owns the rotation pairs (i, i + D/2) for
// i = l, l + 32, ...  so each lane rotates with no exchange and the only
// cross-lane step is the sum of squares. fp32 math, one rounding to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace {

constexpr int kMaxPairsPerLane = 16;  // D <= 1024

__global__ void qk_norm_rope_kernel(__nv_bfloat16 *__restrict__ q,
                                    __nv_bfloat16 *__restrict__ k,
                                    const __nv_bfloat16 *__restrict__ gq,
                                    const __nv_bfloat16 *__restrict__ gk,
                                    const int32_t *__restrict__ pos,
                                    float log2_theta, float eps, int B, int Hq,
                                    int Hkv, int D) {
  pkv_grid_dependency_sync();
  const int warps_per_block = blockDim.x >> 5;
  const long long w = blockIdx.x * 1LL * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int H = Hq + Hkv;
  if (w >= 1LL * B * H) return;
  const int b = static_cast<int>(w / H);
  const int h = static_cast<int>(w % H);
  const bool is_q = h < Hq;
  __nv_bfloat16 *x = is_q ? q + (1LL * b * Hq + h) * D
                          : k + (1LL * b * Hkv + (h - Hq)) * D;
  const __nv_bfloat16 *g = is_q ? gq : gk;
  const int half = D >> 1;

  float lo[kMaxPairsPerLane], hi[kMaxPairsPerLane];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxPairsPerLane; ++j) {
    int i = lane + 32 * j;
    if (i < half) {
      lo[j] = __bfloat162float(x[i]);
      hi[j] = __bfloat162float(x[i + half]);
      ss = fmaf(lo[j], lo[j], ss);
      ss = fmaf(hi[j], hi[j], ss);
    }
  }
  float inv_rms = 1.f;
  if (g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    inv_rms = rsqrtf(ss / static_cast<float>(D) + eps);
  }
  const float p = static_cast<float>(pos[b]);
#pragma unroll
  for (int j = 0; j < kMaxPairsPerLane; ++j) {
    int i = lane + 32 * j;
    if (i < half) {
      float r1 = lo[j], r2 = hi[j];
      if (g) {
        r1 = r1 * inv_rms * __bfloat162float(g[i]);
        r2 = r2 * inv_rms * __bfloat162float(g[i + half]);
      }
      // theta^(-2i/D) = 2^(-(2i/D) log2 theta)
      float inv_freq = exp2f(-(2.0f * i / static_cast<float>(D)) * log2_theta);
      float s, c;
      sincosf(p * inv_freq, &s, &c);
      x[i] = __float2bfloat16_rn(r1 * c - r2 * s);
      x[i + half] = __float2bfloat16_rn(r2 * c + r1 * s);
    }
  }
}

}  // namespace

extern "C" int qk_norm_rope(pkv_bf16 *q, pkv_bf16 *k, const pkv_bf16 *gamma_q,
                            const pkv_bf16 *gamma_k, const int32_t *pos,
                            float theta, float eps, int B, int Hq, int Hkv,
                            int D, void *stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || D < 2 || D % 2 || D > 64 * kMaxPairsPerLane)
    return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope: bad shape (D even, <= 1024)");
  if (!(theta > 0.f)) return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope: theta must be > 0");
  if (!(eps >= 0.f)) return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope: eps must be >= 0");
  if (Hkv > 0 && (gamma_q == nullptr) != (gamma_k == nullptr))
    return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope: give both gains or neither");
  if (B == 0 || Hq + Hkv == 0) return pkv::ok();
  if (!pos || (Hq && !q) || (Hkv && !k))
    return pkv::fail(PKV_E_BAD_ARG, "qk_norm_rope: NULL tensor");
  const long long warps = 1LL * B * (Hq + Hkv);
  const int threads = 256, wpb = threads / 32;
  long long blocks = (warps + wpb - 1) / wpb;
  PKV_CUDA_CHECK(pkv::launch_pdl(
      qk_norm_rope_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
      static_cast<cudaStream_t>(stream), reinterpret_cast<__nv_bfloat16 *>(q),
      reinterpret_cast<__nv_bfloat16 *>(k), reinterpret_cast<const __nv_bfloat16 *>(gamma_q),
      reinterpret_cast<const __nv_bfloat16 *>(gamma_k), pos, log2f(theta), eps, B, Hq, Hkv,
      D));
  return pkv::ok();
}
