// Per-head RMSNorm + rotate-half RoPE of one head vector held by a warp.
//
// Order and convention from "unsloth: compare main...flex-moe-qwen3" ·
// unsloth/inference/flex_gemma4_moe.py · attention forward (q_norm / k_norm
// on the head axis, then rotary) and Rotary helpers (rotate_half =
// cat(-x2, x1); x*cos + rotate_half(x)*sin):
//   r = x * rsqrt(mean(x^2) + eps) * gamma
//   y_i = r_i cos(phi_i) - r_{i+D/2} sin(phi_i)
//   y_{i+D/2} = r_{i+D/2} cos(phi_i) + r_i sin(phi_i),  phi_i = pos*theta^(-2i/D)
//
// Lane l owns the rotation pairs (i, i + D/2) for i = l, l + 32, ... so the
// only cross-lane step is the sum of squares. Every rounding step is spelled
// out with _rn intrinsics (no contraction left to the compiler), and the
// rotation factors (cos phi_i, sin phi_i) are a pure function of (i, D, pos,
// theta) computed by pkv_rope_factor alone, so the standalone qk_norm_rope
// kernel (factors inline) and the fused decode step (each lane's factors
// computed once per row and kept in registers) produce the same bits for the
// same input.
#pragma once

#include <cuda_bf16.h>

// Rotation factors of pair i. Pairs i >= rot_pairs are not rotated (Gemma-4
// proportional RoPE: a zero inverse frequency gives cos 1, sin 0 there).
__device__ __forceinline__ void pkv_rope_factor(int i, int D, float pos, float log2_theta,
                                                int rot_pairs, float &cs, float &sn) {
  if (i >= rot_pairs) {
    cs = 1.f;
    sn = 0.f;
    return;
  }
  // theta^(-2i/D) = 2^(-(2i/D) log2 theta)
  const float e = __fdiv_rn(2.0f * static_cast<float>(i), static_cast<float>(D));
  const float inv_freq = exp2f(-__fmul_rn(e, log2_theta));
  sincosf(__fmul_rn(pos, inv_freq), &sn, &cs);
}

// Norm + rotation with the factors supplied by factor(j, i, cs, sn) for the
// lane's j-th pair i = lane + 32 j. PAIRS >= ceil(D / 64): register slots per
// lane. x and gamma may point to global or
// shared memory; gamma == nullptr skips the norm.
template <int PAIRS, typename Factor>
__device__ __forceinline__ void pkv_norm_rope_core(const __nv_bfloat16 *x,
                                                   const __nv_bfloat16 *g, float eps, int D,
                                                   int lane, Factor factor, float (&lo)[PAIRS],
                                                   float (&hi)[PAIRS]) {
  const int half = D >> 1;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < PAIRS; ++j) {
    const int i = lane + 32 * j;
    if (i < half) {
      lo[j] = __bfloat162float(x[i]);
      hi[j] = __bfloat162float(x[i + half]);
      ss = __fmaf_rn(lo[j], lo[j], ss);
      ss = __fmaf_rn(hi[j], hi[j], ss);
    }
  }
  float inv_rms = 1.f;
  if (g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    inv_rms = rsqrtf(__fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), eps));
  }
#pragma unroll
  for (int j = 0; j < PAIRS; ++j) {
    const int i = lane + 32 * j;
    if (i < half) {
      float r1 = lo[j], r2 = hi[j];
      if (g) {
        r1 = __fmul_rn(__fmul_rn(r1, inv_rms), __bfloat162float(g[i]));
        r2 = __fmul_rn(__fmul_rn(r2, inv_rms), __bfloat162float(g[i + half]));
      }
      float cs, sn;
      factor(j, i, cs, sn);
      lo[j] = __fsub_rn(__fmul_rn(r1, cs), __fmul_rn(r2, sn));
      hi[j] = __fadd_rn(__fmul_rn(r2, cs), __fmul_rn(r1, sn));
    }
  }
}

// Factors computed inline for row position pos.
template <int PAIRS>
__device__ __forceinline__ void pkv_norm_rope_lane(const __nv_bfloat16 *x,
                                                   const __nv_bfloat16 *g, float pos,
                                                   float log2_theta, int rot_pairs, float eps,
                                                   int D, int lane, float (&lo)[PAIRS],
                                                   float (&hi)[PAIRS]) {
  pkv_norm_rope_core<PAIRS>(
      x, g, eps, D, lane,
      [&](int, int i, float &cs, float &sn) {
        pkv_rope_factor(i, D, pos, log2_theta, rot_pairs, cs, sn);
      },
      lo, hi);
}

// RMSNorm without a gain (Gemma-4 v_norm, with_scale=False): the same sum of
// squares and scale as the gained norm above, then one rounding per output.
template <int PAIRS>
__device__ __forceinline__ void pkv_rms_norm_lane(const __nv_bfloat16 *x, float eps, int D,
                                                  int lane, float (&lo)[PAIRS],
                                                  float (&hi)[PAIRS]) {
  const int half = D >> 1;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < PAIRS; ++j) {
    const int i = lane + 32 * j;
    if (i < half) {
      lo[j] = __bfloat162float(x[i]);
      hi[j] = __bfloat162float(x[i + half]);
      ss = __fmaf_rn(lo[j], lo[j], ss);
      ss = __fmaf_rn(hi[j], hi[j], ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  const float inv_rms = rsqrtf(__fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), eps));
#pragma unroll
  for (int j = 0; j < PAIRS; ++j) {
    const int i = lane + 32 * j;
    if (i < half) {
      lo[j] = __fmul_rn(lo[j], inv_rms);
      hi[j] = __fmul_rn(hi[j], inv_rms);
    }
  }
}
