"""Per-head RMSNorm followed by RoPE (oracle; test infrastructure only).

Order and RoPE convention follow "unsloth: compare main...flex-moe-qwen3" ·
unsloth/inference/flex_gemma4_moe.py · "Rotary helpers" (_rotate_half,
_apply_rotary_full) and the attention forward (q_norm / k_norm on the head
axis, then rotary, then the paged write). Qwen3's per-head q/k RMSNorm is the
only architecture-specific branch ("unsloth: compare
main...transformers-continuous-batching-qwen3" · README, Install).

  rotate_half(x) = concat(-x2, x1)        (x1, x2 = the two halves of D)
  rope(x)        = x * cos + rotate_half(x) * sin
  cos, sin       = cos/sin of pos * inv_freq, each frequency used for index
                   i and i + D/2

Gemma-4 variants ("unsloth: compare main...flex-moe-qwen3" · the Gemma-4
notes on two-tier RoPE, per-head Q/K/V RMSNorm and the K=V alternative, and
the Rotary helpers docstring):
  * proportional RoPE rotates the leading rotary_dims of the head dimension
    and passes the rest through; the pages realise this with an inv_freq
    whose tail entries are zero (cos = 1, sin = 0 there);
  * v_norm is RMSNorm without a gain (with_scale=False);
  * with K=V the value is the raw k projection (before k_norm and RoPE),
    followed by v_norm.

Readings where the pages leave a step open (each is pinned by a test):
  * RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma, eps inside the root, the
    gain multiplies directly (not 1 + gamma);
  * inv_freq_i = theta^(-2i/D), i = 0 .. D/2-1 (default RoPE over the full
    head dimension);
  * proportional RoPE keeps those frequencies for the rotated pairs
    i < rotary_dims/2 and sets the rest to zero (the pages name only the
    zeros, not a rescaled exponent);
  * everything is float64 here; the GPU computes in fp32 and rounds once.
"""
from __future__ import annotations

import numpy as np


def rms_norm(x: np.ndarray, gamma: np.ndarray | None, eps: float) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    y = x / np.sqrt(ms + eps)
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64)
    return y


def inv_freq(head_dim: int, theta: float, rotary_dims: int | None = None) -> np.ndarray:
    """theta^(-2i/D) for the rotated pairs i < rotary_dims/2, zero after."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    f = np.power(float(theta), -2.0 * i / head_dim)
    if rotary_dims is not None:
        f[i >= rotary_dims // 2] = 0.0
    return f


def rope(x: np.ndarray, pos, theta: float, rotary_dims: int | None = None) -> np.ndarray:
    """x: [..., D] with a leading batch axis B; pos: [B] (any real values)."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    pos = np.asarray(pos, dtype=np.float64)
    ang = pos.reshape((-1,) + (1,) * (x.ndim - 1)) * inv_freq(D, theta, rotary_dims)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def qk_norm_rope(q, k, gamma_q, gamma_k, pos, theta: float, eps: float,
                 norm: bool = True, rotary_dims: int | None = None):
    """q: [B][Hq][D], k: [B][Hkv][D], pos: [B]. Returns float64 (q', k')."""
    if norm:
        q = rms_norm(q, gamma_q, eps)
        k = rms_norm(k, gamma_k, eps)
    return rope(q, pos, theta, rotary_dims), rope(k, pos, theta, rotary_dims)


def v_norm(v: np.ndarray, eps: float) -> np.ndarray:
    """Scale-free RMSNorm of each head vector: v / sqrt(mean(v^2) + eps)."""
    return rms_norm(v, None, eps)
