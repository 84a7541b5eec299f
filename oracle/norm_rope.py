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

Readings where the pages leave a step open (each is pinned by a test):
  * RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma, eps inside the root, the
    gain multiplies directly (not 1 + gamma);
  * inv_freq_i = theta^(-2i/D), i = 0 .. D/2-1 (default RoPE over the full
    head dimension);
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


def inv_freq(head_dim: int, theta: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """x: [..., D] with a leading batch axis B; pos: [B] (any real values)."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    pos = np.asarray(pos, dtype=np.float64)
    ang = pos.reshape((-1,) + (1,) * (x.ndim - 1)) * inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def qk_norm_rope(q, k, gamma_q, gamma_k, pos, theta: float, eps: float,
                 norm: bool = True):
    """q: [B][Hq][D], k: [B][Hkv][D], pos: [B]. Returns float64 (q', k')."""
    if norm:
        q = rms_norm(q, gamma_q, eps)
        k = rms_norm(k, gamma_k, eps)
    return rope(q, pos, theta), rope(k, pos, theta)
