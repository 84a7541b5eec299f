"""GQA single-token decode attention over a paged cache (oracle).

TEST INFRASTRUCTURE ONLY. Follows "unsloth: compare main...flex-moe-qwen3" ·
unsloth/inference/flex_gemma4_moe.py · the attention forward
(flex_attention(q, k, v, scale, block_mask, enable_gqa=True) with q of shape
(B, Hq, 1, D)) and the decode block masks in _decode_block_mask:

  full layers     keep key kv iff  pos >= kv
  sliding layers  keep key kv iff  pos >= kv and pos - kv < W

with pos the position of the token just appended. Written with
seq_len = pos + 1 that is keys [lo, seq_len), lo = max(0, seq_len - W) when
W > 0, else lo = 0.

Each row's pages are gathered into a contiguous float64 K, V and the output
is computed directly:  o = softmax(scale * K q)^T V,
lse = log sum_j exp(scale * k_j . q).

Readings where the pages leave a step open:
  * GQA: query head h reads kv head h // (Hq / Hkv) (grouped-contiguous, the
    enable_gqa convention);
  * a row with no key to attend (seq_len 0) or a row in the no-op slot 0
    outputs exact zeros and lse = -inf (the pages only say that skipping the
    "row has a key" check produced NaN; see the README's list of options
    that broke correctness);
  * the caller passes scale.
"""
from __future__ import annotations

import numpy as np

from .paged_kv import gather_pages


def decode_attention_row(q_row: np.ndarray, K: np.ndarray, V: np.ndarray,
                         scale: float):
    """One query head against contiguous K, V ([L][D]). Returns (o, lse)."""
    L, D = K.shape
    if L == 0:
        return np.zeros(D), -np.inf
    s = scale * (K @ q_row)
    m = np.max(s)
    p = np.exp(s - m)
    denom = np.sum(p)
    return (p @ V) / denom, m + np.log(denom)


def decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     table: np.ndarray, batch_idx, seq_lens, window: int,
                     scale: float, page_size: int):
    """q: [B][Hq][D] (float), caches: [Hkv][n_pages*page_size][D] (float),
    table: [n_slots][max_pages] int. batch_idx None means slot b for row b.

    Returns (out float64 [B][Hq][D], lse float64 [B][Hq]).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[0]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        slot = b if batch_idx is None else int(batch_idx[b])
        L = int(seq_lens[b])
        if slot == 0 or L <= 0:
            continue
        lo = max(0, L - window) if window > 0 else 0
        for g in range(Hkv):
            K = gather_pages(k_cache, table, slot, g, L, page_size)[lo:L].astype(np.float64)
            V = gather_pages(v_cache, table, slot, g, L, page_size)[lo:L].astype(np.float64)
            for h in range(g * G, (g + 1) * G):
                out[b, h], lse[b, h] = decode_attention_row(q[b, h], K, V, scale)
    return out, lse
