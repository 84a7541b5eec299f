"""Document-causal prefill attention and its block mask over packed tokens (oracle).

TEST INFRASTRUCTURE ONLY. Follows "unsloth: compare
main...transformers-continuous-batching-qwen3" ·
scripts/benchmarks/flex_paged_attention.py ·
PagedKVCache.create_prefill_blockmask_no_paging, and the Gemma-4 inference
script's _create_prefill_sliding_blockmask: L prompt tokens of several
documents are packed into one row ([1, H, L, D]); docs[t] is the document of
token t (not necessarily sorted) and the mask is

    keep (q_idx, kv_idx)  iff  q_idx >= kv_idx  and  docs[q_idx] == docs[kv_idx]
                               [and q_idx - kv_idx < W for a sliding layer]

The attention runs on the packed k/v themselves ("no paging"), with GQA
(query head h reads kv head h // (Hq / Hkv)) as in the decode path:

    o[h, i] = softmax_j(scale * q[h, i] . k[g, j])  over the kept j,  times v

Every query keeps at least itself, so no row is empty.

The block mask is the tiled summary of that mask which create_block_mask
makes: the L x L square is cut into blocks of `block` query rows by `block`
keys (the last row and column of blocks run past L). Per query block it lists,
in ascending order, the key blocks that are FULL (every one of the block's
block x block pairs lies inside L and is kept) and, apart from those, the key
blocks that are PARTIAL (at least one pair inside L is kept). A key block with
no kept pair is in neither list.
"""
from __future__ import annotations

import numpy as np

from .attention import decode_attention_row


def keep_matrix(docs, window: int = 0) -> np.ndarray:
    """The L x L boolean mask: [i, j] is True iff query i keeps key j."""
    docs = np.asarray(docs)
    L = len(docs)
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    keep = (i >= j) & (docs[:, None] == docs[None, :])
    if window > 0:
        keep &= j > i - window          # i - j < W, without an L x L integer temporary
    return keep


def prefill_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, docs, scale: float,
                      window: int = 0):
    """q: [Hq][L][D], k, v: [Hkv][L][D] (float), docs: [L]; window 0 = none.
    Returns float64 [Hq][L][D]. Each query row is the single-query attention
    over its kept keys, in token order."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    keep = keep_matrix(docs, window)
    Hq, L, D = q.shape
    G = Hq // k.shape[0]
    out = np.zeros((Hq, L, D))
    for i in range(L):
        js = np.nonzero(keep[i])[0]
        for h in range(Hq):
            g = h // G
            out[h, i], _ = decode_attention_row(q[h, i], k[g, js], v[g, js], scale)
    return out


def prefill_block_mask(docs, block: int, window: int = 0):
    """Block mask of the document-causal (optionally sliding) mask.

    Returns (kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices):
    the counts are int arrays of length n = ceil(L / block); the index lists
    are Python lists of n ascending int lists (partial and full blocks)."""
    keep = keep_matrix(docs, window)
    L = keep.shape[0]
    n = -(-L // block)
    pad = n * block
    kept = np.zeros((pad, pad), dtype=bool)
    kept[:L, :L] = keep
    inside = np.zeros((pad, pad), dtype=bool)
    inside[:L, :L] = True
    # [qb, r, kb, c] -> per (qb, kb): any kept pair / every pair inside and kept
    kb4 = kept.reshape(n, block, n, block)
    ib4 = inside.reshape(n, block, n, block)
    any_kept = kb4.any(axis=(1, 3))
    full = (kb4 & ib4).all(axis=(1, 3))
    partial = any_kept & ~full
    kv_idx = [[int(x) for x in np.nonzero(partial[qb])[0]] for qb in range(n)]
    full_idx = [[int(x) for x in np.nonzero(full[qb])[0]] for qb in range(n)]
    return (np.array([len(x) for x in kv_idx], dtype=np.int64), kv_idx,
            np.array([len(x) for x in full_idx], dtype=np.int64), full_idx)
