"""Document-causal prefill attention over packed tokens (oracle).

TEST INFRASTRUCTURE ONLY. Follows "unsloth: compare
main...transformers-continuous-batching-qwen3" ·
scripts/benchmarks/flex_paged_attention.py ·
PagedKVCache.create_prefill_blockmask_no_paging: L prompt tokens of several
documents are packed into one row ([1, H, L, D]); docs[t] is the document of
token t (not necessarily sorted) and the mask is

    keep (q_idx, kv_idx)  iff  q_idx >= kv_idx  and  docs[q_idx] == docs[kv_idx]

The attention runs on the packed k/v themselves ("no paging"), with GQA
(query head h reads kv head h // (Hq / Hkv)) as in the decode path:

    o[h, i] = softmax_j(scale * q[h, i] . k[g, j])  over the kept j,  times v

Every query keeps at least itself, so no row is empty.
"""
from __future__ import annotations

import numpy as np

from .attention import decode_attention_row


def prefill_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, docs, scale: float):
    """q: [Hq][L][D], k, v: [Hkv][L][D] (float), docs: [L]. Returns float64
    [Hq][L][D]. Each query row is the single-query attention over its kept
    keys, in token order."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    docs = np.asarray(docs)
    Hq, L, D = q.shape
    G = Hq // k.shape[0]
    out = np.zeros((Hq, L, D))
    for i in range(L):
        keep = np.nonzero((np.arange(L) <= i) & (docs == docs[i]))[0]
        for h in range(Hq):
            g = h // G
            out[h, i], _ = decode_attention_row(q[h, i], k[g, keep], v[g, keep], scale)
    return out
