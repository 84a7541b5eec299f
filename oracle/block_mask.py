"""Logical -> physical block-mask conversion (oracle; test infrastructure only).

Follows "unsloth: compare main...transformers-continuous-batching-qwen3" ·
scripts/benchmarks/flex_paged_attention.py ·
PageTable.convert_logical_block_mask: a BlockMask built over logical
positions (key blocks of page_size tokens, kv_indices of shape
[B, H, ROWS, MAX_BLOCKS]) is re-pointed at the paged cache by sending every
logical key-block index of batch row b through that row's page-table row:

    new_kv_indices[b, h, r, c] = page_table[batch_idx[b], kv_indices[b, h, r, c]]
                                  for c < MAX_BLOCKS,  0 for the columns after

The block counts are unchanged; full and partial index arrays are converted
alike. batch_idx defaults to b.

Error reading (the pages' gather raises on an index outside the table row):
an index outside [0, max_pages_per_seq) gives -1 and ERR_POS; a batch row
whose slot is outside [0, n_slots) gives -1 in all its entries and ERR_SLOT.
Table entries are copied as they are (-1 for an unreserved block included).
"""
from __future__ import annotations

import numpy as np

from .paged_kv import ERR_POS, ERR_SLOT


def convert_logical_block_mask(table: np.ndarray, kv_indices: np.ndarray, batch_idx=None,
                               n_cols: int | None = None):
    """table: int [n_slots][max_pages]; kv_indices: int [B][H][ROWS][M].
    Returns (int64 [B][H][ROWS][n_cols], error bits); n_cols defaults to
    max(M, max_pages)."""
    table = np.asarray(table)
    idx = np.asarray(kv_indices)
    n_slots, max_pages = table.shape
    B, H, R, M = idx.shape
    if n_cols is None:
        n_cols = max(M, max_pages)
    out = np.zeros((B, H, R, n_cols), dtype=np.int64)
    err = 0
    for b in range(B):
        slot = b if batch_idx is None else int(batch_idx[b])
        if slot < 0 or slot >= n_slots:
            out[b, :, :, :M] = -1
            err |= ERR_SLOT
            continue
        for h in range(H):
            for r in range(R):
                for c in range(M):
                    j = int(idx[b, h, r, c])
                    if 0 <= j < max_pages:
                        out[b, h, r, c] = table[slot, j]
                    else:
                        out[b, h, r, c] = -1
                        err |= ERR_POS
    return out, err
