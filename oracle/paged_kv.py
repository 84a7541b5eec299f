"""Decode K/V scatter and page gather (oracle; test infrastructure only).

Follows "unsloth: compare main...transformers-continuous-batching-qwen3" ·
scripts/benchmarks/flex_paged_attention.py · PagedKVCache (cache shape
(1, H, n_pages * page_size, D)) and PageTable.assign (find address):

    block  = input_pos // page_size
    offset = input_pos %  page_size
    row    = page_table[batch_idx, block] * page_size + offset
    cache[:, h, row, :] = value[b, h, :]

Caches here are [H][n_pages * page_size][D] arrays of any element type; the
scatter copies elements unchanged, so bf16 bit patterns (uint16) round-trip
exactly.

Error bits (a reading: the pages raise on bad shapes but say nothing about a
bad table entry during decode). Each invalid token write is skipped and
reported:
    ERR_POS        position negative or beyond the table row
    ERR_PAGE_RANGE table entry >= n_pages
    ERR_PAGE_NEG   table entry < 0 (unreserved block)
    ERR_SLOT       batch index outside [0, n_slots)
"""
from __future__ import annotations

import numpy as np

ERR_POS = 1
ERR_PAGE_RANGE = 2
ERR_PAGE_NEG = 4
ERR_SLOT = 8


def physical_row(table: np.ndarray, slot: int, pos: int, page_size: int) -> int:
    """Physical cache row of logical token `pos` of `slot` (no checks)."""
    page = int(table[slot, pos // page_size])
    return page * page_size + pos % page_size


def _checked_row(table, slot, pos, page_size, n_pages):
    n_slots, max_pages = table.shape
    if slot < 0 or slot >= n_slots:
        return None, ERR_SLOT
    if pos < 0 or pos // page_size >= max_pages:
        return None, ERR_POS
    page = int(table[slot, pos // page_size])
    if page < 0:
        return None, ERR_PAGE_NEG
    if page >= n_pages:
        return None, ERR_PAGE_RANGE
    return page * page_size + pos % page_size, 0


def kv_append(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
              table: np.ndarray, batch_idx, input_pos, page_size: int,
              n_pages: int) -> int:
    """Scatter k[b], v[b] ([B][H][D]) into the caches in place.

    batch_idx None means row b uses slot b. Rows are applied in order b = 0..B-1
    (rows that hit the same address: the last one wins). Returns the OR of
    error bits.
    """
    B = k.shape[0]
    err = 0
    for b in range(B):
        slot = b if batch_idx is None else int(batch_idx[b])
        row, e = _checked_row(table, slot, int(input_pos[b]), page_size, n_pages)
        err |= e
        if row is None:
            continue
        k_cache[:, row, :] = k[b]
        v_cache[:, row, :] = v[b]
    return err


def gather_pages(cache: np.ndarray, table: np.ndarray, slot: int, head: int,
                 length: int, page_size: int) -> np.ndarray:
    """Logical tokens 0..length-1 of `slot` for one head, as a contiguous
    [length][D] copy, read page by page through the table."""
    n_blocks = -(-length // page_size)
    parts = []
    for blk in range(n_blocks):
        page = int(table[slot, blk])
        parts.append(cache[head, page * page_size:(page + 1) * page_size, :])
    if not parts:
        return cache[head, 0:0, :].copy()
    return np.concatenate(parts, axis=0)[:length].copy()
