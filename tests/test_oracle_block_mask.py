"""Pins for the oracle's logical -> physical block-mask conversion (CPU).

"unsloth: compare main...transformers-continuous-batching-qwen3" ·
flex_paged_attention.py · PageTable.convert_logical_block_mask: each logical
key-block index goes through its batch row's page-table row; the columns
after the logical ones are zero."""
import numpy as np
import pytest

import oracle


def test_convert_by_hand():
    """Slot 1 holds pages [5, 2], slot 2 pages [7, 1, 3]; batch row 0 is
    slot 2 and row 1 is slot 1. Logical blocks [[0, 2], [1, 0]] of row 0 are
    pages [[7, 3], [1, 7]]; [[1, 0], [0, 0]] of row 1 are [[2, 5], [5, 5]];
    the two columns after them are 0."""
    table = np.array([[0, 0, 0, 0], [5, 2, -1, -1], [7, 1, 3, -1]])
    idx = np.array([[[[0, 2], [1, 0]]], [[[1, 0], [0, 0]]]])      # [B=2][H=1][R=2][M=2]
    out, err = oracle.convert_logical_block_mask(table, idx, batch_idx=[2, 1], n_cols=4)
    assert err == 0
    assert out.tolist() == [[[[7, 3, 0, 0], [1, 7, 0, 0]]], [[[2, 5, 0, 0], [5, 5, 0, 0]]]]
    # default batch_idx = b (row 0 -> slot 0, the no-op slot of page 0) and
    # default width = the table row's
    out, err = oracle.convert_logical_block_mask(table, idx)
    assert err == 0 and out.shape == (2, 1, 2, 4)
    assert out[0].tolist() == [[[0, 0, 0, 0], [0, 0, 0, 0]]]
    assert out[1].tolist() == [[[2, 5, 0, 0], [5, 5, 0, 0]]]


@pytest.mark.parametrize("seed", range(4))
def test_convert_agrees_with_the_scatter_address(seed):
    """The physical block of logical block j of a slot is the page that the
    decode scatter writes token j * page_size of that slot to."""
    rng = np.random.default_rng(60 + seed)
    n_slots, max_pages, ps, n_pages = 5, 6, 16, 40
    table = np.full((n_slots, max_pages), -1)
    table[0] = 0
    perm = iter(rng.permutation(np.arange(1, n_pages)))
    for s in range(1, n_slots):
        for j in range(int(rng.integers(1, max_pages + 1))):
            table[s, j] = next(perm)
    B, H, R, M = 3, 2, 3, 4
    bidx = rng.integers(1, n_slots, size=B)
    idx = np.zeros((B, H, R, M), dtype=np.int64)
    for b in range(B):
        filled = int(np.sum(table[bidx[b]] >= 0))
        idx[b] = rng.integers(0, filled, size=(H, R, M))
    out, err = oracle.convert_logical_block_mask(table, idx, batch_idx=bidx)
    assert err == 0
    for b in range(B):
        for h in range(H):
            for r in range(R):
                for c in range(M):
                    j = int(idx[b, h, r, c])
                    row = oracle.physical_row(table, int(bidx[b]), j * ps + 3, ps)
                    assert out[b, h, r, c] == row // ps
    assert np.all(out[..., M:] == 0)


def test_convert_errors():
    table = np.array([[0, 0, 0], [4, 6, -1]])
    idx = np.array([[[[0, 3, -1, 2]]]])                               # 3 and -1 outside
    out, err = oracle.convert_logical_block_mask(table, idx, batch_idx=[1])
    assert err == oracle.ERR_POS
    assert out.tolist() == [[[[4, -1, -1, -1]]]]                      # entry 2 is -1 itself
    out, err = oracle.convert_logical_block_mask(table, idx, batch_idx=[2])
    assert err == oracle.ERR_SLOT and np.all(out[..., :4] == -1)
