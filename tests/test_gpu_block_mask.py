"""GPU parity of convert_logical_block_mask with the oracle, through the C
ABI: integer work, so the converted indices and the error word must be
equal, entry for entry."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    return torch.device("cuda:0")


def _table(rng, n_slots, max_pages, n_pages):
    table = np.full((n_slots, max_pages), -1, np.int32)
    table[0] = 0
    perm = iter(rng.permutation(np.arange(1, n_pages)))
    for s in range(1, n_slots):
        for j in range(int(rng.integers(0, max_pages + 1))):
            table[s, j] = next(perm)
    return table


def _run(dev, table, idx, bidx, n_cols):
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = pkv.convert_logical_block_mask(
        torch.from_numpy(idx).to(dev), torch.from_numpy(table).to(dev), table.shape[0],
        table.shape[1], None if bidx is None else torch.from_numpy(bidx).to(dev), n_cols, err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("B,H,R,M,n_cols,with_bidx", [
    (1, 1, 1, 1, None, False), (4, 2, 3, 5, None, True), (8, 8, 16, 16, 64, True),
    (3, 1, 33, 7, 7, False), (64, 1, 1, 16, None, True), (5, 4, 2, 20, None, True)])
def test_convert_equals_oracle(dev, B, H, R, M, n_cols, with_bidx):
    rng = np.random.default_rng(B * 100 + M)
    n_slots, max_pages, n_pages = 70, 16, 70 * 16 + 1
    table = _table(rng, n_slots, max_pages, n_pages)
    idx = rng.integers(0, max_pages, size=(B, H, R, M)).astype(np.int32)
    bidx = rng.integers(0, n_slots, size=B).astype(np.int32) if with_bidx else None
    got, err = _run(dev, table, idx, bidx, n_cols)
    ref, ref_err = oracle.convert_logical_block_mask(table, idx, bidx, n_cols)
    assert err == ref_err == 0
    assert np.array_equal(got, ref)


def test_convert_error_entries(dev):
    """Indices outside the table row and slots outside the table: -1 and the
    same error bits as the oracle."""
    rng = np.random.default_rng(9)
    n_slots, max_pages, n_pages = 6, 8, 60
    table = _table(rng, n_slots, max_pages, n_pages)
    idx = rng.integers(-3, max_pages + 3, size=(4, 2, 3, 6)).astype(np.int32)
    bidx = np.array([1, 7, 5, -1], np.int32)
    got, err = _run(dev, table, idx, bidx, 9)
    ref, ref_err = oracle.convert_logical_block_mask(table, idx, bidx, 9)
    assert ref_err == oracle.ERR_POS | oracle.ERR_SLOT
    assert err == ref_err
    assert np.array_equal(got, ref)


def test_convert_bad_arguments(dev):
    table = torch.zeros((2, 4), dtype=torch.int32, device=dev)
    idx = torch.zeros((1, 1, 1, 5), dtype=torch.int32, device=dev)
    with pytest.raises(pkv.BadArgError):       # n_cols < max_blocks
        pkv.convert_logical_block_mask(idx, table, 2, 4, n_cols=4)
