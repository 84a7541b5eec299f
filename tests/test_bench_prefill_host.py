"""The prefill benchmark's FLOP count (CPU): 4 D Hq per kept (query, key)
pair, with the kept pairs counted in closed form per document, equals a
brute-force count of the oracle's document-causal mask."""
import numpy as np

import bench
import oracle


def test_prefill_flops_equal_kept_pairs_of_the_mask():
    docs, lens = bench.prefill_docs(n_docs=5, seed_salt=3)
    assert len(docs) == int(np.sum(lens)) and np.all((lens >= 100) & (lens <= 400))
    kept = int(oracle.keep_matrix(docs).sum())
    assert bench.prefill_flops(lens, 32, 128) == 4.0 * 128 * 32 * kept


def test_prefill_long_layout():
    docs, lens = bench.prefill_docs(long=True)
    assert list(lens) == [2048] * 8 and len(docs) == 8 * 2048
    assert np.all(np.diff(docs) >= 0)     # documents packed in order
