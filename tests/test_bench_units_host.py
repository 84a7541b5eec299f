"""The benchmark's algorithmic units (CPU): the prefill FLOP count (4 D Hq
per kept pair, kept pairs in closed form per document) equals a brute-force
count of the oracle's document-causal mask, and the decode byte count equals
a key-by-key count."""
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


def test_decode_bytes_equal_a_per_key_count():
    """The decode benchmark's algorithmic bytes: K and V of every attended key
    (the last W with a window), q read and out written once, one int32 table
    entry per distinct page touched, counted here key by key."""
    B, Hq, Hkv, D, ps = 6, 8, 2, 64, 16
    lens = np.array([0, 1, 15, 16, 17, 100])
    for window in (0, 1, 20, 64):
        total = B * Hq * D * 2 * 2
        for L in lens:
            keys = range(max(0, L - window), L) if window > 0 else range(L)
            total += Hkv * len(keys) * D * 2 * 2
            total += 4 * len({k // ps for k in keys})
        assert bench.attn_bytes(lens, B, Hq, Hkv, D, ps, window) == total, window
