"""Pins for the oracle's document-causal prefill attention and block mask (CPU).

Mask of "unsloth: compare main...transformers-continuous-batching-qwen3" ·
flex_paged_attention.py · create_prefill_blockmask_no_paging:
q_idx >= kv_idx and docs[q_idx] == docs[kv_idx]; the sliding variant
(_create_prefill_sliding_blockmask of the Gemma-4 script) adds
q_idx - kv_idx < W.
"""
import math

import numpy as np
import pytest

import oracle


def _kept(i, j, docs, window):
    return j <= i and docs[j] == docs[i] and (window == 0 or i - j < window)


def _brute(q, k, v, docs, scale, window=0):
    """Scalar loops with math.fsum: the mask and softmax written out."""
    Hq, L, D = q.shape
    G = Hq // k.shape[0]
    out = np.zeros((Hq, L, D))
    for h in range(Hq):
        g = h // G
        for i in range(L):
            js = [j for j in range(L) if _kept(i, j, docs, window)]
            s = [scale * math.fsum(q[h, i, d] * k[g, j, d] for d in range(D)) for j in js]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            z = math.fsum(w)
            for d in range(D):
                out[h, i, d] = math.fsum(w[t] * v[g, js[t], d] for t in range(len(js))) / z
    return out


def test_prefill_matches_brute_force_with_unsorted_documents():
    rng = np.random.default_rng(30)
    Hq, Hkv, L, D = 4, 2, 13, 8
    q = rng.standard_normal((Hq, L, D))
    k = rng.standard_normal((Hkv, L, D))
    v = rng.standard_normal((Hkv, L, D))
    docs = np.array([2, 0, 2, 1, 0, 0, 2, 1, 1, 0, 2, 1, 0])    # interleaved, unsorted
    got = oracle.prefill_attention(q, k, v, docs, 0.3)
    assert np.allclose(got, _brute(q, k, v, docs, 0.3), atol=1e-12)
    for w in (1, 3, 6):
        got = oracle.prefill_attention(q, k, v, docs, 0.3, window=w)
        assert np.allclose(got, _brute(q, k, v, docs, 0.3, w), atol=1e-12)


@pytest.mark.parametrize("window", [0, 3])
def test_prefill_rows_equal_decode_attention_of_each_prefix(window):
    """Row i of a document is decode attention of that document's prefix up to
    i (keys 0..i, the last `window` of them on a sliding layer) — an
    independent path through the paged decode oracle and its window."""
    rng = np.random.default_rng(31)
    Hq, Hkv, D, ps = 4, 1, 16, 4
    lens = [9, 5]
    L = sum(lens)
    docs = np.repeat([0, 1], lens)
    q = rng.standard_normal((Hq, L, D))
    k = rng.standard_normal((Hkv, L, D))
    v = rng.standard_normal((Hkv, L, D))
    got = oracle.prefill_attention(q, k, v, docs, 0.25, window=window)
    # lay each document into its own slot's pages (identity placement)
    n_pages = 1 + sum(-(-n // ps) for n in lens)
    kc = np.zeros((Hkv, n_pages * ps, D))
    vc = np.zeros((Hkv, n_pages * ps, D))
    table = np.zeros((3, 4), np.int64)
    page, start = 1, 0
    for s, n in enumerate(lens):
        for blk in range(-(-n // ps)):
            table[s + 1, blk] = page
            rows = slice(blk * ps, min(n, (blk + 1) * ps))
            m = rows.stop - rows.start
            kc[:, page * ps:page * ps + m] = k[:, start + rows.start:start + rows.stop]
            vc[:, page * ps:page * ps + m] = v[:, start + rows.start:start + rows.stop]
            page += 1
        start += n
    start = 0
    for s, n in enumerate(lens):
        for i in range(n):
            qi = q[:, start + i][None]                     # [1][Hq][D]
            ref, _ = oracle.decode_attention(qi, kc, vc, table, [s + 1], [i + 1], window,
                                             0.25, ps)
            assert np.allclose(got[:, start + i], ref[0], atol=1e-12)
        start += n


def test_prefill_first_token_and_document_isolation():
    rng = np.random.default_rng(32)
    Hq, Hkv, L, D = 2, 1, 10, 4
    q = rng.standard_normal((Hq, L, D))
    k = rng.standard_normal((Hkv, L, D))
    v = rng.standard_normal((Hkv, L, D))
    docs = np.array([0, 0, 0, 1, 1, 1, 1, 2, 2, 2])
    got = oracle.prefill_attention(q, k, v, docs, 1.0)
    # a document's first token sees only itself: output = its own v
    for i in (0, 3, 7):
        assert np.allclose(got[:, i], v[0, i], atol=1e-15)
    # changing another document's keys and values leaves a document unchanged
    k2, v2 = k.copy(), v.copy()
    k2[:, 3:7] += 5.0
    v2[:, 3:7] -= 3.0
    got2 = oracle.prefill_attention(q, k2, v2, docs, 1.0)
    assert np.array_equal(got2[:, :3], got[:, :3]) and np.array_equal(got2[:, 7:], got[:, 7:])
    # identical keys inside a document: the output is the running mean of its values
    k3 = np.repeat(k[:, :1], L, axis=1)
    got3 = oracle.prefill_attention(q, k3, v, np.zeros(L, int), 1.0)
    for i in range(L):
        assert np.allclose(got3[:, i], v[0, :i + 1].mean(0), atol=1e-12)


# ---- block mask -------------------------------------------------------------

def _as_lists(bm):
    kv_num, kv_idx, full_num, full_idx = bm
    assert list(kv_num) == [len(x) for x in kv_idx]
    assert list(full_num) == [len(x) for x in full_idx]
    return [list(x) for x in kv_idx], [list(x) for x in full_idx]


def test_block_mask_single_document_by_hand():
    """One document of 200 tokens, blocks of 64: the plain causal pattern.
    Query block qb (rows inside L) has the key blocks before it full and its
    diagonal partial; the last query block (rows 192..255, past L from 200) is
    never full, so all four of its key blocks are partial."""
    part, full = _as_lists(oracle.prefill_block_mask(np.zeros(200, int), 64))
    assert full == [[], [0], [0, 1], []]
    assert part == [[0], [1], [2], [0, 1, 2, 3]]
    # L a multiple of the block: full_num[qb] = qb and one partial (the diagonal)
    kv_num, _, full_num, _ = oracle.prefill_block_mask(np.zeros(256, int), 64)
    assert list(full_num) == [0, 1, 2, 3] and list(kv_num) == [1, 1, 1, 1]


def test_block_mask_two_documents_by_hand():
    """docs = 0 x6, 1 x6 in blocks of 4: block (1, 0) holds rows 4..7 (docs
    0 0 1 1) against keys 0..3 (doc 0): rows 4, 5 keep, rows 6, 7 do not ->
    partial; (2, 0) is doc 1 against doc 0 -> absent; (2, 1) partial; the
    diagonals partial; nothing is full."""
    part, full = _as_lists(oracle.prefill_block_mask([0] * 6 + [1] * 6, 4))
    assert part == [[0], [0, 1], [1, 2]]
    assert full == [[], [], []]


def test_block_mask_sliding_window_by_hand():
    """One document of 16 tokens, blocks of 4. W = 5: (1, 0) has i - j from
    1 to 7, some < 5 -> partial; (2, 0) has i - j >= 5 -> absent. W = 8:
    (1, 0) has every i - j in 1..7 < 8 -> full; (2, 0) has i - j from 5 to
    11 -> partial; (2, 1) full."""
    part, full = _as_lists(oracle.prefill_block_mask(np.zeros(16, int), 4, window=5))
    assert part == [[0], [0, 1], [1, 2], [2, 3]] and full == [[], [], [], []]
    part, full = _as_lists(oracle.prefill_block_mask(np.zeros(16, int), 4, window=8))
    assert part == [[0], [1], [0, 2], [1, 3]]
    assert full == [[], [0], [1], [2]]


@pytest.mark.parametrize("seed", range(6))
def test_block_mask_against_pairwise_loops(seed):
    """Brute force over every pair with scalar loops: a block is full iff all
    of its block x block pairs are inside L and kept, partial iff not full and
    some pair inside L is kept; the lists are ascending and disjoint."""
    rng = np.random.default_rng(40 + seed)
    L = int(rng.integers(1, 40))
    block = int(rng.choice([2, 3, 4, 8]))
    window = int(rng.choice([0, 0, 1, 2, 5, 9]))
    docs = rng.integers(0, int(rng.integers(1, 4)), size=L)
    if seed % 2:
        docs = np.sort(docs)
    part, full = _as_lists(oracle.prefill_block_mask(docs, block, window))
    n = -(-L // block)
    assert len(part) == n and len(full) == n
    for qb in range(n):
        assert part[qb] == sorted(part[qb]) and full[qb] == sorted(full[qb])
        assert not set(part[qb]) & set(full[qb])
        for kb in range(n):
            pairs = [(i, j) for i in range(qb * block, (qb + 1) * block)
                     for j in range(kb * block, (kb + 1) * block)]
            kept = [i < L and j < L and _kept(i, j, docs, window) for i, j in pairs]
            assert (kb in full[qb]) == all(kept)
            assert (kb in part[qb]) == (any(kept) and not all(kept))
