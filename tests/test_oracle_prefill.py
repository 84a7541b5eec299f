"""Pins for the oracle's document-causal prefill attention (CPU).

Mask of "unsloth: compare main...transformers-continuous-batching-qwen3" ·
flex_paged_attention.py · create_prefill_blockmask_no_paging:
q_idx >= kv_idx and docs[q_idx] == docs[kv_idx].
"""
import math

import numpy as np

import oracle


def _brute(q, k, v, docs, scale):
    """Scalar loops with math.fsum: the mask and softmax written out."""
    Hq, L, D = q.shape
    G = Hq // k.shape[0]
    out = np.zeros((Hq, L, D))
    for h in range(Hq):
        g = h // G
        for i in range(L):
            js = [j for j in range(L) if j <= i and docs[j] == docs[i]]
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


def test_prefill_rows_equal_decode_attention_of_each_prefix():
    """Row i of a document is decode attention of that document's prefix up to
    i (keys 0..i) — an independent path through the paged decode oracle."""
    rng = np.random.default_rng(31)
    Hq, Hkv, D, ps = 4, 1, 16, 4
    lens = [9, 5]
    L = sum(lens)
    docs = np.repeat([0, 1], lens)
    q = rng.standard_normal((Hq, L, D))
    k = rng.standard_normal((Hkv, L, D))
    v = rng.standard_normal((Hkv, L, D))
    got = oracle.prefill_attention(q, k, v, docs, 0.25)
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
            ref, _ = oracle.decode_attention(qi, kc, vc, table, [s + 1], [i + 1], 0, 0.25, ps)
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
