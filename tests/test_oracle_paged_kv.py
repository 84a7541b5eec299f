"""Pins for the oracle's decode scatter address map and page gather (CPU).

Address map: "unsloth: compare main...transformers-continuous-batching-qwen3"
· flex_paged_attention.py · PageTable.assign ("find address").
"""
import numpy as np

import oracle


def test_address_closed_form_hand_values():
    # table row of slot 1: logical block 0 -> page 5, block 1 -> page 2
    table = np.array([[0, 0, 0], [5, 2, -1]], dtype=np.int32)
    assert oracle.physical_row(table, 1, 0, 16) == 80
    assert oracle.physical_row(table, 1, 15, 16) == 95
    assert oracle.physical_row(table, 1, 16, 16) == 32
    assert oracle.physical_row(table, 1, 17, 16) == 33
    assert oracle.physical_row(table, 0, 7, 16) == 7      # no-op slot -> page 0


def test_append_writes_only_addressed_rows():
    ps, P, H, D = 4, 6, 2, 3
    table = np.array([[0, 0], [3, 1], [4, -1]], dtype=np.int32)
    kc = np.arange(H * P * ps * D, dtype=np.uint16).reshape(H, P * ps, D)
    vc = kc.copy() + 7
    k = np.array([[[901, 902, 903], [904, 905, 906]],
                  [[911, 912, 913], [914, 915, 916]]], dtype=np.uint16)
    v = k + 1000
    ref_k, ref_v = kc.copy(), vc.copy()
    err = oracle.kv_append(kc, vc, k, v, table, [1, 2], [5, 2], ps, P)
    assert err == 0
    # slot 1, pos 5 -> block 1 -> page 1, offset 1 -> row 5
    # slot 2, pos 2 -> block 0 -> page 4, offset 2 -> row 18
    ref_k[:, 5, :] = k[0]
    ref_v[:, 5, :] = v[0]
    ref_k[:, 18, :] = k[1]
    ref_v[:, 18, :] = v[1]
    assert np.array_equal(kc, ref_k) and np.array_equal(vc, ref_v)


def test_append_error_bits_skip_the_write():
    ps, P = 4, 6
    table = np.array([[0, 0], [3, 9], [-1, -1]], dtype=np.int32)
    kc = np.zeros((1, P * ps, 2), np.uint16)
    vc = kc.copy()
    k = np.ones((5, 1, 2), np.uint16)
    # bad slot, pos beyond table, page >= n_pages, negative page, negative pos
    err = oracle.kv_append(kc, vc, k, k, table, [3, 1, 1, 2, 1], [0, 8, 4, 0, -1], ps, P)
    assert err == (oracle.ERR_SLOT | oracle.ERR_POS | oracle.ERR_PAGE_RANGE
                   | oracle.ERR_PAGE_NEG)
    assert not kc.any() and not vc.any()


def test_append_then_gather_round_trip_under_any_placement():
    rng = np.random.default_rng(11)
    ps, P, H, D, L = 8, 20, 2, 4, 37
    for _ in range(5):
        perm = rng.permutation(np.arange(1, P))[: -(-L // ps)]
        table = np.full((2, 8), -1, np.int32)
        table[0] = 0
        table[1, :len(perm)] = perm
        kc = np.zeros((H, P * ps, D), np.uint16)
        vc = np.zeros_like(kc)
        toks = rng.integers(0, 65535, size=(L, H, D)).astype(np.uint16)
        for t in range(L):
            assert oracle.kv_append(kc, vc, toks[t:t + 1], toks[t:t + 1], table,
                                    [1], [t], ps, P) == 0
        for h in range(H):
            got = oracle.gather_pages(kc, table, 1, h, L, ps)
            assert np.array_equal(got, toks[:, h, :])
