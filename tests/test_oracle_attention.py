"""Pins for the oracle's paged decode attention (CPU).

Semantics: "unsloth: compare main...flex-moe-qwen3" · flex_gemma4_moe.py ·
attention forward (flex_attention with enable_gqa=True, caller's scale) and
_decode_block_mask (full: pos >= kv; sliding: pos >= kv and pos - kv < W).
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _random_paged(rng, B, Hq, Hkv, D, ps, lens, n_pages=None, placement=None):
    n_blocks = [-(-L // ps) for L in lens]
    n_pages = n_pages or (sum(n_blocks) + 3)
    max_pages = max(max(n_blocks), 1)
    pages = placement if placement is not None else rng.permutation(np.arange(1, n_pages))
    table = np.full((B + 1, max_pages), -1, np.int32)
    table[0] = 0
    it = iter(pages)
    for b in range(B):
        for blk in range(n_blocks[b]):
            table[b + 1, blk] = next(it)
    kc = rng.standard_normal((Hkv, n_pages * ps, D))
    vc = rng.standard_normal((Hkv, n_pages * ps, D))
    q = rng.standard_normal((B, Hq, D))
    bidx = np.arange(1, B + 1)
    return q, kc, vc, table, bidx


def _brute(q, kc, vc, table, bidx, lens, W, scale, ps):
    """Scalar loops: the pages' mask predicate per key, math.exp, math.fsum."""
    B, Hq, D = q.shape
    Hkv = kc.shape[0]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -math.inf)
    for b in range(B):
        slot, L = int(bidx[b]), int(lens[b])
        if slot == 0 or L == 0:
            continue
        pos = L - 1
        for h in range(Hq):
            g = h // G
            keys = []
            for kv in range(L):
                keep = pos >= kv and (W <= 0 or pos - kv < W)
                if not keep:
                    continue
                row = int(table[slot, kv // ps]) * ps + kv % ps
                s = scale * math.fsum(q[b, h, d] * kc[g, row, d] for d in range(D))
                keys.append((s, row))
            m = max(s for s, _ in keys)
            w = [math.exp(s - m) for s, _ in keys]
            den = math.fsum(w)
            for d in range(D):
                out[b, h, d] = math.fsum(wi * vc[g, row, d] for wi, (_, row) in zip(w, keys)) / den
            lse[b, h] = m + math.log(den)
    return out, lse


@pytest.mark.parametrize("W", [0, 3, 5, 100])
def test_matches_scalar_brute_force(W):
    rng = np.random.default_rng(10 + W)
    lens = [7, 3, 1, 9]
    q, kc, vc, table, bidx = _random_paged(rng, 4, 4, 2, 8, 4, lens)
    got, glse = oracle.decode_attention(q, kc, vc, table, bidx, lens, W, 0.37, 4)
    ref, rlse = _brute(q, kc, vc, table, bidx, lens, W, 0.37, 4)
    assert np.allclose(got, ref, atol=1e-12, rtol=0)
    assert np.allclose(glse, rlse, atol=1e-12, rtol=0)


def test_page_permutation_leaves_output_unchanged():
    rng = np.random.default_rng(20)
    B, Hq, Hkv, D, ps = 3, 6, 2, 16, 4
    lens = [13, 4, 22]
    q, kc, vc, table, bidx = _random_paged(rng, B, Hq, Hkv, D, ps, lens, n_pages=20)
    ref, rlse = oracle.decode_attention(q, kc, vc, table, bidx, lens, 0, 0.25, ps)
    for seed in range(3):
        perm = np.random.default_rng(seed).permutation(np.arange(1, 20))
        table2 = np.full_like(table, -1)
        table2[0] = 0
        kc2, vc2 = np.zeros_like(kc), np.zeros_like(vc)
        it = iter(perm)
        for b in range(B):
            for blk in range(-(-lens[b] // ps)):
                old, new = table[b + 1, blk], next(it)
                table2[b + 1, blk] = new
                kc2[:, new * ps:(new + 1) * ps] = kc[:, old * ps:(old + 1) * ps]
                vc2[:, new * ps:(new + 1) * ps] = vc[:, old * ps:(old + 1) * ps]
        got, glse = oracle.decode_attention(q, kc2, vc2, table2, bidx, lens, 0, 0.25, ps)
        assert np.array_equal(got, ref) and np.array_equal(glse, rlse)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(21)
    q, kc, vc, table, bidx = _random_paged(rng, 2, 4, 1, 8, 4, [1, 1])
    out, lse = oracle.decode_attention(q, kc, vc, table, bidx, [1, 1], 0, 0.5, 4)
    for b in range(2):
        row = table[b + 1, 0] * 4
        assert np.allclose(out[b], vc[0, row][None, :], atol=1e-15)
        assert np.allclose(lse[b], 0.5 * q[b] @ kc[0, row], atol=1e-13)


def test_identical_keys_give_window_mean_of_values():
    rng = np.random.default_rng(22)
    q, kc, vc, table, bidx = _random_paged(rng, 1, 2, 1, 8, 4, [11])
    kc[:] = kc[0, 0]
    for W in (0, 4, 6):
        out, lse = oracle.decode_attention(q, kc, vc, table, bidx, [11], W, 0.3, 4)
        lo = 0 if W == 0 else 11 - W
        V = oracle.gather_pages(vc, table, 1, 0, 11, 4)[lo:]
        assert np.allclose(out[0], V.mean(0)[None, :], atol=1e-13)
        n = 11 - lo
        assert np.allclose(lse[0], 0.3 * q[0] @ kc[0, 0] + math.log(n), atol=1e-12)


def test_sliding_window_equals_truncation():
    rng = np.random.default_rng(23)
    ps, D = 4, 8
    q, kc, vc, table, bidx = _random_paged(rng, 1, 2, 1, D, ps, [23])
    for W in (1, 5, 8, 22, 23, 40):
        got, glse = oracle.decode_attention(q, kc, vc, table, bidx, [23], W, 0.4, ps)
        n = min(W, 23)
        K = oracle.gather_pages(kc, table, 1, 0, 23, ps)[23 - n:]
        V = oracle.gather_pages(vc, table, 1, 0, 23, ps)[23 - n:]
        # re-page the last n tokens contiguously from page 1, no window
        nb = -(-n // ps)
        kc2 = np.zeros((1, (nb + 1) * ps, D))
        vc2 = np.zeros_like(kc2)
        kc2[0, ps:ps + n], vc2[0, ps:ps + n] = K, V
        t2 = np.array([[0] * nb, list(range(1, nb + 1))], np.int32)
        ref, rlse = oracle.decode_attention(q, kc2, vc2, t2, [1], [n], 0, 0.4, ps)
        assert np.array_equal(got, ref) and np.array_equal(glse, rlse)


def test_matches_torch_sdpa_with_gqa():
    # enable_gqa in torch's SDPA is the grouped-contiguous mapping the pages
    # request; on contiguous keys with no mask both must agree
    rng = np.random.default_rng(24)
    B, Hq, Hkv, D, ps, L = 2, 8, 2, 16, 4, 14
    q, kc, vc, table, bidx = _random_paged(rng, B, Hq, Hkv, D, ps, [L, L])
    out, _ = oracle.decode_attention(q, kc, vc, table, bidx, [L, L], 0, 0.21, ps)
    K = np.stack([np.stack([oracle.gather_pages(kc, table, b + 1, g, L, ps)
                            for g in range(Hkv)]) for b in range(B)])
    V = np.stack([np.stack([oracle.gather_pages(vc, table, b + 1, g, L, ps)
                            for g in range(Hkv)]) for b in range(B)])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, :, None, :], torch.from_numpy(K), torch.from_numpy(V),
        scale=0.21, enable_gqa=True)[:, :, 0, :].numpy()
    assert np.allclose(out, ref, atol=1e-12)


def test_empty_and_noop_rows_are_zero():
    rng = np.random.default_rng(25)
    q, kc, vc, table, bidx = _random_paged(rng, 3, 2, 1, 8, 4, [5, 5, 5])
    bidx = np.array([1, 0, 2])
    out, lse = oracle.decode_attention(q, kc, vc, table, bidx, [5, 5, 0], 0, 0.3, 4)
    assert not out[1].any() and not out[2].any()
    assert np.isneginf(lse[1]).all() and np.isneginf(lse[2]).all()
    assert out[0].any() and np.isfinite(lse[0]).all()
