"""Pins for the oracle's PageTable model (CPU only).

The allocator policy is the one stated on "unsloth: compare
main...transformers-continuous-batching-qwen3" · flex_paged_attention.py ·
class PageTable, with the "+1 capacity" fix of "unsloth: compare
main...flex-moe-qwen3" (commit message). The worked example under
tests/golden was derived by hand from that policy.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pagetable_lifo_example.json")
ERRORS = {"NoSlot": oracle.NoSlot, "NoPages": oracle.NoPages,
          "BadSlot": oracle.BadSlot, "BadArg": oracle.BadArg}


def _load():
    with open(GOLDEN) as f:
        return json.load(f)


def test_worked_example_matches_hand_derivation():
    g = _load()
    pt = oracle.PageTableModel(g["max_batch_size"], g["page_size"], g["n_pages"],
                               g["max_pages_per_seq"])
    assert pt.free_slots == g["initial"]["free_slots"]
    assert pt.free_pages == g["initial"]["free_pages"]
    assert pt.table.tolist() == g["initial"]["table"]
    for i, op in enumerate(g["ops"]):
        before = pt.snapshot()
        if "error" in op:
            with pytest.raises(ERRORS[op["error"]]):
                _apply(pt, op)
            after = pt.snapshot()
            assert _same(before, after), f"op {i} changed state on failure"
        else:
            ret = _apply(pt, op)
            if "ret" in op:
                assert ret == op["ret"], f"op {i}"
        assert pt.table.tolist() == op["table"], f"op {i}"
        assert pt.free_pages == op["free_pages"], f"op {i}"
        assert pt.capacity == op["capacity"], f"op {i}"


def _apply(pt, op):
    if op["op"] == "assign":
        return pt.assign(op["len"])
    if op["op"] == "reserve":
        return pt.reserve(op["slot"], op["len"])
    if op["op"] == "free":
        return pt.free(op["slot"])
    raise ValueError(op)


def _same(a, b):
    ta, *ra = a
    tb, *rb = b
    return np.array_equal(ta, tb) and ra == rb


def test_plus_one_capacity():
    # a user max_batch_size of N yields exactly N concurrent slots 1..N
    for n in (1, 2, 8, 64):
        pt = oracle.PageTableModel(n, 16, 4 * n + 1, 4)
        slots = [pt.assign(1) for _ in range(n)]
        assert slots == list(range(1, n + 1))
        with pytest.raises(oracle.NoSlot):
            pt.assign(1)


def test_slot_reuse_is_lifo():
    pt = oracle.PageTableModel(4, 16, 33, 4)
    s = [pt.assign(5) for _ in range(4)]
    pt.free(s[1])
    pt.free(s[3])
    assert pt.assign(5) == s[3]
    assert pt.assign(5) == s[1]


def _check_invariants(pt):
    owned = [p for sl in range(1, pt.n_slots) for p in pt.pages[sl]]
    assert len(owned) == len(set(owned)), "page owned twice"
    assert not set(owned) & set(pt.free_pages)
    assert 0 not in owned and 0 not in pt.free_pages
    assert len(owned) + len(pt.free_pages) == pt.n_pages - 1
    for sl in range(1, pt.n_slots):
        if pt.is_live(sl):
            assert pt.capacity[sl] == pt.page_size * len(pt.pages[sl])
            row = pt.table[sl]
            n = len(pt.pages[sl])
            assert row[:n].tolist() == pt.pages[sl]
            assert (row[n:] == -1).all()
    assert (pt.table[0] == 0).all()


def test_random_ops_keep_invariants_and_fail_atomically():
    rng = np.random.default_rng(3407)
    pt = oracle.PageTableModel(6, 8, 40, 6)
    for _ in range(3000):
        r = rng.random()
        before = pt.snapshot()
        try:
            if r < 0.4:
                pt.assign(int(rng.integers(0, 60)))
            elif r < 0.7:
                pt.reserve(int(rng.integers(0, 8)), int(rng.integers(0, 60)))
            else:
                pt.free(int(rng.integers(-1, 8)))
        except oracle.PageTableError:
            assert _same(before, pt.snapshot())
        _check_invariants(pt)


def test_can_reserve_agrees_with_reserve():
    rng = np.random.default_rng(7)
    pt = oracle.PageTableModel(3, 16, 12, 5)
    for _ in range(500):
        L = int(rng.integers(0, 90))
        ok = pt.can_reserve(L)
        try:
            s = pt.assign(L)
            assert ok
            if rng.random() < 0.5:
                pt.free(s)
        except (oracle.NoSlot, oracle.NoPages, oracle.BadArg):
            assert not ok
        live = [sl for sl in range(1, pt.n_slots) if pt.is_live(sl)]
        if live:
            sl = live[int(rng.integers(0, len(live)))]
            L2 = int(rng.integers(0, 90))
            ok2 = pt.can_reserve(L2, sl)
            try:
                pt.reserve(sl, L2)
                assert ok2
            except (oracle.NoPages, oracle.BadArg):
                assert not ok2
            if rng.random() < 0.3:
                pt.free(sl)
