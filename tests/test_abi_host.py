"""C-ABI library checks that need no GPU: every declared symbol is exported,
and the host PageTable allocator (host-only mode, no device mirror) matches
the CPU oracle bit for bit."""
import json
import os
import re

import numpy as np
import pytest

import oracle
import workloads as wl

pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pkv.LIB_PATH):
        from paged_kv_decode_pagetable_gb300 import _build
        _build.build()
    return pkv.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(pkv.EXPORTS)


ERRS = {"NoSlot": pkv.NoSlotError, "NoPages": pkv.NoPagesError,
        "BadSlot": pkv.BadSlotError, "BadArg": pkv.BadArgError}


def test_worked_example_through_the_abi(lib):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "pagetable_lifo_example.json")))
    pt = pkv.PageTable(g["max_batch_size"], g["page_size"], g["n_pages"], g["max_pages_per_seq"])
    assert pt.host_table().tolist() == g["initial"]["table"]
    assert pt.free_page_list() == g["initial"]["free_pages"]
    for i, op in enumerate(g["ops"]):
        def run():
            if op["op"] == "assign":
                return pt.assign(op["len"])
            if op["op"] == "reserve":
                return pt.reserve(op["slot"], op["len"])
            return pt.free(op["slot"])
        if "error" in op:
            with pytest.raises(ERRS[op["error"]]):
                run()
        else:
            r = run()
            if "ret" in op:
                assert r == op["ret"], i
        assert pt.host_table().tolist() == op["table"], i
        assert pt.free_page_list() == op["free_pages"], i
        assert [pt.capacity(s) for s in range(pt.n_slots)] == op["capacity"], i


def _compare(pt, model):
    assert np.array_equal(pt.host_table().numpy(), model.table)
    assert pt.free_page_list() == model.free_pages
    for s in range(model.n_slots):
        assert pt.capacity(s) == model.capacity[s]
        assert pt.pages(s) == model.pages[s]


def test_random_ops_match_oracle(lib):
    rng = np.random.default_rng(99)
    pt = pkv.PageTable(5, 8, 33, 6)
    model = oracle.PageTableModel(5, 8, 33, 6)
    for _ in range(2000):
        r = rng.random()
        if r < 0.4:
            args = ("assign", int(rng.integers(0, 56)))
        elif r < 0.7:
            args = ("reserve", int(rng.integers(-1, 7)), int(rng.integers(0, 56)))
        else:
            args = ("free", int(rng.integers(-1, 7)))
        res = []
        for obj, exc in ((model, oracle.PageTableError), (pt, pkv.PkvError)):
            try:
                res.append(("ok", getattr(obj, args[0])(*args[1:])))
            except exc as e:
                res.append(("err", type(e).__name__))
        m, p = res
        assert m[0] == p[0], (args, m, p)
        if m[0] == "ok":
            assert m[1] == p[1]
        else:
            assert m[1].replace("Error", "") == p[1].replace("Error", ""), (m, p)
        if args[0] == "assign" or rng.random() < 0.1:
            _compare(pt, model)
        for L in (0, 7, 30):
            assert pt.can_reserve(L) == model.can_reserve(L)
    _compare(pt, model)


def test_rollout_schedule_tables_match_oracle(lib):
    """The continuous-batching workload (64 slots, 512 steps, refills at once)
    driven through both allocators: identical tables at every step."""
    w = wl.ROLLOUT
    sched = wl.rollout_schedule(w)
    pt = pkv.PageTable(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq)
    model = oracle.PageTableModel(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq)
    slots_p, slots_m, length = [], [], []
    for r in sched.first:
        slots_p.append(pt.assign(r.prompt_len + 1))
        slots_m.append(model.assign(r.prompt_len + 1))
        length.append(r.prompt_len)
    assert slots_p == slots_m
    for t in range(sched.steps):
        for lane in sched.finish[t]:
            pt.free(slots_p[lane])
            model.free(slots_m[lane])
        for lane, r in sched.start[t]:
            slots_p[lane] = pt.assign(r.prompt_len + 1)
            slots_m[lane] = model.assign(r.prompt_len + 1)
            length[lane] = r.prompt_len
        for lane in range(sched.lanes):
            pt.reserve(slots_p[lane], length[lane] + 1)
            model.reserve(slots_m[lane], length[lane] + 1)
            length[lane] += 1
        assert slots_p == slots_m
        assert np.array_equal(pt.host_table().numpy(), model.table), t
    _compare(pt, model)
