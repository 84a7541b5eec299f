"""Host-side engine logic: the CUDA-graph batch buckets and the continuous
batching scheduler of "unsloth: compare main...flex-moe-qwen3" ·
flex_gemma4_moe.py (capture_decode_cudagraph bucket ladder; generate's
admission, growth and newest-first preemption), driven by the real host
PageTable allocator (no GPU)."""
import numpy as np
import pytest

pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")
from paged_kv_decode_pagetable_gb300 import engine  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def lib():
    pkv.load_library()


def test_bucket_ladder_and_lookup():
    assert engine.bucket_ladder(64) == [1, 2, 4, 8, 16, 32, 48, 64]
    assert engine.bucket_ladder(6) == [1, 2, 4]
    assert engine.bucket_ladder(40) == [1, 2, 4, 8, 16, 32]
    lad = engine.bucket_ladder(64)
    assert [engine.bucket_for(b, lad) for b in (1, 3, 8, 9, 17, 64)] == [1, 4, 8, 16, 32, 64]
    with pytest.raises(ValueError):
        engine.bucket_for(65, lad)


def test_preemption_trace_worked_example():
    """Hand-worked trace of the generate loop. Pool: page_size 4, 4 usable
    pages, 2 slots. A and B (prompt 7, 6 new tokens each) are admitted
    together (2 pages each) and prefilled; both decode at length 8. At length
    9 A needs a third page and none is free: A goes back to the front and the
    newest running sequence, B, is preempted and its two pages freed; A takes
    one and decodes alone until it finishes (6 tokens), freeing slot 1. B (now
    prompt + 2 tokens = 9) is re-admitted into slot 1 (LIFO slot stack) with
    3 pages, re-prefilled (its third token) and decoded to 6 tokens, growing
    to a fourth page on the way."""
    pt = pkv.PageTable(2, 4, 5, 8)
    a, b = engine.Sequence(0, 7, 6), engine.Sequence(1, 7, 6)
    slots_at_prefill = []
    cb = engine.ContinuousBatcher(pt, [a, b],
                                  prefill=lambda batch: slots_at_prefill.append(
                                      [(s.rid, s.slot) for s in batch]))
    cb.run()
    assert cb.events == [
        ("prefill", [0, 1]), ("decode", [0, 1]), ("preempt", 1),
        ("decode", [0]), ("decode", [0]), ("decode", [0]), ("decode", [0]), ("finish", 0),
        ("prefill", [1]), ("decode", [1]), ("decode", [1]), ("decode", [1]), ("finish", 1)]
    assert slots_at_prefill == [[(0, 1), (1, 2)], [(1, 1)]]
    assert a.generated == b.generated == 6 and a.finished and b.finished
    assert len(pt.free_page_list()) == 4


def test_scheduler_invariants_random_workload():
    """Every sequence ends with exactly max_new_tokens; at every decode each
    row's slot holds capacity for its length; pages are never over-committed;
    a preemption only happens when a running row could not grow."""
    rng = np.random.default_rng(21)
    ps, n_pages, max_bs, mp = 16, 1 + 40, 8, 16
    pt = pkv.PageTable(max_bs, ps, n_pages, mp)
    seqs = [engine.Sequence(i, int(rng.integers(5, 120)), int(rng.integers(1, 80)))
            for i in range(30)]

    def check_decode(batch):
        for s in batch:
            assert pt.capacity(s.slot) >= s.total_length
        owned = sum(len(pt.pages(s.slot)) for s in batch)
        assert owned <= n_pages - 1

    cb = engine.ContinuousBatcher(pt, seqs, decode=check_decode)
    done = cb.run()
    assert sorted(s.rid for s in done) == list(range(30))
    assert all(s.generated == s.max_new_tokens for s in done)
    assert any(e[0] == "preempt" for e in cb.events)      # the pool is tight enough
    assert len(pt.free_page_list()) == n_pages - 1        # everything returned
