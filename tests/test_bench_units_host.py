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


def test_schedule_sample_spreads_timed_steps_over_the_whole_schedule():
    """The rollout bench times K steps of its fixed 512-step schedule: every
    step exactly once at K = 512, the step in the middle of each of K equal
    stretches below that, every step K/512 times above it."""
    S = 512
    assert list(bench.schedule_sample(S, S)) == list(range(S))
    for K in (1, 3, 20, 100, 511):
        idx = bench.schedule_sample(S, K)
        assert len(idx) == K and np.all(np.diff(idx) > 0)
        for i, t in enumerate(idx):
            assert (i * S) // K <= t < (i + 1) * S / K      # the middle of stretch i
    idx = bench.schedule_sample(S, 3 * S)
    assert np.array_equal(np.bincount(idx, minlength=S), np.full(S, 3))
    assert list(bench.schedule_sample(S, 4, 0.0)) == [0, 128, 256, 384]


def test_rollout_lengths_equal_the_allocator_driven_schedule():
    """The reference arm's per-step lengths (from the schedule alone) equal the
    seq_lens the GPU arm gets from the PageTable-driven schedule, so both arms
    time the same rows."""
    import workloads as wl
    pytest = __import__("pytest")
    pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")
    try:
        pkv.load_library()
    except RuntimeError:
        pytest.skip("libpkv.so not built")
    w = wl.ROLLOUT
    lens = bench.rollout_lengths(w)
    _, _, _, lens_pt = bench.rollout_metadata(w, w.steps)
    assert lens.shape == (512, 64) and np.array_equal(lens, lens_pt)
    assert lens.min() >= 101 and lens.max() <= 1024


def test_prefill_flops_with_a_window_equal_kept_pairs_of_the_mask():
    """The sliding-window count (W(W+1)/2 + (n - W) W kept pairs for a document
    of n > W tokens) equals the oracle mask's kept pairs, for documents both
    shorter and longer than the window."""
    lens = np.array([5, 30, 31, 90, 7])
    docs = np.repeat(np.arange(len(lens)), lens).astype(np.int32)
    for window in (1, 8, 31, 64):
        kept = int(oracle.keep_matrix(docs, window).sum())
        assert bench.prefill_flops(lens, 8, 256, window) == 4.0 * 256 * 8 * kept, window


def test_traffic_records_follow_the_kernel_source(tmp_path, monkeypatch):
    # a record is used only while the hash of the kernel source it names
    # matches; a ratio record scales to the run's mean launch, a bytes record
    # (a fixed workload) is returned as is
    import hashlib
    import json
    csrc = tmp_path / "paged_kv_decode_pagetable_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "decode_attn.cu").write_bytes(b"decode source")
    (csrc / "prefill_tc.cu").write_bytes(b"prefill source")
    h = {n: hashlib.sha256(n.encode()).hexdigest()[:16]
         for n in ("decode source", "prefill source")}
    recs = {"a_decode_attn_128": {"source_sha256_16": h["decode source"],
                                  "dram_over_algorithmic": 1.5},
            "b_prefill_128": {"source_file": "prefill_tc.cu",
                              "source_sha256_16": h["prefill source"],
                              "dram_bytes_per_launch": 1e6},
            "c_prefill_128": {"source_file": "prefill_tc.cu",
                              "source_sha256_16": h["decode source"],
                              "dram_bytes_per_launch": 1e6}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(recs))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("a_decode_attn_128", 2e6) == 3e6
    assert bench.profile_traffic("b_prefill_128") == 1e6
    assert bench.profile_traffic("c_prefill_128") is None      # source changed
    assert bench.profile_traffic("missing") is None
    (csrc / "decode_attn.cu").write_bytes(b"decode source, edited")
    assert bench.profile_traffic("a_decode_attn_128", 2e6) is None
