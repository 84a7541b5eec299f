"""GPU parity of the document-causal prefill path (prefill_block_mask and
prefill_attn) with the float64 oracle, through the C ABI, on the GPU's own
bf16 inputs. Cases span several 64-token blocks with a ragged tail, one
token, a single document, contiguous documents of random lengths, documents
interleaved in no order (the pages do not sort tokens), sliding windows, and
more than 128 key blocks (the builder's second pass).

The block mask is integer work: equal to the oracle's, entry for entry.

Head dims 64 and 128 run on prefill_tc.cu's kernel, 256 and 512 (the Gemma-4
widths) on prefill_tc_wide.cu's. With an even number of query heads per kv
head a work item holds one query block of two heads; otherwise two query
blocks of one head: both are covered.

Attention bar: the decode path's, max abs 1e-2 and mean abs 1e-3, on every
query row that keeps at least 16 keys, and the mean over all rows. Rows with
fewer kept keys (a document's first tokens) may miss 1e-2 without any fault:
with one or two keys the output is about as large as v itself, and rounding
it once to bf16 (half an ulp, 2^-9 relative) plus the bf16 probabilities in
P.V give |o_gpu - o| <= 2^-9 (max|v| + |o|) <= 2^-8 max|v|, about 0.018 for
N(0, 1) values. Those rows are held to 2^-8 max|v| + 2e-3."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import f64

pytestmark = pytest.mark.gpu
pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")
BLOCK = 64


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    return torch.device("cuda:0")


def _docs(rng, kind, L):
    if kind == "one":
        return np.zeros(L, np.int32)
    if kind == "contiguous":
        cuts = np.sort(rng.choice(np.arange(1, L), size=min(5, L - 1), replace=False))
        return np.repeat(np.arange(len(cuts) + 1), np.diff(np.r_[0, cuts, L])).astype(np.int32)
    if kind == "many":      # rollout-like prompts of 100..400 tokens, packed in order
        lens = wl.uniform_lengths(rng, L // 100 + 1, 100, 400)
        return np.repeat(np.arange(len(lens)), lens)[:L].astype(np.int32)
    return rng.integers(0, 4, size=L).astype(np.int32)      # interleaved


def _check_mask(bm, docs, window):
    kv_num, kv_idx, full_num, full_idx = oracle.prefill_block_mask(docs, BLOCK, window)
    g_kv_num = bm.kv_num_blocks.cpu().numpy()
    g_full_num = bm.full_kv_num_blocks.cpu().numpy()
    g_kv = bm.kv_indices.cpu().numpy()
    g_full = bm.full_kv_indices.cpu().numpy()
    assert np.array_equal(g_kv_num, kv_num) and np.array_equal(g_full_num, full_num)
    for qb in range(len(kv_num)):
        assert list(g_kv[qb, :kv_num[qb]]) == kv_idx[qb], qb
        assert list(g_full[qb, :full_num[qb]]) == full_idx[qb], qb


@pytest.mark.parametrize("L,kind,window", [
    (1, "one", 0), (63, "one", 0), (64, "one", 0), (65, "interleaved", 0),
    (300, "contiguous", 0), (777, "interleaved", 0), (200, "one", 64), (777, "contiguous", 37),
    (1000, "interleaved", 130), (4100, "many", 0), (9000, "many", 0), (9000, "many", 512),
    (8400, "interleaved", 0)])
def test_block_mask_equals_oracle(dev, L, kind, window):
    rng = np.random.default_rng(L + window)
    docs = _docs(rng, kind, L)
    bm = pkv.prefill_block_mask(torch.from_numpy(docs).to(dev), window)
    torch.cuda.synchronize()
    _check_mask(bm, docs, window)


def _run(dev, q, k, v, docs, window, scale, bm=None):
    Hq, L, D = q.shape
    if bm is None:
        bm = pkv.prefill_block_mask(torch.from_numpy(docs).to(dev), window)
    out = torch.full((Hq, L, D), float("nan"), dtype=torch.bfloat16, device=dev)
    pkv.prefill_attn(q.to(dev), k.to(dev), v.to(dev), bm, scale, out)
    torch.cuda.synchronize()
    return out, bm


def _compare(got, ref, v, kept):
    """got, ref: [Hq][L][D]; kept: keys kept by each of the L query rows."""
    assert np.isfinite(got).all()
    e = np.abs(got - ref)
    long_rows = np.asarray(kept) >= 16
    assert e.mean() <= 1e-3, float(e.mean())
    if long_rows.any():
        el = e[:, long_rows]
        assert el.max() <= 1e-2, (float(el.max()), int(long_rows.sum()))
    if (~long_rows).any():
        bound = 2.0 ** -8 * float(np.abs(v.double().numpy()).max()) + 2e-3
        es = e[:, ~long_rows]
        assert es.max() <= bound, (float(es.max()), bound)


def _kept(docs, window=0):
    return oracle.keep_matrix(docs, window).sum(axis=1)


@pytest.mark.parametrize("L,Hq,Hkv,D,kind,window", [
    (300, 8, 2, 128, "contiguous", 0), (257, 4, 4, 64, "interleaved", 0),
    (64, 8, 1, 128, "one", 0), (1, 2, 1, 64, "one", 0), (65, 4, 2, 128, "interleaved", 0),
    (777, 16, 4, 128, "contiguous", 0), (200, 6, 3, 64, "contiguous", 0),
    (300, 4, 1, 128, "one", 100), (500, 4, 2, 64, "contiguous", 64),
    (257, 4, 2, 128, "interleaved", 7), (640, 8, 2, 128, "many", 0),
    # odd query heads per kv head: items of two query blocks of one head
    (300, 6, 2, 128, "contiguous", 0), (333, 3, 1, 64, "many", 0), (400, 3, 3, 128, "many", 90),
    # the Gemma-4 widths: sliding layers D=256 (window 512), full layers D=512
    (300, 8, 1, 256, "contiguous", 0), (257, 4, 2, 256, "interleaved", 0),
    (200, 8, 1, 256, "one", 64), (700, 8, 1, 256, "many", 512), (1, 2, 1, 256, "one", 0),
    (300, 8, 1, 512, "contiguous", 0), (65, 4, 1, 512, "interleaved", 0),
    (1, 2, 1, 512, "one", 0), (500, 8, 1, 512, "many", 0), (257, 2, 2, 512, "interleaved", 37),
    (300, 6, 2, 256, "many", 0), (200, 3, 1, 512, "contiguous", 50)])
def test_prefill_attention_parity(dev, L, Hq, Hkv, D, kind, window):
    rng = np.random.default_rng(L * 10 + D + Hq + window)
    q = wl.randn_bf16(rng, (Hq, L, D))
    k = wl.randn_bf16(rng, (Hkv, L, D))
    v = wl.randn_bf16(rng, (Hkv, L, D))
    docs = _docs(rng, kind, L)
    scale = D ** -0.5
    out, _ = _run(dev, q, k, v, docs, window, scale)
    ref = oracle.prefill_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                   docs, scale, window=window)
    _compare(f64(out), ref, v, _kept(docs, window))


def test_prefill_full_size_sampled_documents(dev):
    """The benchmark's launch: 64 packed prompts of U[100, 400] tokens, 32 q /
    8 kv heads, head_dim 128. A document's rows depend on its own tokens only
    (pinned in the oracle tests), so whole documents are checked against the
    oracle run on that document alone: the first, one in the middle and the
    last."""
    rng = np.random.default_rng(77)
    lens = wl.uniform_lengths(rng, 64, 100, 400)
    docs = np.repeat(np.arange(64), lens).astype(np.int32)
    L, Hq, Hkv, D = len(docs), 32, 8, 128
    q = wl.randn_bf16(rng, (Hq, L, D))
    k = wl.randn_bf16(rng, (Hkv, L, D))
    v = wl.randn_bf16(rng, (Hkv, L, D))
    scale = D ** -0.5
    out, bm = _run(dev, q, k, v, docs, 0, scale)
    _check_mask(bm, docs, 0)
    got = f64(out)
    starts = np.r_[0, np.cumsum(lens)]
    for d in (0, 31, 63):
        sl = slice(int(starts[d]), int(starts[d + 1]))
        ref = oracle.prefill_attention(q[:, sl].double().numpy(), k[:, sl].double().numpy(),
                                       v[:, sl].double().numpy(), docs[sl], scale)
        _compare(got[:, sl], ref, v, _kept(docs[sl]))


def test_prefill_mask_lists_are_bounds_safe(dev):
    """List entries outside [0, n) are skipped (the output is bit-identical to
    the unmodified mask's), and a query block whose lists are empty gets
    zeros."""
    rng = np.random.default_rng(5)
    L, Hq, Hkv, D = 300, 4, 2, 128
    q = wl.randn_bf16(rng, (Hq, L, D))
    k = wl.randn_bf16(rng, (Hkv, L, D))
    v = wl.randn_bf16(rng, (Hkv, L, D))
    docs = _docs(rng, "contiguous", L)
    out, bm = _run(dev, q, k, v, docs, 0, 0.1)
    n = bm.kv_num_blocks.numel()
    kv_num = bm.kv_num_blocks.clone()
    kv_idx = bm.kv_indices.clone()
    for qb in range(n):
        c = int(kv_num[qb])
        if c + 2 <= n:
            kv_idx[qb, c] = -3
            kv_idx[qb, c + 1] = n + 5
            kv_num[qb] = c + 2
    bad = pkv.PrefillBlockMask(kv_num, kv_idx, bm.full_kv_num_blocks, bm.full_kv_indices,
                               bm.docs, 0)
    out2, _ = _run(dev, q, k, v, docs, 0, 0.1, bad)
    assert torch.equal(out, out2)
    empty = pkv.PrefillBlockMask(torch.zeros_like(kv_num), kv_idx,
                                 torch.zeros_like(kv_num), bm.full_kv_indices, bm.docs, 0)
    out3, _ = _run(dev, q, k, v, docs, 0, 0.1, empty)
    assert torch.count_nonzero(out3) == 0


def test_prefill_bad_arguments(dev):
    docs = torch.zeros(8, dtype=torch.int32, device=dev)
    bm = pkv.prefill_block_mask(docs)
    q = torch.zeros((2, 8, 96), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pkv.BadArgError):       # D = 96 unsupported (64, 128, 256, 512 are)
        pkv.prefill_attn(q, q, q, bm, 0.1, q.clone())
    q = torch.zeros((3, 8, 64), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((2, 8, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pkv.BadArgError):       # Hq % Hkv != 0
        pkv.prefill_attn(q, k, k, bm, 0.1, q.clone())
    with pytest.raises(pkv.BadArgError):       # negative window
        pkv.prefill_block_mask(docs, -1)
    q = torch.zeros((2, 9, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pkv.BadArgError):       # mask built for another length
        pkv.prefill_attn(q, q, q, bm, 0.1, q.clone())


@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_prefill_rising_scores_rescale_every_tile(dev, D):
    """Scores that climb by about 16 (log2 units) per 64-key tile: every row's
    maximum outgrows the kept one on each new tile, so the kernel rescales
    its running output on every tile (the path random inputs rarely take)."""
    rng = np.random.default_rng(90 + D)
    L, Hq, Hkv = 700, 4, 2
    base = wl.randn_bf16(rng, (D,)).double().numpy()
    base = base / np.sqrt((base ** 2).sum()) * np.sqrt(D)          # |base|^2 = D
    a = np.arange(L) / 64.0                                          # +1 per tile
    q = torch.from_numpy(np.broadcast_to(base, (Hq, L, D)).copy()).to(torch.bfloat16)
    k = torch.from_numpy((a[None, :, None] * base[None, None, :]).repeat(Hkv, 0)).to(torch.bfloat16)
    v = wl.randn_bf16(rng, (Hkv, L, D))
    docs = np.zeros(L, np.int32)
    docs[400:] = 1
    scale = D ** -0.5
    out, _ = _run(dev, q, k, v, docs, 0, scale)
    ref = oracle.prefill_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                   docs, scale)
    _compare(f64(out), ref, v, _kept(docs))


def test_prefill_long_documents_sampled_rows(dev):
    """The long-document launch: 8 documents of 2048 tokens, 32 q / 8 kv
    heads, head_dim 128. Sampled query rows of every document (its first
    tokens, rows across it and its last rows, where 2048 keys are kept) are
    each compared, all heads, with the oracle's single-query attention over
    the row's kept keys; every sampled row keeping 16 or more keys is held to
    max abs 1e-2."""
    from oracle.attention import decode_attention_row
    rng = np.random.default_rng(78)
    L, Hq, Hkv, D, n = 8 * 2048, 32, 8, 128, 2048
    docs = np.repeat(np.arange(8), n).astype(np.int32)
    q = wl.randn_bf16(rng, (Hq, L, D))
    k = wl.randn_bf16(rng, (Hkv, L, D))
    v = wl.randn_bf16(rng, (Hkv, L, D))
    scale = D ** -0.5
    out, bm = _run(dev, q, k, v, docs, 0, scale)
    got = f64(out)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    within = np.r_[0, 1, 15, 16, rng.integers(17, n - 64, size=6), np.arange(n - 64, n, 16),
                   n - 1]
    G = Hq // Hkv
    errs, kept = [], []
    for d in range(8):
        for w_ in within:
            i = d * n + int(w_)
            js = np.arange(d * n, i + 1)
            ref = np.stack([decode_attention_row(qd[h, i], kd[h // G, js], vd[h // G, js],
                                                 scale)[0] for h in range(Hq)])
            errs.append(np.abs(got[:, i] - ref))
            kept.append(len(js))
    e = np.stack(errs, axis=1)                       # [Hq][rows][D]
    long_rows = np.array(kept) >= 16
    assert np.isfinite(got).all()
    assert e[:, long_rows].max() <= 1e-2, float(e[:, long_rows].max())
    assert e.mean() <= 1e-3, float(e.mean())


@pytest.mark.parametrize("D,window", [(256, 512), (512, 0)])
def test_prefill_gemma_layers_sampled_documents(dev, D, window):
    """The Gemma-4 E2B prefill launches: 64 packed prompts of U[100, 400]
    tokens, 8 q heads / 1 kv head, the sliding layer (D=256, window 512) and
    the full layer (D=512). Whole documents are checked against the oracle run
    on that document alone: the first, one in the middle and the last."""
    rng = np.random.default_rng(79 + D)
    lens = wl.uniform_lengths(rng, 64, 100, 400)
    docs = np.repeat(np.arange(64), lens).astype(np.int32)
    L, Hq, Hkv = len(docs), 8, 1
    q = wl.randn_bf16(rng, (Hq, L, D))
    k = wl.randn_bf16(rng, (Hkv, L, D))
    v = wl.randn_bf16(rng, (Hkv, L, D))
    scale = D ** -0.5
    out, bm = _run(dev, q, k, v, docs, window, scale)
    _check_mask(bm, docs, window)
    got = f64(out)
    starts = np.r_[0, np.cumsum(lens)]
    for d in (0, 31, 63):
        sl = slice(int(starts[d]), int(starts[d + 1]))
        ref = oracle.prefill_attention(q[:, sl].double().numpy(), k[:, sl].double().numpy(),
                                       v[:, sl].double().numpy(), docs[sl], scale, window=window)
        _compare(got[:, sl], ref, v, _kept(docs[sl], window))


def test_prefill_more_items_than_the_sorted_schedule_holds(dev):
    """A launch with more work items per CTA than the cost-sorted schedule's
    list holds (256), so every CTA walks its items round-robin instead:
    40,000 packed tokens of U[100, 400]-token documents, 128 q / 64 kv heads
    (one query block of two heads per item, 64 items per row tile, 40,000
    items), head_dim 64. Inputs are drawn on the GPU from a seeded generator;
    sampled rows of every head are compared with the oracle's single-query
    attention over the row's kept keys."""
    from oracle.attention import decode_attention_row
    rng = np.random.default_rng(80)
    lens = wl.uniform_lengths(rng, 200, 100, 400)
    docs = np.repeat(np.arange(len(lens)), lens)[:40000].astype(np.int32)
    L, Hq, Hkv, D = len(docs), 128, 64, 64
    assert L == 40000 and ((L + 63) // 64) * Hkv > 256 * torch.cuda.get_device_properties(
        dev).multi_processor_count
    g = torch.Generator(device=dev)
    g.manual_seed(81)
    q, k, v = (torch.randn((h, L, D), generator=g, device=dev).to(torch.bfloat16)
               for h in (Hq, Hkv, Hkv))
    scale = D ** -0.5
    bm = pkv.prefill_block_mask(torch.from_numpy(docs).to(dev), 0)
    out = torch.full((Hq, L, D), float("nan"), dtype=torch.bfloat16, device=dev)
    pkv.prefill_attn(q, k, v, bm, scale, out)
    torch.cuda.synchronize()
    starts = np.r_[0, np.flatnonzero(np.diff(docs)) + 1]
    rows = np.r_[0, 63, 64, 20000, 39999, rng.integers(1, L - 1, size=11)]
    G = Hq // Hkv
    errs, kept = [], []
    for i in rows:
        j0 = int(starts[np.searchsorted(starts, i, side="right") - 1])
        js = slice(j0, int(i) + 1)
        qd = q[:, i].double().cpu().numpy()
        kd, vd = k[:, js].double().cpu().numpy(), v[:, js].double().cpu().numpy()
        ref = np.stack([decode_attention_row(qd[h], kd[h // G], vd[h // G], scale)[0]
                        for h in range(Hq)])
        got = out[:, i].double().cpu().numpy()
        assert np.isfinite(got).all()
        errs.append(np.abs(got - ref))
        kept.append(int(i) + 1 - j0)
    e = np.stack(errs, axis=1)
    long_rows = np.array(kept) >= 16
    assert e[:, long_rows].max() <= 1e-2, float(e[:, long_rows].max())
    assert e.mean() <= 1e-3, float(e.mean())
