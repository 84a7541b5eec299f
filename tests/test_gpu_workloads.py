"""End-to-end GPU parity on the five workloads (C ABI, real allocator).

Each step runs the layer step as the product does (the fused
paged_decode_step, or the chain qk_norm_rope -> kv_append ->
paged_decode_attn) and is compared with the oracle:
  * the device page table equals the oracle allocator's table (bit-exact);
  * q/k after norm+RoPE are within one bf16 rounding of the oracle (for
    the fused step, which leaves q and k unrotated, the rotation is
    recomputed with qk_norm_rope, whose bits the fused kernel reproduces);
  * the appended cache rows equal the GPU's roped k / raw v (bit-exact);
  * attention equals the oracle fed the GPU's own bf16 q and cache
    (max abs <= 1e-2, mean abs <= 1e-3); on the last step of each workload
    the oracle chain from the raw inputs is held to the same bar.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import assert_attn_close, bits, bits_to_f64, f64

pytestmark = pytest.mark.gpu
pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")
from paged_kv_decode_pagetable_gb300 import engine  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    return torch.device("cuda:0")


def _prefill(rng, pt, caches, slot, n, Hkv, dev):
    """Fill tokens 0..n-1 of a slot with random bf16 K/V through kv_append."""
    if n == 0:
        return
    bidx = torch.full((n,), slot, dtype=torch.int32, device=dev)
    pos = torch.arange(n, dtype=torch.int32, device=dev)
    for kc, vc in caches:
        D = kc.shape[2]
        k = wl.randn_bf16(rng, (n, Hkv, D)).to(dev)
        v = wl.randn_bf16(rng, (n, Hkv, D)).to(dev)
        pkv.kv_append(k, v, bidx, pos, pt.dev_table, pt.n_slots, pt.max_pages_per_seq,
                      pt.page_size, pt.n_pages, kc, vc, None)


def _check_step(w, spec, pt, model, kc, vc, q_raw, k_raw, v_raw, q_gpu, k_gpu, v_gpu, out,
                meta, gq, gk, check_chain):
    table = pt.dev_table.cpu().numpy()
    assert np.array_equal(table, model.table)
    pos = meta.input_pos
    # prologue
    if spec.rope:
        rq, rk = oracle.qk_norm_rope(q_raw.double().numpy(), k_raw.double().numpy(),
                                     None if gq is None else gq.double().numpy(),
                                     None if gk is None else gk.double().numpy(),
                                     pos, spec.theta, w.eps, norm=spec.qk_norm,
                                     rotary_dims=spec.rotary_dims or None)
        rv = (k_raw if spec.k_eq_v else v_raw).double().numpy()
        if spec.v_norm:
            rv = oracle.v_norm(rv, w.eps)
        for got, ref in ((f64(q_gpu), rq), (f64(k_gpu), rk), (f64(v_gpu), rv)):
            assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2e-3).all()
    # appended rows hold exactly the GPU's k and v
    kb, vb = bits(kc), bits(vc)
    for b in range(w.batch):
        row = oracle.physical_row(model.table, int(meta.batch_idx[b]), int(pos[b]), w.page_size)
        assert np.array_equal(kb[:, row, :], bits(k_gpu)[b])
        assert np.array_equal(vb[:, row, :], bits(v_gpu)[b])
    # attention on the GPU's own inputs
    scale = spec.head_dim ** -0.5
    ref, _ = oracle.decode_attention(f64(q_gpu), bits_to_f64(kb), bits_to_f64(vb), model.table,
                                     meta.batch_idx, meta.seq_lens, spec.window, scale,
                                     w.page_size)
    assert_attn_close(f64(out), ref)
    if check_chain and spec.rope:
        # oracle chain from the raw inputs: exact cached prefix, unrounded new rows
        kf, vf = bits_to_f64(kb), bits_to_f64(vb)
        for b in range(w.batch):
            row = oracle.physical_row(model.table, int(meta.batch_idx[b]), int(pos[b]),
                                      w.page_size)
            kf[:, row, :] = rk[b]
            vf[:, row, :] = rv[b]
        ref2, _ = oracle.decode_attention(rq, kf, vf, model.table, meta.batch_idx,
                                          meta.seq_lens, spec.window, scale, w.page_size)
        assert_attn_close(f64(out), ref2)


def _rotated(spec, q_raw, k_raw, v_raw, gq, gk, pos, eps, dev):
    """The q, k and v the step attended with and appended, recomputed with
    qkv_norm_rope on copies of the raw inputs (the chain's in-place results
    and the fused kernel reproduce these bits)."""
    qr, kr = q_raw.to(dev), k_raw.to(dev)
    vr = (k_raw if spec.k_eq_v else v_raw).to(dev)
    if not spec.rope:
        return qr, kr, vr
    g = (lambda t: None if t is None or not spec.qk_norm else t.to(dev))
    pkv.qkv_norm_rope(qr, kr, vr if spec.v_norm else None, g(gq), g(gk), pos, spec.theta, eps,
                      spec.rotary_dims or None)
    return qr, kr, vr


def _specs(w):
    rope = w.name != "tiny"
    return [engine.LayerSpec(l.head_dim, l.theta, l.window, l.qk_norm, rope, l.rotary_dims,
                             l.v_norm, l.k_eq_v) for l in w.layers]


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("name,steps", [("qwen3", 64), ("llama", 4), ("gemma", 2)])
def test_static_workload(dev, name, steps, fused):
    w = wl.WORKLOADS[name]
    rng = np.random.default_rng(w.seed())
    pt = pkv.PageTable(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq, device=dev)
    model = oracle.PageTableModel(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq)
    specs = _specs(w)
    caches = [engine.alloc_cache(w.n_kv_heads, w.n_pages, w.page_size, s.head_dim, dev)
              for s in specs]
    lens0 = wl.static_lengths(w)
    slots = []
    for L in lens0:
        s = pt.assign(int(L) + 1)
        assert s == model.assign(int(L) + 1)
        slots.append(s)
        _prefill(rng, pt, caches, s, int(L), w.n_kv_heads, dev)
    gammas = [(wl.gamma_bf16(rng, s.head_dim), wl.gamma_bf16(rng, s.head_dim)) if s.qk_norm
              else (None, None) for s in specs]
    wss = [engine.AttnWorkspace(w.batch, w.n_q_heads, w.n_kv_heads, s.head_dim,
                                w.max_pages_per_seq, w.page_size, s.window, dev) for s in specs]
    length = [int(L) for L in lens0]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    check_at = {0, steps - 1}
    for t in range(steps):
        for b, s in enumerate(slots):
            pt.reserve(s, length[b] + 1)
            model.reserve(s, length[b] + 1)
        pos = np.array(length, np.int32)
        meta = engine.StepMeta(np.array(slots, np.int32), pos, pos + 1, [])
        d_bidx = torch.from_numpy(meta.batch_idx).to(dev)
        d_pos = torch.from_numpy(pos).to(dev)
        d_lens = torch.from_numpy(meta.seq_lens).to(dev)
        for li, spec in enumerate(specs):
            D = spec.head_dim
            q_raw = wl.randn_bf16(rng, (w.batch, w.n_q_heads, D))
            k_raw = wl.randn_bf16(rng, (w.batch, w.n_kv_heads, D))
            v_raw = wl.randn_bf16(rng, (w.batch, w.n_kv_heads, D))
            q, k, v = q_raw.to(dev), k_raw.to(dev), v_raw.to(dev)
            gq, gk = gammas[li]
            out = torch.empty((w.batch, w.n_q_heads, D), dtype=torch.bfloat16, device=dev)
            kc, vc = caches[li]
            engine.decode_layer_step(spec, pt, kc, vc, q, k, v, d_bidx, d_pos, d_lens, out,
                                     wss[li], None if gq is None else gq.to(dev),
                                     None if gk is None else gk.to(dev), w.eps, err=err,
                                     fused=fused)
            torch.cuda.synchronize()
            if t in check_at:
                qr, kr, vr = _rotated(spec, q_raw, k_raw, v_raw, gq, gk, d_pos, w.eps, dev)
                _check_step(w, spec, pt, model, kc, vc, q_raw, k_raw, v_raw, qr, kr, vr, out,
                            meta, gq, gk, check_chain=(t == steps - 1))
        length = [L + 1 for L in length]
    assert pkv.pkv_read_error_word(err) == 0


def test_tiny_workload_permuted_pages(dev):
    """B=2, 2/1 heads, D=64, page 16, seq_lens {37, 5}, 8 pages placed by a
    seeded permutation; one kv_append then one decode step."""
    w = wl.TINY
    rng = np.random.default_rng(w.seed())
    perm = wl.page_permutation(rng, w.n_pages)
    lens0 = wl.static_lengths(w)
    table = np.full((w.n_slots, w.max_pages_per_seq), -1, np.int32)
    table[0] = 0
    it = iter(perm)
    for b, L in enumerate(lens0 + 1):
        for blk in range(-(-int(L) // w.page_size)):
            table[b + 1, blk] = next(it)
    D = 64
    kc = wl.randn_bf16(rng, (1, w.n_pages * w.page_size, D))
    vc = wl.randn_bf16(rng, (1, w.n_pages * w.page_size, D))
    q = wl.randn_bf16(rng, (2, 2, D))
    k = wl.randn_bf16(rng, (2, 1, D))
    v = wl.randn_bf16(rng, (2, 1, D))
    bidx = np.array([1, 2], np.int32)
    pos = lens0.astype(np.int32)
    d = lambda a: torch.from_numpy(a).to(dev)
    dkc, dvc = kc.to(dev), vc.to(dev)
    pkv.kv_append(k.to(dev), v.to(dev), d(bidx), d(pos), d(table), w.n_slots,
                  w.max_pages_per_seq, w.page_size, w.n_pages, dkc, dvc, None)
    ref_k, ref_v = bits(kc).copy(), bits(vc).copy()
    assert oracle.kv_append(ref_k, ref_v, bits(k), bits(v), table, bidx, pos, w.page_size,
                            w.n_pages) == 0
    assert np.array_equal(bits(dkc), ref_k) and np.array_equal(bits(dvc), ref_v)
    for S in (0, 1, 2, 3):
        nsp = S or pkv.paged_decode_attn_splits(2, 1, D, w.max_pages_per_seq, w.page_size, 0)
        n = pkv.paged_decode_attn_workspace(2, 2, D, nsp)
        ws = torch.zeros(n, dtype=torch.uint8, device=dev) if n else None
        out = torch.empty((2, 2, D), dtype=torch.bfloat16, device=dev)
        pkv.paged_decode_attn(q.to(dev), dkc, dvc, d(table), w.n_slots, w.max_pages_per_seq,
                              w.page_size, w.n_pages, d(bidx), d(pos + 1), 0, 0.125, S, ws, out)
        torch.cuda.synchronize()
        ref, _ = oracle.decode_attention(q.double().numpy(), bits_to_f64(ref_k),
                                         bits_to_f64(ref_v), table, bidx, pos + 1, 0, 0.125,
                                         w.page_size)
        assert_attn_close(f64(out), ref)


@pytest.mark.parametrize("fused", [True, False])
def test_rollout_continuous_batching(dev, fused):
    """64 slots, 512 steps; finished sequences free their slot and pages and
    new prompts take them at once, so placement fragments."""
    w = wl.ROLLOUT
    rng = np.random.default_rng(w.seed())
    sched = wl.rollout_schedule(w)
    pt = pkv.PageTable(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq, device=dev)
    model = oracle.PageTableModel(w.max_batch_size, w.page_size, w.n_pages, w.max_pages_per_seq)
    model_slots = [model.assign(r.prompt_len + 1) for r in sched.first]
    model_len = [r.prompt_len for r in sched.first]
    drv = engine.RolloutDriver(pt, sched)
    assert drv.slots == model_slots
    spec = _specs(w)[0]
    D = spec.head_dim
    kc, vc = engine.alloc_cache(w.n_kv_heads, w.n_pages, w.page_size, D, dev)
    ws = engine.AttnWorkspace(w.batch, w.n_q_heads, w.n_kv_heads, D, w.max_pages_per_seq,
                              w.page_size, 0, dev)
    gq, gk = wl.gamma_bf16(rng, D), wl.gamma_bf16(rng, D)
    dgq, dgk = gq.to(dev), gk.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    check_at = {0, 1, 100, 255, 384, w.steps - 1}
    out = torch.empty((w.batch, w.n_q_heads, D), dtype=torch.bfloat16, device=dev)
    n_admitted = 0
    for t in range(w.steps):
        meta = drv.next_step()
        for lane in sched.finish[t]:
            model.free(model_slots[lane])
        for lane, r in sched.start[t]:
            model_slots[lane] = model.assign(r.prompt_len + 1)
            model_len[lane] = r.prompt_len
        for lane in range(w.batch):
            model.reserve(model_slots[lane], model_len[lane] + 1)
            model_len[lane] += 1
        assert meta.batch_idx.tolist() == model_slots
        for lane, slot, plen in meta.admitted:
            _prefill(rng, pt, [(kc, vc)], slot, plen, w.n_kv_heads, dev)
        n_admitted += len(meta.admitted)
        q_raw = wl.randn_bf16(rng, (w.batch, w.n_q_heads, D))
        k_raw = wl.randn_bf16(rng, (w.batch, w.n_kv_heads, D))
        v_raw = wl.randn_bf16(rng, (w.batch, w.n_kv_heads, D))
        q, k, v = q_raw.to(dev), k_raw.to(dev), v_raw.to(dev)
        d_pos = torch.from_numpy(meta.input_pos).to(dev)
        engine.decode_layer_step(spec, pt, kc, vc, q, k, v,
                                 torch.from_numpy(meta.batch_idx).to(dev), d_pos,
                                 torch.from_numpy(meta.seq_lens).to(dev), out, ws, dgq, dgk,
                                 w.eps, err=err, fused=fused)
        if t in check_at:
            torch.cuda.synchronize()
            qr, kr, vr = _rotated(spec, q_raw, k_raw, v_raw, gq, gk, d_pos, w.eps, dev)
            _check_step(w, spec, pt, model, kc, vc, q_raw, k_raw, v_raw, qr, kr, vr, out, meta,
                        gq, gk, check_chain=(t == w.steps - 1))
        elif t % 16 == 0:
            assert np.array_equal(pt.dev_table.cpu().numpy(), model.table), t
    torch.cuda.synchronize()
    assert pkv.pkv_read_error_word(err) == 0
    assert n_admitted > w.batch + 20     # the schedule really churned slots
