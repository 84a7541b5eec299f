"""GPU parity of each kernel against the CPU oracle, through the C ABI.

Bars: K/V scatter and error words bit-exact; attention max abs <= 1e-2 and
mean abs <= 1e-3 against the float64 oracle fed the same bf16 inputs;
qk_norm_rope within one bf16 rounding of the float64 oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import PagedCase, assert_attn_close, bits, bits_to_f64, f64, run_attn

pytestmark = pytest.mark.gpu

pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    return torch.device("cuda:0")


# ------------------------------------------------------------------ kv_append
@pytest.mark.parametrize("B,Hkv,D,ps", [(2, 1, 64, 16), (8, 8, 128, 64), (5, 2, 256, 32),
                                        (3, 1, 512, 64), (7, 3, 24, 8)])
def test_kv_append_bit_exact(dev, B, Hkv, D, ps):
    rng = np.random.default_rng(100 + B + D)
    P, max_pages = 4 * B + 2, 4
    table = np.full((B + 2, max_pages), -1, np.int32)
    table[0] = 0
    perm = rng.permutation(np.arange(1, P))
    table[1:B + 1] = perm[:4 * B].reshape(B, 4)
    bidx = rng.permutation(np.arange(1, B + 1)).astype(np.int32)
    pos = rng.integers(0, 4 * ps, size=B).astype(np.int32)
    kc = rng.integers(-2**15, 2**15, size=(Hkv, P * ps, D), dtype=np.int16)
    vc = rng.integers(-2**15, 2**15, size=(Hkv, P * ps, D), dtype=np.int16)
    k = rng.integers(-2**15, 2**15, size=(B, Hkv, D), dtype=np.int16)
    v = rng.integers(-2**15, 2**15, size=(B, Hkv, D), dtype=np.int16)
    t = lambda a: torch.from_numpy(a).to(dev)
    d_kc, d_vc = t(kc).view(torch.bfloat16), t(vc).view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.kv_append(t(k).view(torch.bfloat16), t(v).view(torch.bfloat16), t(bidx), t(pos), t(table),
                  B + 2, max_pages, ps, P, d_kc, d_vc, err)
    assert pkv.pkv_read_error_word(err) == 0
    ref_k, ref_v = kc.copy(), vc.copy()
    assert oracle.kv_append(ref_k, ref_v, k, v, table, bidx, pos, ps, P) == 0
    assert np.array_equal(bits(d_kc), ref_k)
    assert np.array_equal(bits(d_vc), ref_v)


def test_kv_append_multi_token_fill_and_identity_batch(dev):
    # prefill-style: many rows share a slot with distinct positions
    rng = np.random.default_rng(7)
    ps, P, D, Hkv, L = 16, 12, 64, 2, 70
    table = np.full((2, 8), -1, np.int32)
    table[0] = 0
    table[1, :5] = [9, 3, 11, 1, 6]
    k = rng.integers(-2**15, 2**15, size=(L, Hkv, D), dtype=np.int16)
    kc = np.zeros((Hkv, P * ps, D), np.int16)
    t = lambda a: torch.from_numpy(a).to(dev)
    d_kc, d_vc = t(kc).view(torch.bfloat16), t(kc.copy()).view(torch.bfloat16)
    bidx = np.ones(L, np.int32)
    pos = np.arange(L, dtype=np.int32)
    pkv.kv_append(t(k).view(torch.bfloat16), t(k).view(torch.bfloat16), t(bidx), t(pos), t(table),
                  2, 8, ps, P, d_kc, d_vc, None)
    got = bits(d_kc)
    for h in range(Hkv):
        assert np.array_equal(oracle.gather_pages(got, table, 1, h, L, ps), k[:, h, :])
    # batch_idx NULL means slot b for row b
    table2 = np.array([[0, 0], [2, 4], [5, 7]], np.int32)
    k2 = rng.integers(-2**15, 2**15, size=(3, Hkv, D), dtype=np.int16)
    pos2 = np.array([3, 20, 31], np.int32)
    d2 = torch.zeros((Hkv, P * ps, D), dtype=torch.bfloat16, device=dev)
    pkv.kv_append(t(k2).view(torch.bfloat16), t(k2).view(torch.bfloat16), None, t(pos2), t(table2),
                  3, 2, ps, P, d2, d2.clone(), None)
    ref = np.zeros((Hkv, P * ps, D), np.int16)
    oracle.kv_append(ref, ref.copy(), k2, k2, table2, None, pos2, ps, P)
    # row 0 writes the dummy page 0 through slot 0
    assert np.array_equal(bits(d2), ref)


def test_kv_append_error_bits_without_fault(dev):
    ps, P, D = 8, 6, 16
    table = np.array([[0, 0], [3, 9], [-1, -1]], np.int32)
    bidx = np.array([3, 1, 1, 2, 1, -1], np.int32)
    pos = np.array([0, 16, 8, 0, -1, 0], np.int32)
    k = np.ones((6, 1, D), np.int16)
    t = lambda a: torch.from_numpy(a).to(dev)
    kc = torch.zeros((1, P * ps, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.kv_append(t(k).view(torch.bfloat16), t(k).view(torch.bfloat16), t(bidx), t(pos), t(table),
                  3, 2, ps, P, kc, vc, err)
    ref_k = np.zeros((1, P * ps, D), np.int16)
    want = oracle.kv_append(ref_k, ref_k.copy(), k, k, table, bidx, pos, ps, P)
    assert pkv.pkv_read_error_word(err) == want
    assert want == (oracle.ERR_SLOT | oracle.ERR_POS | oracle.ERR_PAGE_RANGE | oracle.ERR_PAGE_NEG)
    assert not bits(kc).any() and not bits(vc).any()


def test_kv_append_prefill_packed_documents(dev):
    """The prefill scatter of packed tokens (head-major [Hkv][L][D], one slot
    and position per token, documents interleaved) equals the oracle's scatter
    of the same tokens, bit for bit, with invalid tokens reported and skipped."""
    rng = np.random.default_rng(77)
    Hkv, D, ps, P, max_pages = 3, 128, 16, 40, 6
    table = np.full((5, max_pages), -1, np.int32)
    table[0] = 0
    table[1:5] = rng.permutation(np.arange(1, P))[:4 * max_pages].reshape(4, max_pages)
    lens = [37, 5, 60, 1]                       # prompt lengths of slots 1..4
    slots = np.concatenate([np.full(n, s + 1) for s, n in enumerate(lens)]).astype(np.int32)
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    perm = rng.permutation(len(slots))           # the pages do not sort tokens by document
    slots, pos = slots[perm], pos[perm]
    slots[3], pos[7] = 9, max_pages * ps        # a bad slot and a position past the table
    L = len(slots)
    k = wl.randn_bf16(rng, (Hkv, L, D))
    v = wl.randn_bf16(rng, (Hkv, L, D))
    kc0 = wl.randn_bf16(rng, (Hkv, P * ps, D))
    vc0 = wl.randn_bf16(rng, (Hkv, P * ps, D))
    dkc, dvc = kc0.to(dev), vc0.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    d = lambda a: torch.from_numpy(a).to(dev)
    pkv.kv_append_prefill(k.to(dev), v.to(dev), d(slots), d(pos), d(table), 5, max_pages, ps, P,
                          dkc, dvc, err)
    ref_k, ref_v = bits(kc0).copy(), bits(vc0).copy()
    kt = bits(k).transpose(1, 0, 2).copy()       # token-major for the oracle
    vt = bits(v).transpose(1, 0, 2).copy()
    want = oracle.kv_append(ref_k, ref_v, kt, vt, table, slots, pos, ps, P)
    assert want == pkv.PKV_ERR_SLOT | pkv.PKV_ERR_POS
    assert pkv.pkv_read_error_word(err) == want
    assert np.array_equal(bits(dkc), ref_k) and np.array_equal(bits(dvc), ref_v)


# --------------------------------------------------------------- qk_norm_rope
def _norm_rope_bound(ref):
    # one bf16 rounding (relative 2^-9) of an fp32 result, with slack
    return 2.0 ** -8 * np.abs(ref) + 2e-3


@pytest.mark.parametrize("B,Hq,Hkv,D,theta,norm", [
    (8, 32, 8, 128, 1e6, True), (16, 24, 8, 128, 5e5, False), (3, 8, 1, 256, 1e4, True),
    (2, 8, 1, 512, 1e6, True), (5, 4, 2, 64, 1e4, True), (1, 3, 0, 80, 1e4, True)])
def test_qk_norm_rope_parity(dev, B, Hq, Hkv, D, theta, norm):
    rng = np.random.default_rng(B * 1000 + D)
    q = wl.randn_bf16(rng, (B, Hq, D))
    k = wl.randn_bf16(rng, (B, max(Hkv, 1), D))[:, :Hkv].contiguous()
    gq, gk = wl.gamma_bf16(rng, D), wl.gamma_bf16(rng, D)
    pos = rng.integers(0, 2100, size=B).astype(np.int32)
    pos[0] = 0
    dq, dk = q.to(dev), k.to(dev)
    pkv.qk_norm_rope(dq, dk if Hkv else None, gq.to(dev) if norm else None,
                     gk.to(dev) if (norm and Hkv) else None, torch.from_numpy(pos).to(dev),
                     theta, 1e-6)
    torch.cuda.synchronize()
    rq, rk = oracle.qk_norm_rope(q.double().numpy(), k.double().numpy(),
                                 gq.double().numpy(), gk.double().numpy(), pos, theta, 1e-6,
                                 norm=norm)
    for got, ref in ((f64(dq), rq), (f64(dk), rk)):
        if ref.size == 0:
            continue
        e = np.abs(got - ref)
        assert (e <= _norm_rope_bound(ref)).all(), e.max()
        # one rounding to bf16 averages a quarter ulp: <= 2^-9 of the magnitude
        assert e.mean() <= 2.0 ** -9 * np.abs(ref).mean() + 1e-4


@pytest.mark.parametrize("B,Hq,Hkv,D,theta,rd", [
    (4, 8, 1, 512, 1e6, 128), (6, 8, 1, 256, 1e4, 256), (5, 16, 4, 128, 1e6, 0),
    (3, 6, 2, 64, 1e4, 16)])
def test_qkv_norm_rope_partial_rotary_and_v_norm(dev, B, Hq, Hkv, D, theta, rd):
    """Gemma-4 options: RoPE on the leading rd dims (the rest pass through) and
    the gain-free RMSNorm of v, against the oracle; the pass-through dims of q
    and k equal the normalised inputs rounded once."""
    rng = np.random.default_rng(B * 7000 + D + rd)
    q = wl.randn_bf16(rng, (B, Hq, D))
    k = wl.randn_bf16(rng, (B, Hkv, D))
    v = wl.randn_bf16(rng, (B, Hkv, D), scale=3.0)
    gq, gk = wl.gamma_bf16(rng, D), wl.gamma_bf16(rng, D)
    pos = rng.integers(0, 2100, size=B).astype(np.int32)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    pkv.qkv_norm_rope(dq, dk, dv, gq.to(dev), gk.to(dev), torch.from_numpy(pos).to(dev), theta,
                      1e-6, rd)
    torch.cuda.synchronize()
    rq, rk = oracle.qk_norm_rope(q.double().numpy(), k.double().numpy(), gq.double().numpy(),
                                 gk.double().numpy(), pos, theta, 1e-6, rotary_dims=rd)
    rv = oracle.v_norm(v.double().numpy(), 1e-6)
    for got, ref in ((f64(dq), rq), (f64(dk), rk), (f64(dv), rv)):
        e = np.abs(got - ref)
        assert (e <= _norm_rope_bound(ref)).all(), e.max()
        assert e.mean() <= 2.0 ** -9 * np.abs(ref).mean() + 1e-4
    # with rotary_dims = D the call is qk_norm_rope bit for bit
    if rd == D:
        q2, k2 = q.to(dev), k.to(dev)
        pkv.qk_norm_rope(q2, k2, gq.to(dev), gk.to(dev), torch.from_numpy(pos).to(dev), theta,
                         1e-6)
        torch.cuda.synchronize()
        assert np.array_equal(bits(q2), bits(dq)) and np.array_equal(bits(k2), bits(dk))


# ----------------------------------------------------------- paged attention
ATTN_CASES = [
    # D, Hq, Hkv, ps, lens, window, splits
    (64, 2, 1, 16, [37, 5], 0, 0),
    (64, 2, 1, 16, [37, 5], 0, 1),
    (128, 32, 8, 64, [64, 1000, 1, 63, 65, 513], 0, 0),
    (128, 32, 8, 64, [64, 1000, 1, 63, 65, 513], 0, 3),
    (128, 24, 8, 64, [700, 1024, 512], 0, 1),
    (128, 12, 4, 8, [200, 9, 33], 0, 0),
    (128, 4, 4, 32, [130, 2], 0, 2),
    (256, 8, 1, 64, [2000, 300, 512, 513, 40], 512, 0),
    (256, 8, 1, 64, [2000, 300, 512, 513, 40], 512, 1),
    (256, 8, 1, 128, [777, 1500], 100, 3),
    (512, 8, 1, 64, [2048, 256, 1, 1111], 0, 0),
    (512, 8, 1, 64, [2048, 256, 1, 1111], 0, 1),
    (512, 16, 2, 16, [95, 300], 0, 4),
    (64, 7, 1, 256, [1, 300, 257], 0, 0),
    (128, 40, 8, 64, [333, 64], 65, 0),
    # one long row and few kv heads: the automatic mode cuts a (row, head) into
    # up to 128 parts (more than a warp's worth of flags, several merge batches)
    (128, 8, 1, 64, [8192], 0, 0),
    (64, 4, 2, 64, [5000, 3], 0, 0),
    (512, 8, 1, 64, [4096], 1500, 0),
]


@pytest.mark.parametrize("D,Hq,Hkv,ps,lens,window,splits", ATTN_CASES)
def test_paged_decode_attn_parity(dev, D, Hq, Hkv, ps, lens, window, splits):
    rng = np.random.default_rng(D + Hq + ps + sum(lens) + window)
    case = PagedCase(rng, len(lens), Hq, Hkv, D, ps, lens)
    scale = 1.0 / math.sqrt(D)
    out, err = run_attn(pkv, case, dev, window, scale, splits)
    assert pkv.pkv_read_error_word(err) == 0
    ref, _ = case.oracle(window, scale)
    assert_attn_close(f64(out), ref)


def test_splits_agree_and_many_splits(dev):
    rng = np.random.default_rng(5)
    case = PagedCase(rng, 6, 32, 8, 128, 64, [1000, 17, 640, 64, 129, 900])
    ref, _ = case.oracle(0, 0.0884)
    res = []
    for S in (1, 2, 5, 16, 0):
        out, _ = run_attn(pkv, case, dev, 0, 0.0884, S)
        res.append(f64(out))
        assert_attn_close(res[-1], ref)
    # split counts change the fp32 summation order and the max each split
    # rounds its bf16 P against; outputs (|o| < 1 here) may differ by about
    # one bf16 ulp at unit scale
    for r in res[1:]:
        d = np.abs(r - res[0])
        assert d.max() <= 2.0 ** -8 and d.mean() <= 1e-4, (d.max(), d.mean())


def test_workspace_reused_across_modes_is_left_zero(dev):
    """Cut rows leave their partials in the workspace as self-validating words
    (zero = not yet written) that the reader clears: one workspace serves
    automatic and fixed-split calls in any order, and after every completed
    call its partial area is zero again."""
    rng = np.random.default_rng(15)
    B, Hq, Hkv, D, ps = 5, 32, 8, 128, 64
    case = PagedCase(rng, B, Hq, Hkv, D, ps, [3000, 17, 640, 1900, 129])
    ref, _ = case.oracle(0, 0.0884)
    d = case.device(dev)
    p_auto = pkv.paged_decode_attn_splits(B, Hkv, D, case.max_pages, ps, 0)
    n = max(pkv.paged_decode_attn_workspace(B, Hq, D, P) for P in (p_auto, 5, 2))
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    counts = (B * Hq * 4 + 255) // 256 * 256       # the fixed mode's part counts come first
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for S in (0, 5, 0, 2, 0, 0):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
        pkv.paged_decode_attn(d["q"], d["kc"], d["vc"], d["table"], case.n_slots, case.max_pages,
                              ps, case.P, d["bidx"], d["lens"], 0, 0.0884, S, ws, out, err)
        torch.cuda.synchronize()
        assert pkv.pkv_read_error_word(err) == 0
        assert_attn_close(f64(out), ref)
        assert int(torch.count_nonzero(ws[counts:])) == 0, S


def test_empty_rows_and_noop_slot_give_zeros(dev):
    rng = np.random.default_rng(6)
    case = PagedCase(rng, 4, 8, 2, 128, 16, [50, 50, 50, 50])
    case.slots = np.array([1, 0, 3, 4], np.int32)     # row 1: the no-op slot
    case.lens = np.array([50, 50, 0, 50])             # row 2: empty
    for S in (1, 3):
        out, err = run_attn(pkv, case, dev, 0, 0.1, S)
        got = f64(out)
        assert pkv.pkv_read_error_word(err) == 0
        assert not got[1].any() and not got[2].any()
        ref, _ = case.oracle(0, 0.1)
        assert_attn_close(got, ref)


def test_attention_error_bits_without_fault(dev):
    rng = np.random.default_rng(8)
    case = PagedCase(rng, 3, 4, 1, 64, 16, [40, 40, 40])
    ref, _ = case.oracle(0, 0.125)
    case.table[2, 1] = case.P + 5          # page id beyond the cache
    case.table[3, 2] = -1                  # unreserved block inside the range
    out, err = run_attn(pkv, case, dev, 0, 0.125, 2)
    assert pkv.pkv_read_error_word(err) == (pkv.PKV_ERR_PAGE_RANGE | pkv.PKV_ERR_PAGE_NEG)
    # row 0 does not touch the bad entries and must still be right
    assert_attn_close(f64(out)[0:1], ref[0:1])
    # a length beyond the table row
    case3 = PagedCase(np.random.default_rng(9), 2, 4, 1, 64, 16, [40, 40])
    case3.lens = np.array([40, 40 + 16 * case3.max_pages])
    out, err = run_attn(pkv, case3, dev, 0, 0.125, 1)
    assert pkv.pkv_read_error_word(err) == pkv.PKV_ERR_POS
    # a batch index beyond the table: error bit, zero output for that row
    case3.lens = np.array([40, 40])
    case3.slots = np.array([1, case3.n_slots + 3], np.int32)
    out, err = run_attn(pkv, case3, dev, 0, 0.125, 1)
    assert pkv.pkv_read_error_word(err) == pkv.PKV_ERR_SLOT
    assert not f64(out)[1].any()


def test_bad_arguments_rejected_before_launch(dev):
    rng = np.random.default_rng(10)
    case = PagedCase(rng, 2, 4, 1, 64, 16, [100, 100])     # two 64-key tiles per row
    d = case.device(dev)
    out = torch.empty((2, 4, 64), dtype=torch.bfloat16, device=dev)

    def call(q=d["q"], kc=d["kc"], ps=case.ps, splits=2, ws=None):
        pkv.paged_decode_attn(q, kc, kc, d["table"], case.n_slots, case.max_pages, ps, case.P,
                              d["bidx"], d["lens"], 0, 0.1, splits, ws, out)

    with pytest.raises(pkv.BadArgError):
        call()                                            # split partials need a workspace
    with pytest.raises(pkv.BadArgError):
        call(ps=24, splits=1)                             # page size not a power of two
    with pytest.raises(pkv.BadArgError):
        call(q=torch.empty((2, 20, 64), dtype=torch.bfloat16, device=dev), splits=1)  # 20/1 > 8
    with pytest.raises(pkv.BadArgError):
        kc96 = torch.zeros((1, case.P * case.ps, 96), dtype=torch.bfloat16, device=dev)
        call(q=torch.empty((2, 4, 96), dtype=torch.bfloat16, device=dev), kc=kc96, splits=1)
    with pytest.raises(pkv.BadArgError):
        pkv.paged_decode_attn_splits(2, 0, 64, 4, 16, 0)


def test_graph_replay_is_bit_identical_to_eager(dev):
    """The pages' criterion for eager vs captured decode: exact match."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, ps = 8, 32, 8, 128, 64
    lens0 = rng.integers(64, 1024, size=B)
    case = PagedCase(rng, B, Hq, Hkv, D, ps, lens0 + 1, nan_fill=False)
    d = case.device(dev)
    k_new, v_new = wl.randn_bf16(rng, (B, Hkv, D)).to(dev), wl.randn_bf16(rng, (B, Hkv, D)).to(dev)
    gq, gk = wl.gamma_bf16(rng, D).to(dev), wl.gamma_bf16(rng, D).to(dev)
    pos = torch.from_numpy(lens0.astype(np.int32)).to(dev)
    S = 0    # automatic, length-balanced parts
    P = pkv.paged_decode_attn_splits(B, Hkv, D, case.max_pages, ps, 0)
    ws = torch.zeros(max(pkv.paged_decode_attn_workspace(B, Hq, D, P), 16), dtype=torch.uint8,
                     device=dev)
    bufs = dict(q=d["q"].clone(), k=k_new.clone(), kc=d["kc"].clone(), vc=d["vc"].clone(),
                out=torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev))
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        pkv.qk_norm_rope(bufs["q"], bufs["k"], gq, gk, pos, 1e6, 1e-6)
        pkv.kv_append(bufs["k"], v_new, d["bidx"], pos, d["table"], case.n_slots, case.max_pages,
                      ps, case.P, bufs["kc"], bufs["vc"], err)
        pkv.paged_decode_attn(bufs["q"], bufs["kc"], bufs["vc"], d["table"], case.n_slots,
                              case.max_pages, ps, case.P, d["bidx"], d["lens"], 0, 0.0884, S, ws,
                              bufs["out"], err)

    def reset():
        bufs["q"].copy_(d["q"])
        bufs["k"].copy_(k_new)
        bufs["kc"].copy_(d["kc"])
        bufs["vc"].copy_(d["vc"])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        reset()
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = bufs["out"].clone()
    eager_kc = bufs["kc"].clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        reset()
        bufs["out"].fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(bufs["out"].view(torch.int16), eager.view(torch.int16))
        assert torch.equal(bufs["kc"].view(torch.int16), eager_kc.view(torch.int16))
    assert pkv.pkv_read_error_word(err) == 0


# ------------------------------------------------------ fused prologue
@pytest.mark.parametrize("B,Hq,Hkv,D,ps,norm", [(8, 32, 8, 128, 64, True), (16, 24, 8, 128, 64, False),
                                                (5, 8, 1, 256, 16, True), (3, 8, 1, 512, 64, True),
                                                (4, 6, 3, 64, 8, True)])
def test_fused_prologue_equals_norm_rope_then_append(dev, B, Hq, Hkv, D, ps, norm):
    rng = np.random.default_rng(300 + B + D)
    P, max_pages = 4 * B + 3, 4
    table = np.full((B + 2, max_pages), -1, np.int32)
    table[0] = 0
    table[1:B + 1] = rng.permutation(np.arange(1, P))[:4 * B].reshape(B, 4)
    bidx = rng.permutation(np.arange(1, B + 1)).astype(np.int32)
    pos = rng.integers(0, 4 * ps, size=B).astype(np.int32)
    if B > 3:   # a bad slot, a position past the row and an unreserved block
        bidx[0], pos[1] = B + 5, 4 * ps + 3
        table[bidx[2], pos[2] // ps] = -1
    q = wl.randn_bf16(rng, (B, Hq, D))
    k = wl.randn_bf16(rng, (B, Hkv, D))
    v = wl.randn_bf16(rng, (B, Hkv, D))
    gq, gk = wl.gamma_bf16(rng, D), wl.gamma_bf16(rng, D)
    kc0 = wl.randn_bf16(rng, (Hkv, P * ps, D))
    vc0 = wl.randn_bf16(rng, (Hkv, P * ps, D))
    d = lambda a: torch.from_numpy(a).to(dev)
    outs = []
    for fused in (False, True):
        dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
        kc, vc = kc0.to(dev), vc0.to(dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        g1, g2 = (gq.to(dev), gk.to(dev)) if norm else (None, None)
        if fused:
            pkv.qk_norm_rope_append(dq, dk, dv, g1, g2, d(bidx), d(pos), 1e6, 1e-6, d(table),
                                    B + 2, max_pages, ps, P, kc, vc, err)
        else:
            pkv.qk_norm_rope(dq, dk, g1, g2, d(pos), 1e6, 1e-6)
            pkv.kv_append(dk, dv, d(bidx), d(pos), d(table), B + 2, max_pages, ps, P, kc, vc, err)
        outs.append([bits(t) for t in (dq, dk, kc, vc)] + [pkv.pkv_read_error_word(err)])
    for a, b in zip(outs[0][:4], outs[1][:4]):
        assert np.array_equal(a, b)
    assert outs[0][4] == outs[1][4]
    if B > 3:
        assert outs[1][4] == (pkv.PKV_ERR_SLOT | pkv.PKV_ERR_POS | pkv.PKV_ERR_PAGE_NEG)
