"""GPU parity of the fused decode step (paged_decode_step) through the C ABI.

The fused step must equal the three-call chain qk_norm_rope -> kv_append ->
paged_decode_attn (seq_lens = input_pos + 1) bit for bit: the same output
bits, the same cache bytes and the same error word, with q, k and v left
unchanged. Before the step, every cache row that the step's append will
write holds a NaN, so an attention that read the row without the new token
would fail the comparison. The main case is also checked against the
float64 oracle end to end (max abs <= 1e-2, mean abs <= 1e-3).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import NAN_BF16, PagedCase, assert_attn_close, bits, bits_to_f64

pytestmark = pytest.mark.gpu

pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    return torch.device("cuda:0")


class StepCase:
    """A paged case for one decode step: row b appends at input_pos[b], so
    its pages cover input_pos[b] + 1 tokens; the append rows start as NaN."""

    def __init__(self, seed, B, Hq, Hkv, D, ps, pos, slots=None, norm=True, theta=1e6,
                 rotary_dims=None, v_norm=False, k_eq_v=False):
        rng = np.random.default_rng(seed)
        self.pos = np.asarray(pos, np.int32)
        self.case = PagedCase(rng, B, Hq, Hkv, D, ps, self.pos.astype(np.int64) + 1,
                              slots=slots)
        c = self.case
        for b in range(B):
            s = c.slots[b]
            if s == 0:
                continue
            p = int(self.pos[b])
            row = c.table[s, p // ps] * ps + p % ps
            c.kc_bits[:, row, :] = NAN_BF16
            c.vc_bits[:, row, :] = NAN_BF16
        self.k = wl.randn_bf16(rng, (B, Hkv, D))
        self.v = wl.randn_bf16(rng, (B, Hkv, D))
        self.gq = wl.gamma_bf16(rng, D) if norm else None
        self.gk = wl.gamma_bf16(rng, D) if norm else None
        self.theta = theta
        self.rotary_dims, self.v_norm, self.k_eq_v = rotary_dims, v_norm, k_eq_v

    @property
    def gemma(self):
        return self.rotary_dims is not None or self.v_norm or self.k_eq_v


def _ws(B, Hq, Hkv, D, max_pages, ps, window, splits, dev):
    P = splits or pkv.paged_decode_attn_splits(B, Hkv, D, max_pages, ps, window)
    n = pkv.paged_decode_attn_workspace(B, Hq, D, P)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=dev) if n else None


def run_chain_and_step(sc: StepCase, dev, window, splits, eps=1e-6, table=None):
    c = sc.case
    tbl = torch.from_numpy(c.table if table is None else table).to(dev)
    bidx = torch.from_numpy(c.slots).to(dev)
    pos = torch.from_numpy(sc.pos).to(dev)
    scale = c.D ** -0.5
    g = (lambda t: None if t is None else t.to(dev))
    res = {}
    for mode in ("chain", "step"):
        d = c.device(dev)
        q, k, v = c.q.to(dev), sc.k.to(dev), sc.v.to(dev)
        out = torch.full((c.B, c.Hq, c.D), float("nan"), dtype=torch.bfloat16, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = _ws(c.B, c.Hq, c.Hkv, c.D, c.max_pages, c.ps, window, splits, dev)
        if mode == "chain":
            vv = k.clone() if sc.k_eq_v else v.clone()
            if sc.gemma:
                pkv.qkv_norm_rope(q, k, vv if sc.v_norm else None, g(sc.gq), g(sc.gk), pos,
                                  sc.theta, eps, sc.rotary_dims)
            else:
                pkv.qk_norm_rope(q, k, g(sc.gq), g(sc.gk), pos, sc.theta, eps)
            pkv.kv_append(k, vv, bidx, pos, tbl, c.n_slots, c.max_pages, c.ps, c.P, d["kc"],
                          d["vc"], err)
            pkv.paged_decode_attn(q, d["kc"], d["vc"], tbl, c.n_slots, c.max_pages, c.ps, c.P,
                                  bidx, pos + 1, window, scale, splits, ws, out, err)
        elif sc.gemma:
            pkv.paged_decode_step_ex(q, k, None if sc.k_eq_v else v, g(sc.gq), g(sc.gk), bidx,
                                     pos, sc.theta, eps, sc.rotary_dims, sc.v_norm, sc.k_eq_v,
                                     tbl, c.n_slots, c.max_pages, c.ps, c.P, d["kc"], d["vc"],
                                     window, scale, splits, ws, out, err)
        else:
            pkv.paged_decode_step(q, k, v, g(sc.gq), g(sc.gk), bidx, pos, sc.theta, eps, tbl,
                                  c.n_slots, c.max_pages, c.ps, c.P, d["kc"], d["vc"], window,
                                  scale, splits, ws, out, err)
        torch.cuda.synchronize()
        res[mode] = dict(out=bits(out), kc=bits(d["kc"]), vc=bits(d["vc"]), q=bits(q), k=bits(k),
                         v=bits(v), err=pkv.pkv_read_error_word(err))
    return res


def assert_step_equals_chain(res, sc: StepCase):
    a, b = res["chain"], res["step"]
    assert a["err"] == b["err"], (a["err"], b["err"])
    assert np.array_equal(a["kc"], b["kc"]), "k cache differs"
    assert np.array_equal(a["vc"], b["vc"]), "v cache differs"
    diff = np.argwhere(a["out"] != b["out"])
    assert diff.size == 0, f"{len(diff)} output elements differ, first at {diff[:3].tolist()}"
    # inputs of the fused step are read only
    assert np.array_equal(b["q"], bits(sc.case.q))
    assert np.array_equal(b["k"], bits(sc.k)) and np.array_equal(b["v"], bits(sc.v))


def _positions(rng, B, lo, hi, ps):
    pos = rng.integers(lo, hi, size=B)
    # a new token at the first and at the last row of a 64-key tile and of a page
    edge = [0, 63, 64, ps - 1, ps, 127]
    for i, e in enumerate(edge[:B // 3]):
        pos[i] = min(e, hi - 1)
    return pos.astype(np.int32)


STEP_CASES = [
    # B, Hq, Hkv, D, ps, pos range, window, splits, norm
    (64, 32, 8, 128, 64, (0, 1024), 0, 0, True),     # rollout heads, automatic parts
    (64, 32, 8, 128, 64, (0, 1024), 0, 1, True),     # one part per row: direct output
    (16, 24, 8, 128, 64, (0, 1024), 0, 3, False),    # llama heads, no q/k norm, 3 parts
    (9, 4, 2, 64, 16, (0, 300), 40, 0, True),        # small pages, window
    (6, 8, 1, 256, 64, (0, 2100), 512, 0, True),     # gemma sliding layer
    (4, 8, 1, 512, 64, (0, 2100), 0, 0, True),       # gemma full layer
    (5, 6, 3, 64, 8, (0, 100), 0, 2, True),          # 8-token pages, G = 2
]


@pytest.mark.parametrize("B,Hq,Hkv,D,ps,pr,window,splits,norm", STEP_CASES)
def test_step_equals_chain(dev, B, Hq, Hkv, D, ps, pr, window, splits, norm):
    rng = np.random.default_rng(4000 + B + D + splits)
    pos = _positions(rng, B, pr[0], pr[1], ps)
    sc = StepCase(4100 + B + D, B, Hq, Hkv, D, ps, pos, norm=norm)
    res = run_chain_and_step(sc, dev, window, splits)
    assert res["step"]["err"] == 0
    assert_step_equals_chain(res, sc)


GEMMA_CASES = [
    # B, Hq, Hkv, D, ps, pos range, window, rotary_dims, v_norm, k_eq_v
    (12, 8, 1, 512, 64, (0, 2100), 0, 128, True, True),     # Gemma-4 full layer
    (12, 8, 1, 256, 64, (0, 2100), 512, None, True, False),  # Gemma-4 sliding layer
    (9, 16, 4, 128, 16, (0, 500), 0, 32, False, True),       # K=V without v_norm
    (7, 8, 2, 64, 64, (0, 300), 0, 0, True, False),          # no rotation at all
]


@pytest.mark.parametrize("B,Hq,Hkv,D,ps,pr,window,rd,vn,kv", GEMMA_CASES)
def test_step_gemma_options_equal_chain(dev, B, Hq, Hkv, D, ps, pr, window, rd, vn, kv):
    """paged_decode_step_ex (proportional RoPE, v_norm, K=V) against the chain
    qkv_norm_rope -> kv_append -> paged_decode_attn, bit for bit."""
    rng = np.random.default_rng(4600 + B + D)
    pos = _positions(rng, B, pr[0], pr[1], ps)
    sc = StepCase(4700 + B + D, B, Hq, Hkv, D, ps, pos, rotary_dims=rd, v_norm=vn, k_eq_v=kv)
    res = run_chain_and_step(sc, dev, window, 0)
    assert res["step"]["err"] == 0
    assert_step_equals_chain(res, sc)


def test_step_gemma_full_matches_oracle(dev):
    """The Gemma-4 full-layer step from raw inputs against the oracle: q/k
    RMSNorm, RoPE on the leading 128 of 512 dims, v = v_norm(raw k)."""
    rng = np.random.default_rng(4800)
    B, Hq, Hkv, D, ps = 10, 8, 1, 512, 64
    pos = _positions(rng, B, 0, 2000, ps)
    sc = StepCase(4801, B, Hq, Hkv, D, ps, pos, rotary_dims=128, v_norm=True, k_eq_v=True)
    c = sc.case
    res = run_chain_and_step(sc, dev, 0, 0)
    qd, kd = c.q.double().numpy(), sc.k.double().numpy()
    g = lambda t: t.double().numpy()
    qr, kr = oracle.qk_norm_rope(qd, kd, g(sc.gq), g(sc.gk), sc.pos, sc.theta, 1e-6,
                                 rotary_dims=128)
    vr = oracle.v_norm(kd, 1e-6)
    kc, vc = bits_to_f64(c.kc_bits), bits_to_f64(c.vc_bits)
    assert oracle.kv_append(kc, vc, kr, vr, c.table, c.slots, sc.pos, ps, c.P) == 0
    ref, _ = oracle.decode_attention(qr, kc, vc, c.table, c.slots, sc.pos + 1, 0, D ** -0.5, ps)
    assert_attn_close(bits_to_f64(res["step"]["out"]), ref)


def test_step_matches_oracle_end_to_end(dev):
    """Fused step from raw inputs against the oracle's norm + RoPE, append and
    attention in float64 (the bf16 roundings of q and of the appended k are
    the oracle's own, so this is the end-to-end bar, not bit identity)."""
    rng = np.random.default_rng(4200)
    B, Hq, Hkv, D, ps = 32, 32, 8, 128, 64
    pos = _positions(rng, B, 0, 1024, ps)
    sc = StepCase(4201, B, Hq, Hkv, D, ps, pos)
    c = sc.case
    res = run_chain_and_step(sc, dev, 0, 0)
    qd, kd, vd = (t.double().numpy() for t in (c.q, sc.k, sc.v))
    g = lambda t: t.double().numpy()
    qr, kr = oracle.qk_norm_rope(qd, kd, g(sc.gq), g(sc.gk), sc.pos, sc.theta, 1e-6)
    # append through the oracle's scatter on float64 copies of the caches
    kc, vc = bits_to_f64(c.kc_bits), bits_to_f64(c.vc_bits)
    assert oracle.kv_append(kc, vc, kr, vd, c.table, c.slots, sc.pos, ps, c.P) == 0
    ref, _ = oracle.decode_attention(qr, kc, vc, c.table, c.slots, sc.pos + 1, 0, D ** -0.5, ps)
    got = bits_to_f64(res["step"]["out"])
    assert_attn_close(got, ref)


def test_step_padding_rows_and_error_bits(dev):
    """Padding rows (slot 0) append into the reserved page and output zeros;
    a position past the table, an unreserved append block and an
    out-of-range slot set the same error bits as the chain, with no fault."""
    rng = np.random.default_rng(4300)
    B, Hq, Hkv, D, ps = 12, 16, 4, 128, 64
    pos = _positions(rng, B, 0, 500, ps)
    pos[[3, 7]] = [70, 11]        # distinct rows of the reserved page
    slots = np.arange(1, B + 1, dtype=np.int32)
    slots[[3, 7]] = 0
    sc = StepCase(4301, B, Hq, Hkv, D, ps, pos, slots=slots)
    c = sc.case
    res = run_chain_and_step(sc, dev, 0, 0)
    assert res["step"]["err"] == 0
    assert_step_equals_chain(res, sc)
    out = res["step"]["out"].reshape(B, Hq, D)
    assert (out[[3, 7]] == 0).all()
    # error rows: position past the table, -1 entry at the append block, bad slot
    table = c.table.copy()
    bad = sc.pos.copy()
    bad[0] = c.max_pages * ps + 5
    table[c.slots[1], int(sc.pos[1]) // ps] = -1
    sc.pos = bad
    slots_bad = c.slots.copy()
    slots_bad[2] = c.n_slots + 4
    c.slots = slots_bad
    res = run_chain_and_step(sc, dev, 0, 0, table=table)
    want = pkv.PKV_ERR_POS | pkv.PKV_ERR_PAGE_NEG | pkv.PKV_ERR_SLOT
    assert res["chain"]["err"] == want
    assert_step_equals_chain(res, sc)


def test_step_graph_replay_bit_identical(dev):
    """A CUDA graph of fused steps replays to the same bits as eager calls."""
    rng = np.random.default_rng(4400)
    B, Hq, Hkv, D, ps = 16, 32, 8, 128, 64
    sc = StepCase(4401, B, Hq, Hkv, D, ps, _positions(rng, B, 0, 900, ps))
    c = sc.case
    outs = []
    for graph in (False, True):
        d = c.device(dev)
        q, k, v = c.q.to(dev), sc.k.to(dev), sc.v.to(dev)
        gq, gk = sc.gq.to(dev), sc.gk.to(dev)
        pos = torch.from_numpy(sc.pos).to(dev)
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = _ws(B, Hq, Hkv, D, c.max_pages, ps, 0, 0, dev)

        def step():
            pkv.paged_decode_step(q, k, v, gq, gk, d["bidx"], pos, sc.theta, 1e-6, d["table"],
                                  c.n_slots, c.max_pages, ps, c.P, d["kc"], d["vc"], 0,
                                  D ** -0.5, 0, ws, out, err)

        step()   # first use outside capture
        torch.cuda.synchronize()
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            g.replay()
        else:
            step()
        torch.cuda.synchronize()
        outs.append((bits(out), bits(d["kc"]), pkv.pkv_read_error_word(err)))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
    assert outs[0][2] == outs[1][2] == 0


def test_step_bad_arguments_rejected(dev):
    B, Hq, Hkv, D, ps = 2, 4, 1, 64, 16
    sc = StepCase(4500, B, Hq, Hkv, D, ps, [5, 20])
    c = sc.case
    d = c.device(dev)
    pos = torch.from_numpy(sc.pos).to(dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    q, k, v = c.q.to(dev), sc.k.to(dev), sc.v.to(dev)
    gq = sc.gq.to(dev)
    with pytest.raises(pkv.BadArgError):   # one gain without the other
        pkv.paged_decode_step(q, k, v, gq, None, d["bidx"], pos, 1e4, 1e-6, d["table"],
                              c.n_slots, c.max_pages, ps, c.P, d["kc"], d["vc"], 0, 0.125, 1,
                              None, out)
    with pytest.raises(pkv.BadArgError):   # theta <= 0
        pkv.paged_decode_step(q, k, v, None, None, d["bidx"], pos, 0.0, 1e-6, d["table"],
                              c.n_slots, c.max_pages, ps, c.P, d["kc"], d["vc"], 0, 0.125, 1,
                              None, out)
