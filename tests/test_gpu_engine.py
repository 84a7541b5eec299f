"""GPU check of the bucketed decode graphs (engine.DecodeGraphs): a batch of
B rows replayed through the graph of its bucket (padding rows on the
reserved slot 0) gives the same output bits and the same cache bytes (outside
the reserved page 0) as the eager layer step on the same B rows."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import bits

pytestmark = pytest.mark.gpu
pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")
from paged_kv_decode_pagetable_gb300 import engine  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    return torch.device("cuda:0")


def test_bucketed_graph_replay_equals_eager(dev):
    rng = np.random.default_rng(90)
    max_bs, Hq, Hkv, D, ps, P, mp = 16, 8, 2, 128, 64, 200, 16
    spec = engine.LayerSpec(D, 1e6, 0, True, True)
    pt = pkv.PageTable(max_bs, ps, P, mp, device=dev)
    kc, vc = engine.alloc_cache(Hkv, P, ps, D, dev, fill="randn")
    gq, gk = wl.gamma_bf16(rng, D).to(dev), wl.gamma_bf16(rng, D).to(dev)
    lens = rng.integers(30, 700, size=11)
    slots = [pt.assign(int(L) + 1) for L in lens]
    graphs = engine.DecodeGraphs(spec, pt, kc, vc, Hq, max_bs, dev, gq, gk)
    for B, rows in ((5, [0, 3, 4, 7, 9]), (3, [1, 2, 10]), (11, list(range(11))), (1, [6])):
        q = wl.randn_bf16(rng, (B, Hq, D)).to(dev)
        k = wl.randn_bf16(rng, (B, Hkv, D)).to(dev)
        v = wl.randn_bf16(rng, (B, Hkv, D)).to(dev)
        bidx = torch.tensor([slots[r] for r in rows], dtype=torch.int32, device=dev)
        pos = torch.tensor([int(lens[r]) for r in rows], dtype=torch.int32, device=dev)
        kc_e, vc_e = kc.clone(), vc.clone()
        out_e = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = engine.AttnWorkspace(B, Hq, Hkv, D, mp, ps, 0, dev)
        engine.decode_layer_step(spec, pt, kc_e, vc_e, q, k, v, bidx, pos, pos + 1, out_e, ws,
                                 gq, gk, err=err)
        out_g = graphs.step(q, k, v, bidx, pos)
        torch.cuda.synchronize()
        assert pkv.pkv_read_error_word(err) == 0 and pkv.pkv_read_error_word(graphs.err) == 0
        assert np.array_equal(bits(out_g), bits(out_e)), B
        assert np.array_equal(bits(kc)[:, ps:], bits(kc_e)[:, ps:])
        assert np.array_equal(bits(vc)[:, ps:], bits(vc_e)[:, ps:])
        for r in rows:              # the appended token is now part of the sequence
            lens[r] += 1
            pt.reserve(slots[r], int(lens[r]) + 1)
