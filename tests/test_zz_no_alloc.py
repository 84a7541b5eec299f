"""paged_decode_attn_noalloc: the decode attention entry point for callers
that cannot allocate device memory (a C program with no device allocator
of its own, or a plugin whose host framework owns all device memory and
offers no scratch buffer). It must give the same results as
paged_decode_attn with a caller workspace, call after call, while keeping
its split partials in the library's own fixed device scratch.

This file is named so that pytest collects it last; it also passes when run
alone in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

from gpu_util import PagedCase, assert_attn_close, f64, run_attn

pytestmark = pytest.mark.gpu
pkv = pytest.importorskip("paged_kv_decode_pagetable_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    return torch.device("cuda:0")


def _noalloc(case, dev, window, scale, splits):
    d = case.device(dev)
    out = torch.full((case.B, case.Hq, case.D), float("nan"), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_decode_attn_noalloc(d["q"], d["kc"], d["vc"], d["table"], case.n_slots,
                                  case.max_pages, case.ps, case.P, d["bidx"], d["lens"], window,
                                  scale, splits, out, err)
    torch.cuda.synchronize()
    return out, err


def test_noalloc_matches_workspace_entry_point_on_two_calls(dev):
    # two different problems back to back: the second call must not see the
    # first call's partials left in the shared scratch
    cases = [
        (PagedCase(np.random.default_rng(41), 6, 32, 8, 128, 64, [1000, 17, 640, 64, 129, 900]),
         0, 3),
        (PagedCase(np.random.default_rng(42), 4, 8, 1, 256, 64, [2000, 300, 5, 1024]), 512, 0),
    ]
    for case, window, splits in cases:
        scale = 1.0 / math.sqrt(case.D)
        got, err = _noalloc(case, dev, window, scale, splits)
        assert pkv.pkv_read_error_word(err) == 0
        want, _ = run_attn(pkv, case, dev, window, scale, splits)
        assert_attn_close(f64(got), f64(want))
        ref, _ = case.oracle(window, scale)
        assert_attn_close(f64(got), ref)


def test_noalloc_rejects_partials_beyond_its_scratch(dev):
    case = PagedCase(np.random.default_rng(43), 2, 8, 1, 512, 64, [100, 100])
    d = case.device(dev)
    out = torch.empty((2, 8, 512), dtype=torch.bfloat16, device=dev)
    # 2 rows x 8 heads x 2100 splits x (512 + 1) x 4 bytes > 32 MiB
    with pytest.raises(pkv.BadArgError, match="scratch"):
        pkv.paged_decode_attn_noalloc(d["q"], d["kc"], d["vc"], d["table"], case.n_slots,
                                      case.max_pages, case.ps, case.P, d["bidx"], d["lens"], 0,
                                      0.04, 2100, out)
