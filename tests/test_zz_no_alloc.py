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


def test_noalloc_accepts_split_counts_beyond_the_rows_tiles(dev):
    # num_splits is capped at the tiles of the longest row the table holds
    # (here 2 pages of 64 keys, so 2 parts), as paged_decode_attn caps it: a
    # huge split count needs only a few KB of scratch and gives the same result
    case = PagedCase(np.random.default_rng(44), 3, 16, 2, 128, 64, [100, 7, 128])
    scale = 1.0 / math.sqrt(case.D)
    for _ in range(2):
        got, err = _noalloc(case, dev, 0, scale, 2100)
        assert pkv.pkv_read_error_word(err) == 0
        want, _ = run_attn(pkv, case, dev, 0, scale, 2100)
        assert_attn_close(f64(got), f64(want))
        ref, _ = case.oracle(0, scale)
        assert_attn_close(f64(got), ref)


@pytest.mark.parametrize("splits", [0, 33])
def test_noalloc_rejects_partials_beyond_its_scratch(dev, splits):
    # 64 rows x 8 heads x D=512 with a table of 40 pages of 64 keys: the
    # automatic mode may cut a row into 40 parts, 64*8*40*(512+1)*4 bytes
    # (42 MB); a fixed 33 parts need 64*8*33*513*4 bytes (34.7 MB). Both are
    # beyond the 32 MiB scratch; the call is refused before any launch.
    case = PagedCase(np.random.default_rng(43), 64, 8, 1, 512, 64, [10] * 64, max_pages=40)
    d = case.device(dev)
    out = torch.empty((64, 8, 512), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pkv.BadArgError, match="scratch"):
        pkv.paged_decode_attn_noalloc(d["q"], d["kc"], d["vc"], d["table"], case.n_slots,
                                      case.max_pages, case.ps, case.P, d["bidx"], d["lens"], 0,
                                      0.04, splits, out)


def test_noalloc_accepts_the_largest_split_count_that_fits(dev):
    # the same table with 31 fixed parts: 64*8*31*513*4 bytes plus the part
    # counts, just under 32 MiB, so the call runs and matches paged_decode_attn
    case = PagedCase(np.random.default_rng(45), 64, 8, 1, 512, 64,
                     np.random.default_rng(46).integers(1, 300, size=64), max_pages=40)
    assert pkv.paged_decode_attn_workspace(64, 8, 512, 31) <= 32 << 20
    assert pkv.paged_decode_attn_workspace(64, 8, 512, 32) > 32 << 20
    scale = 1.0 / math.sqrt(case.D)
    got, err = _noalloc(case, dev, 0, scale, 31)
    assert pkv.pkv_read_error_word(err) == 0
    want, _ = run_attn(pkv, case, dev, 0, scale, 31)
    assert_attn_close(f64(got), f64(want))
