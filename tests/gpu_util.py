"""Helpers for the GPU parity tests: seeded paged layouts and oracle checks."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl

NAN_BF16 = np.int16(0x7FC0)   # quiet NaN bit pattern


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def bits_to_f64(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).double().numpy()


class PagedCase:
    """A seeded paged cache: rows 1..B own pages drawn from a permutation of
    1..P-1; every cache element that no row can read (page 0, unused pages,
    positions at or beyond a row's length) holds a NaN so that masking is
    exercised."""

    def __init__(self, rng, B, Hq, Hkv, D, ps, lens, extra_pages=3, slots=None,
                 nan_fill=True, max_pages=None):
        self.B, self.Hq, self.Hkv, self.D, self.ps = B, Hq, Hkv, D, ps
        self.lens = np.asarray(lens, dtype=np.int64)
        nb = [-(-int(L) // ps) for L in self.lens]
        self.P = sum(nb) + extra_pages + 1
        self.max_pages = max_pages or max(max(nb), 1)
        self.slots = np.arange(1, B + 1, dtype=np.int32) if slots is None else np.asarray(slots, np.int32)
        self.n_slots = int(max(self.slots.max(), B)) + 1
        self.table = np.full((self.n_slots, self.max_pages), -1, np.int32)
        self.table[0] = 0
        perm = rng.permutation(np.arange(1, self.P))
        it = iter(perm)
        for b in range(B):
            if self.slots[b] == 0:
                continue
            for blk in range(nb[b]):
                self.table[self.slots[b], blk] = next(it)
        kc = wl.randn_bf16(rng, (Hkv, self.P * ps, D)).view(torch.int16).numpy().copy()
        vc = wl.randn_bf16(rng, (Hkv, self.P * ps, D)).view(torch.int16).numpy().copy()
        if nan_fill:
            readable = np.zeros(self.P * ps, bool)
            for b in range(B):
                if self.slots[b] == 0:
                    continue
                for j in range(int(self.lens[b])):
                    readable[self.table[self.slots[b], j // ps] * ps + j % ps] = True
            kc[:, ~readable, :] = NAN_BF16
            vc[:, ~readable, :] = NAN_BF16
        self.kc_bits, self.vc_bits = kc, vc
        self.q = wl.randn_bf16(rng, (B, Hq, D))

    def device(self, dev):
        return dict(
            q=self.q.to(dev),
            kc=torch.from_numpy(self.kc_bits).view(torch.bfloat16).to(dev),
            vc=torch.from_numpy(self.vc_bits).view(torch.bfloat16).to(dev),
            table=torch.from_numpy(self.table).to(dev),
            bidx=torch.from_numpy(self.slots).to(dev),
            lens=torch.from_numpy(self.lens.astype(np.int32)).to(dev),
        )

    def oracle(self, window, scale, q=None):
        q = self.q.double().numpy() if q is None else q
        return oracle.decode_attention(q, bits_to_f64(self.kc_bits), bits_to_f64(self.vc_bits),
                                       self.table, self.slots, self.lens, window, scale, self.ps)


def run_attn(pkv, case, dev, window, scale, splits, err=None, out=None, q=None):
    d = case.device(dev)
    if q is not None:
        d["q"] = q
    P = splits or pkv.paged_decode_attn_splits(case.B, case.Hkv, case.D, case.max_pages,
                                               case.ps, window)
    ws_n = pkv.paged_decode_attn_workspace(case.B, case.Hq, case.D, P)
    ws = torch.zeros(max(ws_n, 16), dtype=torch.uint8, device=dev) if ws_n else None
    if out is None:
        out = torch.full((case.B, case.Hq, case.D), float("nan"), dtype=torch.bfloat16, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_decode_attn(d["q"], d["kc"], d["vc"], d["table"], case.n_slots, case.max_pages,
                          case.ps, case.P, d["bidx"], d["lens"], window, scale, splits, ws, out,
                          err)
    torch.cuda.synchronize()
    return out, err


def assert_attn_close(got: np.ndarray, ref: np.ndarray, max_abs=1e-2, mean_abs=1e-3):
    assert np.isfinite(got).all(), "non-finite output"
    e = np.abs(got - ref)
    assert e.max() <= max_abs and e.mean() <= mean_abs, (float(e.max()), float(e.mean()))
    return float(e.max()), float(e.mean())
