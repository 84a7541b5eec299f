"""One layer's decode step and a continuous-batching driver over the C ABI.

The step follows the write-then-attend order of "unsloth: compare
main...flex-moe-qwen3" · flex_gemma4_moe.py · attention forward: per-head
q/k RMSNorm, RoPE, the paged write of the new K/V, then attention over keys
0..pos. By default the whole step is one fused libpkv kernel (plus the split
combine); the three separate kernels remain available. Everything runs on
the caller's stream with fixed shapes, so a step can be captured in a CUDA
graph (the pages capture the decode step per batch bucket,
capture_decode_cudagraph).

The driver applies a schedule of finished / admitted requests to the
PageTable the way the pages' generate loop does (free on finish, assign a
new request, grow capacity by reserve before each decode step) and yields
the per-step batch_idx / input_pos / seq_lens.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import (PageTable, kv_append, paged_decode_attn, paged_decode_attn_splits,
               paged_decode_attn_workspace, paged_decode_step, paged_decode_step_ex,
               qk_norm_rope, qkv_norm_rope)


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    head_dim: int
    theta: float
    window: int = 0
    qk_norm: bool = False
    rope: bool = True
    rotary_dims: int = 0      # 0: all of head_dim; fewer: Gemma-4 proportional RoPE
    v_norm: bool = False      # Gemma-4 gain-free RMSNorm of the value
    k_eq_v: bool = False      # Gemma-4 K=V: the value is the raw k projection

    @property
    def gemma_options(self) -> bool:
        return bool(self.rotary_dims) or self.v_norm or self.k_eq_v


def alloc_cache(Hkv: int, n_pages: int, page_size: int, D: int, device, fill: str = "zeros"):
    """K and V caches, bf16 [Hkv][n_pages * page_size][D]."""
    shape = (Hkv, n_pages * page_size, D)
    if fill == "randn":
        k = torch.randn(shape, dtype=torch.bfloat16, device=device)
        v = torch.randn(shape, dtype=torch.bfloat16, device=device)
    else:
        k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
    return k, v


class AttnWorkspace:
    """Split mode and workspace for one (B, Hq, Hkv, D, table, window) shape.

    num_splits 0 is the automatic, length-balanced mode; the workspace is
    sized for the most parts a row can be cut into in that mode."""

    def __init__(self, B, Hq, Hkv, D, max_pages_per_seq, page_size, window, device,
                 num_splits: int = 0):
        self.splits = num_splits
        self.max_parts = num_splits or paged_decode_attn_splits(B, Hkv, D, max_pages_per_seq,
                                                                page_size, window)
        n = paged_decode_attn_workspace(B, Hq, D, self.max_parts)
        self.buf = torch.empty(n, dtype=torch.uint8, device=device) if n else None


def decode_layer_step(spec: LayerSpec, pt: PageTable, k_cache, v_cache, q, k, v, batch_idx,
                      input_pos, seq_lens, out, ws: AttnWorkspace, gamma_q=None, gamma_k=None,
                      eps: float = 1e-6, scale: float | None = None, err=None, stream=None,
                      table=None, fused: bool = True):
    """One layer's decode step: q/k norm + RoPE, K/V append, attention.

    fused (default, rotary layers): one paged_decode_step(_ex) call; q, k and
    v are read only and seq_lens must equal input_pos + 1 (the kernel derives
    it). Otherwise the chain qk_norm_rope (qkv_norm_rope with the Gemma-4
    options) -> kv_append -> paged_decode_attn, which rotates q and k (and
    normalises v) in place; both give the same bits.

    `pt` supplies the table geometry (n_slots, max_pages_per_seq, page_size,
    n_pages) and, unless `table` is given, the device table itself."""
    table = pt.dev_table if table is None else table
    scale = scale if scale is not None else spec.head_dim ** -0.5
    gq = gamma_q if spec.qk_norm else None
    gk = gamma_k if spec.qk_norm else None
    if spec.gemma_options and not spec.rope:
        raise ValueError("rotary_dims, v_norm and k_eq_v need a rotary layer")
    if fused and spec.rope:
        if spec.gemma_options:
            paged_decode_step_ex(q, k, v, gq, gk, batch_idx, input_pos, spec.theta, eps,
                                 spec.rotary_dims or None, spec.v_norm, spec.k_eq_v, table,
                                 pt.n_slots, pt.max_pages_per_seq, pt.page_size, pt.n_pages,
                                 k_cache, v_cache, spec.window, scale, ws.splits, ws.buf, out,
                                 err, stream=stream)
        else:
            paged_decode_step(q, k, v, gq, gk, batch_idx, input_pos, spec.theta, eps, table,
                              pt.n_slots, pt.max_pages_per_seq, pt.page_size, pt.n_pages,
                              k_cache, v_cache, spec.window, scale, ws.splits, ws.buf, out,
                              err, stream=stream)
        return
    if spec.k_eq_v:
        v = k.clone()        # the raw k row, before k is rotated in place
    if spec.gemma_options:
        qkv_norm_rope(q, k, v if spec.v_norm else None, gq, gk, input_pos, spec.theta, eps,
                      spec.rotary_dims or None, stream=stream)
    elif spec.rope:
        qk_norm_rope(q, k, gq, gk, input_pos, spec.theta, eps, stream=stream)
    kv_append(k, v, batch_idx, input_pos, table, pt.n_slots, pt.max_pages_per_seq,
              pt.page_size, pt.n_pages, k_cache, v_cache, err, stream=stream)
    paged_decode_attn(q, k_cache, v_cache, table, pt.n_slots, pt.max_pages_per_seq,
                      pt.page_size, pt.n_pages, batch_idx, seq_lens, spec.window, scale,
                      ws.splits, ws.buf, out, err, stream=stream)


@dataclasses.dataclass
class StepMeta:
    batch_idx: np.ndarray      # int32 [B] slot of each row
    input_pos: np.ndarray      # int32 [B] position of the token appended
    seq_lens: np.ndarray       # int32 [B] input_pos + 1
    admitted: list             # [(lane, slot, prompt_len)] new this step


class RolloutDriver:
    """Applies a workloads.RolloutSchedule to a PageTable (host allocator)."""

    def __init__(self, pt: PageTable, schedule):
        self.pt = pt
        self.sched = schedule
        self.slots = []
        self.length = []
        self.t = 0
        first = []
        for lane, r in enumerate(schedule.first):
            s = pt.assign(r.prompt_len + 1)
            self.slots.append(s)
            self.length.append(r.prompt_len)
            first.append((lane, s, r.prompt_len))
        self.pending = first

    def next_step(self) -> StepMeta:
        t = self.t
        admitted = self.pending
        self.pending = []
        for lane in self.sched.finish[t]:
            self.pt.free(self.slots[lane])
        for lane, r in self.sched.start[t]:
            s = self.pt.assign(r.prompt_len + 1)
            self.slots[lane] = s
            self.length[lane] = r.prompt_len
            admitted.append((lane, s, r.prompt_len))
        pos = np.array(self.length, dtype=np.int32)
        for lane in range(self.sched.lanes):
            self.pt.reserve(self.slots[lane], int(pos[lane]) + 1)
            self.length[lane] += 1
        self.t += 1
        return StepMeta(np.array(self.slots, dtype=np.int32), pos, pos + 1, admitted)
