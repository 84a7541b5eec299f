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
    sized for the most parts a row can be cut into in that mode. It starts
    zeroed: a zero partial word is one not yet written in the current call
    (each call clears what it read, leaving the workspace zero)."""

    def __init__(self, B, Hq, Hkv, D, max_pages_per_seq, page_size, window, device,
                 num_splits: int = 0):
        self.splits = num_splits
        self.max_parts = num_splits or paged_decode_attn_splits(B, Hkv, D, max_pages_per_seq,
                                                                page_size, window)
        n = paged_decode_attn_workspace(B, Hq, D, self.max_parts)
        self.buf = torch.zeros(n, dtype=torch.uint8, device=device) if n else None


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


# --------------------------------------------------------------------------
# Batch buckets and the continuous-batching scheduler
# --------------------------------------------------------------------------

def bucket_ladder(max_bs: int) -> list:
    """The pages' CUDA-graph batch buckets (capture_decode_cudagraph):
    1, 2, 4, 8, then every multiple of 16 up to max_bs."""
    return [b for b in [1, 2, 4, 8] if b <= max_bs] + list(range(16, max_bs + 1, 16))


def bucket_for(B: int, ladder: list) -> int:
    """Smallest bucket holding B rows (a decode batch is padded up to it)."""
    for b in ladder:
        if b >= B:
            return b
    raise ValueError(f"batch {B} exceeds the largest bucket {ladder[-1]}")


@dataclasses.dataclass
class Sequence:
    rid: int
    prompt_len: int
    max_new_tokens: int
    generated: int = 0
    slot: int = -1
    finished: bool = False

    @property
    def total_length(self) -> int:
        return self.prompt_len + self.generated


class ContinuousBatcher:
    """The scheduling of the pages' generate loop ("unsloth: compare
    main...flex-moe-qwen3" · flex_gemma4_moe.py · generate) over a PageTable:

      * admission (prefill first): while the head of the waiting queue fits
        (can_reserve(total_length)), give it a slot reserved for its whole
        length; an admitted batch is prefilled and the loop starts over;
      * decode: each running sequence keeps its capacity or grows it by
        reserve; when it cannot, it goes back to the front of the queue and
        the newest running sequence is preempted (its slot and pages freed,
        it returns to the front of the waiting queue, keeping its tokens);
      * every prefill or decode appends one token; a sequence that reaches
        max_new_tokens finishes and frees its slot.

    The model work is supplied by prefill(batch) and decode(batch) callbacks
    (each gets the Sequence list; decode rows are in running order). events
    records ("prefill" | "decode", [rids]), ("preempt", rid) and ("finish",
    rid) in order."""

    def __init__(self, pt: PageTable, sequences, prefill=None, decode=None):
        import collections
        self.pt = pt
        self.waiting = collections.deque(sequences)
        self.running = collections.deque()
        self.done = []
        self.events = []
        self._prefill = prefill
        self._decode = decode

    def _finish_if_done(self, s: Sequence) -> bool:
        if s.generated >= s.max_new_tokens:
            s.finished = True
            self.done.append(s)
            self.pt.free(s.slot)
            self.events.append(("finish", s.rid))
            s.slot = -1
            return True
        return False

    def step(self) -> bool:
        """One pass of the loop; False once nothing is waiting or running."""
        if not (self.waiting or self.running):
            return False
        batch = []
        while self.waiting and self.pt.can_reserve(self.waiting[0].total_length):
            s = self.waiting.popleft()
            s.slot = self.pt.assign(s.total_length)
            batch.append(s)
        if batch:
            self.events.append(("prefill", [s.rid for s in batch]))
            if self._prefill:
                self._prefill(batch)
            for s in batch:
                s.generated += 1
                if not self._finish_if_done(s):
                    self.running.append(s)
            return True
        decode_batch = []
        while self.running:
            s = self.running.popleft()
            if self.pt.capacity(s.slot) >= s.total_length:
                decode_batch.append(s)
            elif self.pt.can_reserve(s.total_length, s.slot):
                self.pt.reserve(s.slot, s.total_length)
                decode_batch.append(s)
            else:
                self.running.appendleft(s)
                newest = self.running.pop()
                self.waiting.appendleft(newest)
                self.pt.free(newest.slot)
                newest.slot = -1
                self.events.append(("preempt", newest.rid))
        if not decode_batch:
            return True
        self.events.append(("decode", [s.rid for s in decode_batch]))
        if self._decode:
            self._decode(decode_batch)
        for s in decode_batch:
            s.generated += 1
            if not self._finish_if_done(s):
                self.running.append(s)
        return True

    def run(self, max_steps: int = 100000) -> list:
        for _ in range(max_steps):
            if not self.step():
                return self.done
        raise RuntimeError("scheduler did not drain")


class DecodeGraphs:
    """One CUDA graph of the decode layer step per batch bucket, as the pages'
    capture_decode_cudagraph does (graphs over static buffers, replayed after
    copying the step's inputs in). A batch of B rows replays the smallest
    bucket >= B; rows B.. of the bucket are padding rows on slot 0 (the
    reserved slot: no keys, zero output, their append lands in the reserved
    page 0). The page table is read through pt.dev_table, which the host
    allocator updates between steps."""

    def __init__(self, spec: LayerSpec, pt: PageTable, k_cache, v_cache, Hq: int, max_bs: int,
                 device, gamma_q=None, gamma_k=None, eps: float = 1e-6, ladder=None):
        self.spec, self.pt, self.kc, self.vc = spec, pt, k_cache, v_cache
        self.gq, self.gk, self.eps = gamma_q, gamma_k, eps
        self.ladder = ladder or bucket_ladder(max_bs)
        Hkv, D = k_cache.shape[0], k_cache.shape[2]
        bf = dict(dtype=torch.bfloat16, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.q = torch.zeros((max_bs, Hq, D), **bf)
        self.k = torch.zeros((max_bs, Hkv, D), **bf)
        self.v = torch.zeros((max_bs, Hkv, D), **bf)
        self.out = torch.zeros((max_bs, Hq, D), **bf)
        self.batch_idx = torch.zeros(max_bs, **i32)
        self.input_pos = torch.zeros(max_bs, **i32)
        self.seq_lens = torch.ones(max_bs, **i32)
        self.err = torch.zeros(1, **i32)
        self.ws = {b: AttnWorkspace(b, Hq, Hkv, D, pt.max_pages_per_seq, pt.page_size,
                                    spec.window, device) for b in self.ladder}
        self.graphs = {}
        for b in reversed(self.ladder):
            self._call(b)                  # eager first use of every kernel
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._call(b)
            self.graphs[b] = g
        torch.cuda.synchronize()

    def _call(self, b):
        decode_layer_step(self.spec, self.pt, self.kc, self.vc, self.q[:b], self.k[:b],
                          self.v[:b], self.batch_idx[:b], self.input_pos[:b],
                          self.seq_lens[:b], self.out[:b], self.ws[b], self.gq, self.gk,
                          self.eps, err=self.err)

    def step(self, q, k, v, batch_idx, input_pos):
        """Device tensors for B rows; returns the B rows of the output (a view
        of the static buffer, valid until the next step)."""
        B = q.shape[0]
        b = bucket_for(B, self.ladder)
        self.q[:B].copy_(q)
        self.k[:B].copy_(k)
        self.v[:B].copy_(v)
        self.batch_idx[:B].copy_(batch_idx)
        self.input_pos[:B].copy_(input_pos)
        self.seq_lens[:B].copy_(input_pos + 1)
        self.batch_idx[B:b].zero_()
        self.input_pos[B:b].zero_()
        self.seq_lens[B:b].fill_(1)
        self.graphs[b].replay()
        return self.out[:B]
