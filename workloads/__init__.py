"""Seeded synthetic inputs for the paged decode-attention workloads.

This module only draws random numbers and event schedules. It holds none of
the method's arithmetic (no paging, no norm, no rotary, no attention), so both
the CPU oracle and the CUDA path may consume what it produces.

Workloads (head shapes from the Qwen3-4B / Llama-3.2-3B / Gemma-4-E2B
rollouts described on "unsloth: tests @ 35231d4" · Wiring, and on
"unsloth: compare main...transformers-continuous-batching-qwen3" ·
scripts/benchmarks/README.md · Gemma-4 notes). The pages' prompt dataset is
not available here; uniform length draws stand in for it.

  tiny       B=2, Hq=2, Hkv=1, D=64, page 16, seq_lens {37, 5}, 8 physical
             pages placed by a seeded permutation, scale 1/8.
  qwen3      B=8, Hq=32, Hkv=8, D=128, page 64, L0 ~ U[64, 1024], 64 steps,
             q/k RMSNorm (eps 1e-6, gamma = 1 + 0.1 N(0,1)), theta 1e6.
  llama      B=16 (all slots live), Hq=24, Hkv=8, D=128, page 64,
             L ~ U[512, 1024], theta 5e5, no q/k norm.
  rollout    B=64 slots, Qwen3 heads, page 64, max_seq 1024, prompts
             ~ U[100, 400], 512 steps; each sequence stops at a seeded
             length in [L0 + 16, 1024] and its slot is refilled at once.
  gemma      B=64, Hq=8, Hkv=1, page 64, L ~ U[256, 2048]; sliding layer
             D=256, window 512, theta 1e4; full layer D=512, theta 1e6 with
             proportional RoPE over the leading 25% (128 dims) and K=V; q/k
             RMSNorm as qwen3 and the gain-free v RMSNorm on both layers.

The base seed 3407 is the seed the pages' drivers use.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BASE_SEED = 3407


@dataclasses.dataclass(frozen=True)
class LayerShape:
    head_dim: int
    theta: float
    window: int = 0          # <= 0: no sliding window
    qk_norm: bool = False
    rotary_dims: int = 0     # 0: rotary over all of head_dim (proportional RoPE: fewer)
    v_norm: bool = False     # gain-free RMSNorm of the value
    k_eq_v: bool = False     # value taken from the raw k projection


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int               # live rows per decode step
    max_batch_size: int      # user-visible slots (internal rows = +1)
    n_q_heads: int
    n_kv_heads: int
    page_size: int
    n_pages: int             # physical pages including reserved page 0
    max_seq: int             # longest sequence the table must hold
    layers: tuple            # one LayerShape per attention regime
    steps: int
    seed_offset: int
    eps: float = 1e-6

    @property
    def max_pages_per_seq(self) -> int:
        return -(-self.max_seq // self.page_size)

    @property
    def n_slots(self) -> int:
        return self.max_batch_size + 1

    def seed(self, salt: int = 0) -> int:
        return BASE_SEED + 1000 * self.seed_offset + salt


TINY = Workload("tiny", batch=2, max_batch_size=2, n_q_heads=2, n_kv_heads=1,
                page_size=16, n_pages=8, max_seq=48,
                layers=(LayerShape(64, 1e4),), steps=1, seed_offset=1)
QWEN3 = Workload("qwen3", batch=8, max_batch_size=8, n_q_heads=32, n_kv_heads=8,
                 page_size=64, n_pages=8 * 17 + 1, max_seq=1088,
                 layers=(LayerShape(128, 1e6, qk_norm=True),), steps=64, seed_offset=2)
LLAMA = Workload("llama", batch=16, max_batch_size=16, n_q_heads=24, n_kv_heads=8,
                 page_size=64, n_pages=16 * 17 + 1, max_seq=1088,
                 layers=(LayerShape(128, 5e5),), steps=4, seed_offset=3)
ROLLOUT = Workload("rollout", batch=64, max_batch_size=64, n_q_heads=32, n_kv_heads=8,
                   page_size=64, n_pages=64 * 16 + 1, max_seq=1024,
                   layers=(LayerShape(128, 1e6, qk_norm=True),), steps=512, seed_offset=4)
GEMMA = Workload("gemma", batch=64, max_batch_size=64, n_q_heads=8, n_kv_heads=1,
                 page_size=64, n_pages=64 * 33 + 1, max_seq=2112,
                 layers=(LayerShape(256, 1e4, window=512, qk_norm=True, v_norm=True),
                         LayerShape(512, 1e6, qk_norm=True, rotary_dims=128, v_norm=True,
                                    k_eq_v=True)),
                 steps=4, seed_offset=5)

WORKLOADS = {w.name: w for w in (TINY, QWEN3, LLAMA, ROLLOUT, GEMMA)}


# --------------------------------------------------------------------------
# random tensors
# --------------------------------------------------------------------------

def randn_bf16(rng: np.random.Generator, shape, scale: float = 1.0,
               offset: float = 0.0) -> torch.Tensor:
    """N(offset, scale^2) samples rounded to bf16 by torch (CPU tensor)."""
    x = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale)
    x += np.float32(offset)
    return torch.from_numpy(x).to(torch.bfloat16)


def gamma_bf16(rng: np.random.Generator, dim: int) -> torch.Tensor:
    """RMSNorm gains 1 + 0.1 N(0, 1), as bf16."""
    return randn_bf16(rng, (dim,), scale=0.1, offset=1.0)


def uniform_lengths(rng: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi] inclusive."""
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


def page_permutation(rng: np.random.Generator, n_pages: int) -> np.ndarray:
    """A seeded permutation of the usable physical pages 1..n_pages-1."""
    return rng.permutation(np.arange(1, n_pages, dtype=np.int64))


# --------------------------------------------------------------------------
# continuous-batching event schedule (allocator independent)
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Request:
    rid: int
    prompt_len: int
    final_len: int           # total tokens when the sequence stops


@dataclasses.dataclass
class RolloutSchedule:
    """Per-step events for a fixed set of batch lanes.

    Every lane always holds one live request. At the boundary before step t,
    `finish[t]` lists lanes whose request stopped (free its slot, in lane
    order) and `start[t]` lists (lane, Request) pairs admitted in the same
    lane order. Lanes keep their position in the batch, so row b of every
    step is lane b.
    """
    lanes: int
    steps: int
    first: list              # Request per lane at step 0
    finish: list             # list[list[lane]] per step
    start: list              # list[list[(lane, Request)]] per step


def rollout_schedule(w: Workload, steps: int | None = None,
                     prompt_lo: int = 100, prompt_hi: int = 400,
                     min_new: int = 16) -> RolloutSchedule:
    steps = w.steps if steps is None else steps
    rng = np.random.default_rng(w.seed(17))
    rid = 0

    def new_request() -> Request:
        nonlocal rid
        p = int(rng.integers(prompt_lo, prompt_hi + 1))
        f = int(rng.integers(p + min_new, w.max_seq + 1))
        rid += 1
        return Request(rid - 1, p, f)

    first = [new_request() for _ in range(w.batch)]
    cur = list(first)
    length = [r.prompt_len for r in first]   # tokens already in the cache
    finish, start = [], []
    for _t in range(steps):
        fin, st = [], []
        for lane in range(w.batch):
            if length[lane] >= cur[lane].final_len:
                fin.append(lane)
        for lane in fin:
            r = new_request()
            st.append((lane, r))
            cur[lane] = r
            length[lane] = r.prompt_len
        finish.append(fin)
        start.append(st)
        for lane in range(w.batch):
            length[lane] += 1                # this step appends one token
    return RolloutSchedule(w.batch, steps, first, finish, start)


def static_lengths(w: Workload) -> np.ndarray:
    """Initial cached lengths (tokens already in the cache) for the static
    workloads; the first decode step appends at position L0."""
    rng = np.random.default_rng(w.seed(5))
    if w.name == "tiny":
        return np.array([36, 4], dtype=np.int64)
    if w.name == "qwen3":
        return uniform_lengths(rng, w.batch, 64, 1024)
    if w.name == "llama":
        return uniform_lengths(rng, w.batch, 512, 1024)
    if w.name == "gemma":
        return uniform_lengths(rng, w.batch, 256, 2048)
    if w.name == "rollout":
        return np.array([r.prompt_len for r in rollout_schedule(w, 1).first], dtype=np.int64)
    raise KeyError(w.name)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
