"""CPU oracle for paged single-token decode attention — TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 (NumPy) restatement of what the decode hot path
computes, written from the pages' statement of the method:

  * ``pagetable``  — the LIFO slot/page allocator with reserved slot 0 and
    page 0 and the "+1 capacity" rule;
  * ``paged_kv``   — the decode K/V scatter address map and a page gather;
  * ``norm_rope``  — per-head RMSNorm followed by rotate-half RoPE;
  * ``attention``  — GQA decode attention over a gathered, contiguous K/V
    with length and sliding-window masking, plus its log-sum-exp.
  * ``block_mask`` — logical -> physical conversion of a block mask's kv
    indices through the page table;
  * ``prefill``    — document-causal (optionally sliding) attention over packed
    prefill tokens, and its block mask (full / partial key blocks).

Only the test suite, the package smoke check and the benchmark's CPU
baseline may import this package. The product path (the CUDA library and its
Python binding) never imports, links or calls it, and this package imports
nothing from the product path. Every function here is pinned by CPU tests
against values fixed by the pages or by mathematics (worked examples, closed
forms, invariants, brute force, library special cases); none is "parity
unpinned".
"""
from .pagetable import (PageTableModel, NoSlot, NoPages, BadSlot, BadArg,
                        PageTableError)
from .paged_kv import (physical_row, kv_append, gather_pages,
                       ERR_POS, ERR_PAGE_RANGE, ERR_PAGE_NEG, ERR_SLOT)
from .norm_rope import rms_norm, rope, qk_norm_rope, inv_freq, v_norm
from .attention import decode_attention, decode_attention_row
from .prefill import prefill_attention, prefill_block_mask, keep_matrix
from .block_mask import convert_logical_block_mask

__all__ = [
    "PageTableModel", "NoSlot", "NoPages", "BadSlot", "BadArg", "PageTableError",
    "physical_row", "kv_append", "gather_pages",
    "ERR_POS", "ERR_PAGE_RANGE", "ERR_PAGE_NEG", "ERR_SLOT",
    "rms_norm", "rope", "qk_norm_rope", "inv_freq", "v_norm", "prefill_attention",
    "prefill_block_mask", "keep_matrix", "convert_logical_block_mask",
    "decode_attention", "decode_attention_row",
]
