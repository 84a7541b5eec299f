"""PageTable allocator model (oracle; test infrastructure only).

Follows "unsloth: compare main...transformers-continuous-batching-qwen3" ·
scripts/benchmarks/flex_paged_attention.py · class PageTable (__init__,
can_reserve, allocate, reserve, erase), and the "+1 capacity" commit message
on "unsloth: compare main...flex-moe-qwen3" (first section).

Policy, as the pages state it:
  * slot (batch index) 0 is a no-op padding slot and page 0 a dummy page;
    the table row of slot 0 is all page 0;
  * free slots and free pages are LIFO stacks; initially
    free_slots = [N, ..., 1] and free_pages = [P-1, ..., 1], so the first
    pop yields slot 1 / the tail yields the lowest pages;
  * a user max_batch_size of N gives N usable slots: internal rows are N+1;
  * allocate pops a slot, zeroes its capacity and sets its row to -1;
  * reserve(slot, L) grows capacity to >= L in whole pages: k = ceil((L -
    cap) / page_size) pages are taken as the TAIL free_pages[-k:], in list
    order, for logical blocks cap/page_size, ..., and removed from the list;
    if fewer than k pages are free nothing changes and the call fails;
  * erase(slot) pushes the slot back and extends free_pages with the slot's
    pages in reverse order; the device row is left stale until the next
    allocate.

Readings where the pages leave a step open:
  * the table here is [N+1][max_pages_per_seq] rather than [N+1][P]; a
    reserve needing more than max_pages_per_seq pages fails with BadArg;
  * assign(L) = allocate + reserve(L) as one call; if it cannot complete
    (no slot, or too few pages) nothing changes;
  * freeing slot 0, a slot out of range, or a slot that is not allocated
    fails with BadSlot and changes nothing;
  * a freed slot reports capacity 0.
"""
from __future__ import annotations

import copy

import numpy as np


class PageTableError(Exception):
    pass


class NoSlot(PageTableError):
    pass


class NoPages(PageTableError):
    pass


class BadSlot(PageTableError):
    pass


class BadArg(PageTableError):
    pass


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class PageTableModel:
    def __init__(self, max_batch_size: int, page_size: int, n_pages: int,
                 max_pages_per_seq: int):
        if max_batch_size < 1 or page_size < 1 or n_pages < 2 or max_pages_per_seq < 1:
            raise BadArg("bad PageTable geometry")
        self.max_batch_size = max_batch_size
        self.n_slots = max_batch_size + 1            # slot 0 reserved
        self.page_size = page_size
        self.n_pages = n_pages
        self.max_pages_per_seq = max_pages_per_seq
        self.table = np.full((self.n_slots, max_pages_per_seq), -1, dtype=np.int32)
        self.table[0, :] = 0                         # no-op slot -> dummy page 0
        self.capacity = [0] * self.n_slots
        self.pages = [[] for _ in range(self.n_slots)]
        self.free_pages = list(range(n_pages - 1, 0, -1))
        self.free_slots = list(range(max_batch_size, 0, -1))

    # -- queries ----------------------------------------------------------
    @property
    def pages_available(self) -> int:
        return len(self.free_pages)

    def is_live(self, slot: int) -> bool:
        return 1 <= slot < self.n_slots and slot not in self.free_slots

    def _pages_needed(self, slot_capacity: int, seq_len: int) -> int:
        if seq_len <= slot_capacity:
            return 0
        return _ceil_div(seq_len - slot_capacity, self.page_size)

    def can_reserve(self, seq_len: int, slot: int | None = None) -> bool:
        if slot is None:
            k = self._pages_needed(0, seq_len)
            return (self.pages_available * self.page_size >= seq_len
                    and len(self.free_slots) > 0
                    and k <= self.max_pages_per_seq)
        if not self.is_live(slot):
            raise BadSlot(f"slot {slot} is not allocated")
        cap = self.capacity[slot]
        k = self._pages_needed(cap, seq_len)
        return (k <= self.pages_available
                and cap // self.page_size + k <= self.max_pages_per_seq)

    # -- mutations ----------------------------------------------------------
    def _allocate(self) -> int:
        if not self.free_slots:
            raise NoSlot("no free slot")
        slot = self.free_slots.pop()
        self.capacity[slot] = 0
        self.pages[slot] = []
        self.table[slot, :] = -1
        return slot

    def reserve(self, slot: int, seq_len: int) -> None:
        if not self.is_live(slot):
            raise BadSlot(f"slot {slot} is not allocated")
        if seq_len < 0:
            raise BadArg("negative length")
        cap = self.capacity[slot]
        k = self._pages_needed(cap, seq_len)
        if k == 0:
            return
        start = cap // self.page_size
        if start + k > self.max_pages_per_seq:
            raise BadArg("sequence longer than the table row")
        if k > self.pages_available:
            raise NoPages(f"need {k} pages, {self.pages_available} free")
        taken = self.free_pages[-k:]
        self.table[slot, start:start + k] = taken
        self.pages[slot] = self.pages[slot] + taken
        self.free_pages = self.free_pages[:-k]
        self.capacity[slot] = cap + k * self.page_size

    def assign(self, seq_len: int) -> int:
        if seq_len < 0:
            raise BadArg("negative length")
        if not self.free_slots:
            raise NoSlot("no free slot")
        k = self._pages_needed(0, seq_len)
        if k > self.max_pages_per_seq:
            raise BadArg("sequence longer than the table row")
        if k > self.pages_available:
            raise NoPages(f"need {k} pages, {self.pages_available} free")
        slot = self._allocate()
        self.reserve(slot, seq_len)
        return slot

    def free(self, slot: int) -> None:
        if not self.is_live(slot):
            raise BadSlot(f"slot {slot} is not allocated")
        self.free_slots.append(slot)
        self.free_pages.extend(reversed(self.pages[slot]))
        self.pages[slot] = []
        self.capacity[slot] = 0
        # the table row is left stale on purpose (reset at the next allocate)

    # -- test helpers -------------------------------------------------------
    def snapshot(self):
        return copy.deepcopy((self.table, self.capacity, self.pages,
                              self.free_pages, self.free_slots))
