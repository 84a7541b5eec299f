// Host PageTable allocator with an optional device mirror of the table.
//
// Policy from "unsloth: compare main...transformers-continuous-batching-qwen3"
// · scripts/benchmarks/flex_paged_attention.py · class PageTable, with the
// +1 capacity rule from the commit message on "unsloth: compare
// main...flex-moe-qwen3":
//   - slot 0 is a no-op slot whose table row is all page 0; page 0 is a dummy
//     page; user max_batch_size N -> N usable slots 1..N (N+1 rows);
//   - free slots and free pages are LIFO stacks, initially [N..1] and
//     [n_pages-1..1] (the back of each vector is the top);
//   - allocate pops a slot, zeroes its capacity and resets its row to -1;
//   - reserve takes the last k free pages in list order for the next k
//     logical blocks, or fails with no change;
//   - erase pushes the slot and appends its pages in reverse order; the
//     device row stays stale until the slot is allocated again.
// The host keeps the authoritative copy so no call reads device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>
#include <vector>

#include "pkv_internal.h"

struct pkv_pt {
  int max_batch_size = 0;
  int n_slots = 0;
  int page_size = 0;
  int n_pages = 0;
  int max_pages = 0;
  int32_t *dev_table = nullptr;
  cudaStream_t stream = nullptr;
  std::vector<int32_t> table;              // [n_slots][max_pages]
  std::vector<int> capacity;               // tokens per slot
  std::vector<std::vector<int32_t>> pages; // pages per slot, logical order
  std::vector<int32_t> free_pages;         // back = next taken
  std::vector<int> free_slots;             // back = next popped
  std::vector<char> live;                  // slot allocated?
};

namespace {

int pages_needed(int cap, int seq_len, int ps) {
  if (seq_len <= cap) return 0;
  return (seq_len - cap + ps - 1) / ps;
}

int write_row_range(pkv_pt *pt, int slot, int begin, int count) {
  if (!pt->dev_table || count <= 0) return PKV_OK;
  size_t off = static_cast<size_t>(slot) * pt->max_pages + begin;
  PKV_CUDA_CHECK(cudaMemcpyAsync(pt->dev_table + off, pt->table.data() + off,
                                 sizeof(int32_t) * count,
                                 cudaMemcpyHostToDevice, pt->stream));
  return PKV_OK;
}

bool valid_live(const pkv_pt *pt, int slot) {
  return slot >= 1 && slot < pt->n_slots && pt->live[slot];
}

}  // namespace

extern "C" {

int pt_create(int max_batch_size, int page_size, int n_pages,
              int max_pages_per_seq, int32_t *dev_table, void *stream,
              pkv_pt **out) {
  if (!out) return pkv::fail(PKV_E_BAD_ARG, "pt_create: out is NULL");
  if (max_batch_size < 1 || page_size < 1 || n_pages < 2 ||
      max_pages_per_seq < 1)
    return pkv::fail(PKV_E_BAD_ARG,
                     "pt_create: need max_batch_size>=1, page_size>=1, "
                     "n_pages>=2, max_pages_per_seq>=1");
  if (dev_table && (reinterpret_cast<uintptr_t>(dev_table) & 3u))
    return pkv::fail(PKV_E_BAD_ARG, "pt_create: dev_table not 4-byte aligned");
  pkv_pt *pt = new (std::nothrow) pkv_pt();
  if (!pt) return pkv::fail(PKV_E_BAD_ARG, "pt_create: out of host memory");
  pt->max_batch_size = max_batch_size;
  pt->n_slots = max_batch_size + 1;
  pt->page_size = page_size;
  pt->n_pages = n_pages;
  pt->max_pages = max_pages_per_seq;
  pt->dev_table = dev_table;
  pt->stream = static_cast<cudaStream_t>(stream);
  pt->table.assign(static_cast<size_t>(pt->n_slots) * max_pages_per_seq, -1);
  std::fill(pt->table.begin(), pt->table.begin() + max_pages_per_seq, 0);
  pt->capacity.assign(pt->n_slots, 0);
  pt->pages.assign(pt->n_slots, {});
  pt->live.assign(pt->n_slots, 0);
  for (int p = n_pages - 1; p >= 1; --p) pt->free_pages.push_back(p);
  for (int s = max_batch_size; s >= 1; --s) pt->free_slots.push_back(s);
  int st = write_row_range(pt, 0, 0, pt->n_slots * max_pages_per_seq);
  if (st != PKV_OK) {
    delete pt;
    return st;
  }
  *out = pt;
  return pkv::ok();
}

int pt_destroy(pkv_pt *pt) {
  delete pt;
  return pkv::ok();
}

int pt_set_stream(pkv_pt *pt, void *stream) {
  if (!pt) return pkv::fail(PKV_E_BAD_ARG, "pt_set_stream: NULL handle");
  pt->stream = static_cast<cudaStream_t>(stream);
  return pkv::ok();
}

int pt_can_reserve(const pkv_pt *pt, int seq_len, int slot, int *ok) {
  if (!pt || !ok) return pkv::fail(PKV_E_BAD_ARG, "pt_can_reserve: NULL");
  if (slot < 0) {
    int k = pages_needed(0, seq_len, pt->page_size);
    *ok = !pt->free_slots.empty() &&
          static_cast<long long>(pt->free_pages.size()) * pt->page_size >=
              seq_len &&
          k <= pt->max_pages;
    return pkv::ok();
  }
  if (!valid_live(pt, slot))
    return pkv::fail(PKV_E_BAD_SLOT, "pt_can_reserve: slot %d not allocated",
                     slot);
  int cap = pt->capacity[slot];
  int k = pages_needed(cap, seq_len, pt->page_size);
  *ok = k <= static_cast<int>(pt->free_pages.size()) &&
        cap / pt->page_size + k <= pt->max_pages;
  return pkv::ok();
}

static int reserve_impl(pkv_pt *pt, int slot, int seq_len) {
  int cap = pt->capacity[slot];
  int k = pages_needed(cap, seq_len, pt->page_size);
  if (k == 0) return PKV_OK;
  int start = cap / pt->page_size;
  if (start + k > pt->max_pages)
    return pkv::fail(PKV_E_BAD_ARG,
                     "reserve: %d tokens exceed the table row (%d pages)",
                     seq_len, pt->max_pages);
  if (k > static_cast<int>(pt->free_pages.size()))
    return pkv::fail(PKV_E_NO_PAGES, "reserve: need %d pages, %zu free", k,
                     pt->free_pages.size());
  // take the tail free_pages[-k:] in list order for blocks start..start+k-1
  size_t first = pt->free_pages.size() - k;
  int32_t *row = pt->table.data() + static_cast<size_t>(slot) * pt->max_pages;
  for (int i = 0; i < k; ++i) {
    int32_t p = pt->free_pages[first + i];
    row[start + i] = p;
    pt->pages[slot].push_back(p);
  }
  pt->free_pages.resize(first);
  pt->capacity[slot] = cap + k * pt->page_size;
  return PKV_OK;
}

int pt_reserve(pkv_pt *pt, int slot, int seq_len) {
  if (!pt) return pkv::fail(PKV_E_BAD_ARG, "pt_reserve: NULL handle");
  if (!valid_live(pt, slot))
    return pkv::fail(PKV_E_BAD_SLOT, "pt_reserve: slot %d not allocated", slot);
  if (seq_len < 0) return pkv::fail(PKV_E_BAD_ARG, "pt_reserve: negative length");
  int start = pt->capacity[slot] / pt->page_size;
  size_t before = pt->pages[slot].size();
  int st = reserve_impl(pt, slot, seq_len);
  if (st != PKV_OK) return st;
  int added = static_cast<int>(pt->pages[slot].size() - before);
  st = write_row_range(pt, slot, start, added);
  if (st != PKV_OK) return st;
  return pkv::ok();
}

int pt_assign(pkv_pt *pt, int seq_len, int *slot_out) {
  if (!pt || !slot_out) return pkv::fail(PKV_E_BAD_ARG, "pt_assign: NULL");
  if (seq_len < 0) return pkv::fail(PKV_E_BAD_ARG, "pt_assign: negative length");
  if (pt->free_slots.empty())
    return pkv::fail(PKV_E_NO_SLOT, "pt_assign: no free slot");
  int k = pages_needed(0, seq_len, pt->page_size);
  if (k > pt->max_pages)
    return pkv::fail(PKV_E_BAD_ARG,
                     "pt_assign: %d tokens exceed the table row (%d pages)",
                     seq_len, pt->max_pages);
  if (k > static_cast<int>(pt->free_pages.size()))
    return pkv::fail(PKV_E_NO_PAGES, "pt_assign: need %d pages, %zu free", k,
                     pt->free_pages.size());
  int slot = pt->free_slots.back();
  pt->free_slots.pop_back();
  pt->live[slot] = 1;
  pt->capacity[slot] = 0;
  pt->pages[slot].clear();
  int32_t *row = pt->table.data() + static_cast<size_t>(slot) * pt->max_pages;
  std::fill(row, row + pt->max_pages, -1);
  int st = reserve_impl(pt, slot, seq_len);  // cannot fail after the checks
  if (st == PKV_OK) st = write_row_range(pt, slot, 0, pt->max_pages);
  if (st != PKV_OK) return st;
  *slot_out = slot;
  return pkv::ok();
}

int pt_free(pkv_pt *pt, int slot) {
  if (!pt) return pkv::fail(PKV_E_BAD_ARG, "pt_free: NULL handle");
  if (!valid_live(pt, slot))
    return pkv::fail(PKV_E_BAD_SLOT, "pt_free: slot %d not allocated", slot);
  pt->free_slots.push_back(slot);
  pt->live[slot] = 0;
  auto &pg = pt->pages[slot];
  for (auto it = pg.rbegin(); it != pg.rend(); ++it) pt->free_pages.push_back(*it);
  pg.clear();
  pt->capacity[slot] = 0;
  return pkv::ok();
}

int pt_capacity(const pkv_pt *pt, int slot, int *tokens) {
  if (!pt || !tokens) return pkv::fail(PKV_E_BAD_ARG, "pt_capacity: NULL");
  if (slot < 0 || slot >= pt->n_slots)
    return pkv::fail(PKV_E_BAD_SLOT, "pt_capacity: slot %d out of range", slot);
  *tokens = pt->capacity[slot];
  return pkv::ok();
}

int pt_pages(const pkv_pt *pt, int slot, int32_t *host_out, int max, int *n) {
  if (!pt || !n) return pkv::fail(PKV_E_BAD_ARG, "pt_pages: NULL");
  if (slot < 0 || slot >= pt->n_slots)
    return pkv::fail(PKV_E_BAD_SLOT, "pt_pages: slot %d out of range", slot);
  const auto &pg = pt->pages[slot];
  *n = static_cast<int>(pg.size());
  if (host_out)
    for (int i = 0; i < *n && i < max; ++i) host_out[i] = pg[i];
  return pkv::ok();
}

int pt_free_pages(const pkv_pt *pt, int *n) {
  if (!pt || !n) return pkv::fail(PKV_E_BAD_ARG, "pt_free_pages: NULL");
  *n = static_cast<int>(pt->free_pages.size());
  return pkv::ok();
}

int pt_free_page_list(const pkv_pt *pt, int32_t *host_out, int max, int *n) {
  if (!pt || !n) return pkv::fail(PKV_E_BAD_ARG, "pt_free_page_list: NULL");
  *n = static_cast<int>(pt->free_pages.size());
  if (host_out)
    for (int i = 0; i < *n && i < max; ++i) host_out[i] = pt->free_pages[i];
  return pkv::ok();
}

int pt_host_table(const pkv_pt *pt, int32_t *host_out, int max) {
  if (!pt || !host_out) return pkv::fail(PKV_E_BAD_ARG, "pt_host_table: NULL");
  int n = static_cast<int>(pt->table.size());
  if (max < n)
    return pkv::fail(PKV_E_BAD_ARG, "pt_host_table: need %d entries", n);
  std::copy(pt->table.begin(), pt->table.end(), host_out);
  return pkv::ok();
}

}  // extern "C"
