// Work-item order of the persistent prefill kernels (prefill_tc.cu,
// prefill_tc_wide.cu).
//
// An item is one row tile (a 64-row query block, or two for unpaired heads)
// of one head group; its cost is the number of key blocks the block mask
// lists for that row tile, which on packed short documents ranges from 1 to
// about 7 and on one long document from 1 to the document's blocks. Dealing
// the items round-robin in their natural order leaves the busiest CTA
// 10-20% above the mean. Instead every CTA sorts the row tiles by cost,
// largest first (a stable counting sort, so all CTAs agree on the order),
// and takes the sorted positions of a "snake": in round r, CTA c takes
// position r * grid + c for even r and r * grid + (grid - 1 - c) for odd r.
// This is the longest-processing-time-first rule without a shared counter:
// no workspace, no atomics across CTAs, deterministic.
//
// One warp builds the CTA's list after the grid-dependency wait (the block
// mask may come from the kernel just before); the CTA then syncs. A CTA
// that would hold more than kSchedCap items keeps the round-robin order.
#pragma once

#include <cstdint>

namespace {

constexpr int kSchedClasses = 128;   // cost classes: listed key blocks, clamped
constexpr int kSchedCap = 256;       // items one CTA's list can hold

struct SchedSmem {
  int base[kSchedClasses];   // next sorted position of each cost class
  int list[kSchedCap];       // this CTA's items, in processing order
  int count;                 // items in list, or -1: round-robin order
};

// key blocks listed for row tile ct (both query blocks' lists when
// unpaired: the larger of the two, as their union is about that long)
__device__ __forceinline__ int sched_cost(int ct, bool pair, int nblk,
                                          const int32_t *kv_num, const int32_t *full_num) {
  auto listed = [&](int qb) {
    return min(max(__ldcg(kv_num + qb), 0), nblk) + min(max(__ldcg(full_num + qb), 0), nblk);
  };
  int t;
  if (pair) {
    t = listed(ct);
  } else {
    const int q0 = 2 * ct;
    t = listed(q0);
    if (q0 + 1 < nblk) t = max(t, listed(q0 + 1));
  }
  return min(t, kSchedClasses - 1);
}

// Called by all 32 lanes of one warp. Items are numbered as the kernels'
// item decoders expect: item i belongs to row tile nq - 1 - i / per.
__device__ void sched_build(SchedSmem &s, int nq, int per, bool pair, int nblk,
                            const int32_t *kv_num, const int32_t *full_num) {
  static_assert(kSchedClasses == 4 * 32, "four cost classes per lane in the scan");
  const int lane = threadIdx.x & 31;
  const int grid = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int n_items = nq * per;
  const int rounds = (n_items + grid - 1) / grid;
  if (rounds > kSchedCap) {
    if (lane == 0) s.count = -1;
    return;
  }
  for (int i = lane; i < kSchedClasses; i += 32) s.base[i] = 0;
  __syncwarp();
  for (int ct = lane; ct < nq; ct += 32)
    atomicAdd(&s.base[sched_cost(ct, pair, nblk, kv_num, full_num)], 1);
  __syncwarp();
  // base[t] = row tiles of cost above t (lane l scans classes 127 - 4l - i)
  int h[4], sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = s.base[kSchedClasses - 1 - (4 * lane + i)];
    sum += h[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - sum;
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s.base[kSchedClasses - 1 - (4 * lane + i)] = run;
    run += h[i];
  }
  __syncwarp();
  // sorted position of each row tile, in natural item order within a class
  for (int u0 = 0; u0 < nq; u0 += 32) {
    const int u = u0 + lane;   // natural order: row tile nq - 1 - u
    const bool valid = u < nq;
    const int t = valid ? sched_cost(nq - 1 - u, pair, nblk, kv_num, full_num) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, t);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int pos = valid ? s.base[t] + rank : 0;
    __syncwarp();
    if (valid && rank == __popc(peers) - 1) s.base[t] += __popc(peers);
    __syncwarp();
    if (valid) {
      for (int j = 0; j < per; ++j) {
        const int p = pos * per + j;
        const int r = p / grid, k = p - r * grid;
        if (((r & 1) ? grid - 1 - k : k) == c) s.list[r] = u * per + j;
      }
    }
  }
  if (lane == 0) {
    const int r = rounds - 1;
    const int k = (r & 1) ? grid - 1 - c : c;
    s.count = r + (r * grid + k < n_items ? 1 : 0);
  }
}

// this CTA's item count and its it-th item, once sched_build has run
__device__ __forceinline__ int sched_count(const SchedSmem &s, int n_items) {
  if (s.count >= 0) return s.count;
  const int c = static_cast<int>(blockIdx.x);
  return c < n_items ? (n_items - 1 - c) / static_cast<int>(gridDim.x) + 1 : 0;
}
__device__ __forceinline__ int sched_item(const SchedSmem &s, int it) {
  return s.count >= 0 ? s.list[it] : static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x);
}

}  // namespace
