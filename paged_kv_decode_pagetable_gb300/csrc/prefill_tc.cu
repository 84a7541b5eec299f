// prefill_attn on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Same operation and block mask as prefill_attn.cu's header states
// ("unsloth: compare main...transformers-continuous-batching-qwen3" ·
// flex_paged_attention.py · create_prefill_blockmask_no_paging, and the
// sliding variant of the Gemma-4 script): query i keeps key j iff j <= i,
// docs[j] == docs[i] and, with W > 0, i - j < W.
//
// Design: a persistent kernel, one CTA per SM. A work item is two 128-row
// query tiles ("sub-items") of one kv head and the same query rows, one for
// each of two softmax groups: both use every K / V tile the item loads, so
// one group's waits and exchanges overlap the other group's work, and the
// tiles are loaded once for both.
//   warp 16 (producer, one lane): per item, the two Q tiles by TMA, one
//     copy each (4-D map {64 columns, token, head, 64-column atom}: rows
//     past L read zeros), into the groups' Q buffers, then the union of the
//     item's two query blocks' key-block lists (merged on the fly,
//     ascending), each key block's K and V tiles (one copy each) and its 64
//     document ids by TMA into a 3-stage ring, with a small descriptor
//     (block; full / first / last flags; which query block lists it) in the
//     stage; once an item's last tile is issued, the next item's Q tiles are
//     pulled into L2. Items come in the cost-sorted order of
//     prefill_sched.cuh.
//   warps 17, 18 (MMA, one lane each, one warp per softmax group): per tile,
//     the group's S = Q K^T into its own TMEM S buffers (two; M = 128, N =
//     64, K-major SW128 operands), then, one tile behind (at once for an
//     item's last tile), its O += P V (P K-major from the group's shared
//     buffer, V MN-major). The groups share the K / V tiles (a ring stage is
//     free once both groups' P V of it is done) but neither group's MMAs wait
//     for the other group's softmax.
//   warps 0-7 / 8-15 (softmax groups 0 / 1): warps w and w + 4 of a group
//     share the 32 query rows of TMEM lanes 32(w%4)..32(w%4)+31, one row per
//     thread, and split the 64 keys of a tile and the D columns of O in
//     halves. S from TMEM, branch-free masks on partial blocks, the row
//     maximum combined through shared memory, online softmax in the exp2
//     domain with lazy rescaling (O in TMEM is rescaled only when a row's
//     maximum grows by more than 2^8), P as bf16 into the group's swizzled
//     shared buffer (zeros for the rows of a query block that does not list
//     the key block), and the sub-item's O / l to global memory after its
//     last P V.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "pkv_internal.h"
#include "prefill_sched.cuh"
#include "tcgen05.cuh"

namespace {

constexpr int kQR = kTcM;     // query rows per work item
constexpr int kKB = 64;       // keys per tile (the block mask's block)
constexpr int kNS = 3;        // K/V ring stages, shared by the two groups
constexpr int kGroups = 2;    // softmax groups: the CTA's items alternate between them
constexpr int kSplit = 2;                         // warps of a group per TMEM lane group
constexpr int kGroupWarps = 4 * kSplit;           // each: 32 rows x 32 keys of a tile
constexpr int kSoftWarps = kGroups * kGroupWarps;
constexpr int kKW = 64 / kSplit;                  // keys per softmax warp
constexpr int kProdWarp = kSoftWarps, kMmaWarp = kSoftWarps + 1;   // MMA: one warp per group
constexpr int kTCThreads = (kSoftWarps + 1 + kGroups) * 32;
constexpr float kLazyLog2 = 8.f;   // rescale O only when a row maximum grows past 2^8

// tile descriptor flags; kNeed0 / kNeed1: the block is listed for the
// item's first / second 64-row query block (rows of a block that does not
// list it keep nothing there)
constexpr int kFull = 1, kFirst = 2, kLast = 4, kMaskAll = 8, kNeed0 = 16, kNeed1 = 32;

template <int D>
struct TC {
  static constexpr int ATOMS = D / 64;              // 128-byte (64-column) swizzle atoms
  static constexpr int Q_ATOM = kQR * 128;          // bytes of one atom of the Q tile
  static constexpr int KV_ATOM = kKB * 128;
  static constexpr int Q_BYTES = ATOMS * Q_ATOM;
  static constexpr int KV_BYTES = ATOMS * KV_ATOM;
  static constexpr int P_BYTES = kQR * kKB * 2;
  static constexpr int OFF_Q = 0;                             // [kGroups] Q tiles
  static constexpr int OFF_K = OFF_Q + kGroups * Q_BYTES;      // (group x: Q buffer x)
  static constexpr int OFF_V = OFF_K + kNS * KV_BYTES;
  static constexpr int OFF_P = OFF_V + kNS * KV_BYTES;        // [kGroups] P tiles
  static constexpr int OFF_SD = OFF_P + kGroups * P_BYTES;    // int [kNS][64] key documents
  static constexpr int OFF_XCH = OFF_SD + kNS * kKB * 4;      // float [kGroups][2][kSplit][128]
  static constexpr int OFF_META = OFF_XCH + kGroups * 2 * kSplit * kQR * 4;  // int4 [kNS]
  static constexpr int OFF_BAR = OFF_META + kNS * 16;
  // shared: qfull, qempty, kvfull[NS], kvempty[NS], drain[kGroups]; per group:
  // sfull[2], sfree[2], pfull, pvdone, ofree (per item, so that no waiter
  // can fall two phases behind), xbar[4] (the lane groups' exchanges)
  static constexpr int GB = 11;
  static constexpr int N_BAR = 2 + 2 * kNS + kGroups + kGroups * GB;
  static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;       // tmem address, abort flag
  static constexpr int OFF_SCHED = OFF_MISC + 16;            // SchedSmem: this CTA's items
  static constexpr int SMEM = OFF_SCHED + static_cast<int>(sizeof(SchedSmem)) + 1024;
  // per group: S[2] (2 x 64 columns) then O (D <= 128 columns)
  static constexpr int TMEM_COLS = 512, GROUP_COLS = 256, S_COL = 0, O_COL = 128;
  static constexpr int CTAS_PER_SM = 1;
  static_assert(OFF_P % 1024 == 0 && OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "atom alignment");
  static_assert(OFF_SD % 128 == 0, "TMA destination alignment");
  static_assert(O_COL + D <= GROUP_COLS && kGroups * GROUP_COLS <= TMEM_COLS, "TMEM columns");
  static_assert(SMEM <= 232448 / CTAS_PER_SM, "shared memory per SM");
};

// A sub-item fills the 128 rows of the MMA in one of two ways.
//   paired (Hq / Hkv even): one 64-row query block for two query heads h and
//     h + 1 of one kv group, which share the key blocks and the K / V tiles
//     (tile rows 0-63: head h, rows 64-127: head h + 1);
//   unpaired: two consecutive 64-row query blocks of one head (tile row r is
//     query row0 + r); the key blocks visited are the union of the two
//     blocks' lists, some of them needed by one half only.
// Pairing visits each query block's own list once per head pair; on short
// documents the union of two blocks' lists is nearly twice as long.
// A work item is two sub-items of one kv head with the same rows (so the
// same key blocks): heads h0 (group 0) and h1 (group 1). When the kv group
// has an odd number of sub-items, its last item's second sub-item repeats
// the first one and is not written.
struct Item {
  int row0, hk, h0, h1;
  bool two;
};
// work item i: the last row tiles first; the items of one row tile are
// consecutive over the kv heads
__device__ __forceinline__ Item item_of(int i, int nq, int Hkv, int G, bool pair) {
  const int subs = pair ? G / 2 : G;   // sub-items per kv head and row tile
  const int sups = (subs + 1) / 2;     // items per kv head and row tile
  const int per = Hkv * sups;
  const int ct = nq - 1 - i / per;
  const int r = i - (i / per) * per;
  const int hk = r / sups, sp = r - hk * sups;
  const int s0 = 2 * sp, s1 = 2 * sp + 1;
  Item it;
  it.row0 = ct * (pair ? kKB : kQR);
  it.hk = hk;
  it.two = s1 < subs;
  it.h0 = hk * G + (pair ? 2 * s0 : s0);
  it.h1 = it.two ? hk * G + (pair ? 2 * s1 : s1) : it.h0;
  return it;
}
__host__ __device__ constexpr int items_per_tile(int Hkv, int G, bool pair) {
  return Hkv * (((pair ? G / 2 : G) + 1) / 2);
}

template <int D>
__global__ void __launch_bounds__(kTCThreads, TC<D>::CTAS_PER_SM)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmD, const int32_t *__restrict__ docs,
                      const int32_t *__restrict__ kv_num, const int32_t *__restrict__ kv_idx,
                      const int32_t *__restrict__ full_num,
                      const int32_t *__restrict__ full_idx, int nblk, int L, int Hq, int G,
                      int window, float scale_log2, int pair_heads,
                      __nv_bfloat16 *__restrict__ out) {
  using C = TC<D>;
  extern __shared__ uint8_t tc_raw[];
  // 1024-byte aligned base, by offsetting the shared array itself (an integer
  // round trip would hide the state space and turn every access generic)
  uint8_t *sm = tc_raw + ((1024u - (t_smem(tc_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sQ = t_smem(sm + C::OFF_Q), sK = t_smem(sm + C::OFF_K),
                 sV = t_smem(sm + C::OFF_V), sP = t_smem(sm + C::OFF_P),
                 sD = t_smem(sm + C::OFF_SD);
  int4 *meta = reinterpret_cast<int4 *>(sm + C::OFF_META);
  const uint32_t bar0 = t_smem(sm + C::OFF_BAR);
  const uint32_t qfull = bar0, qempty = bar0 + 8, kvfull = bar0 + 16,
                 kvempty = kvfull + 8 * kNS, drain = kvempty + 8 * kNS,
                 gbar0 = drain + 8 * kGroups;
  // the barriers of group x
  auto sfull = [&](int x, int b) { return gbar0 + 8 * C::GB * x + 8 * b; };
  auto sfree = [&](int x, int b) { return gbar0 + 8 * C::GB * x + 16 + 8 * b; };
  auto pfull = [&](int x) { return gbar0 + 8 * C::GB * x + 32; };
  auto pvdone = [&](int x) { return gbar0 + 8 * C::GB * x + 40; };
  auto ofree = [&](int x) { return gbar0 + 8 * C::GB * x + 48; };
  auto xbar = [&](int x, int lg) { return gbar0 + 8 * C::GB * x + 56 + 8 * lg; };
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);

  if (tid == 0) {
    t_bar_init(qfull, 1);
    t_bar_init(qempty, kGroups);   // each group's MMA warp, after the item's last S
    for (int i = 0; i < kNS; ++i) {
      t_bar_init(kvfull + 8 * i, 1);
      t_bar_init(kvempty + 8 * i, kGroups);   // each group's P V of the tile
    }
    for (int x = 0; x < kGroups; ++x) t_bar_init(drain + 8 * x, 1);
    for (int x = 0; x < kGroups; ++x) {
      for (int b = 0; b < 2; ++b) {
        t_bar_init(sfull(x, b), 1);
        t_bar_init(sfree(x, b), kGroupWarps);
      }
      t_bar_init(pfull(x), kGroupWarps);
      t_bar_init(pvdone(x), 1);
      t_bar_init(ofree(x), kGroupWarps);
      for (int i = 0; i < 4; ++i) t_bar_init(xbar(x, i), kSplit);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     t_smem(tslot)),
                 "r"(C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  t_fence_before();
  __syncthreads();
  t_fence_after();
  const uint32_t tmem = *tslot;
  pkv_wait_prior_grid();
  pkv_allow_next_grid();

  const bool pair = pair_heads != 0;
  const int Hkv = Hq / G;
  const int nq = pair ? nblk : (nblk + 1) / 2;   // row tiles of the items
  const int n_items = nq * items_per_tile(Hkv, G, pair);
  SchedSmem &sched = *reinterpret_cast<SchedSmem *>(sm + C::OFF_SCHED);
  if (warp == kProdWarp)
    sched_build(sched, nq, items_per_tile(Hkv, G, pair), pair, nblk, kv_num, full_num);
  __syncthreads();
  const int n_mine = sched_count(sched, n_items);

  if (warp == kProdWarp) {
    // ============================ producer ============================
    if (lane == 0) {
      int g = 0, it = 0;
      bool ok = true;
      for (; it < n_mine && ok; ++it) {
        const int item = sched_item(sched, it);
        const Item w = item_of(item, nq, Hkv, G, pair);
        // both Q tiles of the item (the two groups'), each as two 64-row halves
        // (rows past L read zeros), once the previous item's last S is done
        if (it >= 1 && !t_wait(qempty, it - 1, abort_flag)) break;
        t_expect_tx(qfull, kGroups * C::Q_BYTES);
        // one copy per group: the map's box is {64 columns, rows, heads,
        // atoms} and lands atom by atom, each [128 rows][64 columns]
#pragma unroll
        for (int x = 0; x < kGroups; ++x)
          t_tma_4d(sQ + x * C::Q_BYTES, &tmQ, 0, w.row0, x ? w.h1 : w.h0, 0, qfull);
        // the union of the two query blocks' lists, ascending (paired: one list)
        const int qb0 = w.row0 / kKB, qb1 = pair ? qb0 : qb0 + 1;
        const bool has1 = qb1 < nblk;
        const int32_t *lf0 = full_idx + static_cast<size_t>(qb0) * nblk;
        const int32_t *lp0 = kv_idx + static_cast<size_t>(qb0) * nblk;
        const int32_t *lf1 = has1 ? full_idx + static_cast<size_t>(qb1) * nblk : lf0;
        const int32_t *lp1 = has1 ? kv_idx + static_cast<size_t>(qb1) * nblk : lp0;
        const int cf0 = min(max(full_num[qb0], 0), nblk), cp0 = min(max(kv_num[qb0], 0), nblk);
        const int cf1 = has1 ? min(max(full_num[qb1], 0), nblk) : 0;
        const int cp1 = has1 ? min(max(kv_num[qb1], 0), nblk) : 0;
        int i0 = 0, i1 = 0, i2 = 0, i3 = 0;
        auto head = [&](const int32_t *a, int cnt, int &i) -> int {
          while (i < cnt) {
            const int v = a[i];
            if (v >= 0 && v < nblk) return v;
            ++i;
          }
          return INT_MAX;
        };
        int pend = -1, pend_flags = 0, emitted = 0;
        auto emit = [&](int kb, int flags) -> bool {
          const int s = g % kNS;
          if (g >= kNS && !t_wait(kvempty + 8 * s, g / kNS - 1, abort_flag)) return false;
          meta[s] = make_int4(kb, flags, w.row0, w.hk);
          t_expect_tx(kvfull + 8 * s, 2 * C::KV_BYTES + kKB * 4);
          t_tma_1d(sD + s * kKB * 4, &tmD, kb * kKB, kvfull + 8 * s);   // past L: zeros
          t_tma_4d(sK + s * C::KV_BYTES, &tmK, 0, kb * kKB, w.hk, 0, kvfull + 8 * s);
          t_tma_4d(sV + s * C::KV_BYTES, &tmV, 0, kb * kKB, w.hk, 0, kvfull + 8 * s);
          ++g;
          return true;
        };
        while (ok) {
          const int h0 = head(lf0, cf0, i0), h1 = head(lp0, cp0, i1);
          const int h2 = head(lf1, cf1, i2), h3 = head(lp1, cp1, i3);
          const int kb = min(min(h0, h1), min(h2, h3));
          if (kb == INT_MAX) break;
          const bool in_f0 = h0 == kb, in_f1 = h2 == kb;
          const int need = (h0 == kb || h1 == kb ? kNeed0 : 0) | (h2 == kb || h3 == kb ? kNeed1 : 0);
          if (h0 == kb) ++i0;
          if (h1 == kb) ++i1;
          if (h2 == kb) ++i2;
          if (h3 == kb) ++i3;
          const int flags = ((in_f0 && (!has1 || in_f1)) ? kFull : 0) | need;
          if (pend >= 0) {
            ok = emit(pend, pend_flags | (emitted == 0 ? kFirst : 0));
            ++emitted;
          }
          pend = kb;
          pend_flags = flags;
        }
        if (!ok) break;
        if (pend < 0) {   // no listed block: one fully masked tile, so the rows get zeros
          pend = 0;
          pend_flags = kMaskAll;
        }
        ok = emit(pend, pend_flags | kLast | (emitted == 0 ? kFirst : 0));
        if (ok && it + 1 < n_mine) {   // the next item's Q tiles into L2 meanwhile
          const Item wn = item_of(sched_item(sched, it + 1), nq, Hkv, G, pair);
#pragma unroll
          for (int x = 0; x < kGroups; ++x) t_prefetch_4d(&tmQ, 0, wn.row0, x ? wn.h1 : wn.h0, 0);
        }
      }
    }
  } else if (warp >= kMmaWarp) {
    // ============================== MMA ===============================
    // one warp per softmax group (one lane issues): the group's S of every
    // tile and, one tile behind, its P V; the two groups share the tiles
    // but neither waits for the other's P
    const int x = warp - kMmaWarp;
    if (lane == 0) {
      constexpr uint32_t idS = t_idesc(kKB, 0), idO = t_idesc(D, 1);
      int g = 0, it = 0, npv = 0, nfirst = 0;
      bool ok = true;
      const uint32_t sQx = sQ + x * C::Q_BYTES;
      const uint32_t scol = C::GROUP_COLS * x + C::S_COL, ocol = C::GROUP_COLS * x + C::O_COL;
      // P V of the tile in stage sp into the group's O; an item's first one
      // overwrites O, once the epilogue of the group's previous item has
      // read it
      auto do_pv = [&](int sp, int flags) -> bool {
        if (!t_wait(pfull(x), npv, abort_flag)) return false;
        if ((flags & kFirst) && nfirst >= 1 && !t_wait(ofree(x), nfirst - 1, abort_flag))
          return false;
        t_fence_after();
#pragma unroll
        for (int k = 0; k < kKB / 16; ++k) {
          const uint64_t a = t_desc(sP + x * C::P_BYTES + k * 32, 16, 1024);
          const uint64_t b = t_desc(sV + sp * C::KV_BYTES + k * 2048, C::KV_ATOM, 1024);
          t_mma(tmem + ocol, a, b, idO, (k > 0 || !(flags & kFirst)) ? 1u : 0u);
        }
        t_commit(pvdone(x));
        t_commit(kvempty + 8 * sp);
        ++npv;
        if (flags & kFirst) ++nfirst;
        return true;
      };
      bool pend = false;
      int pstage = 0, pflags = 0;
      for (; it < n_mine && ok; ++it) {
        if (!t_wait(qfull, it, abort_flag)) break;
        int flags = 0;
        do {
          const int s = g % kNS, b = g & 1;
          if (!t_wait(kvfull + 8 * s, g / kNS, abort_flag)) {
            ok = false;
            break;
          }
          flags = meta[s].y;
          if (g >= 2 && !t_wait(sfree(x, b), (g >> 1) - 1, abort_flag)) {
            ok = false;
            break;
          }
          t_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t a = t_desc(sQx + (k >> 2) * C::Q_ATOM + (k & 3) * 32, 16, 1024);
            const uint64_t bd =
                t_desc(sK + s * C::KV_BYTES + (k >> 2) * C::KV_ATOM + (k & 3) * 32, 16, 1024);
            t_mma(tmem + scol + b * kKB, a, bd, idS, k > 0 ? 1u : 0u);
          }
          t_commit(sfull(x, b));
          if (flags & kLast) t_commit(qempty);
          // P V one tile behind S, so that the softmax of this tile overlaps
          // the tensor core; an item's last tile goes at once (its epilogue
          // must not wait for the next item's Q tiles)
          if (pend && !do_pv(pstage, pflags)) {
            ok = false;
            break;
          }
          pend = !(flags & kLast);
          if (pend) {
            pstage = s;
            pflags = flags;
          } else if (!do_pv(s, flags)) {
            ok = false;
            break;
          }
          ++g;
        } while (!(flags & kLast));
      }
      // every issued MMA completes before the TMEM is released
      t_commit(drain + 8 * x);
      t_wait_drain(drain + 8 * x);
    }
  } else {
    // ============================ softmax =============================
    const int x = warp / kGroupWarps;                           // this warp's group
    const int lg = warp & 3, hf = (warp >> 2) & (kSplit - 1);   // lane group, key / column half
    const int row = 32 * lg + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * lg) << 16) + C::GROUP_COLS * x;
    float *xch = reinterpret_cast<float *>(sm + C::OFF_XCH) + x * 2 * kSplit * kQR;
    // exchange number xn of the lane group (the kSplit warps on these rows):
    // each publishes a per-row value, all wait (bounded) for the group's
    // arrivals and read every value; slots alternate, so a slot is rewritten
    // only after every member has read it
    int xn = 0;
    auto exchange = [&](float mine, float (&all)[kSplit]) -> bool {
      const int slot = xn & 1;
      xch[(slot * kSplit + hf) * kQR + row] = mine;
      __syncwarp();
      if (lane == 0) t_arrive(xbar(x, lg));
      if (!t_wait_warp(xbar(x, lg), xn, abort_flag)) return false;
#pragma unroll
      for (int q = 0; q < kSplit; ++q) all[q] = xch[(slot * kSplit + q) * kQR + row];
      ++xn;
      return true;
    };
    constexpr int OH = D / kSplit;                                // O columns of this warp
    const uint32_t ocol = C::O_COL + OH * hf;
    int g = 0;
    bool ok = true;
    for (int it = 0; it < n_mine && ok; ++it) {
      const int item = sched_item(sched, it);
      const Item w = item_of(item, nq, Hkv, G, pair);
      const int hx = x ? w.h1 : w.h0;
      const bool write = x == 0 || w.two;   // a repeated sub-item is not written
      const int qi = pair ? w.row0 + (row & (kKB - 1)) : w.row0 + row;
      const int hrow = pair ? hx + (row >> 6) : hx;   // this row's query head
      const bool valid = qi < L;
      const int dq = valid ? docs[qi] : 0;
      float m = -INFINITY, l = 0.f;   // l: this warp's share of the row sum
      int flags = 0;
      do {
        const int s = g % kNS, b = g & 1;
        if (!t_wait_warp(kvfull + 8 * s, g / kNS, abort_flag)) {
          ok = false;
          break;
        }
        const int4 md = meta[s];
        flags = md.y;
        const int j0 = md.x * kKB + kKW * hf;   // first key of this warp
        const bool partial = !(flags & kFull);
        const int *dks = reinterpret_cast<const int *>(sm + C::OFF_SD) + s * kKB + kKW * hf;
        if (!t_wait_warp(sfull(x, b), g >> 1, abort_flag)) {
          ok = false;
          break;
        }
        t_fence_after();
        float sv[kKW];
        {
          uint32_t r[kKW];
#pragma unroll
          for (int c = 0; c < kKW / 16; ++c)
            t_ld16(trow + C::S_COL + b * kKB + kKW * hf + 16 * c,
                   *reinterpret_cast<uint32_t(*)[16]>(r + 16 * c));
          t_wait_ld();
#pragma unroll
          for (int c = 0; c < kKW; ++c) sv[c] = __uint_as_float(r[c]);
        }
        t_fence_before();   // S buffer b may be overwritten from here
        __syncwarp();
        if (lane == 0) t_arrive(sfree(x, b));
        // a block not listed for this lane group's query block keeps nothing
        // for its rows: P = 0 there, no exchange, no softmax update (all warps
        // of the lane group take this branch together)
        const bool need = (flags & (lg < 2 ? kNeed0 : kNeed1)) != 0;
        float alpha = 1.f;
        bool resc = false;
        if (need) {
          // whether this warp's 32 keys belong to one document (lane l reads
          // key j0 + l's; the whole warp votes, before any per-row branch)
          static_assert(kKW == 32, "one key per lane for the document vote");
          bool one_doc = false, any_kept = true;
          int d0 = 0;
          if (partial && !(flags & kMaskAll)) {
            const int dl = dks[lane];
            d0 = __shfl_sync(0xffffffffu, dl, 0);
            one_doc = __all_sync(0xffffffffu, dl == d0);
          }
          if (flags & kMaskAll) {
#pragma unroll
            for (int c = 0; c < kKW; ++c) sv[c] = -INFINITY;
          } else if (partial && one_doc) {
            // one document: the row keeps a contiguous range of these keys,
            // [lo, hi] (causal, inside L, inside the window), or none. On the
            // FMA pipe: key c is outside iff |c - mid| - half >= 1, so the
            // saturated difference is exactly 1 there and 0 inside, and the
            // score moves down by 2^100 (its exponential is 0 as for -inf; a
            // warp that keeps nothing reports -inf as its maximum, below)
            const int lo = max((window > 0 ? qi - window + 1 : 0) - j0, 0);
            const int hi = min(min(qi, L - 1) - j0, kKW - 1);
            any_kept = valid && d0 == dq && lo <= hi;
            const float mid = any_kept ? 0.5f * static_cast<float>(lo + hi) : -256.f;
            const float half = any_kept ? 0.5f * static_cast<float>(hi - lo) : 0.f;
#pragma unroll
            for (int c = 0; c < kKW; ++c) {
              const float outside = __saturatef(fabsf(static_cast<float>(c) - mid) - half);
              sv[c] = fmaf(outside, -0x1p100f, sv[c]);
            }
          } else if (partial) {
#pragma unroll
            for (int c = 0; c < kKW; ++c) {
              const int key = j0 + c;   // every term evaluated: no branch per element
              const bool keep = valid & (key <= qi) & (key < L) & (dks[c] == dq) &
                                ((window == 0) | (qi - key < window));
              sv[c] = keep ? sv[c] : -INFINITY;
            }
          }
          // raw-score maximum of this warp's keys (two chains of three-input
          // maxima), then of the row
          static_assert(kKW % 4 == 0 && kKW >= 8, "max chains");
          float x0 = t_max3(sv[0], sv[1], sv[2]), x1 = t_max3(sv[3], sv[4], sv[5]);
#pragma unroll
          for (int c = 6; c + 3 < kKW; c += 4) {
            x0 = t_max3(x0, sv[c], sv[c + 1]);
            x1 = t_max3(x1, sv[c + 2], sv[c + 3]);
          }
          x0 = t_max3(x0, sv[kKW - 2], sv[kKW - 1]);
          float mall[kSplit];
          if (!exchange(any_kept ? fmaxf(x0, x1) : -INFINITY, mall)) {
            ok = false;
            break;
          }
          float mraw = mall[0];
#pragma unroll
          for (int q = 1; q < kSplit; ++q) mraw = fmaxf(mraw, mall[q]);
          const float mt = mraw * scale_log2;   // -inf stays -inf (scale > 0)
          // lazy online softmax: a stale maximum is kept unless the new one
          // exceeds it by more than 2^8 (O and l use the same maximum, so the
          // result is exact either way); the lane group's warps decide alike
          if (mt != -INFINITY) {
            if (m == -INFINITY) {
              m = mt;
            } else if (mt > m + kLazyLog2) {
              alpha = exp2f(m - mt);
              m = mt;
              resc = true;
            }
          }
          const float mneg = m == -INFINITY ? 0.f : -m;
          // masked scores are -inf: exp2 gives 0 (the scale and the sums two
          // lanes per packed instruction, each rounded as the scalar form)
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int c = 0; c < kKW; c += 4) {
            float y0, y1, y2, y3;
            t_fma2(y0, y1, sv[c], sv[c + 1], scale_log2, mneg);
            t_fma2(y2, y3, sv[c + 2], sv[c + 3], scale_log2, mneg);
            sv[c] = t_ex2(y0);
            sv[c + 1] = t_ex2(y1);
            sv[c + 2] = t_ex2(y2);
            sv[c + 3] = t_ex2(y3);
            t_add2(s0, s1, sv[c], sv[c + 1]);
            t_add2(s2, s3, sv[c + 2], sv[c + 3]);
          }
          l = l * alpha + ((s0 + s1) + (s2 + s3));
        }
        // the group's P buffer and O are free once its previous P V is done
        if (g >= 1 && !t_wait_warp(pvdone(x), g - 1, abort_flag)) {
          ok = false;
          break;
        }
        if (__any_sync(0xffffffffu, resc)) {   // this warp's columns of O *= alpha
          t_fence_after();
#pragma unroll
          for (int c = 0; c < OH / 16; ++c) {
            uint32_t r[16];
            t_ld16(trow + ocol + 16 * c, r);
            t_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            t_st16(trow + ocol + 16 * c, r);
          }
          t_wait_st();
        }
        {   // this warp's keys are 16-byte chunks (kKW / 8) hf .. of the row
          uint8_t *prow = sm + C::OFF_P + x * C::P_BYTES + row * 128;
#pragma unroll
          for (int q4 = 0; q4 < kKW / 8; ++q4) {
            const int ch = (kKW / 8) * hf + q4;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (need) {
              v.x = t_pack(sv[8 * q4 + 0], sv[8 * q4 + 1]);
              v.y = t_pack(sv[8 * q4 + 2], sv[8 * q4 + 3]);
              v.z = t_pack(sv[8 * q4 + 4], sv[8 * q4 + 5]);
              v.w = t_pack(sv[8 * q4 + 6], sv[8 * q4 + 7]);
            }
            *reinterpret_cast<uint4 *>(prow + ((ch ^ (row & 7)) << 4)) = v;
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        t_fence_before();
        __syncwarp();
        if (lane == 0) t_arrive(pfull(x));
        if (flags & kLast) {   // the row sum, then O / l once this last P V is done
          float lall[kSplit];
          if (!exchange(l, lall)) {
            ok = false;
            break;
          }
          float lt = lall[0];   // the same order in every warp of the lane group
#pragma unroll
          for (int q = 1; q < kSplit; ++q) lt += lall[q];
          const float il = lt > 0.f ? 1.f / lt : 0.f;
          if (!t_wait_warp(pvdone(x), g, abort_flag)) {
            ok = false;
            break;
          }
          t_fence_after();
          // O / l as bf16, 32 columns per round, through this warp's 64
          // bytes of each of its rows in the group's P buffer (idle until
          // this warp writes its next P): each lane writes its row's chunks,
          // then reads back so that four lanes store 64 contiguous bytes of
          // one row (8 rows per store instead of 32)
          static_assert(OH % 32 == 0, "32-column rounds");
          uint8_t *pbuf = sm + C::OFF_P + x * C::P_BYTES;
#pragma unroll 1
          for (int c0 = 0; c0 < OH / 16; c0 += 2) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t r[16];
              t_ld16(trow + ocol + 16 * (c0 + h), r);
              t_wait_ld();
#pragma unroll
              for (int jj = 0; jj < 2; ++jj) {
                const uint32_t *e = r + 8 * jj;
                uint4 v;
                v.x = t_pack(__uint_as_float(e[0]) * il, __uint_as_float(e[1]) * il);
                v.y = t_pack(__uint_as_float(e[2]) * il, __uint_as_float(e[3]) * il);
                v.z = t_pack(__uint_as_float(e[4]) * il, __uint_as_float(e[5]) * il);
                v.w = t_pack(__uint_as_float(e[6]) * il, __uint_as_float(e[7]) * il);
                const int j = 2 * h + jj;
                *reinterpret_cast<uint4 *>(pbuf + row * 128 + (((4 * hf + j) ^ (row & 7)) << 4)) = v;
              }
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = 32 * lg + 8 * i + (lane >> 2), j = lane & 3;
              const uint4 v = *reinterpret_cast<const uint4 *>(
                  pbuf + rr * 128 + (((4 * hf + j) ^ (rr & 7)) << 4));
              const int qr = __shfl_sync(0xffffffffu, qi, 8 * i + (lane >> 2));   // row rr's
              const int hr = __shfl_sync(0xffffffffu, hrow, 8 * i + (lane >> 2));
              if (write && qr < L) {
                *reinterpret_cast<uint4 *>(out + (static_cast<size_t>(hr) * L + qr) * D + OH * hf +
                                           16 * c0 + 8 * j) = v;
              }
            }
            __syncwarp();
          }
          t_fence_before();
          __syncwarp();
          if (lane == 0) t_arrive(ofree(x));
        }
        ++g;
      } while (!(flags & kLast));
    }
    if (!ok || *abort_flag) {   // a wait gave up: mark this group's rows as failed
      for (int it = 0; it < n_mine; ++it) {
        const int item = sched_item(sched, it);
        const Item w = item_of(item, nq, Hkv, G, pair);
        if (x == 1 && !w.two) continue;
        const int qi = pair ? w.row0 + (row & (kKB - 1)) : w.row0 + row;
        if (qi >= L) continue;
        const int hrow = pair ? (x ? w.h1 : w.h0) + (row >> 6) : (x ? w.h1 : w.h0);
        __nv_bfloat16 *orow = out + (static_cast<size_t>(hrow) * L + qi) * D + OH * hf;
        for (int c = 0; c < OH; ++c) orow[c] = __float2bfloat16_rn(NAN);
      }
    }
  }
  t_fence_before();
  __syncthreads();
  t_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::TMEM_COLS));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn tc_encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

namespace pkv {
// 1-D map over the int32 document ids, 64-id boxes; ids past L read zeros
int prefill_docs_map(CUtensorMap *tm, const int32_t *docs, int L) {
  EncodeTiledFn fn = tc_encode_fn();
  if (!fn) return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[1] = {static_cast<cuuint64_t>(L)};
  cuuint64_t strides[1] = {0};
  cuuint32_t box[1] = {static_cast<cuuint32_t>(kKB)};
  cuuint32_t estr[1] = {1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_INT32, 1, const_cast<int32_t *>(docs), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled (docs) failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

// 3-D map {column, token, head} over a [heads][L][D] bf16 tensor with
// [box_rows][64] boxes, 128-byte swizzle; tokens past L read zeros
int prefill_head_map(CUtensorMap *tm, const void *base, int heads, int L, int D, int box_rows) {
  EncodeTiledFn fn = tc_encode_fn();
  if (!fn) return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(D) * 2 * L};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

}  // namespace pkv

namespace pkv {
// 4-D map over a [heads][L][D] bf16 tensor as {64 columns, token, head,
// 64-column atom}: one box of {64, box_rows, box_heads, box_atoms} lands in
// shared memory as box_atoms atoms, each [box_heads][box_rows][64] with the
// 128-byte swizzle (the operand layout of a 64- or 128-row tile); tokens
// past L read zeros
int prefill_atoms_map(CUtensorMap *tm, const void *base, int heads, int L, int D, int box_rows,
                      int box_heads, int box_atoms) {
  EncodeTiledFn fn = tc_encode_fn();
  if (!fn) return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[4] = {64u, static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(D / 64)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(D) * 2 * L, 128u};
  cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_atoms)};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled (atoms) failed (%d)", static_cast<int>(r));
  return PKV_OK;
}
}  // namespace pkv

// Launch of the tcgen05 prefill kernel (declared in pkv_internal.h); the
// public entry point prefill_attn validates the arguments first.
namespace pkv {
template <int D>
int launch_prefill_tc(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                      const int32_t *docs, const int32_t *kv_num, const int32_t *kv_idx,
                      const int32_t *full_num, const int32_t *full_idx, int L, int Hq, int Hkv,
                      int window, float scale, pkv_bf16 *out, cudaStream_t s) {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  PKV_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return pkv::fail(PKV_E_CUDA, "device id out of range");
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      PKV_CUDA_CHECK(cudaFuncSetAttribute(prefill_tc_kernel<D>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          TC<D>::SMEM));
      done[dev] = true;
    }
  }
  const int n = (L + kKB - 1) / kKB;
  const int G = Hq / Hkv;
  const bool pair = G % 2 == 0;
  // a group's Q tile: paired, 64 rows of two heads; otherwise 128 rows of one
  CUtensorMap tmQ, tmK, tmV, tmD;
  int st = prefill_atoms_map(&tmQ, q, Hq, L, D, pair ? kKB : kQR, pair ? 2 : 1, D / 64);
  if (st == PKV_OK) st = prefill_atoms_map(&tmK, k, Hkv, L, D, kKB, 1, D / 64);
  if (st == PKV_OK) st = prefill_atoms_map(&tmV, v, Hkv, L, D, kKB, 1, D / 64);
  if (st == PKV_OK) st = prefill_docs_map(&tmD, docs, L);
  if (st != PKV_OK) return st;
  const long long items = 1LL * (pair ? n : (n + 1) / 2) * items_per_tile(Hkv, G, pair);
  const long long cap = 1LL * TC<D>::CTAS_PER_SM * pkv::sm_count();
  const int grid = static_cast<int>(items < cap ? items : cap);
  PKV_CUDA_CHECK(pkv::launch_pdl(prefill_tc_kernel<D>, dim3(grid), dim3(kTCThreads), TC<D>::SMEM,
                                 s, tmQ, tmK, tmV, tmD, docs, kv_num, kv_idx, full_num, full_idx, n, L,
                                 Hq, G, window, scale * 1.4426950408889634f, pair ? 1 : 0,
                                 reinterpret_cast<__nv_bfloat16 *>(out)));
  return PKV_OK;
}
template int launch_prefill_tc<64>(const pkv_bf16 *, const pkv_bf16 *, const pkv_bf16 *,
                                   const int32_t *, const int32_t *, const int32_t *,
                                   const int32_t *, const int32_t *, int, int, int, int, float,
                                   pkv_bf16 *, cudaStream_t);
template int launch_prefill_tc<128>(const pkv_bf16 *, const pkv_bf16 *, const pkv_bf16 *,
                                    const int32_t *, const int32_t *, const int32_t *,
                                    const int32_t *, const int32_t *, int, int, int, int, float,
                                    pkv_bf16 *, cudaStream_t);
}  // namespace pkv
