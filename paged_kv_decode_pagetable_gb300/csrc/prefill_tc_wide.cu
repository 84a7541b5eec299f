// prefill_attn for the wide head dims of the Gemma-4 layers (D = 256 on the
// sliding layers, D = 512 on the full ones), on tcgen05, TMEM and TMA.
//
// Same operation and block mask as prefill_attn.cu's header states
// ("unsloth: compare main...transformers-continuous-batching-qwen3" ·
// flex_paged_attention.py · create_prefill_blockmask_no_paging, and the
// sliding variant of the Gemma-4 script): query i keeps key j iff j <= i,
// docs[j] == docs[i] and, with W > 0, i - j < W.
//
// Why a second kernel: at these widths a 128-row Q tile (64 / 128 KB) and
// 64-key K and V tiles no longer fit shared memory beside a ring, and the
// fp32 output of 128 rows x 512 columns alone fills the 512 TMEM columns.
// So here:
//   * the output columns are cut into halves of DO = 256: a work item is
//     (128 query rows, query head, output half); D = 256 has one half, D = 512
//     two, each computing the scores over the full D;
//   * Q is not kept: each key tile's scores S = Q K^T are accumulated over D
//     in 64-column chunks, every chunk bringing its Q and K slices by TMA
//     through a 5-stage ring (Q is re-read from L2 once per key tile);
//   * the V tile (64 keys x DO columns), the tile's 64 document ids and its
//     descriptor come through a separate 2-stage ring;
//   * TMEM: S in two 64-column buffers, one O of DO columns (384 of 512).
// The producer, the softmax (16 warps, lazy rescaling, exp2 domain, P as
// bf16 in a swizzled shared buffer), the work order and the failure handling
// are those of prefill_tc.cu; two MMA warps issue, one every tile's S and
// the other its P V; an item's output is written after the next item's first
// tile, and the next item's first P V waits for it (one O buffer).
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

constexpr int wQR = kTcM;     // query rows per work item
constexpr int wKB = 64;       // keys per tile (the block mask's block)
constexpr int wDO = 256;      // output columns per work item
constexpr int wNSQ = 5;       // Q / K chunk ring stages
constexpr int wNSV = 2;       // V ring stages
constexpr int wSplit = 4;                  // softmax warps per TMEM lane group
constexpr int wSoftWarps = 4 * wSplit;
constexpr int wKW = 64 / wSplit;           // keys per softmax warp
// MMA: one warp issuing S, one issuing P V
constexpr int wProdWarp = wSoftWarps, wMmaWarp = wSoftWarps + 1;
constexpr int wThreads = (wSoftWarps + 3) * 32;
constexpr float wLazyLog2 = 8.f;
constexpr int wFull = 1, wFirst = 2, wLast = 4, wMaskAll = 8, wNeed0 = 16, wNeed1 = 32;

template <int D>
struct TW {
  static constexpr int NCH = D / 64;               // 64-column chunks of the score contraction
  static constexpr int NOC = D / wDO;              // output halves (work items per row block)
  static constexpr int Q_CH = wQR * 128;           // one chunk of the Q tile (SW128 atom)
  static constexpr int K_CH = wKB * 128;           // one chunk of the K tile
  static constexpr int QK_STAGE = Q_CH + K_CH;
  static constexpr int V_ATOM = wKB * 128;
  static constexpr int V_BYTES = (wDO / 64) * V_ATOM;
  static constexpr int P_BYTES = wQR * wKB * 2;
  static constexpr int OFF_QK = 0;
  static constexpr int OFF_V = OFF_QK + wNSQ * QK_STAGE;
  static constexpr int OFF_P = OFF_V + wNSV * V_BYTES;
  static constexpr int OFF_SD = OFF_P + 2 * P_BYTES;              // int [wNSV][64] key documents
  static constexpr int OFF_XCH = OFF_SD + wNSV * wKB * 4;          // float [2][wSplit][128]
  static constexpr int OFF_META = OFF_XCH + 2 * wSplit * wQR * 4;  // int4 [wNSV]
  static constexpr int OFF_BAR = OFF_META + wNSV * 16;
  // qkfull[NSQ] qkempty[NSQ] dfull[NSV] vfull[NSV] vempty[NSV] sfull[2] sfree[2]
  // pfull[2] pvdone[2] ofree drain[2] xbar[4]
  static constexpr int N_BAR = 2 * wNSQ + 3 * wNSV + 8 + 3 + 4;
  static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
  static constexpr int OFF_SCHED = OFF_MISC + 16;   // SchedSmem: this CTA's items
  static constexpr int SMEM = OFF_SCHED + static_cast<int>(sizeof(SchedSmem)) + 1024;
  static constexpr int TMEM_COLS = 512;   // S[2] (2 x 64) + O (256)
  static constexpr int S_COL = 0, O_COL = 128;
  static_assert(OFF_V % 1024 == 0 && OFF_P % 1024 == 0 && QK_STAGE % 1024 == 0, "atoms");
  static_assert(OFF_SD % 128 == 0, "TMA destination alignment");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// The 128 rows of an item: paired (Hq / Hkv even) one 64-row query block of
// query heads h and h + 1 (rows 0-63 / 64-127), which share the key blocks
// and the K / V tiles; unpaired two consecutive 64-row query blocks of head h
// (the union of their key lists is visited).
struct WItem {
  int row0, h, oc;
};
// work item i: the last query blocks first; the items of one query block
// (pair) are consecutive over (head, output half)
__device__ __forceinline__ WItem witem_of(int i, int nq, int Hq, int noc, bool pair) {
  WItem it;
  const int per = (pair ? Hq / 2 : Hq) * noc;
  const int ct = nq - 1 - i / per;
  const int r = i - (i / per) * per;
  it.row0 = ct * (pair ? wKB : wQR);
  const int hi = r / noc;
  it.h = pair ? 2 * hi : hi;
  it.oc = r - hi * noc;
  return it;
}

template <int D>
__global__ void __launch_bounds__(wThreads, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmD, const int32_t *__restrict__ docs,
                        const int32_t *__restrict__ kv_num, const int32_t *__restrict__ kv_idx,
                        const int32_t *__restrict__ full_num,
                        const int32_t *__restrict__ full_idx, int nblk, int L, int Hq, int G,
                        int window, float scale_log2, int pair_heads,
                        __nv_bfloat16 *__restrict__ out) {
  using C = TW<D>;
  extern __shared__ uint8_t tw_raw[];
  uint8_t *sm = tw_raw + ((1024u - (t_smem(tw_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sQK = t_smem(sm + C::OFF_QK), sV = t_smem(sm + C::OFF_V),
                 sP = t_smem(sm + C::OFF_P), sD = t_smem(sm + C::OFF_SD);
  int4 *meta = reinterpret_cast<int4 *>(sm + C::OFF_META);
  const uint32_t bar0 = t_smem(sm + C::OFF_BAR);
  const uint32_t qkfull = bar0, qkempty = qkfull + 8 * wNSQ, dfull = qkempty + 8 * wNSQ,
                 vfull = dfull + 8 * wNSV, vempty = vfull + 8 * wNSV, sfull = vempty + 8 * wNSV,
                 sfree = sfull + 16, pfull = sfree + 16, pvdone = pfull + 16, ofree = pvdone + 16,
                 drain = ofree + 8, xbar = drain + 16;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);

  if (tid == 0) {
    for (int i = 0; i < wNSQ; ++i) {
      t_bar_init(qkfull + 8 * i, 1);
      t_bar_init(qkempty + 8 * i, 1);
    }
    for (int i = 0; i < wNSV; ++i) {
      t_bar_init(dfull + 8 * i, 1);
      t_bar_init(vfull + 8 * i, 1);
      t_bar_init(vempty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      t_bar_init(sfull + 8 * i, 1);
      t_bar_init(sfree + 8 * i, wSoftWarps);
      t_bar_init(pfull + 8 * i, wSoftWarps);
      t_bar_init(pvdone + 8 * i, 1);
    }
    t_bar_init(ofree, wSoftWarps);
    t_bar_init(drain, 1);
    t_bar_init(drain + 8, 1);
    for (int i = 0; i < 4; ++i) t_bar_init(xbar + 8 * i, wSplit);
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
  const int nq = pair ? nblk : (nblk + 1) / 2;   // row tiles of the items
  const int n_items = nq * (pair ? Hq / 2 : Hq) * C::NOC;
  SchedSmem &sched = *reinterpret_cast<SchedSmem *>(sm + C::OFF_SCHED);
  if (warp == wProdWarp)
    sched_build(sched, nq, (pair ? Hq / 2 : Hq) * C::NOC, pair, nblk, kv_num, full_num);
  __syncthreads();
  const int n_mine = sched_count(sched, n_items);

  if (warp == wProdWarp) {
    // ============================ producer ============================
    if (lane == 0) {
      int gq = 0, gv = 0;
      bool ok = true;
      for (int it = 0; it < n_mine && ok; ++it) {
        const int item = sched_item(sched, it);
        const WItem w = witem_of(item, nq, Hq, C::NOC, pair);
        const int hk = w.h / G;   // = (h + 1) / G when paired
        // the union of the two halves' lists, ascending (paired: one list)
        const int qb0 = w.row0 / wKB, qb1 = pair ? qb0 : qb0 + 1;
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
            const int x = a[i];
            if (x >= 0 && x < nblk) return x;
            ++i;
          }
          return INT_MAX;
        };
        int pend = -1, pend_flags = 0, emitted = 0;
        // one key tile: its Q / K chunks, then its V tile, document ids and
        // descriptor
        auto emit = [&](int kb, int flags) -> bool {
          for (int c = 0; c < C::NCH; ++c) {
            const int s = gq % wNSQ;
            if (gq >= wNSQ && !t_wait(qkempty + 8 * s, gq / wNSQ - 1, abort_flag)) return false;
            const uint32_t dst = sQK + s * C::QK_STAGE;
            t_expect_tx(qkfull + 8 * s, C::QK_STAGE);
            // the chunk's 128 Q rows in one copy (rows past L read zeros)
            t_tma_4d(dst, &tmQ, 0, w.row0, w.h, c, qkfull + 8 * s);
            t_tma_3d(dst + C::Q_CH, &tmK, 64 * c, kb * wKB, hk, qkfull + 8 * s);
            ++gq;
          }
          const int s = gv % wNSV;
          if (gv >= wNSV && !t_wait(vempty + 8 * s, gv / wNSV - 1, abort_flag)) return false;
          meta[s] = make_int4(kb, flags, w.row0, w.h);
          t_expect_tx(dfull + 8 * s, wKB * 4);
          t_tma_1d(sD + s * wKB * 4, &tmD, kb * wKB, dfull + 8 * s);   // past L: zeros
          t_expect_tx(vfull + 8 * s, C::V_BYTES);
          t_tma_4d(sV + s * C::V_BYTES, &tmV, 0, kb * wKB, hk, w.oc * (wDO / 64), vfull + 8 * s);
          ++gv;
          return true;
        };
        while (ok) {
          const int h0 = head(lf0, cf0, i0), h1 = head(lp0, cp0, i1);
          const int h2 = head(lf1, cf1, i2), h3 = head(lp1, cp1, i3);
          const int kb = min(min(h0, h1), min(h2, h3));
          if (kb == INT_MAX) break;
          const bool in_f0 = h0 == kb, in_f1 = h2 == kb;
          const int need =
              (h0 == kb || h1 == kb ? wNeed0 : 0) | (h2 == kb || h3 == kb ? wNeed1 : 0);
          if (h0 == kb) ++i0;
          if (h1 == kb) ++i1;
          if (h2 == kb) ++i2;
          if (h3 == kb) ++i3;
          const int flags = ((in_f0 && (!has1 || in_f1)) ? wFull : 0) | need;
          if (pend >= 0) {
            ok = emit(pend, pend_flags | (emitted == 0 ? wFirst : 0));
            ++emitted;
          }
          pend = kb;
          pend_flags = flags;
        }
        if (!ok) break;
        if (pend < 0) {   // no listed block: one fully masked tile, so the rows get zeros
          pend = 0;
          pend_flags = wMaskAll;
        }
        ok = emit(pend, pend_flags | wLast | (emitted == 0 ? wFirst : 0));
      }
    }
  } else if (warp >= wMmaWarp) {
    // ============================== MMA ===============================
    // one warp (one lane issues) for the S of every tile and one for the
    // P V, so that a tile's S streams in while the previous P V waits for
    // its P
    const bool pv_warp = warp != wMmaWarp;
    if (lane == 0) {
      constexpr uint32_t idS = t_idesc(wKB, 0), idO = t_idesc(wDO, 1);
      int g = 0;
      bool ok = true;
      if (!pv_warp) {
        int gq = 0;
        for (int it = 0; it < n_mine && ok; ++it) {
          int flags = 0;
          do {
            const int b = g & 1, sv = g % wNSV;
            if (g >= 2 && !t_wait(sfree + 8 * b, (g >> 1) - 1, abort_flag)) {
              ok = false;
              break;
            }
            for (int c = 0; c < C::NCH && ok; ++c) {
              const int s = gq % wNSQ;
              if (!t_wait(qkfull + 8 * s, gq / wNSQ, abort_flag)) {
                ok = false;
                break;
              }
              t_fence_after();
              const uint32_t base = sQK + s * C::QK_STAGE;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t a = t_desc(base + k * 32, 16, 1024);
                const uint64_t bd = t_desc(base + C::Q_CH + k * 32, 16, 1024);
                t_mma(tmem + C::S_COL + b * wKB, a, bd, idS, (c > 0 || k > 0) ? 1u : 0u);
              }
              t_commit(qkempty + 8 * s);
              ++gq;
            }
            if (!ok) break;
            t_commit(sfull + 8 * b);
            // the tile's flags (for the item's end), staged with its V tile
            if (!t_wait(dfull + 8 * sv, g / wNSV, abort_flag)) {
              ok = false;
              break;
            }
            flags = meta[sv].y;
            ++g;
          } while (!(flags & wLast));
        }
      } else {
        // P V of tile g into O once its P is written; an item's first one
        // overwrites O once the previous item's output has been read out
        int pv_item = 0;
        for (int it = 0; it < n_mine && ok; ++it) {
          int flags = 0;
          do {
            const int bp = g & 1, sv = g % wNSV;
            if (!t_wait(dfull + 8 * sv, g / wNSV, abort_flag)) {
              ok = false;
              break;
            }
            flags = meta[sv].y;
            if (!t_wait(pfull + 8 * bp, g >> 1, abort_flag) ||
                ((flags & wFirst) && pv_item > 0 && !t_wait(ofree, pv_item - 1, abort_flag)) ||
                !t_wait(vfull + 8 * sv, g / wNSV, abort_flag)) {
              ok = false;
              break;
            }
            t_fence_after();
#pragma unroll
            for (int k = 0; k < wKB / 16; ++k) {
              const uint64_t a = t_desc(sP + bp * C::P_BYTES + k * 32, 16, 1024);
              const uint64_t bv = t_desc(sV + sv * C::V_BYTES + k * 2048, C::V_ATOM, 1024);
              t_mma(tmem + C::O_COL, a, bv, idO, (k > 0 || !(flags & wFirst)) ? 1u : 0u);
            }
            t_commit(pvdone + 8 * bp);
            t_commit(vempty + 8 * sv);
            if (flags & wLast) ++pv_item;
            ++g;
          } while (!(flags & wLast));
        }
      }
      // every issued MMA completes before the TMEM is released
      const uint32_t dr = drain + (pv_warp ? 8 : 0);
      t_commit(dr);
      t_wait_drain(dr);
    }
  } else {
    // ============================ softmax =============================
    const int lg = warp & 3, hf = warp >> 2;          // lane group, key / column quarter
    const int row = 32 * lg + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * lg) << 16);
    float *xch = reinterpret_cast<float *>(sm + C::OFF_XCH);
    int xn = 0;
    auto exchange = [&](float mine, float (&all)[wSplit]) -> bool {
      const int slot = xn & 1;
      xch[(slot * wSplit + hf) * wQR + row] = mine;
      __syncwarp();
      if (lane == 0) t_arrive(xbar + 8 * lg);
      if (!t_wait_warp(xbar + 8 * lg, xn, abort_flag)) return false;
#pragma unroll
      for (int q = 0; q < wSplit; ++q) all[q] = xch[(slot * wSplit + q) * wQR + row];
      ++xn;
      return true;
    };
    constexpr int OH = wDO / wSplit;                // O columns of this warp
    const uint32_t ocol = C::O_COL + OH * hf;
    bool ep = false;
    int ep_g = 0, ep_it = 0, ep_qi = 0, ep_h = 0, ep_oc = 0;
    float ep_il = 0.f;
    auto epilogue = [&]() -> bool {
      if (!t_wait_warp(pvdone + 8 * (ep_g & 1), ep_g >> 1, abort_flag)) return false;
      t_fence_after();
      // O / l as bf16, 16 columns per round, through this warp's 32 bytes
      // of each of its rows in the idle P buffer (the previous item's last
      // tile's, whose P V is done): each lane writes its row's two chunks,
      // then two lanes store 32 contiguous bytes of one row (16 rows per
      // store instead of 32)
      uint8_t *pbuf = sm + C::OFF_P + (ep_g & 1) * C::P_BYTES;
      const float il = ep_il;
#pragma unroll 1
      for (int c = 0; c < OH / 16; ++c) {
        uint32_t r[16];
        t_ld16(trow + ocol + 16 * c, r);
        t_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const uint32_t *e = r + 8 * jj;
          uint4 v;
          v.x = t_pack(__uint_as_float(e[0]) * il, __uint_as_float(e[1]) * il);
          v.y = t_pack(__uint_as_float(e[2]) * il, __uint_as_float(e[3]) * il);
          v.z = t_pack(__uint_as_float(e[4]) * il, __uint_as_float(e[5]) * il);
          v.w = t_pack(__uint_as_float(e[6]) * il, __uint_as_float(e[7]) * il);
          *reinterpret_cast<uint4 *>(pbuf + row * 128 + (((2 * hf + jj) ^ (row & 7)) << 4)) = v;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int src = 16 * i + (lane >> 1), jj = lane & 1, rr = 32 * lg + src;
          const uint4 v =
              *reinterpret_cast<const uint4 *>(pbuf + rr * 128 + (((2 * hf + jj) ^ (rr & 7)) << 4));
          const int qr = __shfl_sync(0xffffffffu, ep_qi, src);   // row rr's
          const int hr = __shfl_sync(0xffffffffu, ep_h, src);
          if (qr < L)
            *reinterpret_cast<uint4 *>(out + (static_cast<size_t>(hr) * L + qr) * D + ep_oc * wDO +
                                       OH * hf + 16 * c + 8 * jj) = v;
        }
        __syncwarp();
      }
      t_fence_before();
      __syncwarp();
      if (lane == 0) t_arrive(ofree);
      ep = false;
      (void)ep_it;
      return true;
    };
    int g = 0, it = -1;
    bool ok = true;
    for (int wi = 0; wi < n_mine && ok; ++wi) {
      const int item = sched_item(sched, wi);
      ++it;
      const WItem w = witem_of(item, nq, Hq, C::NOC, pair);
      const int qi = pair ? w.row0 + (row & (wKB - 1)) : w.row0 + row;
      const int hrow = pair ? w.h + (row >> 6) : w.h;   // this row's query head
      const bool valid = qi < L;
      const int dq = valid ? docs[qi] : 0;
      float m = -INFINITY, l = 0.f;
      int flags = 0;
      do {
        const int sv = g % wNSV, b = g & 1;
        if (!t_wait_warp(dfull + 8 * sv, g / wNSV, abort_flag)) {
          ok = false;
          break;
        }
        const int4 md = meta[sv];
        flags = md.y;
        const int j0 = md.x * wKB + wKW * hf;
        const bool partial = !(flags & wFull);
        if (!t_wait_warp(sfull + 8 * b, g >> 1, abort_flag)) {
          ok = false;
          break;
        }
        const int *dks = reinterpret_cast<const int *>(sm + C::OFF_SD) + sv * wKB + wKW * hf;
        t_fence_after();
        float svv[wKW];
        {
          uint32_t r[16];
          t_ld16(trow + C::S_COL + b * wKB + wKW * hf, r);
          t_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) svv[j] = __uint_as_float(r[j]);
        }
        t_fence_before();
        __syncwarp();
        if (lane == 0) t_arrive(sfree + 8 * b);
        const bool need = (flags & (lg < 2 ? wNeed0 : wNeed1)) != 0;
        if (!need) {
          if (g >= 2 && !t_wait_warp(pvdone + 8 * b, (g >> 1) - 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t *prow = sm + C::OFF_P + b * C::P_BYTES + row * 128;
#pragma unroll
          for (int q4 = 0; q4 < wKW / 8; ++q4) {
            const int ch = (wKW / 8) * hf + q4;
            *reinterpret_cast<uint4 *>(prow + ((ch ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
          }
        } else {
          if (flags & wMaskAll) {
#pragma unroll
            for (int c = 0; c < wKW; ++c) svv[c] = -INFINITY;
          } else if (partial && window == 0 && j0 + wKW <= w.row0 && valid) {
#pragma unroll
            for (int c = 0; c < wKW; ++c) svv[c] = dks[c] == dq ? svv[c] : -INFINITY;
          } else if (partial) {
#pragma unroll
            for (int c = 0; c < wKW; ++c) {
              const int key = j0 + c;
              const bool keep = valid & (key <= qi) & (key < L) & (dks[c] == dq) &
                                ((window == 0) | (qi - key < window));
              svv[c] = keep ? svv[c] : -INFINITY;
            }
          }
          // two chains of three-input maxima
          static_assert(wKW % 4 == 0 && wKW >= 8, "max chains");
          float x0 = t_max3(svv[0], svv[1], svv[2]), x1 = t_max3(svv[3], svv[4], svv[5]);
#pragma unroll
          for (int c = 6; c + 3 < wKW; c += 4) {
            x0 = t_max3(x0, svv[c], svv[c + 1]);
            x1 = t_max3(x1, svv[c + 2], svv[c + 3]);
          }
          x0 = t_max3(x0, svv[wKW - 2], svv[wKW - 1]);
          float mall[wSplit];
          if (!exchange(fmaxf(x0, x1), mall)) {
            ok = false;
            break;
          }
          float mraw = mall[0];
#pragma unroll
          for (int q = 1; q < wSplit; ++q) mraw = fmaxf(mraw, mall[q]);
          const float mt = mraw * scale_log2;
          float alpha = 1.f;
          bool resc = false;
          if (mt != -INFINITY) {
            if (m == -INFINITY) {
              m = mt;
            } else if (mt > m + wLazyLog2) {
              alpha = exp2f(m - mt);
              m = mt;
              resc = true;
            }
          }
          const float mneg = m == -INFINITY ? 0.f : -m;
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int c = 0; c < wKW; c += 4) {   // packed scale and sums, as in prefill_tc.cu
            float y0, y1, y2, y3;
            t_fma2(y0, y1, svv[c], svv[c + 1], scale_log2, mneg);
            t_fma2(y2, y3, svv[c + 2], svv[c + 3], scale_log2, mneg);
            svv[c] = t_ex2(y0);
            svv[c + 1] = t_ex2(y1);
            svv[c + 2] = t_ex2(y2);
            svv[c + 3] = t_ex2(y3);
            t_add2(s0, s1, svv[c], svv[c + 1]);
            t_add2(s2, s3, svv[c + 2], svv[c + 3]);
          }
          l = l * alpha + ((s0 + s1) + (s2 + s3));
          if (__any_sync(0xffffffffu, resc)) {   // this warp's columns of O *= alpha
            if (!t_wait_warp(pvdone + 8 * ((g - 1) & 1), (g - 1) >> 1, abort_flag)) {
              ok = false;
              break;
            }
            t_fence_after();
#pragma unroll
            for (int c = 0; c < OH / 16; ++c) {
              uint32_t r[16];
              t_ld16(trow + ocol + 16 * c, r);
              t_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
              t_st16(trow + ocol + 16 * c, r);
            }
            t_wait_st();
          }
          if (g >= 2 && !t_wait_warp(pvdone + 8 * b, (g >> 1) - 1, abort_flag)) {
            ok = false;
            break;
          }
          {
            uint8_t *prow = sm + C::OFF_P + b * C::P_BYTES + row * 128;
#pragma unroll
            for (int q4 = 0; q4 < wKW / 8; ++q4) {
              const int ch = (wKW / 8) * hf + q4;
              uint4 v;
              v.x = t_pack(svv[8 * q4 + 0], svv[8 * q4 + 1]);
              v.y = t_pack(svv[8 * q4 + 2], svv[8 * q4 + 3]);
              v.z = t_pack(svv[8 * q4 + 4], svv[8 * q4 + 5]);
              v.w = t_pack(svv[8 * q4 + 6], svv[8 * q4 + 7]);
              *reinterpret_cast<uint4 *>(prow + ((ch ^ (row & 7)) << 4)) = v;
            }
          }
        }   // need
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        t_fence_before();
        __syncwarp();
        if (lane == 0) t_arrive(pfull + 8 * b);
        if (ep && !epilogue()) {   // the previous item's output
          ok = false;
          break;
        }
        if (flags & wLast) {
          float lall[wSplit];
          if (!exchange(l, lall)) {
            ok = false;
            break;
          }
          float lt = lall[0];
#pragma unroll
          for (int q = 1; q < wSplit; ++q) lt += lall[q];
          ep = true;
          ep_g = g;
          ep_it = it;
          ep_qi = qi;
          ep_h = hrow;
          ep_oc = w.oc;
          ep_il = lt > 0.f ? 1.f / lt : 0.f;
        }
        ++g;
      } while (!(flags & wLast));
    }
    if (ok && ep && !epilogue()) ok = false;
    if (!ok || *abort_flag) {   // a wait gave up: mark this CTA's rows as failed
      for (int wi = 0; wi < n_mine; ++wi) {
        const int item = sched_item(sched, wi);
        const WItem w = witem_of(item, nq, Hq, C::NOC, pair);
        const int qi = pair ? w.row0 + (row & (wKB - 1)) : w.row0 + row;
        if (qi >= L) continue;
        const int hrow = pair ? w.h + (row >> 6) : w.h;
        __nv_bfloat16 *orow = out + (static_cast<size_t>(hrow) * L + qi) * D + w.oc * wDO + OH * hf;
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

}  // namespace

namespace pkv {
template <int D>
int launch_prefill_wide(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
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
      PKV_CUDA_CHECK(cudaFuncSetAttribute(prefill_wide_kernel<D>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          TW<D>::SMEM));
      done[dev] = true;
    }
  }
  CUtensorMap tmQ, tmK, tmV, tmD;
  const bool pair_q = (Hq / Hkv) % 2 == 0;
  // a Q chunk: 64 rows of two heads (paired) or 128 rows of one; a V tile:
  // 64 keys x the 256 columns of an output half
  int st = prefill_atoms_map(&tmQ, q, Hq, L, D, pair_q ? wKB : wQR, pair_q ? 2 : 1, 1);
  if (st == PKV_OK) st = prefill_head_map(&tmK, k, Hkv, L, D, wKB);
  if (st == PKV_OK) st = prefill_atoms_map(&tmV, v, Hkv, L, D, wKB, 1, wDO / 64);
  if (st == PKV_OK) st = prefill_docs_map(&tmD, docs, L);
  if (st != PKV_OK) return st;
  const int n = (L + wKB - 1) / wKB;
  const int G = Hq / Hkv;
  const bool pair = G % 2 == 0;
  const long long items =
      (pair ? 1LL * n * (Hq / 2) : 1LL * ((n + 1) / 2) * Hq) * TW<D>::NOC;
  const long long cap = pkv::sm_count();
  const int grid = static_cast<int>(items < cap ? items : cap);
  PKV_CUDA_CHECK(pkv::launch_pdl(prefill_wide_kernel<D>, dim3(grid), dim3(wThreads),
                                 TW<D>::SMEM, s, tmQ, tmK, tmV, tmD, docs, kv_num, kv_idx,
                                 full_num, full_idx, n, L, Hq, G, window,
                                 scale * 1.4426950408889634f, pair ? 1 : 0,
                                 reinterpret_cast<__nv_bfloat16 *>(out)));
  return PKV_OK;
}
template int launch_prefill_wide<256>(const pkv_bf16 *, const pkv_bf16 *, const pkv_bf16 *,
                                      const int32_t *, const int32_t *, const int32_t *,
                                      const int32_t *, const int32_t *, int, int, int, int, float,
                                      pkv_bf16 *, cudaStream_t);
template int launch_prefill_wide<512>(const pkv_bf16 *, const pkv_bf16 *, const pkv_bf16 *,
                                      const int32_t *, const int32_t *, const int32_t *,
                                      const int32_t *, const int32_t *, int, int, int, int, float,
                                      pkv_bf16 *, cudaStream_t);
}  // namespace pkv
