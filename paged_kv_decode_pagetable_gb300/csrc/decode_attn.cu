// paged_decode_attn: split-KV GQA decode attention over a paged bf16 cache.
//
// Semantics: "unsloth: compare main...flex-moe-qwen3" · unsloth/inference/
// flex_gemma4_moe.py · attention forward (flex_attention(q, k, v, scale,
// block_mask, enable_gqa=True), q of shape (B, Hq, 1, D)) and
// _decode_block_mask (full layers: pos >= kv; sliding: also pos - kv < W).
// With L = pos + 1 the keys of row b are [lo, L), lo = max(0, L - W).
//
// Design (GB300):
//   * grid (split, kv head, row); one CTA of 4 warps streams its share of
//     the row's keys once for all G <= 8 query heads of the GQA group;
//   * keys are processed in tiles of 64; each tile's K and V are staged in
//     shared memory by TMA (cp.async.bulk.tensor, 128-byte swizzle), one
//     box per (page segment, 64-column chunk), with separate K / V
//     mbarriers and an NS-deep ring so the next tiles are in flight while
//     the current one is computed;
//   * S^T = K q^T and O^T = V^T P^T run on the tensor cores
//     (mma.sync m16n8k16 bf16 -> fp32) with keys / head-dim on M and the
//     query heads on N, so no head padding beyond N = 8 is paid;
//   * online softmax in the exp2 domain with a CTA-wide running max; P is
//     exchanged through a 1 KB shared buffer;
//   * each split writes an fp32 partial output and its log2-sum-exp; a
//     combine kernel merges splits (skipped when there is one split);
//   * every wait is bounded; a wait that gives up sets PKV_ERR_TIMEOUT and
//     the CTA drains its copies and exits. Invalid table entries are
//     reported through the error word and never dereferenced.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "pkv_internal.h"

namespace {

constexpr int kT = 64;          // keys per tile
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxG = 8;        // query heads per kv head (MMA N)
constexpr int kSpinLimit = 1 << 21;

template <int D>
struct Cfg {
  static constexpr int NS = D <= 64 ? 4 : D <= 128 ? 3 : D <= 256 ? 2 : 1;
  static constexpr int CHUNKS = D / 64;             // 128-byte column chunks
  static constexpr int CHUNK_BYTES = kT * 128;      // one chunk of one tile
  static constexpr int STAGE_BYTES = kT * D * 2;
  static constexpr int OFF_V = NS * STAGE_BYTES;
  static constexpr int OFF_P = 2 * NS * STAGE_BYTES;
  static constexpr int OFF_RED = OFF_P + kT * 16;            // 2 x [4][8] f32
  static constexpr int OFF_BAR = OFF_RED + 2 * kWarps * kMaxG * 4;
  static constexpr int OFF_MASK = OFF_BAR + 2 * NS * 8;      // 2 x NS u32
  static constexpr int OFF_FLAG = OFF_MASK + 2 * NS * 4;
  static constexpr int SMEM = OFF_FLAG + 16 + 1024;          // + alignment slack
  static constexpr int MIN_BLOCKS = D <= 128 ? 2 : 1;
};

// ---------------------------------------------------------------- PTX ----
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after kSpinLimit polls (each poll may suspend the
// thread for a hardware-defined interval).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm,
                                            int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                        uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// byte offset of 16-byte chunk `chunk` (8 bf16 along D) of tile row `r`
// inside one stage laid out by TMA with SWIZZLE_128B: column chunks of 64
// elements are separate [kT][128 B] blocks; inside a 1024-byte atom the
// 16-byte unit index is XORed with the row index mod 8.
__device__ __forceinline__ uint32_t swz(int r, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (kT * 128) + r * 128 +
                               (((chunk & 7) ^ (r & 7)) << 4));
}

// ------------------------------------------------------------- kernel ----
template <int D>
__global__ void __launch_bounds__(kThreads, Cfg<D>::MIN_BLOCKS)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __nv_bfloat16 *__restrict__ q,
                        const int32_t *__restrict__ table, int n_slots,
                        int max_pages, int log2_ps, int n_pages,
                        const int32_t *__restrict__ batch_idx,
                        const int32_t *__restrict__ seq_lens, int window,
                        float scale_log2, int Hq, int G, int S,
                        float *__restrict__ o_part, float *__restrict__ lse_part,
                        __nv_bfloat16 *__restrict__ out, int32_t *__restrict__ err) {
  using C = Cfg<D>;
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int ps = 1 << log2_ps;
  const bool reporter = (s == 0 && g == 0 && tid == 0);

  // ---- this CTA's key range (identical in every thread) ----
  int slot = batch_idx ? batch_idx[b] : b;
  int L = seq_lens[b];
  bool empty = false;
  if (slot < 0 || slot >= n_slots) {
    if (reporter && err) atomicOr(err, PKV_ERR_SLOT);
    empty = true;
  }
  const int Lmax = max_pages << log2_ps;
  if (L > Lmax || L < 0) {
    if (reporter && err) atomicOr(err, PKV_ERR_POS);
    L = L < 0 ? 0 : Lmax;
  }
  if (slot == 0 || L <= 0) empty = true;
  const int lo = window > 0 ? max(0, L - window) : 0;
  const int t_first = lo / kT, t_end = (L + kT - 1) / kT;
  const int per = (t_end - t_first + S - 1) / S;
  const int ta = t_first + s * per, tb = min(t_end, ta + per);
  const int k0 = max(lo, ta * kT), k1 = min(L, tb * kT);
  const size_t head0 = static_cast<size_t>(b) * Hq + static_cast<size_t>(g) * G;

  if (empty || ta >= tb) {
    if (S == 1) {
      for (int i = tid; i < G * D; i += kThreads)
        out[head0 * D + i] = __float2bfloat16_rn(0.f);
    } else if (tid < G) {
      lse_part[(head0 + tid) * S + s] = -INFINITY;
    }
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_u32(sm), sV = sK + C::OFF_V, sP = sK + C::OFF_P;
  float *red_max = reinterpret_cast<float *>(sm + C::OFF_RED);
  float *red_sum = red_max + kWarps * kMaxG;
  const uint32_t barK = sK + C::OFF_BAR, barV = barK + C::NS * 8;
  uint32_t *kmask = reinterpret_cast<uint32_t *>(sm + C::OFF_MASK);
  uint32_t *vmask = kmask + C::NS;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_FLAG);

  const int box_rows = ps < kT ? ps : kT;
  const int boxes = kT / box_rows;
  const uint32_t all_boxes = boxes == 32 ? 0xffffffffu : ((1u << boxes) - 1u);
  const int n_local = tb - ta;
  const int32_t *trow = table + static_cast<size_t>(slot) * max_pages;

  // producer (thread 0): stage tile t of K (is_v=0) or V (is_v=1)
  auto issue = [&](int t, int stage, int is_v) {
    const CUtensorMap *tm = is_v ? &tmV : &tmK;
    const uint32_t dst0 = (is_v ? sV : sK) + stage * C::STAGE_BYTES;
    const uint32_t bar = (is_v ? barV : barK) + stage * 8;
    uint32_t mask = 0;
    int rows[kT / 8];
    for (int i = 0; i < boxes; ++i) {
      const int key = t * kT + i * box_rows;
      rows[i] = -1;
      if (key + box_rows <= k0 || key >= k1) continue;
      const int page = trow[key >> log2_ps];
      if (page < 0) {
        if (err) atomicOr(err, PKV_ERR_PAGE_NEG);
        continue;
      }
      if (page >= n_pages) {
        if (err) atomicOr(err, PKV_ERR_PAGE_RANGE);
        continue;
      }
      rows[i] = ((g * n_pages + page) << log2_ps) + (key & (ps - 1));
      mask |= 1u << i;
    }
    (is_v ? vmask : kmask)[stage] = mask;
    mbar_expect_tx(bar, static_cast<uint32_t>(__popc(mask)) * C::CHUNKS * box_rows * 128);
    for (int i = 0; i < boxes; ++i) {
      if (rows[i] < 0) continue;
#pragma unroll
      for (int cc = 0; cc < C::CHUNKS; ++cc)
        tma_load_2d(dst0 + cc * C::CHUNK_BYTES + i * box_rows * 128, tm, cc * 64,
                    rows[i], bar);
    }
  };

  if (tid == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(barK + i * 8, 1);
      mbar_init(barV + i * 8, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  __syncthreads();
  // copies issued / completions observed, tracked by thread 0 only
  int issued_k = 0, issued_v = 0, waited_k = 0, waited_v = 0;
  if (tid == 0) {
    for (; issued_k < min(C::NS, n_local); ++issued_k) issue(ta + issued_k, issued_k, 0);
    for (; issued_v < min(C::NS - 1, n_local); ++issued_v) issue(ta + issued_v, issued_v, 1);
  }

  // Q^T as MMA B fragments (N = head gid, K = head dim), zero for gid >= G
  constexpr int KS = D / 16;
  uint32_t qb[KS][2];
  {
    const bool hv = gid < G;
    const uint32_t *qrow =
        reinterpret_cast<const uint32_t *>(q + (head0 + (hv ? gid : 0)) * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[ks][0] = hv ? qrow[(16 * ks + 2 * tig) >> 1] : 0u;
      qb[ks][1] = hv ? qrow[(16 * ks + 8 + 2 * tig) >> 1] : 0u;
    }
  }

  constexpr int MT = D / 64;  // 16-row m-tiles of this warp's D/4 slice
  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;
  const int h0 = 2 * tig, h1 = 2 * tig + 1;
  const bool hv0 = h0 < G, hv1 = h1 < G;
  int lt = 0;
  bool aborted = false;

  for (; lt < n_local; ++lt) {
    const int t = ta + lt, st = lt % C::NS;
    const uint32_t par = (lt / C::NS) & 1;
    if (mbar_wait(barK + st * 8, par))
      waited_k = lt + 1;
    else
      *abort_flag = 1;
    const uint32_t km = kmask[st];
    const uint32_t kbase = sK + st * C::STAGE_BYTES;

    // ---- S^T[16 keys x 8 heads] for keys 16*warp .. +15 of the tile ----
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int mi = lane >> 3;
      const int r = 16 * warp + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + swz(r, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
        mma_bf16(sacc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
      }
    }
    const int kr_lo = 16 * warp + gid, kr_hi = kr_lo + 8;
    const int key_lo = t * kT + kr_lo, key_hi = t * kT + kr_hi;
    const bool v_lo = key_lo >= k0 && key_lo < k1 && ((km >> (kr_lo / box_rows)) & 1u);
    const bool v_hi = key_hi >= k0 && key_hi < k1 && ((km >> (kr_hi / box_rows)) & 1u);
    float s00 = (v_lo && hv0) ? sacc[0] * scale_log2 : -INFINITY;
    float s01 = (v_lo && hv1) ? sacc[1] * scale_log2 : -INFINITY;
    float s10 = (v_hi && hv0) ? sacc[2] * scale_log2 : -INFINITY;
    float s11 = (v_hi && hv1) ? sacc[3] * scale_log2 : -INFINITY;
    float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    if (gid == 0) {
      red_max[warp * kMaxG + h0] = mx0;
      red_max[warp * kMaxG + h1] = mx1;
    }
    __syncthreads();  // (1) K stage consumed; maxima visible
    if (*abort_flag) {
      aborted = true;
      break;
    }
    if (tid == 0) {
      fence_proxy_async();
      if (issued_k < n_local) {
        issue(ta + issued_k, issued_k % C::NS, 0);
        ++issued_k;
      }
      if (issued_v < n_local && issued_v <= lt + C::NS - 1) {
        issue(ta + issued_v, issued_v % C::NS, 1);
        ++issued_v;
      }
    }
    float mt0 = red_max[h0], mt1 = red_max[h1];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      mt0 = fmaxf(mt0, red_max[w * kMaxG + h0]);
      mt1 = fmaxf(mt1, red_max[w * kMaxG + h1]);
    }
    const float mn0 = fmaxf(m_run0, mt0), mn1 = fmaxf(m_run1, mt1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float p00 = exp2f(s00 - mu0), p01 = exp2f(s01 - mu1);
    const float p10 = exp2f(s10 - mu0), p11 = exp2f(s11 - mu1);
    {
      uint32_t *pt = reinterpret_cast<uint32_t *>(sm + C::OFF_P);
      pt[kr_lo * 4 + tig] = pack_bf16(p00, p01);
      pt[kr_hi * 4 + tig] = pack_bf16(p10, p11);
    }
    float sm0 = p00 + p10, sm1 = p01 + p11;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      sm0 += __shfl_xor_sync(0xffffffffu, sm0, off);
      sm1 += __shfl_xor_sync(0xffffffffu, sm1, off);
    }
    if (gid == 0) {
      red_sum[warp * kMaxG + h0] = sm0;
      red_sum[warp * kMaxG + h1] = sm1;
    }
    // ---- V tile: wait, then clear rows of keys outside [k0, k1) ----
    if (mbar_wait(barV + st * 8, par))
      waited_v = lt + 1;
    else
      *abort_flag = 1;
    const uint32_t vm = vmask[st];
    const uint32_t vbase = sV + st * C::STAGE_BYTES;
    const bool full_tile = t * kT >= k0 && t * kT + kT <= k1 && vm == all_boxes;
    if (!full_tile) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int i = tid; i < kT * (D / 8); i += kThreads) {
        const int r = i / (D / 8), c = i % (D / 8);
        const int key = t * kT + r;
        const bool valid = key >= k0 && key < k1 && ((vm >> (r / box_rows)) & 1u);
        if (!valid)
          *reinterpret_cast<uint4 *>(sm + C::OFF_V + st * C::STAGE_BYTES +
                                     (c >> 3) * (kT * 128) + r * 128 + (c & 7) * 16) = z;
      }
      fence_proxy_async();
    }
    __syncthreads();  // (2) P, sums and V visible
    if (*abort_flag) {
      aborted = true;
      break;
    }
    float ts0 = 0.f, ts1 = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      ts0 += red_sum[w * kMaxG + h0];
      ts1 += red_sum[w * kMaxG + h1];
    }
    const float al0 = exp2f(m_run0 - mu0), al1 = exp2f(m_run1 - mu1);
    l_run0 = l_run0 * al0 + ts0;
    l_run1 = l_run1 * al1 + ts1;
    m_run0 = mn0;
    m_run1 = mn1;
    // ---- O^T[warp's D/4 slice x 8 heads] += V^T P^T ----
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      o[mt][0] *= al0;
      o[mt][1] *= al1;
      o[mt][2] *= al0;
      o[mt][3] *= al1;
    }
#pragma unroll
    for (int kp = 0; kp < kT / 32; ++kp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sP + (32 * kp + lane) * 16, b0, b1, b2, b3);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int ks = 2 * kp + half;
        const uint32_t bb0 = half ? b2 : b0, bb1 = half ? b3 : b1;
        const int mi = lane >> 3;
        const int r = 16 * ks + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int dchunk = (warp * (D / 4) + 16 * mt) / 8 + (mi & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vbase + swz(r, dchunk), a0, a1, a2, a3);
          mma_bf16(o[mt], a0, a1, a2, a3, bb0, bb1);
        }
      }
    }
  }

  if (aborted) {
    if (tid == 0) {
      if (err) atomicOr(err, PKV_ERR_TIMEOUT);
      // drain every copy still in flight before the CTA's smem is released
      for (int i = waited_k; i < issued_k; ++i)
        (void)mbar_wait(barK + (i % C::NS) * 8, (i / C::NS) & 1);
      for (int i = waited_v; i < issued_v; ++i)
        (void)mbar_wait(barV + (i % C::NS) * 8, (i / C::NS) & 1);
    }
    return;
  }

  // ---- epilogue ----
  const float il0 = l_run0 > 0.f ? 1.f / l_run0 : 0.f;
  const float il1 = l_run1 > 0.f ? 1.f / l_run1 : 0.f;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const int d = warp * (D / 4) + 16 * mt + gid;
    if (S == 1) {
      if (hv0) {
        out[(head0 + h0) * D + d] = __float2bfloat16_rn(o[mt][0] * il0);
        out[(head0 + h0) * D + d + 8] = __float2bfloat16_rn(o[mt][2] * il0);
      }
      if (hv1) {
        out[(head0 + h1) * D + d] = __float2bfloat16_rn(o[mt][1] * il1);
        out[(head0 + h1) * D + d + 8] = __float2bfloat16_rn(o[mt][3] * il1);
      }
    } else {
      if (hv0) {
        float *op = o_part + ((head0 + h0) * S + s) * D;
        op[d] = o[mt][0] * il0;
        op[d + 8] = o[mt][2] * il0;
      }
      if (hv1) {
        float *op = o_part + ((head0 + h1) * S + s) * D;
        op[d] = o[mt][1] * il1;
        op[d + 8] = o[mt][3] * il1;
      }
    }
  }
  if (S > 1 && warp == 0 && gid == 0) {
    if (hv0) lse_part[(head0 + h0) * S + s] = l_run0 > 0.f ? m_run0 + log2f(l_run0) : -INFINITY;
    if (hv1) lse_part[(head0 + h1) * S + s] = l_run1 > 0.f ? m_run1 + log2f(l_run1) : -INFINITY;
  }
}

// Merge the splits of one (row, head): weights 2^(lse_s - max), skipping
// empty splits (lse = -inf); a row with no key gives zeros.
__global__ void combine_kernel(const float *__restrict__ o_part,
                               const float *__restrict__ lse_part,
                               __nv_bfloat16 *__restrict__ out, int rows, int S,
                               int D) {
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float *lse = lse_part + static_cast<size_t>(r) * S;
  float m = -INFINITY;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, lse[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const float *op = o_part + static_cast<size_t>(r) * S * D;
  __nv_bfloat16 *orow = out + static_cast<size_t>(r) * D;
  for (int d = 4 * lane; d < D; d += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        const float l = lse[s];
        if (l == -INFINITY) continue;
        const float w = exp2f(l - m);
        const float4 v = *reinterpret_cast<const float4 *>(op + static_cast<size_t>(s) * D + d);
        wsum += w;
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2 packed;
    packed.x = pack_bf16(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(orow + d) = packed;
  }
}

// ------------------------------------------------------------- host ----
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                   void *, const cuuint64_t *, const cuuint64_t *,
                                   const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map over a cache viewed as [rows][D] bf16 with [box_rows][64] boxes.
int make_cache_map(CUtensorMap *tm, const void *base, long long rows, int D,
                   int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

template <int D>
int set_smem_attr() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  PKV_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return pkv::fail(PKV_E_CUDA, "device id out of range");
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    PKV_CUDA_CHECK(cudaFuncSetAttribute(decode_split_kernel<D>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Cfg<D>::SMEM));
    done[dev] = true;
  }
  return PKV_OK;
}

template <int D>
int launch_split(const CUtensorMap &tmK, const CUtensorMap &tmV, const pkv_bf16 *q,
                 const int32_t *table, int n_slots, int max_pages, int log2_ps,
                 int n_pages, const int32_t *batch_idx, const int32_t *seq_lens,
                 int window, float scale_log2, int B, int Hq, int Hkv, int S,
                 float *o_part, float *lse_part, pkv_bf16 *out, int32_t *err,
                 cudaStream_t stream) {
  int st = set_smem_attr<D>();
  if (st != PKV_OK) return st;
  dim3 grid(S, Hkv, B);
  decode_split_kernel<D><<<grid, kThreads, Cfg<D>::SMEM, stream>>>(
      tmK, tmV, reinterpret_cast<const __nv_bfloat16 *>(q), table, n_slots, max_pages,
      log2_ps, n_pages, batch_idx, seq_lens, window, scale_log2, Hq, Hq / Hkv, S,
      o_part, lse_part, reinterpret_cast<__nv_bfloat16 *>(out), err);
  PKV_CUDA_CHECK(cudaGetLastError());
  return PKV_OK;
}

int ctas_per_sm(int D) { return D <= 64 ? 3 : D <= 128 ? 2 : 1; }

int auto_splits(int B, int Hkv, int D, int max_pages, int page_size, int window) {
  long long max_keys = 1LL * max_pages * page_size;
  if (window > 0 && window < max_keys) max_keys = window + kT - 1;
  int max_tiles = static_cast<int>((max_keys + kT - 1) / kT);
  int sms = pkv::sm_count();
  if (sms <= 0) sms = 148;
  long long target = 2LL * sms * ctas_per_sm(D);
  long long work = 1LL * (B > 0 ? B : 1) * Hkv;
  int S = static_cast<int>((target + work - 1) / work);
  int cap = (max_tiles + 1) / 2;  // at least ~2 tiles per split
  if (S > cap) S = cap;
  if (S < 1) S = 1;
  return S;
}

}  // namespace

extern "C" {

size_t paged_decode_attn_workspace(int B, int Hq, int D, int num_splits) {
  if (num_splits <= 1 || B <= 0 || Hq <= 0 || D <= 0) return 0;
  size_t rows = static_cast<size_t>(B) * Hq * num_splits;
  size_t o_bytes = rows * D * sizeof(float);
  o_bytes = (o_bytes + 15) & ~size_t(15);
  return o_bytes + rows * sizeof(float);
}

int paged_decode_attn_splits(int B, int Hkv, int D, int max_pages_per_seq,
                             int page_size, int window, int *num_splits) {
  if (!num_splits || Hkv < 1 || max_pages_per_seq < 1 || page_size < 1)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn_splits: bad argument");
  *num_splits = auto_splits(B, Hkv, D, max_pages_per_seq, page_size, window);
  return pkv::ok();
}

int paged_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                      const pkv_bf16 *v_cache, const int32_t *dev_table,
                      int n_slots, int max_pages_per_seq, int page_size,
                      int n_pages, const int32_t *batch_idx,
                      const int32_t *seq_lens, int window, float scale, int B,
                      int Hq, int Hkv, int D, int num_splits, void *workspace,
                      size_t workspace_bytes, pkv_bf16 *out, int32_t *err_word,
                      void *stream) {
  if (D != 64 && D != 128 && D != 256 && D != 512)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: D must be 64, 128, 256 or 512");
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv || Hq / Hkv > kMaxG)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: need Hq %% Hkv == 0 and Hq/Hkv <= %d", kMaxG);
  if (!pkv::is_pow2(page_size) || page_size < 8)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: page_size must be a power of two >= 8");
  if (B < 0 || n_slots < 1 || max_pages_per_seq < 1 || n_pages < 1 || num_splits < 0)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: bad size argument");
  if (B > 65535 || Hkv > 65535)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: B and Hkv must be <= 65535");
  if (static_cast<long long>(max_pages_per_seq) * page_size > (1LL << 30))
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: table row too long");
  const long long rows = 1LL * Hkv * n_pages * page_size;
  if (rows >= (1LL << 31))
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: cache has too many rows");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: scale must be finite and > 0");
  if (B == 0) return pkv::ok();
  if (!q || !k_cache || !v_cache || !dev_table || !seq_lens || !out)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: NULL tensor");
  if (!pkv::aligned16(q) || !pkv::aligned16(out) || !pkv::aligned16(k_cache) ||
      !pkv::aligned16(v_cache))
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: tensors must be 16-byte aligned");
  int S = num_splits ? num_splits
                     : auto_splits(B, Hkv, D, max_pages_per_seq, page_size, window);
  if (S > 65535) return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: too many splits");
  const size_t need = paged_decode_attn_workspace(B, Hq, D, S);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: workspace needs %zu bytes", need);
    if (!pkv::aligned16(workspace))
      return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn: workspace must be 16-byte aligned");
  }
  float *o_part = static_cast<float *>(workspace);
  float *lse_part = nullptr;
  if (need > 0) {
    size_t o_bytes = static_cast<size_t>(B) * Hq * S * D * sizeof(float);
    o_bytes = (o_bytes + 15) & ~size_t(15);
    lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_bytes);
  }
  const int box_rows = page_size < kT ? page_size : kT;
  CUtensorMap tmK, tmV;
  int st = make_cache_map(&tmK, k_cache, rows, D, box_rows);
  if (st != PKV_OK) return st;
  st = make_cache_map(&tmV, v_cache, rows, D, box_rows);
  if (st != PKV_OK) return st;
  int log2_ps = 0;
  while ((1 << log2_ps) < page_size) ++log2_ps;
  const float scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (D) {
    case 64:
      st = launch_split<64>(tmK, tmV, q, dev_table, n_slots, max_pages_per_seq, log2_ps,
                            n_pages, batch_idx, seq_lens, window, scale_log2, B, Hq, Hkv,
                            S, o_part, lse_part, out, err_word, s);
      break;
    case 128:
      st = launch_split<128>(tmK, tmV, q, dev_table, n_slots, max_pages_per_seq, log2_ps,
                             n_pages, batch_idx, seq_lens, window, scale_log2, B, Hq, Hkv,
                             S, o_part, lse_part, out, err_word, s);
      break;
    case 256:
      st = launch_split<256>(tmK, tmV, q, dev_table, n_slots, max_pages_per_seq, log2_ps,
                             n_pages, batch_idx, seq_lens, window, scale_log2, B, Hq, Hkv,
                             S, o_part, lse_part, out, err_word, s);
      break;
    default:
      st = launch_split<512>(tmK, tmV, q, dev_table, n_slots, max_pages_per_seq, log2_ps,
                             n_pages, batch_idx, seq_lens, window, scale_log2, B, Hq, Hkv,
                             S, o_part, lse_part, out, err_word, s);
      break;
  }
  if (st != PKV_OK) return st;
  if (S > 1) {
    const int rows_bh = B * Hq;
    const int wpb = 4;
    combine_kernel<<<(rows_bh + wpb - 1) / wpb, wpb * 32, 0, s>>>(
        o_part, lse_part, reinterpret_cast<__nv_bfloat16 *>(out), rows_bh, S, D);
    PKV_CUDA_CHECK(cudaGetLastError());
  }
  return pkv::ok();
}

}  // extern "C"
