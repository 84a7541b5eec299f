// prefill_block_mask + prefill_attn: document-causal attention over packed
// prefill tokens, driven by a block mask.
//
// Semantics: "unsloth: compare main...transformers-continuous-batching-qwen3"
// · scripts/benchmarks/flex_paged_attention.py ·
// PagedKVCache.create_prefill_blockmask_no_paging, and the sliding variant
// _create_prefill_sliding_blockmask of the Gemma-4 inference script. L prompt
// tokens of several documents are packed into one row; docs[t] is the
// document of token t (in any order) and query i keeps key j iff j <= i,
// docs[j] == docs[i] and, with a window W > 0, i - j < W. The attention runs
// on the packed q, k, v themselves ("no paging"), with GQA (query head h
// reads kv head h / (Hq / Hkv)).
//
// The block mask is the tiled summary create_block_mask makes of that mask,
// at the attention kernel's own tile (64 query rows x 64 keys): per query
// block, the ascending lists of FULL key blocks (all 64 x 64 pairs inside L
// and kept: no masking needed) and PARTIAL ones (some pair kept). It depends
// only on docs and W, so one build serves every layer and head of a batch.
// prefill_block_mask_kernel: one CTA per query block; each thread summarises
// one key block's document range, the blocks whose range meets the query
// block's are tested pair by pair by a warp (ballots), and the flags are
// compacted in ascending order by ballot prefix counts.
//
// prefill_attn_kernel: a flash-attention forward on the tensor cores
// (mma.sync m16n8k16, bf16 -> fp32). One CTA of four warps per (64 query
// rows, query head); each warp owns 16 rows. It visits only the listed key
// blocks (full ones first, then partial ones), each 64-token K/V tile
// double-buffered in shared memory with cp.async (16-byte chunks,
// XOR-swizzled rows, so the ldmatrix reads are conflict-free; tokens past L
// zero-filled), the block index two tiles ahead read early. Per tile the warp
// computes S = Q K^T, masks partial tiles (causal, document, window, inside
// L), keeps an online softmax in the exp2 domain and adds P V, with P taken
// straight from the S accumulators as the A operand. In a partial tile each
// warp skips the 16-key groups that cannot hold a kept pair for any of its 16
// rows (after its last row, outside the window, or with document ids outside
// its rows' range): half of a diagonal tile's work on average. The CTAs of the last
// query blocks are scheduled first.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "pkv_internal.h"

namespace {

constexpr int kBM = 64;   // query rows per CTA
constexpr int kBN = 64;   // keys per tile
constexpr int kPWarps = 4;
constexpr int kPThreads = kPWarps * 32;

template <int D>
struct PCfg {
  static constexpr int ROWB = D * 2;
  static constexpr int CH = D / 8;              // 16-byte chunks per row
  static constexpr int TILE = kBN * ROWB;
  // K buffers 0 and 1, then V buffers 0 and 1. The Q tile (kBM == kBN rows)
  // shares K buffer 1: it is read into registers before that buffer's first
  // fill.
  static constexpr int OFF_K = 0;
  static constexpr int OFF_Q = TILE;
  static constexpr int OFF_V = OFF_K + 2 * TILE;
  static constexpr int OFF_DQ = OFF_V + 2 * TILE;        // int [kBM]
  static constexpr int OFF_DK = OFF_DQ + kBM * 4;        // int [2][kBN]
  static constexpr int SMEM = OFF_DK + 2 * kBN * 4;
  // CTAs per SM the launch bounds ask for: registers and shared memory allow
  // 3 at D = 128 (66 KB each) and 4 at D = 64
  static constexpr int MIN_CTAS = D == 128 ? 3 : 4;
};

__device__ __forceinline__ uint32_t p_smem(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// byte offset of 16-byte chunk c of row r, rows of D bf16, chunk index XORed
// with the row's low three bits
template <int D>
__device__ __forceinline__ uint32_t p_swz(int r, int c) {
  return static_cast<uint32_t>(r * (D * 2) + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void p_ldsm_x4(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void p_ldsm_x4_t(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void p_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                      uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t p_pack(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// rows [row0, row0 + 64) of a [L][D] head into a swizzled tile, and their
// document ids (tokens past L: zeros and document INT_MIN)
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const __nv_bfloat16 *head, int row0,
                                          int L, int *dtile, const int32_t *docs, int tid) {
  using C = PCfg<D>;
  for (int i = tid; i < kBN * C::CH; i += kPThreads) {
    const int r = i / C::CH, c = i - r * C::CH;
    const int row = row0 + r;
    const bool ok = row < L;
    cp_async16(dst + p_swz<D>(r, c), head + static_cast<size_t>(ok ? row : 0) * D + c * 8, ok);
  }
  for (int r = tid; r < kBN; r += kPThreads) {
    const int row = row0 + r;
    dtile[r] = row < L ? docs[row] : (-2147483647 - 1);
  }
}

// ---------------------------------------------------------------------------
// Block mask builder
// ---------------------------------------------------------------------------
constexpr int kMThreads = 128;   // key blocks summarised per pass

__global__ void __launch_bounds__(kMThreads)
    prefill_block_mask_kernel(const int32_t *__restrict__ docs, int L, int n, int window,
                              int32_t *__restrict__ kv_num, int32_t *__restrict__ kv_idx,
                              int32_t *__restrict__ full_num, int32_t *__restrict__ full_idx) {
  __shared__ int s_qd[kBM];
  __shared__ int s_cand[kMThreads];
  __shared__ uint8_t s_flag[kMThreads];
  __shared__ int s_ncand, s_qlo, s_qhi;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pkv_wait_prior_grid();
  pkv_allow_next_grid();
  const int qb = blockIdx.x, row0 = qb * kBM;
  const int nq = min(kBM, L - row0);
  if (tid < kBM) s_qd[tid] = tid < nq ? docs[row0 + tid] : 0;
  __syncthreads();
  if (warp == 0) {   // document range of the query block's rows inside L
    int lo = 2147483647, hi = -2147483647 - 1;
    for (int r = lane; r < nq; r += 32) {
      lo = min(lo, s_qd[r]);
      hi = max(hi, s_qd[r]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      s_qlo = lo;
      s_qhi = hi;
    }
  }
  // rows of this block that are inside L: lane and lane + 32
  const int qd0 = s_qd[lane], qd1 = s_qd[lane + 32];
  const int qi0 = row0 + lane, qi1 = qi0 + 32;
  const bool qv0 = lane < nq, qv1 = lane + 32 < nq;
  int kb_lo = 0;   // no key before row0 - W + 1 is kept
  if (window > 0 && row0 - window + 1 > 0) kb_lo = (row0 - window + 1) / kBN;
  int np = 0, nf = 0;   // list lengths so far (kept by warp 0)
  int32_t *prow = kv_idx + static_cast<size_t>(qb) * n;
  int32_t *frow = full_idx + static_cast<size_t>(qb) * n;
  for (int c0 = kb_lo; c0 <= qb; c0 += kMThreads) {
    if (tid == 0) s_ncand = 0;
    s_flag[tid] = 0;
    __syncthreads();   // s_qlo / s_qhi visible; s_ncand reset
    const int kb = c0 + tid;
    if (kb <= qb) {
      const int j0 = kb * kBN, nk = min(kBN, L - j0);
      int lo = 2147483647, hi = -2147483647 - 1;
      for (int r = 0; r < nk; ++r) {
        const int d = __ldg(docs + j0 + r);
        lo = min(lo, d);
        hi = max(hi, d);
      }
      if (lo <= s_qhi && s_qlo <= hi) s_cand[atomicAdd(&s_ncand, 1)] = kb;
    }
    __syncthreads();
    const int nc = s_ncand;
    for (int c = warp; c < nc; c += kMThreads / 32) {   // exact test, one warp per block
      const int kbc = s_cand[c], j0 = kbc * kBN;
      const bool kv0 = j0 + lane < L, kv1 = j0 + lane + 32 < L;
      const int kd0 = kv0 ? docs[j0 + lane] : 0, kd1 = kv1 ? docs[j0 + lane + 32] : 0;
      bool any = false, all = nq == kBM && j0 + kBN <= L;
#pragma unroll 4
      for (int t = 0; t < kBN; ++t) {
        const int kd = __shfl_sync(0xffffffffu, t < 32 ? kd0 : kd1, t & 31);
        const int j = j0 + t;
        const bool in = j < L;
        const bool k0 = qv0 && in && j <= qi0 && kd == qd0 && (window == 0 || qi0 - j < window);
        const bool k1 = qv1 && in && j <= qi1 && kd == qd1 && (window == 0 || qi1 - j < window);
        any |= k0 || k1;
        all &= k0 && k1;
      }
      any = __any_sync(0xffffffffu, any);
      all = __all_sync(0xffffffffu, all);
      if (lane == 0) s_flag[kbc - c0] = all ? 2 : (any ? 1 : 0);
    }
    __syncthreads();
    if (warp == 0) {   // ascending compaction of this pass's flags
      const unsigned lt = (1u << lane) - 1u;
#pragma unroll
      for (int g = 0; g < kMThreads / 32; ++g) {
        const int kbg = c0 + g * 32 + lane;
        const int f = kbg <= qb ? s_flag[g * 32 + lane] : 0;
        const unsigned mp = __ballot_sync(0xffffffffu, f == 1);
        const unsigned mf = __ballot_sync(0xffffffffu, f == 2);
        if (f == 1) prow[np + __popc(mp & lt)] = kbg;
        if (f == 2) frow[nf + __popc(mf & lt)] = kbg;
        np += __popc(mp);
        nf += __popc(mf);
      }
    }
    __syncthreads();   // flags and candidates are rewritten by the next pass
  }
  if (tid == 0) {
    kv_num[qb] = np;
    full_num[qb] = nf;
  }
}

// ---------------------------------------------------------------------------
// Attention
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kPThreads, PCfg<D>::MIN_CTAS)
    prefill_attn_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                        const __nv_bfloat16 *__restrict__ v, const int32_t *__restrict__ docs,
                        const int32_t *__restrict__ kv_num, const int32_t *__restrict__ kv_idx,
                        const int32_t *__restrict__ full_num,
                        const int32_t *__restrict__ full_idx, int nblk, int L, int Hq, int G,
                        int window, float scale_log2, __nv_bfloat16 *__restrict__ out) {
  using C = PCfg<D>;
  constexpr int KS = D / 16;   // k-steps of Q K^T
  constexpr int NO = D / 8;    // n-tiles of O
  extern __shared__ __align__(128) uint8_t psm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  pkv_wait_prior_grid();
  pkv_allow_next_grid();

  const int qt = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);  // heavy first
  const int h = blockIdx.y, g = h / G;
  const int row0 = qt * kBM;
  const __nv_bfloat16 *qh = q + static_cast<size_t>(h) * L * D;
  const __nv_bfloat16 *kh = k + static_cast<size_t>(g) * L * D;
  const __nv_bfloat16 *vh = v + static_cast<size_t>(g) * L * D;
  const uint32_t s0 = p_smem(psm), sQ = s0 + C::OFF_Q, sK = s0 + C::OFF_K, sV = s0 + C::OFF_V;
  int *dq = reinterpret_cast<int *>(psm + C::OFF_DQ);
  int *dk = reinterpret_cast<int *>(psm + C::OFF_DK);

  // the block lists of this query block (entries outside [0, n) are skipped)
  const int32_t *frow = full_idx + static_cast<size_t>(qt) * nblk;
  const int32_t *prow = kv_idx + static_cast<size_t>(qt) * nblk;
  const int fn = min(max(full_num[qt], 0), nblk), pn = min(max(kv_num[qt], 0), nblk);
  const int total = fn + pn;
  auto block_at = [&](int t) -> int {
    const int x = t < fn ? frow[t] : prow[t - fn];
    return x >= 0 && x < nblk ? x : -1;
  };
  int cur = total > 0 ? block_at(0) : -1;
  int nxt = total > 1 ? block_at(1) : -1;

  load_tile<D>(sQ, qh, row0, L, dq, docs, tid);
  if (total > 0) {
    load_tile<D>(sK, kh, max(cur, 0) * kBN, L, dk, docs, tid);
    load_tile<D>(sV, vh, max(cur, 0) * kBN, L, dk, docs, tid);
  }
  cp_commit();

  uint32_t qa[KS][4];
  float o[NO][4];
#pragma unroll
  for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int qi0 = row0 + warp * 16 + gid, qi1 = qi0 + 8;
  int dq0 = 0, dq1 = 0;
  // this warp's rows inside L and the range of their document ids
  const int rlo = row0 + warp * 16, rhi = min(rlo + 15, L - 1);
  int wdlo = 2147483647, wdhi = -2147483647 - 1;
  if (total == 0) cp_wait<0>();

  for (int t = 0; t < total; ++t) {
    const int nn = t + 2 < total ? block_at(t + 2) : -1;   // read two tiles ahead
    const int buf = t & 1;
    if (t > 0) {
      if (t + 1 < total) {   // the next key tile into the other buffer
        const int nb = buf ^ 1;
        load_tile<D>(sK + nb * C::TILE, kh, max(nxt, 0) * kBN, L, dk + nb * kBN, docs, tid);
        load_tile<D>(sV + nb * C::TILE, vh, max(nxt, 0) * kBN, L, dk + nb * kBN, docs, tid);
        cp_commit();
        cp_wait<1>();
      } else {
        cp_wait<0>();
      }
      __syncthreads();
    } else {
      // Q and the first tile; Q goes to registers, then K buffer 1 (where Q
      // sits) takes the second tile
      cp_wait<0>();
      __syncthreads();
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
        p_ldsm_x4(sQ + p_swz<D>(warp * 16 + (lane & 15), 2 * ks + (lane >> 4)), qa[ks][0],
                  qa[ks][1], qa[ks][2], qa[ks][3]);
      dq0 = dq[warp * 16 + gid];
      dq1 = dq[warp * 16 + gid + 8];
      const int dr = (lane & 15) <= rhi - rlo ? dq[warp * 16 + (lane & 15)] : dq[warp * 16];
      wdlo = dr;
      wdhi = dr;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        wdlo = min(wdlo, __shfl_xor_sync(0xffffffffu, wdlo, o));
        wdhi = max(wdhi, __shfl_xor_sync(0xffffffffu, wdhi, o));
      }
      __syncthreads();   // every warp holds its Q fragments
      if (total > 1) {
        load_tile<D>(sK + C::TILE, kh, max(nxt, 0) * kBN, L, dk + kBN, docs, tid);
        load_tile<D>(sV + C::TILE, vh, max(nxt, 0) * kBN, L, dk + kBN, docs, tid);
        cp_commit();
      }
    }
    const int *dkt = dk + buf * kBN;
    const bool full = t < fn;
    const int j0 = cur * kBN;
    // 16-key groups of this tile that may hold a kept pair for one of this
    // warp's rows (bit g: keys j0 + 16g .. j0 + 16g + 15); a group whose keys
    // all come after the warp's last row, all fall outside the window, lie
    // past L, or whose document ids miss the rows' id range adds nothing
    int act = 0;
    if (cur >= 0 && rlo < L) {
      act = 0xf;
      if (!full) {
        int lo0 = dkt[lane], hi0 = lo0, lo1 = dkt[lane + 32], hi1 = lo1;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {   // within each half-warp
          lo0 = min(lo0, __shfl_xor_sync(0xffffffffu, lo0, o));
          hi0 = max(hi0, __shfl_xor_sync(0xffffffffu, hi0, o));
          lo1 = min(lo1, __shfl_xor_sync(0xffffffffu, lo1, o));
          hi1 = max(hi1, __shfl_xor_sync(0xffffffffu, hi1, o));
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int src = (g & 1) << 4;
          const int glo = __shfl_sync(0xffffffffu, g < 2 ? lo0 : lo1, src);
          const int ghi = __shfl_sync(0xffffffffu, g < 2 ? hi0 : hi1, src);
          const int kf = j0 + 16 * g;
          const bool may = kf <= rhi && (window == 0 || kf + 15 > rlo - window) &&
                           ghi >= wdlo && glo <= wdhi;
          if (!may) act &= ~(1 << g);
        }
      }
    }
    if (act) {
      const uint32_t kb = sK + buf * C::TILE, vb = sV + buf * C::TILE;
      // ---- S = Q K^T: 16 rows x 64 keys per warp, active key groups only ----
      float s[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        if (!((act >> np) & 1)) continue;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t b0, b1, b2, b3;
          p_ldsm_x4(kb + p_swz<D>(np * 16 + (lane & 7) + ((lane >> 4) << 3),
                                  2 * ks + ((lane >> 3) & 1)),
                    b0, b1, b2, b3);
          p_mma(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          p_mma(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
      // ---- masks (partial blocks: causal, document, window, inside L) and the
      //      online softmax ----
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kl = n * 8 + 2 * tig + e, key = j0 + kl;
          bool v0 = true, v1 = true;
          if (!((act >> (n >> 1)) & 1)) {
            v0 = v1 = false;
          } else if (!full) {
            const int dkey = dkt[kl];
            v0 = key <= qi0 && key < L && dkey == dq0 && (window == 0 || qi0 - key < window);
            v1 = key <= qi1 && key < L && dkey == dq1 && (window == 0 || qi1 - key < window);
          }
          s[n][e] = v0 ? s[n][e] * scale_log2 : -INFINITY;
          s[n][2 + e] = v1 ? s[n][2 + e] * scale_log2 : -INFINITY;
          mx0 = fmaxf(mx0, s[n][e]);
          mx1 = fmaxf(mx1, s[n][2 + e]);
        }
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        s[n][0] = exp2f(s[n][0] - mu0);
        s[n][1] = exp2f(s[n][1] - mu0);
        s[n][2] = exp2f(s[n][2] - mu1);
        s[n][3] = exp2f(s[n][3] - mu1);
        rs0 += s[n][0] + s[n][1];
        rs1 += s[n][2] + s[n][3];
      }
      l0 = l0 * al0 + rs0;   // per-thread partial sums; the quad sum is taken at the end
      l1 = l1 * al1 + rs1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int n = 0; n < NO; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
      // ---- O += P V: P from the S accumulators, V^T fragments by ldmatrix.trans ----
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        if (!((act >> kq) & 1)) continue;   // P is zero there
        const uint32_t a0 = p_pack(s[2 * kq][0], s[2 * kq][1]);
        const uint32_t a1 = p_pack(s[2 * kq][2], s[2 * kq][3]);
        const uint32_t a2 = p_pack(s[2 * kq + 1][0], s[2 * kq + 1][1]);
        const uint32_t a3 = p_pack(s[2 * kq + 1][2], s[2 * kq + 1][3]);
#pragma unroll
        for (int dp = 0; dp < NO / 2; ++dp) {
          uint32_t b0, b1, b2, b3;
          p_ldsm_x4_t(vb + p_swz<D>(kq * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                    2 * dp + (lane >> 4)),
                      b0, b1, b2, b3);
          p_mma(o[2 * dp], a0, a1, a2, a3, b0, b1);
          p_mma(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();   // this buffer is refilled in the next iteration
    cur = nxt;
    nxt = nn;
  }

  // ---- epilogue: 1 / row sum, bf16, rows inside L ----
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const float il0 = l0 > 0.f ? 1.f / l0 : 0.f, il1 = l1 > 0.f ? 1.f / l1 : 0.f;
  __nv_bfloat16 *oh = out + static_cast<size_t>(h) * L * D;
#pragma unroll
  for (int n = 0; n < NO; ++n) {
    const int d = n * 8 + 2 * tig;
    if (qi0 < L)
      *reinterpret_cast<uint32_t *>(oh + static_cast<size_t>(qi0) * D + d) =
          p_pack(o[n][0] * il0, o[n][1] * il0);
    if (qi1 < L)
      *reinterpret_cast<uint32_t *>(oh + static_cast<size_t>(qi1) * D + d) =
          p_pack(o[n][2] * il1, o[n][3] * il1);
  }
}

template <int D>
int launch_prefill(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v, const int32_t *docs,
                   const int32_t *kv_num, const int32_t *kv_idx, const int32_t *full_num,
                   const int32_t *full_idx, int L, int Hq, int Hkv, int window, float scale,
                   pkv_bf16 *out, cudaStream_t s) {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  PKV_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return pkv::fail(PKV_E_CUDA, "device id out of range");
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      PKV_CUDA_CHECK(cudaFuncSetAttribute(prefill_attn_kernel<D>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          PCfg<D>::SMEM));
      done[dev] = true;
    }
  }
  const int n = (L + kBM - 1) / kBM;
  const dim3 grid(n, Hq);
  PKV_CUDA_CHECK(pkv::launch_pdl(prefill_attn_kernel<D>, grid, dim3(kPThreads), PCfg<D>::SMEM,
                                 s, reinterpret_cast<const __nv_bfloat16 *>(q),
                                 reinterpret_cast<const __nv_bfloat16 *>(k),
                                 reinterpret_cast<const __nv_bfloat16 *>(v), docs, kv_num, kv_idx,
                                 full_num, full_idx, n, L, Hq, Hq / Hkv, window,
                                 scale * 1.4426950408889634f,
                                 reinterpret_cast<__nv_bfloat16 *>(out)));
  return PKV_OK;
}

}  // namespace

extern "C" int prefill_block_mask(const int32_t *docs, int L, int window,
                                  int32_t *kv_num_blocks, int32_t *kv_indices,
                                  int32_t *full_kv_num_blocks, int32_t *full_kv_indices,
                                  void *stream) {
  if (L < 0 || L > 0x7fffffff - kBM || window < 0)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_block_mask: bad L or window");
  if (L == 0) return pkv::ok();
  if (!docs || !kv_num_blocks || !kv_indices || !full_kv_num_blocks || !full_kv_indices)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_block_mask: NULL pointer");
  const int n = (L + kBM - 1) / kBM;
  PKV_CUDA_CHECK(pkv::launch_pdl(prefill_block_mask_kernel, dim3(n), dim3(kMThreads), 0,
                                 static_cast<cudaStream_t>(stream), docs, L, n, window,
                                 kv_num_blocks, kv_indices, full_kv_num_blocks,
                                 full_kv_indices));
  return pkv::ok();
}

extern "C" int prefill_attn(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                            const int32_t *docs, const int32_t *kv_num_blocks,
                            const int32_t *kv_indices, const int32_t *full_kv_num_blocks,
                            const int32_t *full_kv_indices, int L, int Hq, int Hkv, int D,
                            int window, float scale, pkv_bf16 *out, void *stream) {
  if (D != 64 && D != 128)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: D must be 64 or 128");
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: need Hq %% Hkv == 0");
  if (L < 0 || L > 0x7fffffff - kBM || Hq > 65535 || window < 0)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: bad size or window");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: scale must be finite and > 0");
  if (L == 0) return pkv::ok();
  if (!q || !k || !v || !docs || !out || !kv_num_blocks || !kv_indices || !full_kv_num_blocks ||
      !full_kv_indices)
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: NULL pointer");
  if (!pkv::aligned16(q) || !pkv::aligned16(k) || !pkv::aligned16(v) || !pkv::aligned16(out))
    return pkv::fail(PKV_E_BAD_ARG, "prefill_attn: tensors must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int st =
      D == 64 ? launch_prefill<64>(q, k, v, docs, kv_num_blocks, kv_indices, full_kv_num_blocks,
                                   full_kv_indices, L, Hq, Hkv, window, scale, out, s)
              : launch_prefill<128>(q, k, v, docs, kv_num_blocks, kv_indices,
                                    full_kv_num_blocks, full_kv_indices, L, Hq, Hkv, window,
                                    scale, out, s);
  if (st != PKV_OK) return st;
  return pkv::ok();
}
