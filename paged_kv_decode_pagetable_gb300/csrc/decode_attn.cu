// paged_decode_attn: split-KV GQA decode attention over a paged bf16 cache.
//
// Semantics: "unsloth: compare main...flex-moe-qwen3" · unsloth/inference/
// flex_gemma4_moe.py · attention forward (flex_attention(q, k, v, scale,
// block_mask, enable_gqa=True), q of shape (B, Hq, 1, D)) and
// _decode_block_mask (full layers: pos >= kv; sliding: also pos - kv < W).
// With L = pos + 1 the keys of row b are [lo, L), lo = max(0, L - W).
//
// Design (GB300):
//   * work: the key tiles (64 keys) of every (row, kv head). In the default
//     (balanced) mode the (row, kv head, tile) sequence is laid on a cost
//     line from the actual lengths and every persistent CTA takes an equal
//     share of it; a fixed split count (each row cut into S equal parts) is
//     also accepted. A (row, head) finished inside one CTA writes the output
//     directly; one that straddles CTAs leaves fp32 partials + log2-sum-exp
//     that the CTA holding its first part merges (a combine kernel, with a
//     fixed split count). Each partial word is stored as the complement of
//     its bits, so a zero word is one not yet written: the reader polls the
//     data itself (no flag, no release fence) and clears it after use;
//   * persistent CTAs (a fixed grid of SMs x CTAs/SM), each with one
//     producer warp and four consumer warps. The producer streams, across
//     all of the CTA's work without pausing, the query rows (cp.async.bulk)
//     and the K and V tiles (cp.async.bulk.tensor, one box per page segment
//     and 64-column chunk, 128-byte swizzle) into rings of shared-memory
//     stages guarded by full / empty mbarriers, looking up the page ids of
//     the next run of tiles before it waits on the current one;
//   * the kernel and the combine are launched as programmatic dependents of
//     the previous kernel in the stream (griddepcontrol), so launch latency
//     and barrier set-up overlap the previous kernel's tail;
//   * consumers compute S^T = K q^T and O^T = V^T P^T on the tensor cores
//     (mma.sync m16n8k16 bf16 -> fp32) with keys / head-dim on M and the
//     <= 8 query heads of the GQA group on N, with an online softmax in the
//     exp2 domain and a CTA-wide running max (P through a 1 KB buffer);
//   * every mbarrier wait is bounded; a wait that gives up sets
//     PKV_ERR_TIMEOUT, the CTA stops issuing, drains its copies and exits.
//     Invalid table entries are reported in the error word and never
//     dereferenced.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "norm_rope.cuh"
#include "pkv_internal.h"

namespace {

constexpr int kT = 64;               // keys per tile
constexpr int kCWarps = 4;           // consumer warps
constexpr int kCThreads = kCWarps * 32;
constexpr int kThreads = kCThreads + 32;   // + producer warp
constexpr int kMaxG = 8;             // query heads per kv head (MMA N)
constexpr int kMaxRows = 512;        // rows per call (row cache kept in smem)
constexpr int kSpinLimit = 1 << 22;
// Balanced split cost model, in quarter tiles: a key tile costs kTileCost and
// starting a (row, kv head) costs kUnitCost more (its query load, table
// lookups, epilogue and the tail of its partly used last tile). A
// least-squares fit of per-CTA end times (%globaltimer) on the rollout gave
// 0.93 us per tile and 0.75 us per unit for the attention kernel, 1.31 us per
// unit for the fused step (which also rotates the unit's query rows). Both
// kernels use one value, so that they cut rows at the same places and the
// fused step stays bit-identical to the separate calls.
constexpr int kTileCost = 4;
constexpr int kUnitCost = 4;
// Shortest share of the cost line a CTA gets (at least one tile's cost): a
// call too small to give every CTA this much leaves the last CTAs idle
// rather than cutting rows into many short parts.
constexpr int kMinShare = kTileCost;

template <int D>
struct Cfg {
  static constexpr int NS = D <= 64 ? 6 : D <= 128 ? 3 : D <= 256 ? 3 : 1;
  static constexpr int CHUNKS = D / 64;             // 128-byte column chunks
  static constexpr int CHUNK_BYTES = kT * 128;      // one column chunk of a tile
  static constexpr int STAGE_BYTES = kT * D * 2;
  static constexpr int Q_ROW = D * 2 + 16;          // padded: conflict-free B-fragment loads
  static constexpr int Q_BYTES = kMaxG * Q_ROW;
  // one Q stage: the G query rows, then (fused step) the raw k and v rows of
  // the token the unit appends
  static constexpr int Q_STAGE = Q_BYTES + 4 * D;
  static constexpr int OFF_V = NS * STAGE_BYTES;
  static constexpr int OFF_Q = 2 * NS * STAGE_BYTES;
  static constexpr int OFF_P = OFF_Q + 2 * Q_STAGE;
  static constexpr int OFF_RED = OFF_P + kT * 16;                // 2 x [4][8] f32
  static constexpr int OFF_BAR = OFF_RED + 2 * kCWarps * kMaxG * 4;
  static constexpr int N_BARS = 4 * NS + 4;
  static constexpr int OFF_MASK = OFF_BAR + N_BARS * 8;           // 2 x NS u32
  static constexpr int OFF_MISC = OFF_MASK + 2 * NS * 4;          // abort flag
  static constexpr int OFF_DESC = OFF_MISC + 16;                  // Unit [2] (48 B each)
  static constexpr int OFF_ROWS = OFF_DESC + 2 * 48;              // int2 [kMaxRows]
  static constexpr int OFF_PRE = OFF_ROWS + kMaxRows * 8;         // int [kMaxRows + 1]
  static constexpr int OFF_PRC = OFF_PRE + (kMaxRows + 1) * 4;    // int [kMaxRows + 1]
  // fused step only: the norm gains (bf16 [D] each)
  static constexpr int OFF_GAM = (OFF_PRC + (kMaxRows + 1) * 4 + 15) & ~15;
  static constexpr int SMEM = OFF_GAM + 4 * D + 1024;  // + alignment
  static constexpr int CTAS_PER_SM = D <= 128 ? 2 : 1;
};
// shared memory per SM on sm_103a: 228 KB, of which 1 KB is reserved per CTA
static_assert(Cfg<64>::CTAS_PER_SM * (Cfg<64>::SMEM + 1024) <= 228 * 1024, "D=64 residency");
static_assert(Cfg<128>::CTAS_PER_SM * (Cfg<128>::SMEM + 1024) <= 228 * 1024, "D=128 residency");
static_assert(Cfg<256>::SMEM <= 227 * 1024 && Cfg<512>::SMEM <= 227 * 1024, "smem per CTA");

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
// Raises the transaction count of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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
// Bounded wait. Gives up after kSpinLimit polls (each poll may suspend the
// thread for a hardware-defined time) or as soon as the CTA aborts.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int *abort_flag) {
  for (int i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && *abort_flag) return false;
  }
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
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm,
                                            int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCThreads) : "memory");
}
// consumer_sync that also returns the OR of `v` over the consumer threads
__device__ __forceinline__ bool consumer_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kCThreads)
      : "memory");
  return r != 0;
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

// Byte offset of 16-byte chunk `chunk` (8 bf16 along D) of tile row `r` in a
// stage written by TMA with SWIZZLE_128B: 64-column chunks are separate
// [kT][128 B] blocks; inside a 1024-byte atom the 16-byte unit index is
// XORed with the row index mod 8.
__device__ __forceinline__ uint32_t swz(int r, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (kT * 128) + r * 128 +
                               (((chunk & 7) ^ (r & 7)) << 4));
}

// ------------------------------------------------------- row geometry ----
struct Problem {
  const int32_t *table, *batch_idx, *seq_lens;
  int len_bias;       // L = seq_lens[b] + len_bias (1 when seq_lens holds input_pos)
  int n_slots, max_pages, log2_ps, n_pages, window, B, Hq, Hkv, G;
  int fixed_splits;   // > 0: each row cut into at most this many parts; 0: balanced
  int max_parts;      // partial slots per (row, kv head) in the workspace
  int unit_cost;      // balanced mode: cost of starting a (row, kv head), quarter tiles
};

struct RowInfo {
  int slot, L, lo, t_first, n_tiles;
  bool clamped;   // L was cut to the table's capacity (position error)
};

// The row cache keeps {slot or -1, L}; bit 31 of L marks a clamped length.
constexpr int kClampBit = static_cast<int>(0x80000000u);

// Row b's slot, clamped length and key-tile range, read from global memory;
// errors are reported by the caller-selected thread.
__device__ __forceinline__ RowInfo row_info(const Problem &p, int b, int32_t *err,
                                            bool report) {
  RowInfo r;
  r.slot = p.batch_idx ? p.batch_idx[b] : b;
  const int raw = p.seq_lens[b];
  r.L = raw < 0x7fffffff ? raw + p.len_bias : raw;
  r.clamped = false;
  bool empty = false;
  if (r.slot < 0 || r.slot >= p.n_slots) {
    if (report && err) atomicOr(err, PKV_ERR_SLOT);
    empty = true;
  }
  const int Lmax = p.max_pages << p.log2_ps;
  if (r.L > Lmax || r.L < 0) {
    if (report && err) atomicOr(err, PKV_ERR_POS);
    r.clamped = r.L > Lmax;
    r.L = r.L < 0 ? 0 : Lmax;
  }
  if (r.slot == 0 || r.L <= 0) empty = true;
  r.lo = p.window > 0 ? max(0, r.L - p.window) : 0;
  r.t_first = r.lo / kT;
  r.n_tiles = empty ? 0 : (r.L + kT - 1) / kT - r.t_first;
  return r;
}

// Same, from the per-CTA shared-memory copy {slot, clamped L}.
__device__ __forceinline__ RowInfo row_cached(const Problem &p, int2 c) {
  RowInfo r;
  r.slot = c.x;
  r.L = c.y & ~kClampBit;
  r.lo = p.window > 0 ? max(0, r.L - p.window) : 0;
  r.t_first = r.lo / kT;
  r.n_tiles = (r.slot <= 0 || r.L <= 0) ? 0 : (r.L + kT - 1) / kT - r.t_first;
  return r;
}

__device__ __forceinline__ int fixed_parts(int n_tiles, int S) {
  if (n_tiles <= 0) return 0;
  const int ch = (n_tiles + S - 1) / S;
  return (n_tiles + ch - 1) / ch;
}

// Inputs of the fused decode step (qk_norm_rope + kv_append + attention);
// unused by the plain attention kernel.
struct StepArgs {
  const __nv_bfloat16 *k_new, *v_new;     // [B][Hkv][D], not modified
  const __nv_bfloat16 *gamma_q, *gamma_k; // [D] each, or both NULL (no norm)
  float log2_theta, eps;
  __nv_bfloat16 *k_cache, *v_cache;       // the caches the tensor maps read
  int rot_pairs;   // rotated pairs (D/2 = full RoPE; fewer: Gemma-4 proportional RoPE)
  int v_norm;      // value gets the gain-free RMSNorm (Gemma-4 v_norm)
  int k_eq_v;      // value is the raw k row (Gemma-4 K=V), not v_new
};

// Cache row of token `pos` of `slot` with kv_append's checks in its order
// (slot, position, negative page, page range); -1 and the error bit if the
// token cannot be written.
__device__ __forceinline__ long long append_row(const Problem &p, int slot, int pos,
                                                int &bits) {
  bits = 0;
  if (slot < 0 || slot >= p.n_slots) {
    bits = PKV_ERR_SLOT;
    return -1;
  }
  if (pos < 0 || (pos >> p.log2_ps) >= p.max_pages) {
    bits = PKV_ERR_POS;
    return -1;
  }
  const int page = __ldg(p.table + static_cast<size_t>(slot) * p.max_pages + (pos >> p.log2_ps));
  if (page < 0) {
    bits = PKV_ERR_PAGE_NEG;
    return -1;
  }
  if (page >= p.n_pages) {
    bits = PKV_ERR_PAGE_RANGE;
    return -1;
  }
  return (static_cast<long long>(page) << p.log2_ps) + (pos & ((1 << p.log2_ps) - 1));
}

// Norm + RoPE of the new k of (row b, kv head g) by one warp, the value
// (v_new or, with K=V, the raw k row; gain-free RMSNorm when v_norm), then
// the kv_append write of k and v at cache row `row` (>= 0). Used for rows
// that have no keys to attend to (padding rows), whose append no unit
// performs.
template <int D>
__device__ __forceinline__ void step_append_head(const Problem &p, const StepArgs &sa, int b,
                                                 int g, float fpos, long long row, int lane) {
  constexpr int PAIRS = (D / 2 + 31) / 32;
  constexpr int half = D / 2;
  const size_t src = (static_cast<size_t>(b) * p.Hkv + g) * D;
  float lo[PAIRS], hi[PAIRS];
  pkv_norm_rope_lane<PAIRS>(sa.k_new + src, sa.gamma_k, fpos, sa.log2_theta, sa.rot_pairs,
                            sa.eps, D, lane, lo, hi);
  const size_t dst = (static_cast<size_t>(g) * p.n_pages * (1 << p.log2_ps) + row) * D;
#pragma unroll
  for (int j = 0; j < PAIRS; ++j) {
    const int i = lane + 32 * j;
    if (i < half) {
      sa.k_cache[dst + i] = __float2bfloat16_rn(lo[j]);
      sa.k_cache[dst + i + half] = __float2bfloat16_rn(hi[j]);
    }
  }
  const __nv_bfloat16 *vsrc = (sa.k_eq_v ? sa.k_new : sa.v_new) + src;
  if (sa.v_norm) {
    pkv_rms_norm_lane<PAIRS>(vsrc, sa.eps, D, lane, lo, hi);
#pragma unroll
    for (int j = 0; j < PAIRS; ++j) {
      const int i = lane + 32 * j;
      if (i < half) {
        sa.v_cache[dst + i] = __float2bfloat16_rn(lo[j]);
        sa.v_cache[dst + i + half] = __float2bfloat16_rn(hi[j]);
      }
    }
  } else {
    const uint4 *vs = reinterpret_cast<const uint4 *>(vsrc);
    for (int c = lane; c < D / 8; c += 32)
      reinterpret_cast<uint4 *>(sa.v_cache + dst)[c] = __ldg(vs + c);
  }
}

// Largest b in [0, B) with scale * arr[b] <= x, for a non-decreasing arr
// with arr[0] = 0 <= x, found by the whole (converged) warp: each lane tests
// one row of every 32 and the ballots are counted. The host guarantees
// Hkv * (tiles of all rows) and the matching costs stay below 2^31.
__device__ __forceinline__ int find_row_warp(const int *arr, int B, int scale, int x, int lane) {
  int count = 0;
  for (int base = 0; base < B; base += 32) {
    const int b = base + lane;
    const unsigned le = __ballot_sync(0xffffffffu, b < B && scale * arr[b] <= x);
    count += __popc(le);
    if (le != 0xffffffffu) break;   // monotone: no later row qualifies
  }
  return count - 1;
}

// floor(x / d) for 0 <= x < n * d with a small n (a kv-head index), by ballot
// when n <= 32; the warp must be converged and the arguments uniform.
__device__ __forceinline__ int small_quotient_warp(int x, int d, int n, int lane) {
  if (n > 32) return x / d;
  return __popc(__ballot_sync(0xffffffffu, lane < n && lane * d <= x)) - 1;
}

// The shares of the balanced cost line: CTA c owns cost positions
// [bound(c), bound(c + 1)) with bound(c) = floor(c * num / den), clipped to
// the line's length. Shares are at least one tile's cost long, so every CTA
// strictly between the first and the last owner of a (row, head) owns one of
// its tiles. Equal fractional shares (num = cost, den = grid) are used when
// the line is long enough, else shares of kMinShare (num = kMinShare,
// den = 1), leaving the CTAs past the line's end idle.
struct Share {
  long long num;
  int den;
};
__device__ __forceinline__ int share_bound(const Share &s, int c, int cost) {
  const long long v = static_cast<long long>(c) * s.num / s.den;
  return v < cost ? static_cast<int>(v) : cost;
}
// CTA owning cost position x: the largest c with bound(c) <= x.
__device__ __forceinline__ int share_owner(const Share &s, int x) {
  return static_cast<int>((static_cast<long long>(x + 1) * s.den + s.num - 1) / s.num) - 1;
}

// A run of key tiles of one (row, kv head) processed by one CTA. The
// producer computes each unit once and hands it to the consumers in shared
// memory with the unit's query rows (b < 0: no more units).
struct Unit {
  int b, g, slot, ta, tb, k0, k1, part, parts;
  // fused step, unit holding the row's last tile: cache row of the appended
  // token (kv_append's address), -1 if its page entry is invalid, -2 if its
  // position is past the table (both errors are reported by the attention's
  // own checks of the same row); -1 for every other unit
  int app;
};
static_assert(sizeof(Unit) <= 48, "unit descriptor slot");

// Walks this CTA's units. Balanced mode: the (row, kv head, tile) sequence
// is flattened and laid on a cost line where each tile costs kTileCost and
// each (row, head) unit_cost more before its first tile; the line is cut into
// one share per CTA, [bound(c), bound(c + 1)), and every CTA owns the tiles
// whose cost position falls in its share, a contiguous run of the flattened
// sequence. A (row, head) that straddles CTAs is cut into parts: its first
// part is the last unit of its CTA and every later part is the first unit of
// its own CTA, so the first part's CTA finds the later parts' partials ready
// when it ends and merges them itself. Fixed mode: units are (row, part,
// head) with each row cut into at most S equal parts, dealt out in equal
// counts, and merged by the combine kernel.
struct UnitIter {
  int pos, end;     // balanced: flattened tile index; fixed: unit index
  Share sh;         // balanced: the shares of the cost line
  int hb, hg, ht;   // balanced: (row, head, tile) of pos when already known; hb < 0 if not
};

// Cost position of the first tile of (row b, head g): prc is the prefix of
// per-row head costs (kTileCost * tiles + unit_cost for rows with tiles).
__device__ __forceinline__ int head_cost_start(const Problem &p, const int *prc, int b, int g) {
  return p.Hkv * prc[b] + g * (prc[b + 1] - prc[b]) + p.unit_cost;
}

// The CTA's range: flattened indices of the first tiles whose cost positions
// are >= x0 and >= x1 (x0 <= x1), found in one warp-wide pass over the rows;
// the (row, head, tile) of the first bound is kept for the first unit.
__device__ __forceinline__ void locate_range(const Problem &p, const int *pre, const int *prc,
                                             int x0, int x1, int lane, UnitIter &it) {
  int n0 = 0, n1 = 0;   // rows whose cost start is <= x0, <= x1
  for (int base = 0; base < p.B; base += 32) {
    const int b = base + lane;
    const int v = b < p.B ? p.Hkv * prc[b] : 0x7fffffff;
    const unsigned m0 = __ballot_sync(0xffffffffu, v <= x0);
    const unsigned m1 = __ballot_sync(0xffffffffu, v <= x1);
    n0 += __popc(m0);
    n1 += __popc(m1);
    if (m1 != 0xffffffffu) break;   // monotone, and m0 is a subset of m1
  }
  const int total_cost = p.Hkv * prc[p.B];
  it.hb = -1;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int x = k ? x1 : x0;
    int flat = p.Hkv * pre[p.B];
    if (x < total_cost) {
      const int b = (k ? n1 : n0) - 1;
      const int W = prc[b + 1] - prc[b], T = pre[b + 1] - pre[b];
      const int within = x - p.Hkv * prc[b];
      const int g = small_quotient_warp(within, W, p.Hkv, lane), r = within - g * W;
      const int j = r <= p.unit_cost ? 0 : (r - p.unit_cost + kTileCost - 1) / kTileCost;
      flat = p.Hkv * pre[b] + g * T + j;
      if (k == 0 && j < T) {
        it.hb = b;
        it.hg = g;
        it.ht = j;
      }
    }
    if (k) it.end = flat; else it.pos = flat;
  }
}

// Called by the converged producer warp with uniform arguments.
__device__ __forceinline__ bool next_unit(const Problem &p, const int2 *rows, const int *pre,
                                          const int *prc, UnitIter &it, Unit &w, int lane) {
  if (it.pos >= it.end) return false;
  if (p.fixed_splits == 0) {
    int b, t0;
    if (it.hb >= 0) {   // located with the CTA's range
      b = it.hb;
      w.g = it.hg;
      t0 = it.ht;
      it.hb = -1;
    } else {
      b = find_row_warp(pre, p.B, p.Hkv, it.pos, lane);
      const int within = it.pos - p.Hkv * pre[b];
      const int T = pre[b + 1] - pre[b];
      w.g = small_quotient_warp(within, T, p.Hkv, lane);
      t0 = within - w.g * T;
    }
    const RowInfo r = row_cached(p, rows[b]);
    const int tiles = pre[b + 1] - pre[b];
    const int n = min(tiles - t0, it.end - it.pos);
    const int c0 = head_cost_start(p, prc, b, w.g);
    const int first_cta = share_owner(it.sh, c0);
    w.b = b;
    w.slot = r.slot;
    w.ta = r.t_first + t0;
    w.tb = w.ta + n;
    w.parts = share_owner(it.sh, c0 + kTileCost * (tiles - 1)) - first_cta + 1;
    w.part = static_cast<int>(blockIdx.x) - first_cta;   // this CTA owns the unit's tiles
    w.k0 = max(r.lo, w.ta * kT);
    w.k1 = min(r.L, w.tb * kT);
    it.pos += n;
  } else {
    const int rc = it.pos / p.Hkv;
    w.g = it.pos - rc * p.Hkv;
    const int b = find_row_warp(pre, p.B, 1, rc, lane);
    const RowInfo r = row_cached(p, rows[b]);
    const int ch = (r.n_tiles + p.fixed_splits - 1) / p.fixed_splits;
    w.b = b;
    w.slot = r.slot;
    w.part = rc - pre[b];
    w.parts = pre[b + 1] - pre[b];
    w.ta = r.t_first + w.part * ch;
    w.tb = min(r.t_first + r.n_tiles, w.ta + ch);
    w.k0 = max(r.lo, w.ta * kT);
    w.k1 = min(r.L, w.tb * kT);
    it.pos += 1;
  }
  return true;
}

// Partials of cut (row, head)s carry their own validity. A part stores each
// fp32 word of its partial (normalised o, lse) as the bitwise complement of
// the float's bits, so a stored word is never 0 (its float would have the
// bits 0xffffffff, a NaN that arithmetic never yields; such a NaN is stored
// as the canonical one), and the workspace holds 0 wherever nothing of this
// call has been written yet. The reader polls the words themselves with
// relaxed gpu-scope loads until none is 0, decodes them and writes 0 back,
// so a completed call leaves the partial area zero for the next one. No
// flag, fence or release is needed: each word is its own message.
constexpr int kPollLimit = 1 << 21;
__device__ __forceinline__ uint32_t part_enc(float v) {
  const uint32_t u = __float_as_uint(v);
  return ~(u == 0xffffffffu ? 0x7fffffffu : u);
}
__device__ __forceinline__ float part_dec(uint32_t w) { return __uint_as_float(~w); }
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const float *a) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_gpu(float *a, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
// The words of one (row, kv head)'s partial records that a consumer thread
// owns: for part j, o[k] of m-tile mt (query heads h0 / h1, columns
// dbase + 16 mt (+ 8)) and the lse of h0 / h1, in the thread's MMA fragment
// order.
struct PartView {
  float *o, *lse;      // the record of part 0
  int G, D, h0, h1, dbase;
  bool hv0, hv1;
  __device__ __forceinline__ bool valid(int k) const { return (k & 1) ? hv1 : hv0; }
  __device__ __forceinline__ float *ow(int j, int mt, int k) const {
    return o + static_cast<size_t>(j) * G * D + ((k & 1) ? h1 : h0) * D + dbase + 16 * mt +
           ((k & 2) ? 8 : 0);
  }
  __device__ __forceinline__ float *lw(int j, int k) const {
    return lse + static_cast<size_t>(j) * G + (k ? h1 : h0);
  }
};
// Loads parts j0 .. j0 + NB - 1; absent parts and heads get the encoding of
// (o = 0, lse = -inf), which merges as nothing and is never waited on.
template <int NB, int MT>
__device__ __forceinline__ void part_load(const PartView &v, int j0, int parts,
                                          uint32_t (&w)[NB][MT][4], uint32_t (&l)[NB][2]) {
#pragma unroll
  for (int jj = 0; jj < NB; ++jj) {
    const bool jv = j0 + jj < parts;
#pragma unroll
    for (int k = 0; k < 2; ++k)
      l[jj][k] = jv && v.valid(k) ? ld_relaxed_gpu(v.lw(j0 + jj, k)) : part_enc(-INFINITY);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        w[jj][mt][k] = jv && v.valid(k) ? ld_relaxed_gpu(v.ow(j0 + jj, mt, k)) : part_enc(0.f);
  }
}
// Waits until no loaded word is 0 (the part has not written it yet),
// re-loading only those; false if it gives up (kPollLimit polls, or the CTA
// aborts).
template <int NB, int MT>
__device__ __forceinline__ bool part_wait(const PartView &v, int j0, uint32_t (&w)[NB][MT][4],
                                          uint32_t (&l)[NB][2], volatile int *abort_flag) {
  for (int i = 0;; ++i) {
    bool ready = true;
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
      ready = ready && l[jj][0] != 0u && l[jj][1] != 0u;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k) ready = ready && w[jj][mt][k] != 0u;
    }
    if (ready) return true;
    if (i >= kPollLimit || *abort_flag) return false;
    __nanosleep(64);
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (l[jj][k] == 0u) l[jj][k] = ld_relaxed_gpu(v.lw(j0 + jj, k));
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (w[jj][mt][k] == 0u) w[jj][mt][k] = ld_relaxed_gpu(v.ow(j0 + jj, mt, k));
    }
  }
}
// Clears part j's o words of this thread (each has this one reader).
template <int MT>
__device__ __forceinline__ void part_clear(const PartView &v, int j) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (v.valid(k)) st_relaxed_gpu(v.ow(j, mt, k), 0u);
}

// ------------------------------------------------------------- kernel ----
template <int D, bool STEP>
__global__ void __launch_bounds__(kThreads, Cfg<D>::CTAS_PER_SM)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmK3,
                       const __grid_constant__ CUtensorMap tmV3,
                       const __nv_bfloat16 *__restrict__ q, const Problem p,
                       float scale_log2, float *__restrict__ o_part,
                       float *__restrict__ lse_part, int *__restrict__ parts_out,
                       __nv_bfloat16 *__restrict__ out,
                       int32_t *__restrict__ err, const StepArgs sa) {
  using Cf = Cfg<D>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_u32(sm), sV = sK + Cf::OFF_V, sQ = sK + Cf::OFF_Q;
  const uint32_t sP = sK + Cf::OFF_P;
  float *red_max = reinterpret_cast<float *>(sm + Cf::OFF_RED);
  float *red_sum = red_max + kCWarps * kMaxG;
  const uint32_t bar0 = sK + Cf::OFF_BAR;
  // barrier layout: fullK[NS] emptyK[NS] fullV[NS] emptyV[NS] fullQ[2] emptyQ[2]
  const uint32_t fullK = bar0, emptyK = bar0 + 8 * Cf::NS, fullV = bar0 + 16 * Cf::NS,
                 emptyV = bar0 + 24 * Cf::NS, fullQ = bar0 + 32 * Cf::NS,
                 emptyQ = fullQ + 16;
  uint32_t *kmask = reinterpret_cast<uint32_t *>(sm + Cf::OFF_MASK);
  uint32_t *vmask = kmask + Cf::NS;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + Cf::OFF_MISC);
  int2 *rows = reinterpret_cast<int2 *>(sm + Cf::OFF_ROWS);
  int *pre = reinterpret_cast<int *>(sm + Cf::OFF_PRE);
  int *prc = reinterpret_cast<int *>(sm + Cf::OFF_PRC);
  Unit *udesc = reinterpret_cast<Unit *>(sm + Cf::OFF_DESC);

  // ---- set-up: barriers, row cache, per-row tile or part prefix sums ----
  if (tid == 0) {
    for (int i = 0; i < Cf::NS; ++i) {
      mbar_init(fullK + 8 * i, 1);
      mbar_init(emptyK + 8 * i, 1);
      mbar_init(fullV + 8 * i, 1);
      mbar_init(emptyV + 8 * i, kCWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(fullQ + 8 * i, 1);
      mbar_init(emptyQ + 8 * i, kCWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
  }
  // Warm L2 with the row metadata and the page table while the previous
  // kernel finishes (prefetches only pull lines into L2, the point of
  // coherence).
  //
  // The set-up below (row cache, prefix sums, the producer's share of the
  // cost line and its first unit's page entries; in the fused step the
  // consumers' loads of the norm gains) runs before the grid dependency wait
  // and reads only seq_lens, batch_idx, the page table, the gains and shared
  // memory. That is safe because the kernels that may still be
  // running when this grid starts never write those: a kernel without
  // programmatic launch completes before its successor starts; the kernels
  // of this library release their dependents only after their own wait
  // returned, except the combine, which releases them at once and writes
  // only its output (so at most the combine and the attention kernel before
  // it can still be running). A kernel that writes them and releases its
  // dependents early must not precede this one (the header states this).
  // Global writes, the query and the cache come after the wait.
  {
    const int gt = blockIdx.x * kThreads + tid, gs = gridDim.x * kThreads;
    for (int i = gt * 32; i < p.B; i += gs * 32) {
      prefetch_l2(p.seq_lens + i);
      if (p.batch_idx) prefetch_l2(p.batch_idx + i);
    }
    const long long tbl = 1LL * p.n_slots * p.max_pages;
    const long long tlim = tbl < (1LL << 20) ? tbl : (1LL << 20);
    for (long long i = 32LL * gt; i < tlim; i += 32LL * gs) prefetch_l2(p.table + i);
  }
  for (int b = tid; b < p.B; b += kThreads) {
    const RowInfo r = row_info(p, b, err, blockIdx.x == 0);
    rows[b] = make_int2(r.n_tiles > 0 ? r.slot : -1, r.L | (r.clamped ? kClampBit : 0));
    pre[b + 1] = p.fixed_splits > 0 ? fixed_parts(r.n_tiles, p.fixed_splits) : r.n_tiles;
    prc[b + 1] = r.n_tiles > 0 ? kTileCost * r.n_tiles + p.unit_cost : 0;
  }
  __syncthreads();
  if (warp < 2) {  // inclusive scans of pre[1..B] (warp 0) and prc[1..B] (warp 1)
    int *arr = warp == 0 ? pre : prc;
    int carry = 0;
#pragma unroll 1
    for (int base = 0; base < p.B; base += 32) {
      const int i = base + lane;
      int v = i < p.B ? arr[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (i < p.B) arr[i + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) arr[0] = 0;
    __syncwarp();
  }
  __syncthreads();
  UnitIter it0, itp;
  {
    const int total = p.Hkv * pre[p.B];
    if (p.fixed_splits == 0) {
      const int grid = static_cast<int>(gridDim.x);
      const int cost = p.Hkv * prc[p.B];
      // at least one tile per share, so that every CTA between the first and
      // the last owner of a (row, head) owns one of its tiles
      if (cost >= kMinShare * grid) {
        it0.sh.num = cost;
        it0.sh.den = grid;
      } else {
        it0.sh.num = kMinShare;
        it0.sh.den = 1;
      }
      it0.pos = it0.end = 0;   // the producer warp finds its range (locate_range)
      it0.hb = -1;
    } else {
      it0.sh.num = 1;
      it0.sh.den = 1;
      it0.hb = -1;
      it0.pos = static_cast<int>(1LL * total * blockIdx.x / gridDim.x);
      it0.end = static_cast<int>(1LL * total * (blockIdx.x + 1) / gridDim.x);
    }
    itp = it0;   // the producer's share of the cost line (shared memory only)
    if (warp == kCWarps && p.fixed_splits == 0) {
      const int cost = p.Hkv * prc[p.B];
      const int c = static_cast<int>(blockIdx.x);
      locate_range(p, pre, prc, share_bound(itp.sh, c, cost), share_bound(itp.sh, c + 1, cost),
                   lane, itp);
    }
    // fused step, consumers: the norm gains are loaded before the dependency
    // wait (like the row metadata, no kernel that can still run writes them)
    // and stored to shared memory after it and after the next grid's release
    // (read after the first unit's barrier)
    constexpr int GPT = (D + kCThreads - 1) / kCThreads;   // gain elements per thread
    __nv_bfloat16 gqv[GPT], gkv[GPT];
    if constexpr (STEP) {
      if (warp < kCWarps && sa.gamma_q) {
#pragma unroll
        for (int e = 0; e < GPT; ++e) {
          const int i = tid + e * kCThreads;
          if (i < D) {
            gqv[e] = sa.gamma_q[i];
            gkv[e] = sa.gamma_k[i];
          }
        }
      }
    }
    // the consumer warps wait here; the producer warp also looks up its first
    // unit and that unit's pages first, and waits just before its first copy
    if (warp < kCWarps) {
      pkv_wait_prior_grid();
      pkv_allow_next_grid();
    }
    if constexpr (STEP) {
      if (warp < kCWarps && sa.gamma_q) {
        __nv_bfloat16 *gs = reinterpret_cast<__nv_bfloat16 *>(sm + Cf::OFF_GAM);
#pragma unroll
        for (int e = 0; e < GPT; ++e) {
          const int i = tid + e * kCThreads;
          if (i < D) {
            gs[i] = gqv[e];
            gs[D + i] = gkv[e];
          }
        }
      }
    }
    if (parts_out && warp < kCWarps) {  // fixed mode: parts per (row, kv head) for the combine
      for (int rh = blockIdx.x + gridDim.x * tid; rh < p.B * p.Hkv; rh += gridDim.x * kCThreads) {
        const int b = rh / p.Hkv;
        parts_out[rh] = pre[b + 1] - pre[b];
      }
    }
  }

  if constexpr (STEP) {
  }

  // rows with no key: zero output (rows spread over the CTAs); in the fused
  // step their new token is still appended as kv_append would (padding rows
  // write into the reserved page of slot 0)
  if (warp < kCWarps) {
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
      if (pre[b + 1] != pre[b]) continue;
      __nv_bfloat16 *o = out + static_cast<size_t>(b) * p.Hq * D;
      for (int i = tid; i < p.Hq * D; i += kCThreads) o[i] = __float2bfloat16_rn(0.f);
      if constexpr (STEP) {
        const int slot = p.batch_idx ? __ldg(p.batch_idx + b) : b;
        const int pos = __ldg(p.seq_lens + b);
        int bits;
        const long long row = append_row(p, slot, pos, bits);
        if (bits) {
          if (tid == 0 && err) atomicOr(err, bits);
        } else {
          for (int g = warp; g < p.Hkv; g += kCWarps)
            step_append_head<D>(p, sa, b, g, static_cast<float>(pos), row, lane);
        }
      }
    }
  }

  const int ps = 1 << p.log2_ps;
  const int box_rows = ps < kT ? ps : kT;
  const int boxes = kT / box_rows;
  const uint32_t all_boxes = (1u << boxes) - 1u;

  if (warp == kCWarps) {
    // ======================== producer (one warp) ========================
    // Lane j looks up box j of a unit (a page segment of one tile); the
    // lookups for the next unit are issued before the current unit's copies
    // so that their latency hides behind the ring that is already in flight.
    // box_page issues the table load only; box_row checks the entry when
    // it is used, so a look-ahead load never stalls the warp.
    auto box_page = [&](const Unit &u, int j) -> int {
      const int n_boxes = (u.tb - u.ta) * boxes;
      if (j >= n_boxes) return -1;
      const int t = u.ta + j / boxes, i = j % boxes;
      const int key = t * kT + i * box_rows;
      if (key + box_rows <= u.k0 || key >= u.k1) return -1;
      const int32_t *trow = p.table + static_cast<size_t>(u.slot) * p.max_pages;
      return __ldg(trow + (key >> p.log2_ps));
    };
    auto box_row = [&](const Unit &u, int j, int page) -> int {
      const int n_boxes = (u.tb - u.ta) * boxes;
      if (j >= n_boxes) return -1;
      const int t = u.ta + j / boxes, i = j % boxes;
      const int key = t * kT + i * box_rows;
      if (key + box_rows <= u.k0 || key >= u.k1) return -1;
      if (page < 0) {
        if (err) atomicOr(err, PKV_ERR_PAGE_NEG);
        return -1;
      }
      if (page >= p.n_pages) {
        if (err) atomicOr(err, PKV_ERR_PAGE_RANGE);
        return -1;
      }
      return ((u.g * p.n_pages + page) << p.log2_ps) + (key & (ps - 1));
    };
    UnitIter it = itp;
    Unit w, wn;
    int it_k = 0, it_v = 0, it_q = 0;
    bool ok = true;
    bool have = next_unit(p, rows, pre, prc, it, w, lane);
    int page_first = have ? box_page(w, lane) : -1;
    pkv_wait_prior_grid();
    while (ok && have) {
      bool have_next = false, looked_ahead = false;
      int page_next = -1;
      const int n_boxes = (w.tb - w.ta) * boxes;
      // query rows of the GQA group, one bulk copy per head into padded rows
      {
        const int qs = it_q & 1;
        // fused step: the unit that holds the row's last tile also gets the
        // raw k and v rows of the token it appends
        const int c_b = rows[w.b].y;
        const bool kv_rows = STEP && w.k1 == (c_b & ~kClampBit);
        if (lane == 0) {
          ok = mbar_wait(emptyQ + 8 * qs, ((it_q >> 1) & 1) ^ 1, abort_flag);
          if (ok) {
            w.app = -1;
            if (kv_rows) {
              if (c_b < 0) {
                w.app = -2;
              } else {
                const int pos = (c_b & ~kClampBit) - 1;
                const int page = __ldg(p.table + static_cast<size_t>(w.slot) * p.max_pages +
                                       (pos >> p.log2_ps));
                if (page >= 0 && page < p.n_pages)
                  w.app = (page << p.log2_ps) + (pos & (ps - 1));
              }
            }
            udesc[qs] = w;   // published to the consumers by the arrive below
            mbar_expect_tx(fullQ + 8 * qs,
                           static_cast<uint32_t>((p.G + (kv_rows ? 2 : 0)) * D * 2));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t qdst = sQ + qs * Cf::Q_STAGE;
        if (lane < p.G)
          bulk_load(qdst + lane * Cf::Q_ROW,
                    q + ((static_cast<size_t>(w.b) * p.Hq + static_cast<size_t>(w.g) * p.G +
                          lane) * D),
                    static_cast<uint32_t>(D * 2), fullQ + 8 * qs);
        if constexpr (STEP) {
          if (kv_rows && (lane == 30 || lane == 31)) {
            const size_t src = (static_cast<size_t>(w.b) * p.Hkv + w.g) * D;
            bulk_load(qdst + Cf::Q_BYTES + (lane - 30) * D * 2,
                      lane == 30 || sa.k_eq_v ? sa.k_new + src : sa.v_new + src,
                      static_cast<uint32_t>(D * 2), fullQ + 8 * qs);
          }
        }
        ++it_q;
      }
      for (int base = 0; base < n_boxes && ok; base += 32) {
        const int row = box_row(w, base + lane, base == 0 ? page_first : box_page(w, base + lane));
        const int tiles_here = min(32, n_boxes - base) / boxes;
        for (int tt = 0; tt < tiles_here && ok; ++tt) {
          uint32_t mask = 0;
          int r0 = -1, r1 = -1, r2 = -1, r3 = -1, r4 = -1, r5 = -1, r6 = -1, r7 = -1;
#pragma unroll
          for (int i = 0; i < kT / 8; ++i) {
            const int v = __shfl_sync(0xffffffffu, row, (tt * boxes + (i < boxes ? i : 0)) & 31);
            const int rv = i < boxes ? v : -1;
            if (rv >= 0) mask |= 1u << i;
            switch (i) {
              case 0: r0 = rv; break; case 1: r1 = rv; break; case 2: r2 = rv; break;
              case 3: r3 = rv; break; case 4: r4 = rv; break; case 5: r5 = rv; break;
              case 6: r6 = rv; break; default: r7 = rv; break;
            }
          }
          if (lane == 0) {
            const uint32_t bytes =
                static_cast<uint32_t>(__popc(mask)) * Cf::CHUNKS * box_rows * 128;
            // One box per tile (pages of >= 64 keys): a tile whose keys end
            // (or start) inside it is loaded as the 64 rows ending at its
            // last key (starting at its first key); rows outside the page are
            // zero-filled by the copy and never read from memory. Shared
            // memory row r then holds key t*64 + r + off.
            int off = 0;
            if (boxes == 1 && Cf::NS > 1) {   // (a one-stage ring gains nothing: D=512)
              const int t = w.ta + base + tt;
              const int lo_r = max(w.k0 - t * kT, 0), hi_r = min(w.k1 - t * kT, kT);
              if (hi_r < kT && (lo_r == 0 || hi_r <= kT - lo_r)) off = hi_r - kT;
              else if (lo_r > 0) off = lo_r;
            }
            const uint32_t mword = mask | (static_cast<uint32_t>(off & 0xff) << 8);
            for (int kv = 0; kv < 2 && ok; ++kv) {
              const int itx = kv ? it_v : it_k;
              const int st = itx % Cf::NS;
              const uint32_t par = ((itx / Cf::NS) & 1) ^ 1;
              if (!mbar_wait((kv ? emptyV : emptyK) + 8 * st, par, abort_flag)) {
                ok = false;
                break;
              }
              (kv ? vmask : kmask)[st] = mword;
              const uint32_t full = (kv ? fullV : fullK) + 8 * st;
              mbar_expect_tx(full, bytes);
              const uint32_t dst0 = (kv ? sV : sK) + st * Cf::STAGE_BYTES;
              const CUtensorMap *tm = kv ? &tmV : &tmK;
              if (boxes == 1 && off != 0) {   // 3-D map {column, row in page, page}
                const CUtensorMap *tm3 = kv ? &tmV3 : &tmK3;
                if (r0 >= 0) {
#pragma unroll
                  for (int cc = 0; cc < Cf::CHUNKS; ++cc)
                    tma_load_3d(dst0 + cc * Cf::CHUNK_BYTES, tm3, cc * 64,
                                (r0 & (ps - 1)) + off, r0 >> p.log2_ps, full);
                }
              } else {            // 2-D map {column, cache row}
#pragma unroll
                for (int i = 0; i < kT / 8; ++i) {
                  const int rv = i == 0 ? r0 : i == 1 ? r1 : i == 2 ? r2 : i == 3 ? r3
                               : i == 4 ? r4 : i == 5 ? r5 : i == 6 ? r6 : r7;
                  if (rv < 0) continue;
#pragma unroll
                  for (int cc = 0; cc < Cf::CHUNKS; ++cc)
                    tma_load_2d(dst0 + cc * Cf::CHUNK_BYTES + i * box_rows * 128, tm, cc * 64,
                                rv, full);
                }
              }
              if (kv) ++it_v; else ++it_k;
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!looked_ahead) {  // next unit's table lookups, once this one is moving
            looked_ahead = true;
            have_next = next_unit(p, rows, pre, prc, it, wn, lane);
            page_next = have_next ? box_page(wn, lane) : -1;
          }
        }
      }
      if (!looked_ahead) {
        have_next = next_unit(p, rows, pre, prc, it, wn, lane);
        page_next = have_next ? box_page(wn, lane) : -1;
      }
      w = wn;
      page_first = page_next;
      have = have_next;
    }
    if (lane != 0) return;
    if (ok) {   // end-of-work descriptor in the next Q stage
      const int qs = it_q & 1;
      ok = mbar_wait(emptyQ + 8 * qs, ((it_q >> 1) & 1) ^ 1, abort_flag);
      if (ok) {
        udesc[qs].b = -1;
        mbar_arrive(fullQ + 8 * qs);
        ++it_q;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      if (err) atomicOr(err, PKV_ERR_TIMEOUT);
    }
    // drain: the last phase armed on every stage must land before exit
    volatile int no_abort = 0;
    for (int s = 0; s < Cf::NS; ++s) {
      if (it_k > s) {
        const int last = s + ((it_k - 1 - s) / Cf::NS) * Cf::NS;
        (void)mbar_wait(fullK + 8 * s, (last / Cf::NS) & 1, &no_abort);
      }
      if (it_v > s) {
        const int last = s + ((it_v - 1 - s) / Cf::NS) * Cf::NS;
        (void)mbar_wait(fullV + 8 * s, (last / Cf::NS) & 1, &no_abort);
      }
    }
    for (int s = 0; s < 2; ++s) {
      if (it_q > s) {
        const int last = s + ((it_q - 1 - s) / 2) * 2;
        (void)mbar_wait(fullQ + 8 * s, (last / 2) & 1, &no_abort);
      }
    }
    return;
  }

  // ============================== consumers ==============================
  const int gid = lane >> 2, tig = lane & 3;
  const int h0 = 2 * tig, h1 = 2 * tig + 1;
  const bool hv0 = h0 < p.G, hv1 = h1 < p.G;
  constexpr int KS = D / 16;
  constexpr int MT = D / 64;  // 16-row m-tiles of this warp's D/4 slice
  int it = 0, it_q = 0;
  bool failed = false;
  // fused step: this lane's rotation factors and the row they belong to
  constexpr int PAIRS = (D / 2 + 31) / 32;
  float cf[PAIRS], sf[PAIRS];
  int fac_b = -1;

  while (true) {
    uint32_t qb[KS][2];
    const int qs = it_q & 1;
    const uint8_t *qstage = sm + Cf::OFF_Q + qs * Cf::Q_STAGE;
    int patch = -1;   // fused step: row of the appended token in the unit's last tile
    // the unit comes from the producer with its query rows; all consumer
    // threads leave the loop together (end of work, or a wait that gave up)
    const bool q_ok = mbar_wait(fullQ + 8 * qs, (it_q >> 1) & 1, abort_flag);
    Unit w;
    w.b = -1;
    if (q_ok) w = udesc[qs];
    if (consumer_sync_or(!q_ok || w.b < 0)) {
      if (!q_ok) {
        failed = true;
        *abort_flag = 1;
      }
      break;
    }
    {
      if constexpr (STEP) {
        // Rotate the raw query rows in place. Lane l of every warp rotates
        // the pairs (l + 32 j, l + 32 j + D/2) of its rows, so each lane needs
        // only its own pairs' factors: computed in registers, once per row
        // (consecutive units of one row reuse them). The unit that holds the
        // row's last tile also rotates the new k in place, writes k and v to
        // their cache row (the kv_append of the chain) and later patches both
        // into that tile, whose TMA copy may predate the write.
        const int c_b = rows[w.b].y;
        const int L_b = c_b & ~kClampBit;
        const int app_b = w.app;
        const int pos_b = c_b < 0 ? __ldg(p.seq_lens + w.b) : L_b - 1;
        if (w.b != fac_b) {
          const float fpos = static_cast<float>(pos_b);
#pragma unroll
          for (int j = 0; j < PAIRS; ++j) {
            const int i = lane + 32 * j;
            if (i < D / 2) pkv_rope_factor(i, D, fpos, sa.log2_theta, sa.rot_pairs, cf[j], sf[j]);
          }
          fac_b = w.b;
        }
        const __nv_bfloat16 *gq =
            sa.gamma_q ? reinterpret_cast<const __nv_bfloat16 *>(sm + Cf::OFF_GAM) : nullptr;
        auto rotate_row = [&](__nv_bfloat16 *x, const __nv_bfloat16 *g, float (&lo)[PAIRS],
                              float (&hi)[PAIRS]) {
          pkv_norm_rope_core<PAIRS>(
              x, g, sa.eps, D, lane,
              [&](int j, int, float &cs, float &sn) {
                cs = cf[j];
                sn = sf[j];
              },
              lo, hi);
#pragma unroll
          for (int j = 0; j < PAIRS; ++j) {
            const int i = lane + 32 * j;
            if (i < D / 2) {
              x[i] = __float2bfloat16_rn(lo[j]);
              x[i + D / 2] = __float2bfloat16_rn(hi[j]);
            }
          }
        };
        for (int h = warp; h < p.G; h += kCWarps) {
          float lo[PAIRS], hi[PAIRS];
          rotate_row(reinterpret_cast<__nv_bfloat16 *>(sm + Cf::OFF_Q + qs * Cf::Q_STAGE +
                                                       h * Cf::Q_ROW),
                     gq, lo, hi);
        }
        const bool append = w.k1 == L_b && app_b >= 0;
        if (append && warp == p.G % kCWarps) {
          __nv_bfloat16 *kx =
              reinterpret_cast<__nv_bfloat16 *>(sm + Cf::OFF_Q + qs * Cf::Q_STAGE + Cf::Q_BYTES);
          float lo[PAIRS], hi[PAIRS];
          rotate_row(kx, gq ? gq + D : nullptr, lo, hi);
          if (sa.v_norm) {   // the value row, in place: gain-free RMSNorm
            __nv_bfloat16 *vx = kx + D;
            pkv_rms_norm_lane<PAIRS>(vx, sa.eps, D, lane, lo, hi);
#pragma unroll
            for (int j = 0; j < PAIRS; ++j) {
              const int i = lane + 32 * j;
              if (i < D / 2) {
                vx[i] = __float2bfloat16_rn(lo[j]);
                vx[i + D / 2] = __float2bfloat16_rn(hi[j]);
              }
            }
          }
          __syncwarp();
          const size_t dst = (static_cast<size_t>(w.g) * p.n_pages * (1 << p.log2_ps) +
                              static_cast<size_t>(app_b)) * D;
          const uint4 *ks = reinterpret_cast<const uint4 *>(kx);
          const uint4 *vs = reinterpret_cast<const uint4 *>(kx + D);
          for (int c = lane; c < D / 8; c += 32) {
            reinterpret_cast<uint4 *>(sa.k_cache + dst)[c] = ks[c];
            reinterpret_cast<uint4 *>(sa.v_cache + dst)[c] = vs[c];
          }
        }
        fence_proxy_async();
        consumer_sync();
        if (append) patch = pos_b & (kT - 1);
      }
      const bool hv = gid < p.G;
      const uint32_t *qrow =
          reinterpret_cast<const uint32_t *>(qstage + (hv ? gid : 0) * Cf::Q_ROW);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[ks][0] = hv ? qrow[(16 * ks + 2 * tig) >> 1] : 0u;
        qb[ks][1] = hv ? qrow[(16 * ks + 8 + 2 * tig) >> 1] : 0u;
      }
      // a fused-step unit that appends the row's new token keeps the stage
      // (its k / v rows) until the unit ends; every other unit frees it now
      if (!STEP || patch < 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(emptyQ + 8 * qs);
      }
      ++it_q;
    }
    float o[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;

    // The first part of a (row, head) cut across CTAs (balanced mode) is its
    // CTA's last unit and merges the later parts at its end. The first PF
    // later parts are loaded when the unit's last tile starts, so that
    // partials already written arrive with that tile; the rest follow at the
    // end, JB per round trip to L2.
    constexpr int JB = D <= 128 ? 4 : D == 256 ? 2 : 1;
    constexpr int PF = 1;
    const bool merge = p.fixed_splits == 0 && w.parts > 1 && w.part == 0;
    PartView pv;
    {
      const size_t rec = (static_cast<size_t>(w.b) * p.Hkv + w.g) * p.max_parts;
      pv.o = o_part + rec * p.G * D;
      pv.lse = lse_part + rec * p.G;
      pv.G = p.G;
      pv.D = D;
      pv.h0 = h0;
      pv.h1 = h1;
      pv.hv0 = hv0;
      pv.hv1 = hv1;
      pv.dbase = warp * (D / 4) + gid;
    }
    uint32_t wp[PF][MT][4], lp[PF][2];   // words of parts 1 .. PF

    for (int t = w.ta; t < w.tb; ++t, ++it) {
      if (merge && t == w.tb - 1) part_load<PF, MT>(pv, 1, w.parts, wp, lp);
      const int st = it % Cf::NS;
      const uint32_t par = (it / Cf::NS) & 1;
      if (!mbar_wait(fullK + 8 * st, par, abort_flag)) {
        failed = true;
        *abort_flag = 1;
      }
      const uint32_t km = kmask[st];
      const int off = static_cast<int8_t>((km >> 8) & 0xffu);   // smem row r holds key t*kT + r + off
      const int tlo = max(w.k0, t * kT), thi = min(w.k1, t * kT + kT);
      const uint32_t kbase = sK + st * Cf::STAGE_BYTES;
      const bool patch_here = STEP && patch >= 0 && t == w.tb - 1;
      const int prow = patch - off;   // shared-memory row of the appended token
      if (patch_here && warp == (prow >> 4)) {  // this warp's 16 keys hold the new token
        const uint4 *src = reinterpret_cast<const uint4 *>(qstage + Cf::Q_BYTES);
        for (int c = lane; c < D / 8; c += 32)
          *reinterpret_cast<uint4 *>(sm + st * Cf::STAGE_BYTES + swz(prow, c)) = src[c];
        fence_proxy_async();
        __syncwarp();
      }

      // ---- S^T[16 keys x 8 heads], keys 16*warp .. +15 of the tile ----
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
      const int key_lo = t * kT + kr_lo + off, key_hi = t * kT + kr_hi + off;
      const bool v_lo = key_lo >= tlo && key_lo < thi && ((km >> (kr_lo / box_rows)) & 1u);
      const bool v_hi = key_hi >= tlo && key_hi < thi && ((km >> (kr_hi / box_rows)) & 1u);
      const float s00 = (v_lo && hv0) ? sacc[0] * scale_log2 : -INFINITY;
      const float s01 = (v_lo && hv1) ? sacc[1] * scale_log2 : -INFINITY;
      const float s10 = (v_hi && hv0) ? sacc[2] * scale_log2 : -INFINITY;
      const float s11 = (v_hi && hv1) ? sacc[3] * scale_log2 : -INFINITY;
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
      consumer_sync();  // (1) K stage consumed; maxima visible
      if (tid == 0) mbar_arrive(emptyK + 8 * st);
      float mt0 = red_max[h0], mt1 = red_max[h1];
#pragma unroll
      for (int ww = 1; ww < kCWarps; ++ww) {
        mt0 = fmaxf(mt0, red_max[ww * kMaxG + h0]);
        mt1 = fmaxf(mt1, red_max[ww * kMaxG + h1]);
      }
      const float mn0 = fmaxf(m_run0, mt0), mn1 = fmaxf(m_run1, mt1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float p00 = exp2f(s00 - mu0), p01 = exp2f(s01 - mu1);
      const float p10 = exp2f(s10 - mu0), p11 = exp2f(s11 - mu1);
      {
        uint32_t *pt = reinterpret_cast<uint32_t *>(sm + Cf::OFF_P);
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
      // ---- V tile: wait, then clear the rows of keys outside [k0, k1) ----
      if (!mbar_wait(fullV + 8 * st, par, abort_flag)) {
        failed = true;
        *abort_flag = 1;
      }
      const uint32_t vm = vmask[st];   // same row offset as the K tile
      const uint32_t vbase = sV + st * Cf::STAGE_BYTES;
      const bool full_tile = off == 0 && t * kT >= w.k0 && t * kT + kT <= w.k1 &&
                             (vm & 0xffu) == all_boxes;
      if (!full_tile) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int i = tid; i < kT * (D / 8); i += kCThreads) {
          const int r = i / (D / 8), c = i % (D / 8);
          const int key = t * kT + r + off;
          const bool valid = key >= tlo && key < thi && ((vm >> (r / box_rows)) & 1u);
          if (!valid)
            *reinterpret_cast<uint4 *>(sm + Cf::OFF_V + st * Cf::STAGE_BYTES +
                                       (c >> 3) * (kT * 128) + r * 128 + (c & 7) * 16) = z;
        }
        fence_proxy_async();
      }
      if (patch_here && tid < D / 8) {
        const uint4 *src = reinterpret_cast<const uint4 *>(qstage + Cf::Q_BYTES + D * 2);
        *reinterpret_cast<uint4 *>(sm + Cf::OFF_V + st * Cf::STAGE_BYTES + swz(prow, tid)) =
            src[tid];
        fence_proxy_async();
      }
      consumer_sync();  // (2) P, sums and V visible
      float ts0 = 0.f, ts1 = 0.f;
#pragma unroll
      for (int ww = 0; ww < kCWarps; ++ww) {
        ts0 += red_sum[ww * kMaxG + h0];
        ts1 += red_sum[ww * kMaxG + h1];
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
      __syncwarp();
      if (lane == 0) mbar_arrive(emptyV + 8 * st);
    }
    if (STEP && patch >= 0) {   // the unit's Q stage (and its k / v rows) is free
      __syncwarp();
      if (lane == 0) mbar_arrive(emptyQ + 8 * qs);
    }

    if (failed) continue;
    // ---- epilogue ----
    // A (row, head) done inside one CTA writes its output directly. A later
    // part of a cut one (every part, in the fixed mode) writes its partial:
    // o / l and lse = m + log2(l) per head, encoded, in the (row, kv head)'s
    // record for that part, and goes on at once. The first part of a cut one
    // (balanced mode) merges the later parts' partials into its own running
    // state and writes the output.
    const size_t head0 = static_cast<size_t>(w.b) * p.Hq + static_cast<size_t>(w.g) * p.G;
    if (w.parts > 1 && !merge) {
      const float il0 = l_run0 > 0.f ? 1.f / l_run0 : 0.f;
      const float il1 = l_run1 > 0.f ? 1.f / l_run1 : 0.f;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (pv.valid(k))
            st_relaxed_gpu(pv.ow(w.part, mt, k), part_enc(o[mt][k] * ((k & 1) ? il1 : il0)));
      if (warp == 0 && gid == 0) {
        if (hv0)
          st_relaxed_gpu(pv.lw(w.part, 0),
                         part_enc(l_run0 > 0.f ? m_run0 + log2f(l_run0) : -INFINITY));
        if (hv1)
          st_relaxed_gpu(pv.lw(w.part, 1),
                         part_enc(l_run1 > 0.f ? m_run1 + log2f(l_run1) : -INFINITY));
      }
      continue;
    }
    if (merge) {
      // fold one part (normalised o, lse) into the running (m, l, unnormalised o)
      auto merge_in = [&](float ls0, float ls1, const uint32_t (&v)[MT][4]) {
        const float mn0 = fmaxf(m_run0, ls0), mn1 = fmaxf(m_run1, ls1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float a0 = exp2f(m_run0 - mu0), b0 = exp2f(ls0 - mu0);
        const float a1 = exp2f(m_run1 - mu1), b1 = exp2f(ls1 - mu1);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          o[mt][0] = fmaf(o[mt][0], a0, part_dec(v[mt][0]) * b0);
          o[mt][2] = fmaf(o[mt][2], a0, part_dec(v[mt][2]) * b0);
          o[mt][1] = fmaf(o[mt][1], a1, part_dec(v[mt][1]) * b1);
          o[mt][3] = fmaf(o[mt][3], a1, part_dec(v[mt][3]) * b1);
        }
        l_run0 = fmaf(l_run0, a0, b0);
        l_run1 = fmaf(l_run1, a1, b1);
        m_run0 = mn0;
        m_run1 = mn1;
      };
      auto give_up = [&]() {
        failed = true;
        *abort_flag = 1;
        if (err) atomicOr(err, PKV_ERR_TIMEOUT);
      };
      if (part_wait<PF, MT>(pv, 1, wp, lp, abort_flag)) {
#pragma unroll
        for (int jj = 0; jj < PF; ++jj) {
          merge_in(part_dec(lp[jj][0]), part_dec(lp[jj][1]), wp[jj]);
          if (1 + jj < w.parts) part_clear<MT>(pv, 1 + jj);
        }
      } else {
        give_up();
      }
      for (int j0 = 1 + PF; j0 < w.parts && !failed; j0 += JB) {
        uint32_t wb[JB][MT][4], lb[JB][2];
        part_load<JB, MT>(pv, j0, w.parts, wb, lb);
        if (!part_wait<JB, MT>(pv, j0, wb, lb, abort_flag)) {
          give_up();
          break;
        }
#pragma unroll
        for (int jj = 0; jj < JB; ++jj) {
          merge_in(part_dec(lb[jj][0]), part_dec(lb[jj][1]), wb[jj]);
          if (j0 + jj < w.parts) part_clear<MT>(pv, j0 + jj);
        }
      }
      // every consumer thread of a head has read its lse words: clear them
      // (the merge unit is the CTA's last, so this barrier costs no overlap)
      consumer_sync();
      if (failed) continue;
      if (warp == 0 && gid == 0) {
        for (int j = 1; j < w.parts; ++j) {
          if (hv0) st_relaxed_gpu(pv.lw(j, 0), 0u);
          if (hv1) st_relaxed_gpu(pv.lw(j, 1), 0u);
        }
      }
    }
    const float il0 = l_run0 > 0.f ? 1.f / l_run0 : 0.f;
    const float il1 = l_run1 > 0.f ? 1.f / l_run1 : 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int d = warp * (D / 4) + 16 * mt + gid;
      if (hv0) {
        out[(head0 + h0) * D + d] = __float2bfloat16_rn(o[mt][0] * il0);
        out[(head0 + h0) * D + d + 8] = __float2bfloat16_rn(o[mt][2] * il0);
      }
      if (hv1) {
        out[(head0 + h1) * D + d] = __float2bfloat16_rn(o[mt][1] * il1);
        out[(head0 + h1) * D + d + 8] = __float2bfloat16_rn(o[mt][3] * il1);
      }
    }
  }
}

// Fixed split mode: merge the parts of one (row, head) with weights
// 2^(lse_c - max), skipping parts without keys (lse = -inf). (Row, head)
// pairs handled by one CTA were written by the attention kernel itself. One
// warp per (row, head); lane l merges output columns 4l + 128c. The part
// count, the log-sum-exps and the first two partials are loaded together, so
// a two-part merge needs one round trip to L2 after the attention kernel
// completes. Part s of query head hi of (row b, kv head g) sits in record
// (b * Hkv + g) * max_parts + s: o at [hi][D] of a [G][D] block, lse at [hi],
// every word encoded (part_enc); the merge clears the words it read, so the
// partial area is zero again for the next call.
__device__ __forceinline__ float4 part_dec4(float4 v) {
  return make_float4(part_dec(__float_as_uint(v.x)), part_dec(__float_as_uint(v.y)),
                     part_dec(__float_as_uint(v.z)), part_dec(__float_as_uint(v.w)));
}
template <int D>
__global__ void combine_kernel(float *__restrict__ o_part, float *__restrict__ lse_part,
                               const int *__restrict__ parts_in, const Problem p,
                               __nv_bfloat16 *__restrict__ out) {
  constexpr int CH = (D + 127) / 128;   // float4 column chunks per lane
  // The next kernel may start (and plan) as soon as every CTA of this grid
  // is running; it waits for this grid to complete before it touches the
  // workspace or the output.
  pkv_allow_next_grid();
  pkv_wait_prior_grid();
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= p.B * p.Hq) return;
  const int b = r / p.Hq, hh = r - b * p.Hq, g = hh / p.G, hi = hh - g * p.G;
  const size_t rec = (static_cast<size_t>(b) * p.Hkv + g) * p.max_parts;
  const size_t pstride = static_cast<size_t>(p.G) * D;     // floats between parts
  float *lse = lse_part + rec * p.G + hi;                    // part s at lse[s * G]
  float *op = o_part + rec * pstride + static_cast<size_t>(hi) * D;
  const int parts = __ldcg(parts_in + b * p.Hkv + g);
  float my_lse = lane < p.max_parts ? part_dec(__float_as_uint(__ldcg(lse + lane * p.G)))
                                    : -INFINITY;
  float4 v0[CH], v1[CH];   // parts 0 and 1 (max_parts >= 2 whenever this kernel runs)
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int d = 4 * lane + 128 * c;
    if (d < D) {
      v0[c] = part_dec4(__ldcg(reinterpret_cast<const float4 *>(op + d)));
      v1[c] = part_dec4(__ldcg(reinterpret_cast<const float4 *>(op + pstride + d)));
    }
  }
  if (parts <= 1) return;
  if (lane >= parts) my_lse = -INFINITY;
  float m = my_lse;
  for (int s = 32 + lane; s < parts; s += 32)
    m = fmaxf(m, part_dec(__float_as_uint(__ldcg(lse + s * p.G))));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  __nv_bfloat16 *orow = out + static_cast<size_t>(r) * D;
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  // every lane runs every iteration (the shuffles name the whole warp); at
  // D = 64 lanes 16-31 own no column and only skip the memory accesses
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int d = 4 * lane + 128 * c;
    const bool dv = d < D;
    float4 acc = zero4;
    float wsum = 0.f;
    for (int s = 0; s < parts; ++s) {
      const float l = s < 32 ? __shfl_sync(0xffffffffu, my_lse, s)
                             : part_dec(__float_as_uint(__ldcg(lse + s * p.G)));
      if (!dv) continue;
      const float4 v =
          s == 0   ? v0[c]
          : s == 1 ? v1[c]
                   : part_dec4(__ldcg(reinterpret_cast<const float4 *>(op + s * pstride + d)));
      // each lane reads its own columns: clear them now
      *reinterpret_cast<float4 *>(op + s * pstride + d) = zero4;
      if (m == -INFINITY) continue;
      const float wgt = l == -INFINITY ? 0.f : exp2f(l - m);
      wsum += wgt;
      acc.x = fmaf(wgt, v.x, acc.x);
      acc.y = fmaf(wgt, v.y, acc.y);
      acc.z = fmaf(wgt, v.z, acc.z);
      acc.w = fmaf(wgt, v.w, acc.w);
    }
    if (!dv) continue;
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2 packed;
    packed.x = pack_bf16(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(orow + d) = packed;
  }
  // every lane has read every lse word it needs
  __syncwarp();
  for (int s = lane; s < parts; s += 32) lse[s * p.G] = 0.f;
}

// Clears the partial area of a workspace when the error word reports a wait
// that gave up (such a call may leave written, unread partials behind).
__global__ void scrub_after_timeout_kernel(uint32_t *__restrict__ base, size_t words,
                                           const int32_t *__restrict__ err) {
  if (!(__ldcg(err) & PKV_ERR_TIMEOUT)) return;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < words;
       i += stride)
    base[i] = 0u;
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
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Map over a cache of `rows` rows of D bf16 in pages of page_size rows, with
// [box_rows][64] boxes: a 2-D map {column, row}, or (paged) a 3-D map
// {column, row in page, page}, so that a box starting before or ending after
// its page reads zeros there instead of the neighbouring page (out-of-range
// elements are filled, not loaded). Full tiles use the 2-D map; the partly
// used tiles at a row's ends use the 3-D one.
int make_cache_map(CUtensorMap *tm, const void *base, long long rows, int D,
                   int box_rows, int page_size, bool paged) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(paged ? page_size : rows),
                        static_cast<cuuint64_t>(paged ? rows / page_size : 1)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(D) * 2 * page_size};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, paged ? 3 : 2,
                  const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return pkv::fail(PKV_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return PKV_OK;
}

template <int D, bool STEP>
int set_smem_attr() {
  static std::mutex mu;
  static bool done[64] = {false};
  int dev = 0;
  PKV_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return pkv::fail(PKV_E_CUDA, "device id out of range");
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    PKV_CUDA_CHECK(cudaFuncSetAttribute(decode_attn_kernel<D, STEP>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Cfg<D>::SMEM));
    done[dev] = true;
  }
  return PKV_OK;
}

template <int D, bool STEP>
int launch_attn(const CUtensorMap &tmK, const CUtensorMap &tmV, const CUtensorMap &tmK3,
                const CUtensorMap &tmV3, const pkv_bf16 *q,
                const Problem &p, float scale_log2, float *o_part, float *lse_part,
                int *parts, pkv_bf16 *out, int32_t *err, const StepArgs &sa,
                cudaStream_t stream) {
  int st = set_smem_attr<D, STEP>();
  if (st != PKV_OK) return st;
  const int sms = pkv::sm_count();
  if (sms <= 0) return pkv::fail(PKV_E_CUDA, "paged_decode_attn: no SM count");
  const int grid = sms * Cfg<D>::CTAS_PER_SM;
  PKV_CUDA_CHECK(pkv::launch_pdl(decode_attn_kernel<D, STEP>, dim3(grid), dim3(kThreads),
                                 Cfg<D>::SMEM, stream, tmK, tmV, tmK3, tmV3,
                                 reinterpret_cast<const __nv_bfloat16 *>(q), p, scale_log2,
                                 o_part, lse_part, parts,
                                 reinterpret_cast<__nv_bfloat16 *>(out), err, sa));
  return PKV_OK;
}

// Upper bound on the parts a row is cut into: the fixed split count, or in
// the automatic mode one part per 64-key tile of the longest possible row.
int max_parts_for(int max_pages, int page_size, int window, int num_splits) {
  const long long max_keys = 1LL * max_pages * page_size;
  long long tiles = (max_keys + kT - 1) / kT;
  if (window > 0 && window < max_keys) tiles = (window + kT - 1) / kT + 1;
  if (num_splits > 0) return static_cast<int>(num_splits < tiles ? num_splits : tiles);
  return static_cast<int>(tiles);
}

}  // namespace

static size_t parts_bytes(int B, int Hq) {
  return (static_cast<size_t>(B) * Hq * sizeof(int) + 255) & ~size_t(255);
}

int pkv::decode_max_parts(int max_pages_per_seq, int page_size, int window, int num_splits) {
  if (max_pages_per_seq < 1 || page_size < 1 || num_splits < 0) return 0;
  return max_parts_for(max_pages_per_seq, page_size, window, num_splits);
}

extern "C" {

// Workspace layout, with P the parts a (row, kv head) may be cut into:
//   [parts per (row, kv head) for the fixed mode's combine: B*Hq ints, 256-byte padded]
//   [o_part: B*Hkv*P records of G*D words, = B*Hq*P*D]
//   [lse_part: B*Hkv*P records of G words, = B*Hq*P]
// Counts are written before they are read. The partial words (part_enc)
// must be zero before the first call; every call that completes without
// PKV_ERR_TIMEOUT leaves them zero again.

size_t paged_decode_attn_workspace(int B, int Hq, int D, int num_splits) {
  if (num_splits <= 1 || B <= 0 || Hq <= 0 || D <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * num_splits;
  return parts_bytes(B, Hq) + rows * D * sizeof(float) + rows * sizeof(float);
}

int paged_decode_attn_splits(int B, int Hkv, int D, int max_pages_per_seq,
                             int page_size, int window, int *num_splits) {
  if (!num_splits || Hkv < 1 || max_pages_per_seq < 1 || page_size < 1 || B < 0 || D < 1)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_attn_splits: bad argument");
  *num_splits = max_parts_for(max_pages_per_seq, page_size, window, 0);
  return pkv::ok();
}

}  // extern "C"

int pkv::decode_scrub_after_timeout(void *workspace, int B, int Hq, int D, int parts,
                                   const int32_t *err_word, cudaStream_t stream) {
  if (!workspace || !err_word || paged_decode_attn_workspace(B, Hq, D, parts) == 0)
    return PKV_OK;
  const size_t rows = static_cast<size_t>(B) * Hq * parts;
  const size_t words = rows * D + rows;   // o_part, then lse_part
  uint32_t *base =
      reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + parts_bytes(B, Hq));
  const int sms = pkv::sm_count();
  if (sms <= 0) return pkv::fail(PKV_E_CUDA, "paged_decode_attn: no SM count");
  scrub_after_timeout_kernel<<<sms, 256, 0, stream>>>(base, words, err_word);
  PKV_CUDA_CHECK(cudaGetLastError());
  return PKV_OK;
}


namespace {

// Argument checks, tensor maps, problem set-up and the launches shared by
// paged_decode_attn (sa == nullptr; seq_lens = lengths) and the fused
// paged_decode_step (seq_lens = input positions, lengths = positions + 1).
int decode_common(const char *fn, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                  const pkv_bf16 *v_cache, const int32_t *dev_table, int n_slots,
                  int max_pages_per_seq, int page_size, int n_pages,
                  const int32_t *batch_idx, const int32_t *seq_lens, int window, float scale,
                  int B, int Hq, int Hkv, int D, int num_splits, void *workspace,
                  size_t workspace_bytes, pkv_bf16 *out, int32_t *err_word,
                  const StepArgs *sa, void *stream) {
  if (D != 64 && D != 128 && D != 256 && D != 512)
    return pkv::fail(PKV_E_BAD_ARG, "%s: D must be 64, 128, 256 or 512", fn);
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv || Hq / Hkv > kMaxG)
    return pkv::fail(PKV_E_BAD_ARG, "%s: need Hq %% Hkv == 0 and Hq/Hkv <= %d", fn, kMaxG);
  if (!pkv::is_pow2(page_size) || page_size < 8)
    return pkv::fail(PKV_E_BAD_ARG, "%s: page_size must be a power of two >= 8", fn);
  if (B < 0 || n_slots < 1 || max_pages_per_seq < 1 || n_pages < 1 || num_splits < 0)
    return pkv::fail(PKV_E_BAD_ARG, "%s: bad size argument", fn);
  if (B > kMaxRows)
    return pkv::fail(PKV_E_BAD_ARG, "%s: B must be <= %d", fn, kMaxRows);
  if (static_cast<long long>(max_pages_per_seq) * page_size > (1LL << 30))
    return pkv::fail(PKV_E_BAD_ARG, "%s: table row too long", fn);
  const long long rows = 1LL * Hkv * n_pages * page_size;
  if (rows >= (1LL << 31))
    return pkv::fail(PKV_E_BAD_ARG, "%s: cache has too many rows", fn);
  if (!(scale > 0.f) || !std::isfinite(scale))
    return pkv::fail(PKV_E_BAD_ARG, "%s: scale must be finite and > 0", fn);
  if (sa) {
    if (!(sa->log2_theta > -INFINITY) || !std::isfinite(sa->log2_theta))
      return pkv::fail(PKV_E_BAD_ARG, "%s: theta must be finite and > 0", fn);
    if (!(sa->eps >= 0.f))
      return pkv::fail(PKV_E_BAD_ARG, "%s: eps must be >= 0", fn);
    if ((sa->gamma_q == nullptr) != (sa->gamma_k == nullptr))
      return pkv::fail(PKV_E_BAD_ARG, "%s: give both gains or neither", fn);
  }
  if (B == 0) return pkv::ok();
  if (!q || !k_cache || !v_cache || !dev_table || !seq_lens || !out)
    return pkv::fail(PKV_E_BAD_ARG, "%s: NULL tensor", fn);
  if (sa && (!sa->k_new || !sa->v_new))
    return pkv::fail(PKV_E_BAD_ARG, "%s: NULL tensor", fn);
  if (!pkv::aligned16(q) || !pkv::aligned16(out) || !pkv::aligned16(k_cache) ||
      !pkv::aligned16(v_cache) ||
      (sa && (!pkv::aligned16(sa->k_new) || !pkv::aligned16(sa->v_new))))
    return pkv::fail(PKV_E_BAD_ARG, "%s: tensors must be 16-byte aligned", fn);
  {
    const long long row_tiles = (1LL * max_pages_per_seq * page_size + kT - 1) / kT + 1;
    if (1LL * B * Hkv * (kTileCost * row_tiles + kUnitCost) >= (1LL << 31))
      return pkv::fail(PKV_E_BAD_ARG, "%s: B * Hkv * tiles per row too large", fn);
  }
  const int max_parts = max_parts_for(max_pages_per_seq, page_size, window, num_splits);
  const size_t need = paged_decode_attn_workspace(B, Hq, D, max_parts);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return pkv::fail(PKV_E_BAD_ARG, "%s: workspace needs %zu bytes", fn, need);
    if (!pkv::aligned16(workspace))
      return pkv::fail(PKV_E_BAD_ARG, "%s: workspace must be 16-byte aligned", fn);
  }
  int *parts = nullptr;
  float *o_part = nullptr, *lse_part = nullptr;
  if (need > 0) {
    parts = static_cast<int *>(workspace);
    o_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + parts_bytes(B, Hq));
    lse_part = o_part + static_cast<size_t>(B) * Hq * max_parts * D;
  }
  const int box_rows = page_size < kT ? page_size : kT;
  CUtensorMap tmK, tmV, tmK3, tmV3;
  int st = make_cache_map(&tmK, k_cache, rows, D, box_rows, page_size, false);
  if (st != PKV_OK) return st;
  st = make_cache_map(&tmV, v_cache, rows, D, box_rows, page_size, false);
  if (st != PKV_OK) return st;
  if (box_rows == kT) {
    st = make_cache_map(&tmK3, k_cache, rows, D, box_rows, page_size, true);
    if (st != PKV_OK) return st;
    st = make_cache_map(&tmV3, v_cache, rows, D, box_rows, page_size, true);
    if (st != PKV_OK) return st;
  } else {
    tmK3 = tmK;
    tmV3 = tmV;
  }
  int log2_ps = 0;
  while ((1 << log2_ps) < page_size) ++log2_ps;
  Problem p;
  p.table = dev_table;
  p.batch_idx = batch_idx;
  p.seq_lens = seq_lens;
  p.len_bias = sa ? 1 : 0;
  p.n_slots = n_slots;
  p.max_pages = max_pages_per_seq;
  p.log2_ps = log2_ps;
  p.n_pages = n_pages;
  p.window = window;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  // with at most one part per row no partial is ever written
  p.fixed_splits = max_parts == 1 ? 1 : num_splits;
  p.max_parts = max_parts;
  p.unit_cost = kUnitCost;
  // the balanced mode merges cut rows inside the attention kernel; only the
  // fixed mode needs the per-row part counts and the combine kernel
  const bool combine = p.fixed_splits > 0 && max_parts > 1;
  if (!combine) parts = nullptr;
  const float scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const StepArgs none = {};
  const StepArgs &a = sa ? *sa : none;
#define PKV_LAUNCH(DD)                                                                        \
  st = sa ? launch_attn<DD, true>(tmK, tmV, tmK3, tmV3, q, p, scale_log2, o_part, lse_part,    \
                                  parts, out, err_word, a, s)                                 \
          : launch_attn<DD, false>(tmK, tmV, tmK3, tmV3, q, p, scale_log2, o_part, lse_part,   \
                                   parts, out, err_word, a, s)
  switch (D) {
    case 64: PKV_LAUNCH(64); break;
    case 128: PKV_LAUNCH(128); break;
    case 256: PKV_LAUNCH(256); break;
    default: PKV_LAUNCH(512); break;
  }
#undef PKV_LAUNCH
  if (st != PKV_OK) return st;
  if (combine) {
    const int rows_bh = B * Hq;
    const int wpb = 4;
    auto *kern = D == 64    ? combine_kernel<64>
                 : D == 128 ? combine_kernel<128>
                 : D == 256 ? combine_kernel<256>
                            : combine_kernel<512>;
    PKV_CUDA_CHECK(pkv::launch_pdl(kern, dim3((rows_bh + wpb - 1) / wpb), dim3(wpb * 32), 0, s,
                                   o_part, lse_part,
                                   static_cast<const int *>(parts), p,
                                   reinterpret_cast<__nv_bfloat16 *>(out)));
  }
  return pkv::ok();
}

}  // namespace

extern "C" {

int paged_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                      const pkv_bf16 *v_cache, const int32_t *dev_table,
                      int n_slots, int max_pages_per_seq, int page_size,
                      int n_pages, const int32_t *batch_idx,
                      const int32_t *seq_lens, int window, float scale, int B,
                      int Hq, int Hkv, int D, int num_splits, void *workspace,
                      size_t workspace_bytes, pkv_bf16 *out, int32_t *err_word,
                      void *stream) {
  return decode_common("paged_decode_attn", q, k_cache, v_cache, dev_table, n_slots,
                       max_pages_per_seq, page_size, n_pages, batch_idx, seq_lens, window,
                       scale, B, Hq, Hkv, D, num_splits, workspace, workspace_bytes, out,
                       err_word, nullptr, stream);
}

int paged_decode_step_ex(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                         const pkv_bf16 *gamma_q, const pkv_bf16 *gamma_k,
                         const int32_t *batch_idx, const int32_t *input_pos, float theta,
                         float eps, int rotary_dims, int v_norm, int k_eq_v,
                         const int32_t *dev_table, int n_slots, int max_pages_per_seq,
                         int page_size, int n_pages, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                         int window, float scale, int B, int Hq, int Hkv, int D,
                         int num_splits, void *workspace, size_t workspace_bytes,
                         pkv_bf16 *out, int32_t *err_word, void *stream) {
  if (!(theta > 0.f) || !std::isfinite(theta))
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_step: theta must be finite and > 0");
  if (rotary_dims < 0 || rotary_dims > D || rotary_dims % 2)
    return pkv::fail(PKV_E_BAD_ARG, "paged_decode_step: rotary_dims must be even and in [0, D]");
  StepArgs sa;
  sa.k_new = reinterpret_cast<const __nv_bfloat16 *>(k);
  sa.v_new = reinterpret_cast<const __nv_bfloat16 *>(k_eq_v ? k : v);
  sa.gamma_q = reinterpret_cast<const __nv_bfloat16 *>(gamma_q);
  sa.gamma_k = reinterpret_cast<const __nv_bfloat16 *>(gamma_k);
  sa.log2_theta = log2f(theta);
  sa.eps = eps;
  sa.k_cache = reinterpret_cast<__nv_bfloat16 *>(k_cache);
  sa.v_cache = reinterpret_cast<__nv_bfloat16 *>(v_cache);
  sa.rot_pairs = rotary_dims / 2;
  sa.v_norm = v_norm ? 1 : 0;
  sa.k_eq_v = k_eq_v ? 1 : 0;
  return decode_common("paged_decode_step", q, k_cache, v_cache, dev_table, n_slots,
                       max_pages_per_seq, page_size, n_pages, batch_idx, input_pos, window,
                       scale, B, Hq, Hkv, D, num_splits, workspace, workspace_bytes, out,
                       err_word, &sa, stream);
}

int paged_decode_step(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                      const pkv_bf16 *gamma_q, const pkv_bf16 *gamma_k,
                      const int32_t *batch_idx, const int32_t *input_pos, float theta,
                      float eps, const int32_t *dev_table, int n_slots,
                      int max_pages_per_seq, int page_size, int n_pages, pkv_bf16 *k_cache,
                      pkv_bf16 *v_cache, int window, float scale, int B, int Hq, int Hkv,
                      int D, int num_splits, void *workspace, size_t workspace_bytes,
                      pkv_bf16 *out, int32_t *err_word, void *stream) {
  return paged_decode_step_ex(q, k, v, gamma_q, gamma_k, batch_idx, input_pos, theta, eps, D, 0,
                              0, dev_table, n_slots, max_pages_per_seq, page_size, n_pages,
                              k_cache, v_cache, window, scale, B, Hq, Hkv, D, num_splits,
                              workspace, workspace_bytes, out, err_word, stream);
}

}  // extern "C"
