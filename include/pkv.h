/*
 * pkv.h — C ABI of libpkv: paged-KV single-token decode attention on one
 * GB300 (sm_103a).
 *
 * The method follows three public web pages:
 *   [P1] "unsloth: compare main...flex-moe-qwen3" (commit message on the
 *        PageTable +1 capacity fix; unsloth/inference/flex_gemma4_moe.py:
 *        rotary helpers, attention forward, decode block masks, CUDA-graph
 *        capture and the continuous-batching loop);
 *   [P3] "unsloth: compare main...transformers-continuous-batching-qwen3"
 *        (scripts/benchmarks/flex_paged_attention.py: PagedKVCache and
 *        PageTable; scripts/benchmarks/README.md).
 *
 * Conventions shared by every call
 *   - Every call returns an int status: PKV_OK (0) or a negative PKV_E_*.
 *     A failed call leaves all state unchanged and records a message that
 *     pkv_last_error() returns (thread-local).
 *   - bf16 tensors are passed as pkv_bf16 (the raw 16-bit pattern).
 *   - Device pointers are caller-owned (allocated by the caller, e.g. with
 *     PyTorch). No call allocates or frees device memory.
 *   - Kernels are enqueued asynchronously on the given stream (a
 *     cudaStream_t passed as void*; NULL = legacy default stream). Only
 *     pkv_read_error_word() synchronizes.
 *   - Kernel launches use a grid that depends only on the scalar arguments,
 *     and read per-step metadata (positions, lengths, table) from device
 *     memory, so a fixed-shape call can be captured in a CUDA graph.
 *   - Kernels are launched with programmatic dependent launch: each waits
 *     for the kernel before it (griddepcontrol.wait) before it touches
 *     memory that kernel may write, so in-stream order is kept. The decode
 *     attention and the fused step read seq_lens, batch_idx and the page
 *     table BEFORE that wait, to plan their work while earlier kernels
 *     drain. So those three must be written by copies or by kernels that do
 *     not let their dependents start early (ordinary kernels); none of this
 *     library's kernels writes them.
 *   - Device-side faults are never raised on purpose: an invalid index read
 *     from device memory sets a bit in the caller's int32 error word
 *     (atomic OR) and the access is skipped.
 *
 * Cache layout (per layer, [P3] PagedKVCache): k_cache and v_cache are bf16
 * [Hkv][n_pages * page_size][D], row-major. Physical page p of kv head g is
 * the contiguous block of rows [p*page_size, (p+1)*page_size) of head g.
 * The page table is int32 [n_slots][max_pages_per_seq], row-major, with
 * n_slots = max_batch_size + 1; entry [s][j] is the physical page holding
 * logical tokens [j*page_size, (j+1)*page_size) of slot s, or -1.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16;
typedef struct pkv_pt pkv_pt;

/* status codes */
#define PKV_OK 0
#define PKV_E_NO_SLOT (-1)   /* no free slot */
#define PKV_E_NO_PAGES (-2)  /* too few free pages */
#define PKV_E_BAD_SLOT (-3)  /* slot 0, out of range, or not allocated */
#define PKV_E_BAD_ARG (-4)   /* shape, alignment, or pointer argument */
#define PKV_E_CUDA (-5)      /* a CUDA runtime call failed */

/* device error-word bits */
#define PKV_ERR_POS 1          /* position negative or beyond the table row */
#define PKV_ERR_PAGE_RANGE 2   /* table entry >= n_pages */
#define PKV_ERR_PAGE_NEG 4     /* table entry < 0 (unreserved block) */
#define PKV_ERR_SLOT 8         /* batch index outside [0, n_slots) */
#define PKV_ERR_TIMEOUT 16     /* a bounded wait on a copy gave up */

/* ---------------------------------------------------------------------
 * PageTable allocator (host) — [P3] PageTable.__init__ / can_reserve /
 * allocate / reserve / erase, with the +1 capacity rule of [P1]'s commit
 * message.
 *
 * Slot 0 is a no-op padding slot and page 0 a dummy page; row 0 of the
 * table is all 0. Slots 1..max_batch_size are usable. Free slots and free
 * pages are LIFO stacks (initially [N..1] and [n_pages-1..1]). reserve takes
 * the last k entries of the free-page list, in list order, for the next k
 * logical blocks; free pushes the slot and appends the slot's pages in
 * reverse order. A freed slot's device row is left stale until it is
 * assigned again.
 *
 * Device mirror: if dev_table is non-NULL it must point to caller-owned
 * int32 device memory of n_slots * max_pages_per_seq entries, 4-byte
 * aligned. pt_create writes the whole table; pt_assign writes the assigned
 * row; pt_reserve writes the new entries. These are cudaMemcpyAsync copies
 * from pageable host memory on the handle's stream: they may synchronize
 * with that stream, and must not be issued while the stream is capturing a
 * CUDA graph. With dev_table NULL the allocator is host-only (no CUDA call).
 * ------------------------------------------------------------------- */
int pt_create(int max_batch_size, int page_size, int n_pages,
              int max_pages_per_seq, int32_t *dev_table, void *stream,
              pkv_pt **out);
int pt_destroy(pkv_pt *pt);
int pt_set_stream(pkv_pt *pt, void *stream);
/* slot < 0: can a new request of seq_len tokens be admitted (a free slot
 * and enough pages)?  slot >= 1: can that live slot grow to seq_len? */
int pt_can_reserve(const pkv_pt *pt, int seq_len, int slot, int *ok);
/* allocate a slot and reserve seq_len tokens for it (all or nothing) */
int pt_assign(pkv_pt *pt, int seq_len, int *slot_out);
/* grow a live slot's capacity to >= seq_len (no-op if it already fits) */
int pt_reserve(pkv_pt *pt, int slot, int seq_len);
/* release a live slot and its pages */
int pt_free(pkv_pt *pt, int slot);
/* tokens reserved for a slot (0 for a free slot) */
int pt_capacity(const pkv_pt *pt, int slot, int *tokens);
/* pages of a slot in logical order (host mirror); *n receives the count */
int pt_pages(const pkv_pt *pt, int slot, int32_t *host_out, int max, int *n);
int pt_free_pages(const pkv_pt *pt, int *n);
/* the free-page stack, bottom first (the next reserve takes from the end) */
int pt_free_page_list(const pkv_pt *pt, int32_t *host_out, int max, int *n);
/* copy of the host mirror, n_slots * max_pages_per_seq entries */
int pt_host_table(const pkv_pt *pt, int32_t *host_out, int max);

/* ---------------------------------------------------------------------
 * kv_append — decode scatter of the step's new K/V ([P3] PageTable.assign):
 *   block = input_pos[b] / page_size, offset = input_pos[b] % page_size,
 *   row   = table[batch_idx[b]][block] * page_size + offset,
 *   k_cache[h][row][:] = k[b][h][:], v_cache[h][row][:] = v[b][h][:].
 * k, v: bf16 [B][Hkv][D]; batch_idx (NULL = identity) and input_pos: int32
 * [B]; rows may share a slot (a multi-token fill). Rows whose address is
 * invalid set PKV_ERR_* bits in err_word (may be NULL) and are skipped.
 * Requires D % 8 == 0 and 16-byte aligned k, v, k_cache, v_cache.
 * ------------------------------------------------------------------- */
int kv_append(const pkv_bf16 *k, const pkv_bf16 *v, const int32_t *batch_idx,
              const int32_t *input_pos, int B, const int32_t *dev_table,
              int n_slots, int max_pages_per_seq, int page_size, int n_pages,
              pkv_bf16 *k_cache, pkv_bf16 *v_cache, int Hkv, int D,
              int32_t *err_word, void *stream);

/* kv_append_prefill — the prefill scatter of [P3] PageTable
 * (assign_prefill_no_paging): L packed tokens, token j with its own slot
 * batch_idx[j] and position input_pos[j], k and v head-major bf16
 * [Hkv][L][D] (the pages' [1, H, L, D]). Same address map, checks and error
 * bits as kv_append, which this is with the head-major layout. */
int kv_append_prefill(const pkv_bf16 *k, const pkv_bf16 *v, const int32_t *batch_idx,
                      const int32_t *input_pos, int L, const int32_t *dev_table,
                      int n_slots, int max_pages_per_seq, int page_size, int n_pages,
                      pkv_bf16 *k_cache, pkv_bf16 *v_cache, int Hkv, int D,
                      int32_t *err_word, void *stream);

/* ---------------------------------------------------------------------
 * qk_norm_rope — per-head RMSNorm then RoPE, in place ([P1] attention
 * forward: q_norm / k_norm on the head axis before rotary; rotary helpers
 * _rotate_half / _apply_rotary_full):
 *   r = x / sqrt(mean(x^2) + eps) * gamma        (skipped if gamma is NULL)
 *   phi_i = pos[b] * theta^(-2i/D),  i < D/2
 *   y_i = r_i cos phi_i - r_{i+D/2} sin phi_i
 *   y_{i+D/2} = r_{i+D/2} cos phi_i + r_i sin phi_i
 * q: bf16 [B][Hq][D], k: bf16 [B][Hkv][D] (k may be NULL with Hkv 0),
 * gamma_q / gamma_k: bf16 [D] or NULL, pos: int32 [B]. Arithmetic is fp32
 * with a single rounding to bf16 per output. Requires D even, 2 <= D <= 1024,
 * theta > 0.
 * ------------------------------------------------------------------- */
int qk_norm_rope(pkv_bf16 *q, pkv_bf16 *k, const pkv_bf16 *gamma_q,
                 const pkv_bf16 *gamma_k, const int32_t *pos, float theta,
                 float eps, int B, int Hq, int Hkv, int D, void *stream);

/* ---------------------------------------------------------------------
 * qkv_norm_rope — qk_norm_rope with the Gemma-4 options of [P1] (two-tier
 * RoPE, per-head Q/K/V RMSNorm, Rotary helpers docstring):
 *   - rotary_dims (even, 0..D): only pairs i < rotary_dims/2 rotate, the
 *     rest pass through, as a zero inverse frequency does ("proportional"
 *     RoPE; rotary_dims = D is qk_norm_rope's full RoPE). Rotated pairs keep
 *     the full-dimension frequency theta^(-2i/D).
 *   - v (bf16 [B][Hkv][D], may be NULL): normalised in place without a gain,
 *     v / sqrt(mean(v^2) + eps) (v_norm, with_scale=False).
 * Other arguments as in qk_norm_rope; same arithmetic, one bf16 rounding.
 * ------------------------------------------------------------------- */
int qkv_norm_rope(pkv_bf16 *q, pkv_bf16 *k, pkv_bf16 *v, const pkv_bf16 *gamma_q,
                  const pkv_bf16 *gamma_k, const int32_t *pos, float theta,
                  float eps, int rotary_dims, int B, int Hq, int Hkv, int D,
                  void *stream);

/* ---------------------------------------------------------------------
 * qk_norm_rope_append — qk_norm_rope followed by kv_append in one kernel
 * (the write-then-attend prologue of [P1]'s attention forward: q/k norm,
 * rotary, then the paged write of [P3] PageTable.assign). Results are
 * identical to the two calls in sequence: q and k are rotated in place, then
 * k (rotated) and v (unchanged) are scattered to row
 * table[batch_idx[b]][input_pos[b] / page_size] * page_size + input_pos[b] %
 * page_size of every kv head's cache, with the same checks and error bits.
 * pos for the rotation is input_pos. Requires Hkv >= 1, D even <= 1024,
 * theta > 0; gains both given or both NULL (no norm).
 * ------------------------------------------------------------------- */
int qk_norm_rope_append(pkv_bf16 *q, pkv_bf16 *k, const pkv_bf16 *v,
                        const pkv_bf16 *gamma_q, const pkv_bf16 *gamma_k,
                        const int32_t *batch_idx, const int32_t *input_pos,
                        float theta, float eps, int B, int Hq, int Hkv, int D,
                        const int32_t *dev_table, int n_slots,
                        int max_pages_per_seq, int page_size, int n_pages,
                        pkv_bf16 *k_cache, pkv_bf16 *v_cache, int32_t *err_word,
                        void *stream);

/* ---------------------------------------------------------------------
 * paged_decode_attn — GQA single-token decode attention over the paged
 * cache ([P1] attention forward: flex_attention(q, k, v, scale,
 * block_mask, enable_gqa=True) with the decode masks of _decode_block_mask).
 * For row b: slot = batch_idx[b] (NULL = b), L = seq_lens[b] (tokens
 * including the one just appended, i.e. input_pos + 1), keys
 * j in [lo, L) with lo = max(0, L - window) if window > 0 else 0.
 * Query head h reads kv head h / (Hq / Hkv).
 *   out[b][h] = sum_j softmax_j(scale * q[b][h] . k_j) v_j
 * Rows with L <= 0 or slot 0 give exact zeros.
 *
 * Split-KV: the (row, kv head) key ranges are cut into parts of whole
 * 64-key tiles processed by persistent CTAs; a row cut into several parts
 * gets fp32 partial outputs and log-sum-exps in the workspace. num_splits 0
 * (automatic) lays the tiles of the call on one line from the actual
 * lengths, on the device, and gives every CTA an equal share of it; the CTA
 * holding the first part of a cut row merges the later parts (each the first
 * work of its own CTA) itself, so no second kernel runs. num_splits S > 0
 * cuts every row into at most S equal parts that a combine kernel merges.
 * The workspace must hold paged_decode_attn_workspace(B, Hq, D, P) bytes
 * (16-byte aligned; may be NULL when that is 0), with P = S for a fixed
 * split count or P = paged_decode_attn_splits(...) for the automatic mode.
 * It holds the partials, each word of which tells by itself whether it has
 * been written in this call (a reader waits for it and clears it after
 * use): zero the workspace once before its first use (e.g. cudaMemset).
 * Every call leaves it zero again, except a call that reports
 * PKV_ERR_TIMEOUT in the error word, after which the workspace must be
 * zeroed again. Calls sharing one workspace must not overlap on the GPU.
 * q: bf16 [B][Hq][D], out: bf16 [B][Hq][D], caches and table as above.
 * Requires D in {64, 128, 256, 512}, 1 <= Hq/Hkv <= 8, Hq % Hkv == 0,
 * page_size a power of two >= 8, B <= 512, and 16-byte aligned q, out,
 * caches.
 * Table entries that are negative or >= n_pages inside a row's key range
 * set PKV_ERR_PAGE_* (that row's output is then unspecified); L beyond
 * max_pages_per_seq * page_size sets PKV_ERR_POS and is clamped.
 * ------------------------------------------------------------------- */
int paged_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                      const pkv_bf16 *v_cache, const int32_t *dev_table,
                      int n_slots, int max_pages_per_seq, int page_size,
                      int n_pages, const int32_t *batch_idx,
                      const int32_t *seq_lens, int window, float scale, int B,
                      int Hq, int Hkv, int D, int num_splits, void *workspace,
                      size_t workspace_bytes, pkv_bf16 *out,
                      int32_t *err_word, void *stream);
/* the most parts a row can be cut into by the automatic mode (num_splits 0):
 * one per 64-key tile of the longest row the table allows (of the window plus
 * one when window > 0); size the workspace with it */
int paged_decode_attn_splits(int B, int Hkv, int D, int max_pages_per_seq,
                             int page_size, int window, int *num_splits);
/* workspace bytes for up to num_splits parts per row (0 when num_splits <= 1) */
size_t paged_decode_attn_workspace(int B, int Hq, int D, int num_splits);

/* ---------------------------------------------------------------------
 * paged_decode_step — one decode layer step in one pass: the write-then-
 * attend order of [P1]'s attention forward (q/k norm, rotary, the paged
 * write of [P3] PageTable.assign, then flex_attention over the pages).
 * Results equal the sequence
 *   qk_norm_rope(q', k', gamma_q, gamma_k, input_pos, theta, eps, ...)
 *   kv_append(k', v, batch_idx, input_pos, ...)
 *   paged_decode_attn(q', ..., seq_lens = input_pos + 1, ...)
 * on copies q', k' of q and k: the caches receive the same bytes, out the
 * same bits, err_word the same bits. q, k and v are inputs only (not
 * rotated in place). The rotated query never leaves the SM; the rotated key
 * is written to its cache row by the CTA that reads the row's last key tile,
 * which also uses it directly, so no second pass over the cache is needed.
 * Rows must name distinct slots (two rows appending into one slot would
 * each see an unspecified subset of the other's new token). Arguments as in
 * the three calls; requires gains both given or both NULL (no norm),
 * theta > 0, eps >= 0, 16-byte aligned k and v. The workspace is sized as for
 * paged_decode_attn.
 * ------------------------------------------------------------------- */
int paged_decode_step(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                      const pkv_bf16 *gamma_q, const pkv_bf16 *gamma_k,
                      const int32_t *batch_idx, const int32_t *input_pos,
                      float theta, float eps, const int32_t *dev_table,
                      int n_slots, int max_pages_per_seq, int page_size,
                      int n_pages, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                      int window, float scale, int B, int Hq, int Hkv, int D,
                      int num_splits, void *workspace, size_t workspace_bytes,
                      pkv_bf16 *out, int32_t *err_word, void *stream);
/* paged_decode_step_ex — paged_decode_step with the Gemma-4 options of
 * qkv_norm_rope ([P1] two-tier RoPE, v_norm, K=V alternative): rotary_dims
 * as in qkv_norm_rope; v_norm != 0 normalises the appended value without a
 * gain; k_eq_v != 0 takes the value from the raw k row (before k_norm and
 * RoPE) instead of v, which may then be NULL. Equals qkv_norm_rope (on
 * copies, with v' = copy of k when k_eq_v) -> kv_append -> paged_decode_attn
 * bit for bit. paged_decode_step is this call with rotary_dims = D,
 * v_norm = k_eq_v = 0. */
int paged_decode_step_ex(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                         const pkv_bf16 *gamma_q, const pkv_bf16 *gamma_k,
                         const int32_t *batch_idx, const int32_t *input_pos,
                         float theta, float eps, int rotary_dims, int v_norm,
                         int k_eq_v, const int32_t *dev_table, int n_slots,
                         int max_pages_per_seq, int page_size, int n_pages,
                         pkv_bf16 *k_cache, pkv_bf16 *v_cache, int window,
                         float scale, int B, int Hq, int Hkv, int D,
                         int num_splits, void *workspace, size_t workspace_bytes,
                         pkv_bf16 *out, int32_t *err_word, void *stream);

/* ---------------------------------------------------------------------
 * convert_logical_block_mask — re-points a block mask built over logical
 * positions at the paged cache ([P3] PageTable.convert_logical_block_mask):
 *   new_kv_indices[b][h][r][c] = table[slot_b][kv_indices[b][h][r][c]]
 *       for c < max_blocks, and 0 for max_blocks <= c < n_cols,
 * slot_b = batch_idx[b] (batch_idx NULL: slot_b = b). The key-block size of
 * the mask must equal page_size (the caller's contract, as on the pages).
 * kv_indices: int32 [B][H][rows][max_blocks]; new_kv_indices: int32
 * [B][H][rows][n_cols], n_cols >= max_blocks (the pages use the table
 * width). The block counts are unchanged (reuse them); convert full and
 * partial index arrays with one call each. Device pointers, caller-owned.
 * Table entries are copied as they are (-1 for an unreserved block). An
 * index outside [0, max_pages_per_seq) gives -1 and PKV_ERR_POS; a slot
 * outside [0, n_slots) gives -1 for all of that row's entries and
 * PKV_ERR_SLOT (err_word may be NULL). One kernel. Errors: PKV_E_BAD_ARG
 * for a bad shape or a NULL pointer, PKV_E_CUDA on a launch failure.
 * ------------------------------------------------------------------- */
int convert_logical_block_mask(const int32_t *dev_table, int n_slots,
                               int max_pages_per_seq, const int32_t *batch_idx,
                               int B, int H, int rows, int max_blocks,
                               const int32_t *kv_indices, int n_cols,
                               int32_t *new_kv_indices, int32_t *err_word,
                               void *stream);

/* ---------------------------------------------------------------------
 * Document-causal prefill attention over L packed prompt tokens
 * ([P3] PagedKVCache.create_prefill_blockmask_no_paging; the sliding
 * variant is [P1] _create_prefill_sliding_blockmask): docs[t] is the
 * document id of token t (any order); query i keeps key j iff j <= i,
 * docs[j] == docs[i] and, when window W > 0, i - j < W. W = 0 means no
 * window.
 *
 * PKV_PREFILL_BLOCK is the block of the block mask and the attention
 * kernel's tile: 64 query rows by 64 keys. n = ceil(L / 64).
 * ------------------------------------------------------------------- */
#define PKV_PREFILL_BLOCK 64

/* prefill_block_mask — the block mask of that mask (create_block_mask's
 * BlockMask with B = 1, H = None): for query block qb,
 *   full_kv_indices[qb][0 .. full_kv_num_blocks[qb])  the key blocks whose
 *       64 x 64 pairs all lie inside L and are all kept (no masking needed),
 *   kv_indices[qb][0 .. kv_num_blocks[qb])            the other key blocks
 *       with at least one kept pair inside L,
 * both ascending. The counts are int32 [n]; the index arrays int32 [n][n]
 * (row stride n; entries past a row's count are left unwritten). docs:
 * int32 [L] device. All four outputs are device memory the caller owns. It
 * depends only on docs and W, so one build serves every layer and head.
 * One kernel; L = 0 launches nothing. Errors: PKV_E_BAD_ARG for L < 0,
 * L > INT_MAX - 64, W < 0 or a NULL pointer; PKV_E_CUDA on a launch
 * failure. */
int prefill_block_mask(const int32_t *docs, int L, int window,
                       int32_t *kv_num_blocks, int32_t *kv_indices,
                       int32_t *full_kv_num_blocks, int32_t *full_kv_indices,
                       void *stream);

/* prefill_attn — the attention itself, on the packed tensors (no paging):
 * q bf16 [Hq][L][D], k and v bf16 [Hkv][L][D] (the pages' [1, H, L, D]),
 * docs int32 [L], out bf16 [Hq][L][D]; query head h reads kv head
 * h / (Hq / Hkv).  out[h][i] = sum_j softmax_j(scale * q[h][i] . k_j) v_j
 * over the kept j. The four block-mask arrays are those prefill_block_mask
 * writes for the same docs, L and W: only the listed key blocks are
 * visited, partial ones masked by the rule above, full ones unmasked (a
 * block listed as full that is not makes its pairs count as kept; list
 * entries outside [0, n) are skipped, so no list can make a read go out of
 * bounds; the lists are expected ascending, as prefill_block_mask writes
 * them). A row with no visited key gets zeros. Requires D in {64, 128,
 * 256, 512} (256 and 512: the Gemma-4 sliding and full layers), Hq % Hkv ==
 * 0, Hq <= 65535, ceil(L / 128) * Hq (twice that at D = 512) < 2^31,
 * 16-byte aligned q, k, v, out and docs, scale finite and > 0. One kernel
 * (tcgen05 MMAs with TMEM accumulators, one persistent CTA per SM over work
 * items of 128 query rows and one head; at D = 256 and 512 the scores are
 * accumulated over D in 64-column chunks and an item writes one 256-column
 * half of the output); no workspace. Errors: PKV_E_BAD_ARG for the above or
 * a NULL pointer, PKV_E_CUDA on a launch failure. */
int prefill_attn(const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                 const int32_t *docs, const int32_t *kv_num_blocks,
                 const int32_t *kv_indices, const int32_t *full_kv_num_blocks,
                 const int32_t *full_kv_indices, int L, int Hq, int Hkv, int D,
                 int window, float scale, pkv_bf16 *out, void *stream);

/* ---------------------------------------------------------------------
 * paged_decode_attn_noalloc — paged_decode_attn without a caller workspace.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory (a plain C program linking only this
 * library with no device allocator, or a plugin whose host framework owns
 * all device memory and hands out no scratch). Same arguments and results
 * as paged_decode_attn minus workspace / workspace_bytes. The split
 * partials go to a fixed 32 MiB scratch array in the library's device
 * image, held by every GPU that loads the library until the process exits;
 * a call whose partials need more fails with PKV_E_BAD_ARG. The need is
 * paged_decode_attn_workspace(B, Hq, D, parts) with parts = num_splits
 * capped at the 64-key tiles of the longest row the table holds (the
 * automatic count of paged_decode_attn_splits when num_splits is 0), the
 * same cap paged_decode_attn applies. The first call on a device looks up the scratch address
 * (cudaGetSymbolAddress) with that device current; make it before any
 * stream capture begins. All calls share the scratch: calls whose kernels
 * overlap on the GPU race and must be serialized by the caller. The
 * scratch starts zeroed and every completed call leaves it zero; each call
 * first launches a small kernel on the caller's stream that clears it only
 * when *err_word holds PKV_ERR_TIMEOUT (a call that gave up on a wait can
 * leave partials behind; with err_word NULL nothing is checked). No device
 * memory is allocated.
 * ------------------------------------------------------------------- */
int paged_decode_attn_noalloc(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                              const pkv_bf16 *v_cache, const int32_t *dev_table,
                              int n_slots, int max_pages_per_seq, int page_size,
                              int n_pages, const int32_t *batch_idx,
                              const int32_t *seq_lens, int window, float scale,
                              int B, int Hq, int Hkv, int D, int num_splits,
                              pkv_bf16 *out, int32_t *err_word, void *stream);

/* ---------------------------------------------------------------------
 * Utilities
 * ------------------------------------------------------------------- */
/* synchronize the stream, then copy the device error word to *host_out */
int pkv_read_error_word(const int32_t *err_word, void *stream,
                        int32_t *host_out);
/* message of the last failed call on this thread ("" if none) */
const char *pkv_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
