/*
 * pkv.h -- C ABI of the paged K/V attention library for GB300 (sm_103a).
 *
 * The library covers the data-parallel hot path of attention read through a
 * paged K/V cache, as described by two TensorRT-LLM pull-request pages:
 *
 *   [VG] "Paged causal K/V cache and cached attention for VisualGen"
 *        (pull request 19938), and
 *   [SP] "Support shared-prefix attention for n-sample requests in FMHA"
 *        (pull request 20841).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *    never allocates, frees, synchronises or reads device memory back on the
 *    host: each call validates its arguments on the host, enqueues its kernels
 *    on `stream` (a cudaStream_t; NULL = the legacy default stream) and returns.
 *    This is the CUDA-graph rule of [VG] Description, Cache ("CUDA-graph safe"
 *    bullet): every kernel input lives in caller-owned device memory, so a
 *    captured call replays with whatever those buffers hold.
 *  - Validation failures return a status before anything is enqueued; the
 *    reason is available from pkv_last_error() (thread-local).  Empty inputs
 *    (zero tokens, rows or heads) return PKV_OK without a launch ([VG] per-file
 *    notes on rotateRows: no-op cases).
 *  - Strides are in ELEMENTS, not bytes.
 *  - Paged pool layout: K and V are separate pools of `num_pages` pages; page
 *    p starts at element p * page_stride and holds `page_size` slots of
 *    [num_kv_heads][head_dim] contiguous elements (token-major).  Slot id
 *    s = page * page_size + offset ([VG] Description, Cache: slot ids are
 *    view_page * tokens_per_page + slot).  page_stride >= page_size *
 *    num_kv_heads * head_dim, so one allocation may hold K and V interleaved
 *    per page.
 *  - Device-side indices (slots, block-table entries, source indices) are the
 *    caller's responsibility, as in [VG] (per-file notes on scatterKvSlots:
 *    device slot indices are not range-checked).  With PKV_FLAG_CHECKED the
 *    kernels range-check them, skip the offending access and OR an error bit
 *    into *err (a device int32 the caller zeroes); nothing faults.
 *  - Duplicate destination slots in one scatter race: the value left in the
 *    slot is unspecified ([VG] per-file notes on scatterKvSlots).
 *  - Calls are not internally synchronised with each other; calls on
 *    different streams that touch the same memory race.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1, /* a pointer, size or stride is not valid     */
    PKV_ERR_UNSUPPORTED = 2, /* valid, but not a combination built here    */
    PKV_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
    PKV_ERR_CUDA = 4         /* a CUDA runtime/driver call failed          */
} pkv_status;

typedef enum { PKV_BF16 = 0, PKV_F16 = 1, PKV_F32 = 2 } pkv_dtype;

typedef enum {
    PKV_MASK_NONE = 0,         /* every key of the sequence is visible       */
    PKV_MASK_CAUSAL = 1,       /* row i sees keys 0 .. kv_len - q_real + i   */
    PKV_MASK_BLOCK_CAUSAL = 2  /* full within a causal block, causal across  */
} pkv_mask;

/* flags */
#define PKV_FLAG_CHECKED 0x1u     /* range-check device indices, report in *err */
#define PKV_FLAG_SIMT_ONLY 0x2u   /* paged_attention: use the generic SIMT kernel
                                     (a slow cross-check of the fast kernels)   */
/* paged_attention, test of the failure path: the decode kernel's consumer warps
 * wait on a barrier that nothing completes, give up after ~20 us, set
 * PKV_ERRBIT_TIMEOUT in *err (required) and wind down as after a real timeout
 * (the producer's ring waits are ~20 us too; every copy already issued is
 * waited for before a CTA exits).  The outputs are unspecified.  Only calls
 * that run the decode kernel accept it (else PKV_ERR_UNSUPPORTED). */
#define PKV_FLAG_TEST_WAIT_TIMEOUT 0x4u
/* paged_attention: run the tensor-core tiles as one CTA per tile pair (keys
 * split as planned); the default, and what PKV_FLAG_STREAM_K is measured
 * against */
#define PKV_FLAG_TILE_GRID 0x8u
/* paged_attention: when the two-tile kernel runs with the automatic split
 * count, schedule it stream-K style instead: one persistent CTA per SM runs
 * one whole tile pair of the first wave and then a contiguous share of the
 * remaining pairs' 128-key tiles; pairs split between CTAs leave partial
 * states that a reduce merges (a planner, the persistent launch and the
 * reduce: three launches).  Results agree with the grid within the attention
 * tolerances.  Slower than the grid on the workloads measured here (identical
 * tile pairs run at SM-dependent speeds that static shares cannot absorb), so
 * not the default; a tuning aid for other GPUs and shapes */
#define PKV_FLAG_STREAM_K 0x10u

/* bits OR-ed into *err in checked mode */
#define PKV_ERRBIT_SLOT 0x1       /* scatter slot >= num_pages * page_size      */
#define PKV_ERRBIT_SRC 0x2        /* scatter source index out of range          */
#define PKV_ERRBIT_PAGE 0x4       /* block-table entry outside [0, num_pages)   */
#define PKV_ERRBIT_LEN 0x8        /* kv_len / q rows beyond the host bounds      */
/* set in any mode: a device wait gave up (about 2 s; see PKV_FLAG_TEST_WAIT_TIMEOUT)
   and the kernel wound down; the call's results are invalid */
#define PKV_ERRBIT_TIMEOUT 0x10

/* Human-readable name of a status, and the last validation message of this thread. */
const char* pkv_status_string(pkv_status status);
const char* pkv_last_error(void);

/*
 * kv_scatter_slots -- write new K/V token rows into pool slots.
 *
 * [VG] Description, Cache ("Chunk K/V write" bullet) and the per-file notes on
 * scatterKvSlots: one kernel reads each source row once, with any token/head
 * stride (so K/V sliced from a fused QKV tensor need no copy), and writes it to
 * one or two pool slots; optional source indices.
 *
 * For t in [0, num_tokens):  src = src_idx ? src_idx[t] : t;
 *   if slots[t] >= 0:            K/V pool slot slots[t]  <- k_src/v_src row src
 *   if slots2 && slots2[t] >= 0: K/V pool slot slots2[t] <- the same row
 * A row is [num_kv_heads][head_dim] elements; source element (t, h, d) is at
 * t * src_token_stride + h * src_head_stride + d (K and V share the strides).
 * Negative slots are skipped (padding rows).  Values are copied bit for bit.
 *
 *  k_src, v_src   device, num_src_rows rows (dtype elements)
 *  slots          device int64 [num_tokens]; slots2 and src_idx: device int64
 *                 [num_tokens] or NULL
 *  k_pool, v_pool device pools (layout above)
 *  dtype          element type (only its size matters: 2 or 4 bytes)
 *  err            device int32, required with PKV_FLAG_CHECKED, else ignored
 */
pkv_status kv_scatter_slots(const void* k_src, const void* v_src, int64_t num_tokens,
                            int64_t num_src_rows, int num_kv_heads, int head_dim,
                            int64_t src_token_stride, int64_t src_head_stride,
                            const int64_t* slots, const int64_t* slots2,
                            const int64_t* src_idx, void* k_pool, void* v_pool,
                            int64_t num_pages, int page_size, int64_t page_stride,
                            pkv_dtype dtype, unsigned flags, int32_t* err, void* stream);

/*
 * paged_attention -- attention of packed query rows over K/V read page by page
 * through per-sequence block tables.
 *
 * [VG] Description, Attention: paged attention over per-block rows, 32-token
 * pages, a real-token seq_len separate from the growing key count, padding rows
 * neither attended nor attending and returned as zeros; frame-causal blocks
 * (Cache, frame-causal bullet).  [SP]: the shared-prefix and private-tail
 * calls each return the output and its LSE for an exact merge.
 *
 * Sequence b owns query rows q_indptr[b] .. q_indptr[b+1]-1 and kv_lens[b]
 * keys; logical key j is slot block_table[b * block_table_stride + j / page_size]
 * * page_size + j % page_size.  The first q_real[b] rows are real (q_real NULL:
 * all rows), row i at absolute position kv_lens[b] - q_real[b] + i (the new
 * tokens are the last keys of their row, [VG] Cache, "Exact window" bullet).
 * Query head h reads K/V head h / (num_q_heads / num_kv_heads).
 * Visible keys of real row i: mask NONE: all kv_len; CAUSAL: the first
 * kv_len - q_real + i + 1; BLOCK_CAUSAL (block size causal_block > 0): the
 * first kv_len - q_real + min(q_real, (i / causal_block + 1) * causal_block).
 *
 *   out[r, h, :] = sum_j softmax_j(scale * q[r,h] . k_j) v_j   (visible j)
 *   lse[r, h]    = ln sum_j exp(scale * q[r,h] . k_j)          (natural log)
 * Padding rows and rows with no visible key: out = 0, lse = -inf.
 *
 *  q            device bf16; element (row, h, d) at row*q_token_stride +
 *               h*q_head_stride + d (d contiguous, 16-byte aligned rows)
 *  k_pool/v_pool device bf16 pools; page_size must be 32
 *  block_table  device int32 [batch][block_table_stride]; entries past a
 *               row's last page are never read
 *  kv_lens      device int32 [batch]; q_indptr device int32 [batch + 1];
 *  q_real       device int32 [batch] or NULL
 *  batch, max_q_rows, max_kv_len: HOST upper bounds of batch size, rows per
 *               sequence and keys per sequence; they size the grid, so a call
 *               captured in a CUDA graph stays valid while the device values
 *               stay within them (keys beyond max_kv_len are not attended)
 *  head_dim     64 or 128; num_q_heads % num_kv_heads == 0
 *  scale        softmax scale; <= 0 selects 1/sqrt(head_dim)
 *  out          device [total_rows][num_q_heads][head_dim], bf16 or f32 (dense)
 *  lse          device f32 [total_rows][num_q_heads] or NULL
 *  workspace    device scratch of paged_attention_workspace_size(...) bytes
 *               (256-byte aligned); may be NULL when that size is 0.  It holds
 *               the decode kernel's scheduling state (counters, the planned
 *               order of its work units) and the split partial states; each
 *               call initialises what it uses, so it needs no clearing, but one
 *               workspace must not serve two calls in flight at once
 *  num_splits   key splits per sequence (split-KV); 0 = chosen from the bounds
 *               and the current device's SM count ([SP] commit notes on
 *               generation split-KV: split only when the grid under-fills the
 *               SMs, chunks of at least 512 tokens)
 *
 * The split choice, and with it the workspace size, depends on the SM count
 * of the device current at the call (152 when no device can be queried), so
 * size the workspace with the device current that the call will use.
 */
size_t paged_attention_workspace_size(int batch, int max_q_rows, int num_q_heads,
                                      int num_kv_heads, int head_dim, int max_kv_len,
                                      int num_splits, unsigned flags);

/*
 * pkv_plan_attention -- the launch plan paged_attention makes for these host
 * bounds on a GPU with num_sms SMs (<= 0: the current device's count): which
 * kernel runs (*kernel: a pkv_kernel value), the key splits per sequence and
 * keys per split, and the workspace bytes (what paged_attention_workspace_size
 * returns when num_sms is the current device's).  Host only: reads no device
 * memory and launches nothing.  PKV_ERR_INVALID_ARG for non-positive sizes,
 * head counts that do not divide, or a null output pointer.
 */
typedef enum {
    PKV_KERNEL_NONE = 0,
    PKV_KERNEL_DECODE = 1, /* persistent split-KV decode kernel (SIMT, TMA-fed)   */
    PKV_KERNEL_TILE = 2,   /* tcgen05 / TMEM tile kernel (+ split reduce)         */
    PKV_KERNEL_SIMT = 3,   /* generic kernel (PKV_FLAG_SIMT_ONLY, other shapes)   */
    PKV_KERNEL_TILE_STREAM_K = 4 /* tile kernel on the stream-K schedule
                                    (PKV_FLAG_STREAM_K): planner, persistent
                                    CTAs, merge of split tile pairs */
} pkv_kernel;

pkv_status pkv_plan_attention(int batch, int max_q_rows, int num_q_heads, int num_kv_heads,
                              int head_dim, int max_kv_len, int num_splits, unsigned flags,
                              int num_sms, int* kernel, int* splits, int* split_keys,
                              size_t* workspace_bytes);

pkv_status paged_attention(const void* q, int64_t q_token_stride, int64_t q_head_stride,
                           const void* k_pool, const void* v_pool, int64_t num_pages,
                           int page_size, int64_t page_stride, const int32_t* block_table,
                           int64_t block_table_stride, const int32_t* kv_lens,
                           const int32_t* q_indptr, const int32_t* q_real, int batch,
                           int max_q_rows, int max_kv_len, int num_q_heads, int num_kv_heads,
                           int head_dim, pkv_mask mask, int causal_block, float scale,
                           void* out, pkv_dtype out_dtype, float* lse, void* workspace,
                           size_t workspace_bytes, int num_splits, unsigned flags,
                           int32_t* err, void* stream);

/*
 * rope_write_kv_paged -- rotary embedding of this step's queries (in place)
 * and keys, with the rotated keys and the values written into pool slots, in
 * one launch (the step that precedes paged_attention).
 *
 * [SP] commit notes: RoPE and the K/V write are one kernel (rope_write_kv_paged:
 * Q rotated in place, the rotated K and V written straight to the pool; NeoX
 * RoPE with no or linear scaling; RoPE at the absolute positions, the write at
 * the slot of the table).  NeoX pairs are (x[i], x[i + D/2]):
 *     out[i]       = x[i] cos - x[i + D/2] sin
 *     out[i + D/2] = x[i + D/2] cos + x[i] sin
 * with the angle of token t's position positions[t] and pair i read from the
 * caller's table cos_sin[positions[t]][i] (cos) and [D/2 + i] (sin), so any
 * frequency base or linear scaling lives in the table.
 *
 * For t in [0, num_tokens): every query head of row t is rotated in place
 * (q: bf16, q_token_stride / q_head_stride); if slots[t] >= 0, the rotated K
 * heads of source row t are written to pool slot slots[t] of k_pool and the V
 * heads, unrotated and bit for bit, to v_pool (k_src / v_src are not
 * modified).  Results are rounded to bf16 from fp32 arithmetic.
 *
 *  cos_sin       device f32 [max_position][head_dim], 16-byte aligned
 *  positions     device int64 [num_tokens]; outside [0, max_position) they are
 *                clamped (and flagged with PKV_FLAG_CHECKED)
 *  head_dim      a multiple of 16; q / sources 16-byte aligned, strides
 *                multiples of 8 elements
 */
pkv_status rope_write_kv_paged(void* q, int64_t q_token_stride, int64_t q_head_stride,
                               int num_q_heads, const void* k_src, const void* v_src,
                               int64_t src_token_stride, int64_t src_head_stride,
                               int64_t num_tokens, int num_kv_heads, int head_dim,
                               const int64_t* positions, const float* cos_sin,
                               int64_t max_position, const int64_t* slots, void* k_pool,
                               void* v_pool, int64_t num_pages, int page_size,
                               int64_t page_stride, unsigned flags, int32_t* err, void* stream);

/*
 * copy_kv_slots -- copy whole slot rows from one pool slot to another, in
 * every layer's K and V pool.
 *
 * [VG] Description, Cache (a pool-to-pool copy, copy_kv_slots_, fills the
 * private pages of the causal blocks at commit) and the per-file notes on
 * causalLayout.cu (copies across layers, K/V and heads; sentinel entries).
 * For c in [0, num_copies) with src_slots[c] >= 0 and dst_slots[c] >= 0, and
 * every layer l in [0, num_layers): slot dst_slots[c] of layer l's K pool (at
 * k_pool + l * layer_stride elements) <- its slot src_slots[c]; same for V.
 * A negative entry is a sentinel and is skipped.  Source and destination slots
 * must be disjoint and destinations distinct: otherwise the result is
 * unspecified (copies run concurrently).
 *
 *  dtype      element type (only its size matters); a slot row
 *             (num_kv_heads * head_dim elements) must be a multiple of 16 bytes
 */
pkv_status copy_kv_slots(void* k_pool, void* v_pool, int num_layers, int64_t layer_stride,
                         int64_t num_pages, int page_size, int64_t page_stride, int num_kv_heads,
                         int head_dim, pkv_dtype dtype, const int64_t* src_slots,
                         const int64_t* dst_slots, int64_t num_copies, unsigned flags,
                         int32_t* err, void* stream);

/*
 * causal_layout -- the per-block rows of a forward over exact windows,
 * computed on the device (at commit: nothing is uploaded from the host).
 *
 * [VG] Description, Cache ("Exact window" bullet and the commit bullet: a
 * layout kernel reads the table and rewrites every per-block tensor in place;
 * a pool-to-pool copy fills the private pages) and the review notes on the
 * private pages (committed_private: copies of committed tokens, made at
 * commit; current_private: copies of earlier blocks' tokens of the same
 * forward, written every forward).
 *
 * The cache is one long sequence [fixed region | committed history | staged
 * tokens]: positions [0, pin_tokens) are the fixed region, *committed tokens
 * of history follow (a device int64, advanced by the caller at commit), then
 * the forward's num_staged staged tokens, cut into causal blocks of
 * block_size (the last one shorter).  Block k attends to the fixed region,
 * the window_tokens tokens just before its first token (never reaching into
 * the fixed region) and its own tokens; the window slides with the block.
 * table[lp] is the physical page of logical page lp (slot of logical
 * position p = table[p / 32] * 32 + p % 32); private_pages[k * private_stride
 * + i] are block k's reserved pages.
 *
 * Row k (rows[k * row_stride ...], -1 after its last page): every logical
 * page fully visible to the block that ends at or before the block's first
 * token, by reference and in logical order, then the block's private pages,
 * which hold every other visible token in logical order (the visible tokens
 * of the fixed-region tail, of the window-start page and of the block's
 * start page, then the block's own tokens, which are the row's last keys).
 * kv_lens[k] = the row's keys; q_indptr[k] = the block's first staged token,
 * q_indptr[num_blocks] = num_staged.  Attention over the rows with
 * PKV_MASK_NONE, q_indptr as the query ranges and all rows real then reads
 * exactly each block's window, each key once.
 *
 * Writes that fill the private region:
 *  - staged_slots[t] = the slot of staged token t's own logical position,
 *    staged_slots2[t] = its slot in its block's private region: the two
 *    destinations of kv_scatter_slots for the forward's K/V;
 *  - committed_src/dst[k * PKV_LAYOUT_COMMITTED_PER_BLOCK + c]: slot-to-slot
 *    copies of committed tokens into block k's private region, for
 *    copy_kv_slots at commit (all layers);
 *  - current_src_idx/dst[k * PKV_LAYOUT_CURRENT_PER_BLOCK + c]: earlier
 *    blocks' staged tokens (index into the forward's staged K/V) into block
 *    k's private region, for kv_scatter_slots with src_idx every forward.
 * Unused list entries are -1 (both fields), which both consumers skip.
 *
 *  page_size          32
 *  capacities         committed_capacity >= num_blocks *
 *                     PKV_LAYOUT_COMMITTED_PER_BLOCK, current_capacity >=
 *                     num_blocks * PKV_LAYOUT_CURRENT_PER_BLOCK (checked)
 *  private_stride     block k needs ceil((private tokens) / 32) pages, at most
 *                     ceil((3 * 31 + block_size) / 32): besides its own tokens a
 *                     block copies the visible part of at most three partly
 *                     visible pages
 *  err                nullable device int32: a row longer than row_stride or a
 *                     private region larger than private_stride pages ORs
 *                     PKV_ERRBIT_LEN (the row is truncated, the overflowing
 *                     private tokens skipped); a logical page at or past
 *                     num_logical_pages ORs PKV_ERRBIT_PAGE (its entries -1).
 */
#define PKV_LAYOUT_COMMITTED_PER_BLOCK 93 /* 3 partly visible pages x 31 */
#define PKV_LAYOUT_CURRENT_PER_BLOCK 62  /* 2 partly visible pages x 31 */

pkv_status causal_layout(const int32_t* table, int64_t num_logical_pages, const int64_t* committed,
                         int64_t pin_tokens, int64_t window_tokens, int num_staged, int block_size,
                         const int32_t* private_pages, int private_stride, int page_size,
                         int32_t* rows, int64_t row_stride, int32_t* kv_lens, int32_t* q_indptr,
                         int64_t* staged_slots, int64_t* staged_slots2, int64_t* committed_src,
                         int64_t* committed_dst, int64_t committed_capacity,
                         int64_t* current_src_idx, int64_t* current_dst, int64_t current_capacity,
                         int32_t* err, void* stream);

/*
 * plan_shared_prefix -- group the rows of a batch that share their leading
 * pages, on the device, once per step.
 *
 * [SP] commit notes: rows whose K/V block tables start with identical pages
 * are grouped, each group's shared pages read once and merged with every
 * row's private tail; a device kernel builds each row's page table from its
 * group's shared run onward and its K/V length past the run; the grouping
 * depends on every block-table entry it reads.
 *
 * Row r has kv_lens[r] keys, the last q_indptr[r+1] - q_indptr[r] of them
 * this step's tokens; its whole committed pages are (kv - q) / 32.  Rows with
 * at least one committed page and the same first page form a group (ordered
 * by their first row; members by row index).  A group's shared run is the
 * longest run of leading pages identical in every member, at most the
 * smallest member's committed pages; a row alone has run 0.
 *
 * Outputs (device, caller-allocated, all rewritten; groups g < *num_groups):
 *  group_rows[g * group_row_stride ...]  the run's pages, then every member's
 *                                        tail pages in member order, then -1
 *  run_lens[g]          32 * run pages (0 for g >= *num_groups)
 *  group_indptr[g]      members of group g are perm[group_indptr[g] ..
 *                       group_indptr[g + 1]); batch from *num_groups on
 *  perm[i], group_of[r] rows in group order; a row's group
 *  tail_start[r], tail_lens[r]  first page of row r's tail in its group's row;
 *                       keys of its tail (kv_lens[r] - run_lens[group])
 *  num_groups           device int32
 *
 *  batch          <= 1024 (one CTA plans the whole batch)
 *  max_pages      pages of block_table a row may use (<= block_table_stride)
 *  group_row_stride  >= the longest group row: max_pages * (largest group)
 *                 is always enough; a longer row ORs PKV_ERRBIT_LEN into *err
 *                 (nullable) and is truncated
 */
pkv_status plan_shared_prefix(const int32_t* block_table, int64_t block_table_stride,
                              const int32_t* kv_lens, const int32_t* q_indptr, int batch,
                              int max_pages, int32_t* group_rows, int64_t group_row_stride,
                              int32_t* run_lens, int32_t* group_indptr, int32_t* perm,
                              int32_t* group_of, int32_t* tail_start, int32_t* tail_lens,
                              int32_t* num_groups, int32_t* err, void* stream);

/*
 * shared_prefix_attention -- attention of a grouped batch (plan_shared_prefix)
 * in one launch: every query token attends to its group's shared run and its
 * own tail in a single online softmax, each group's shared pages read once
 * per group (and K/V head) instead of once per row; no merge step.
 *
 * [SP] commit notes: n-sample rows grouped by identical leading pages, the
 * shared pages read once and merged with every row's private tail; a fused
 * kernel does prefix, tail and merge for up to 16 query tokens per row (so
 * speculative verification steps of K draft tokens + 1 are served too).
 * Here the merge is exact by construction: the run and the tail are two key
 * ranges of one softmax.
 *
 * Row r's query tokens are q[q_indptr[r] .. q_indptr[r+1]) (the row's last
 * keys); token i of ql attends to keys [0, run_lens[g]) of its group row g
 * and to [32 * tail_start[r], 32 * tail_start[r] + tail_lens[r] - ql + i + 1)
 * (causal inside the tail).  Outputs are written at the tokens' own
 * positions: out [tokens][num_q_heads][head_dim], lse [tokens][num_q_heads]
 * (natural log; nullable).
 *
 *  group_rows ... num_groups   as written by plan_shared_prefix (device)
 *  batch            rows of the plan (= group slots)
 *  max_q_len        >= every row's query tokens (<= 16 is what the pages serve)
 *  max_group_tokens >= the query tokens of any group (sizes the grid)
 *  max_group_keys   >= the longest group row in keys (sizes the key splits)
 *  head_dim 128, num_q_heads / num_kv_heads in {1, 2, 4, 8, 16} (tensor-core
 *  tiles); other shapes return PKV_ERR_UNSUPPORTED.
 *  workspace        shared_prefix_attention_workspace_size bytes (256-aligned)
 *                   for the key splits it chooses; may be 0 bytes
 */
size_t shared_prefix_attention_workspace_size(int batch, int max_q_len, int max_group_tokens,
                                              int max_group_keys, int num_q_heads,
                                              int num_kv_heads, int head_dim, int num_splits);
pkv_status shared_prefix_attention(const void* q, int64_t q_token_stride, int64_t q_head_stride,
                                   const void* k_pool, const void* v_pool, int64_t num_pages,
                                   int page_size, int64_t page_stride, const int32_t* group_rows,
                                   int64_t group_row_stride, const int32_t* run_lens,
                                   const int32_t* group_indptr, const int32_t* perm,
                                   const int32_t* tail_start, const int32_t* tail_lens,
                                   const int32_t* num_groups, const int32_t* q_indptr, int batch,
                                   int max_q_len, int max_group_tokens, int max_group_keys,
                                   int num_q_heads, int num_kv_heads, int head_dim, float scale,
                                   void* out, pkv_dtype out_dtype, float* lse, void* workspace,
                                   size_t workspace_bytes, int num_splits, unsigned flags,
                                   int32_t* err, void* stream);

/*
 * paged_attention_no_alloc -- paged_attention for callers that cannot allocate.
 *
 * The pages describe no such entry point; it exists for callers that have no
 * workspace to give: code enqueuing work during CUDA-graph capture (where
 * cudaMalloc is not allowed), servers that fix device memory at start-up and
 * allow no allocator calls per request, and hosts that pass only input and
 * output pointers.  Same arguments, results and errors as paged_attention,
 * without workspace / workspace_bytes: the scratch is a device array inside
 * the library of PKV_NO_ALLOC_SCRATCH_BYTES (32 MiB), present on every GPU
 * that loads the library until the process exits.
 *
 *  - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *  - A call needing more scratch than the array holds (what
 *    paged_attention_workspace_size reports for the same arguments) returns
 *    PKV_ERR_WORKSPACE with a message, before anything is enqueued.
 *  - The first call with a given device current looks up the array's address
 *    on that device; make that first call before any stream capture.  The
 *    address is looked up again when that device's context has changed since
 *    (a cudaDeviceReset in between), so such a call must also come before
 *    any capture.
 *  - Every call on a device uses the same array and leaves its contents
 *    behind (what must start at zero is cleared by each call), so calls that
 *    can overlap on the GPU (unordered streams) race and must be serialised.
 */
#define PKV_NO_ALLOC_SCRATCH_BYTES ((size_t)32 << 20)

pkv_status paged_attention_no_alloc(const void* q, int64_t q_token_stride, int64_t q_head_stride,
                                    const void* k_pool, const void* v_pool, int64_t num_pages,
                                    int page_size, int64_t page_stride,
                                    const int32_t* block_table, int64_t block_table_stride,
                                    const int32_t* kv_lens, const int32_t* q_indptr,
                                    const int32_t* q_real, int batch, int max_q_rows,
                                    int max_kv_len, int num_q_heads, int num_kv_heads,
                                    int head_dim, pkv_mask mask, int causal_block, float scale,
                                    void* out, pkv_dtype out_dtype, float* lse, int num_splits,
                                    unsigned flags, int32_t* err, void* stream);

/*
 * merge_attn_states -- exact merge of two attention states over disjoint key
 * sets (shared-prefix state with private-tail state).
 *
 * [SP] commit notes: the prefix and the tail attention each return an output
 * and its LSE and one merge joins them; an empty run has LSE -inf.  Per (row,
 * head):  m = max(La, Lb), wa = e^(La-m), wb = e^(Lb-m),
 *         out = (wa*Oa + wb*Ob) / (wa + wb),  lse_out = m + ln(wa + wb);
 * both empty (-inf): out = 0, lse_out = -inf.
 *
 *  o_a, o_b     device [rows][num_heads][head_dim] of in_dtype (bf16 or f32)
 *  lse_a, lse_b device f32 [rows][num_heads] (natural log)
 *  o_out        device [rows][num_heads][head_dim] of out_dtype; may alias o_a
 *  lse_out      device f32 or NULL; may alias lse_a
 *  head_dim     a multiple of 4, at most 512
 */
pkv_status merge_attn_states(const void* o_a, const float* lse_a, const void* o_b,
                             const float* lse_b, pkv_dtype in_dtype, int64_t rows,
                             int num_heads, int head_dim, void* o_out, pkv_dtype out_dtype,
                             float* lse_out, void* stream);

/*
 * rotate_rows -- rotate every row of a 2-D buffer left in place.
 *
 * [VG] Description, Cache: eviction is an in-place rotation on the device (op
 * rotate_rows_), and the per-file notes on rotateRows: supported element sizes,
 * shifts, strided rows, no-op cases.  For every row r:
 *     x[r][c] <- x[r][(c + shift) mod cols]      (c in [0, cols))
 * i.e. torch.roll(row, -shift).  Any shift (negative, or beyond cols) is taken
 * modulo cols.  Elements are opaque groups of elem_size bytes, elem_size in
 * {1, 2, 4, 8, 16}; row r starts at byte r * row_stride * elem_size.  rows == 0
 * or cols <= 1: no launch.  Rows must not overlap.
 */
pkv_status rotate_rows(void* x, int64_t rows, int64_t cols, int64_t row_stride,
                       int elem_size, int64_t shift, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
