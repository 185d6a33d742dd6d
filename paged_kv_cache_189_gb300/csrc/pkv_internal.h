// pkv_internal.h -- host-side launcher interfaces between the C-ABI layer
// (pkv_api.cpp: validation, dispatch, tensor maps) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Record a validation message for pkv_last_error() and return the status.
pkv_status report(pkv_status status, const char* message);

// ---------------------------- scatter --------------------------------------
struct ScatterArgs {
    const void* k_src;
    const void* v_src;
    int64_t num_tokens, num_src_rows;
    int num_kv_heads, head_dim, elem_size;
    int64_t src_token_stride, src_head_stride;  // elements
    const int64_t* slots;
    const int64_t* slots2;
    const int64_t* src_idx;
    void* k_pool;
    void* v_pool;
    int64_t num_pages;
    int page_size;
    int64_t page_stride;  // elements
    bool checked;
    int32_t* err;
};
cudaError_t launch_scatter(const ScatterArgs& a, cudaStream_t s);

// ---------------------------- rope + paged write -----------------------------
struct RopeArgs {
    void* q;
    int64_t q_token_stride, q_head_stride;
    int num_q_heads;
    const void* k_src;
    const void* v_src;
    int64_t src_token_stride, src_head_stride;
    int64_t num_tokens;
    int num_kv_heads, head_dim;
    const int64_t* positions;
    const float* cos_sin;  // [max_position][head_dim]: cos of the D/2 pairs, then their sin
    int64_t max_position;
    const int64_t* slots;
    void* k_pool;
    void* v_pool;
    int64_t num_pages;
    int page_size;
    int64_t page_stride;
    bool checked;
    int32_t* err;
};
cudaError_t launch_rope_write(const RopeArgs& a, cudaStream_t s);

// ---------------------------- pool-to-pool slot copy --------------------------
struct PlanArgs {
    const int32_t* block_table;
    int64_t block_table_stride;
    const int32_t* kv_lens;
    const int32_t* q_indptr;
    int batch, max_pages;
    int32_t* group_rows;
    int64_t group_row_stride;
    int32_t* run_lens;
    int32_t* group_indptr;
    int32_t* perm;
    int32_t* group_of;
    int32_t* tail_start;
    int32_t* tail_lens;
    int32_t* num_groups;
    int32_t* err;
};
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s);

struct LayoutArgs {
    const int32_t* table;
    int64_t num_logical_pages;
    const int64_t* committed;  // device scalar
    int64_t pin, window;
    int num_staged, block_size, num_blocks;
    const int32_t* private_pages;
    int private_stride;
    int32_t* rows;
    int64_t row_stride;
    int32_t* kv_lens;
    int32_t* q_indptr;
    int64_t* staged_slots;
    int64_t* staged_slots2;
    int64_t* com_src;
    int64_t* com_dst;
    int64_t* cur_src;
    int64_t* cur_dst;
    int32_t* err;
};
cudaError_t launch_causal_layout(const LayoutArgs& a, cudaStream_t s);

struct CopySlotsArgs {
    void* k_pool;
    void* v_pool;
    int num_layers;
    int64_t layer_stride;  // elements between layers' pools
    int64_t num_pages;
    int page_size;
    int64_t page_stride;
    int num_kv_heads, head_dim, elem_size;
    const int64_t* src_slots;
    const int64_t* dst_slots;
    int64_t num_copies;
    bool checked;
    int32_t* err;
};
cudaError_t launch_copy_slots(const CopySlotsArgs& a, cudaStream_t s);

// ---------------------------- rotate ---------------------------------------
// Rotation in units of `unit` bytes (1, 2, 4, 8 or 16); cols, shift and
// row_stride are already expressed in units, 0 < shift < cols.
cudaError_t launch_rotate(void* x, int64_t rows, int64_t cols, int64_t row_stride, int unit,
                          int64_t shift, cudaStream_t s);

// ---------------------------- merge ----------------------------------------
cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b,
                         const float* lse_b, bool in_f32, int64_t rows, int num_heads,
                         int head_dim, void* o_out, bool out_f32, float* lse_out,
                         cudaStream_t s);

// ---------------------------- attention ------------------------------------
// Everything the attention kernels need, resolved on the host.
struct AttnParams {
    const void* q;
    int64_t q_token_stride, q_head_stride;
    const void* k_pool;
    const void* v_pool;
    int64_t num_pages;
    int64_t page_stride;
    const int32_t* block_table;
    int64_t block_table_stride;
    const int32_t* kv_lens;
    const int32_t* q_indptr;
    const int32_t* q_real;
    int batch, max_q_rows, max_kv_len;
    int num_q_heads, num_kv_heads, head_dim;
    int mask, causal_block;
    float scale_log2;  // softmax scale * log2(e)
    void* out;
    bool out_f32;
    float* lse;
    int num_splits;
    int split_keys;    // keys per split (multiple of the key tile)
    float* ws_o;       // [rows_bound][Hq][splits][D] partial outputs (splits > 1)
    float* ws_lse;     // [rows_bound][Hq][splits]
    int* ws_counters;  // decode: [0] unit ticket, [1 + b*Hkv + h] finished splits
    bool planned;      // decode: units taken from the planned order (else split-major)
    bool checked;
    int32_t* err;
    // two-tile kernel, stream-K schedule (sk_ctas > 0): one persistent CTA per
    // SM, each taking a contiguous range of the units' key tiles (a unit = a
    // tile pair of one sequence and K/V head); units split between CTAs leave
    // partial states in per-CTA fragment slots that a reduce merges
    int sk_ctas;          // persistent CTAs (the grid)
    int sk_units;         // tile pairs x K/V heads x sequences
    int sk_tiles_x;       // tile pairs per sequence
    int sk_dp;            // the first sk_dp units run whole, unit c on CTA c (0 or sk_ctas)
    int* sk_unit_off;     // [units - sk_dp + 1] weighted key-tile offsets of the shared units
    int* sk_cta_off;      // [ctas + 1] each CTA's share of them (planner)
    int4* sk_dir;         // [ctas][2] partial fragments: (unit, j0, j1, key tiles of the unit)
    float* sk_frag_o;     // [ctas][2][256 rows][D] normalised partial outputs
    float* sk_frag_lse;   // [ctas][2][256 rows] their LSEs (natural log)
    // decode kernel, PKV_FLAG_TEST_WAIT_TIMEOUT: consumers wait on a barrier
    // nothing completes (short limit) and the producer's ring waits are short
    bool test_wait_timeout;
    // one-tile kernel: block z takes the (z / num_splits)-th sequence by key
    // count, longest first, so that a grid of several waves starts with them
    bool order_by_keys;
    // shared-prefix groups (grouped tile mode, grp_perm != nullptr): block_table
    // holds the group rows, batch is the number of group slots, q_indptr the
    // original rows' query tokens; kv_lens and q_real are not used
    const int32_t* grp_run_lens;    // [groups] keys of each group's shared run
    const int32_t* grp_indptr;      // [groups + 1] members in grp_perm
    const int32_t* grp_perm;        // rows in group order
    const int32_t* grp_tail_start;  // [rows] first page of the row's tail in its group row
    const int32_t* grp_tail_lens;   // [rows] keys of the row's tail
    const int32_t* grp_num_groups;  // device scalar
    int grp_max_tokens;             // host bound on the query tokens of one group
};

// Decode kernel (one query row per sequence), split-KV, SIMT; K/V pages
// arrive by TMA.  tmap_k / tmap_v are CUtensorMap (128 bytes each).
cudaError_t launch_decode(const AttnParams& p, const void* tmap_k, const void* tmap_v,
                          cudaStream_t s);
bool decode_supported(int head_dim, int group);
size_t decode_sched_bytes(int batch, int num_kv_heads, int splits);  // scheduling region of the workspace

// Generic SIMT kernel: any rows, masks, group sizes; no splits.  A slow
// cross-check of the fast kernels and the path for shapes they do not cover.
cudaError_t launch_attn_simt(const AttnParams& p, cudaStream_t s);

// Grouped mode of the one-tile tensor-core kernel: one CTA per (group, tile of
// the group's query tokens, K/V head); each row attends to its group's shared
// run and its own tail in one online softmax.
cudaError_t launch_attn_tc_grouped(const AttnParams& p, const void* tmap_k, const void* tmap_v,
                                   cudaStream_t s);

// Tensor-core tile kernel (tcgen05 / TMEM, TMA-fed) for many query rows.
cudaError_t launch_attn_tc(const AttnParams& p, const void* tmap_q, const void* tmap_k,
                           const void* tmap_v, cudaStream_t s);
bool attn_tc_supported(int head_dim, int group);
int attn_tc_rows_per_tile(int group);  // query tokens per 128-row tile

// n-way merge of split partials into out / lse.
cudaError_t launch_split_reduce(const AttnParams& p, cudaStream_t s);

// Stream-K schedule of the two-tile kernel: whether a call takes it, and the
// workspace it needs (unit offsets, fragment directory, fragments).
bool attn_tc_two_tile(int max_q_rows, int group);
size_t attn_tc_sk_bytes(int units, int ctas, int head_dim);

}  // namespace pkv
