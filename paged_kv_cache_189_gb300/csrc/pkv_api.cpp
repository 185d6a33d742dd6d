// pkv_api.cpp -- the C ABI: argument validation, kernel choice, split-KV
// planning, TMA tensor maps, status strings.  Nothing here touches device
// memory; every check runs on the host before anything is enqueued.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

thread_local std::string g_last_error;

pkv_status fail(pkv_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pkv_status fail(pkv_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

pkv_status ok() {
    g_last_error.clear();
    return PKV_OK;
}

pkv_status from_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

int elem_size(pkv_dtype d) {
    switch (d) {
        case PKV_BF16: return 2;
        case PKV_F16: return 2;
        case PKV_F32: return 4;
    }
    return 0;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library needs no link-time dependency on libcuda.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// One K (or V) pool as a 4-D tensor {D, Hkv, page slots, pages}; a box is
// 64 columns x 1 head x 32 slots x 1 page (4 KiB), 128-byte swizzled.
pkv_status make_pool_map(CUtensorMap* m, const void* base, int D, int Hkv, int page_size,
                         int64_t num_pages, int64_t page_stride) {
    auto fn = encode_fn();
    if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                          static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(num_pages)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(Hkv) * D * 2,
                             static_cast<cuuint64_t>(page_stride) * 2};
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(page_size), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled(pool) failed: %d", (int)r);
    return PKV_OK;
}

enum class Kernel { kNone, kDecode, kSimt, kTile };

struct Plan {
    Kernel kernel = Kernel::kNone;
    int splits = 1;
    int split_keys = 0;
    size_t ws_bytes = 0;
    // stream-K schedule of the two-tile kernel (sk_ctas > 0)
    int sk_ctas = 0, sk_units = 0, sk_tiles_x = 0;
};


constexpr int kDecodeSplitKeys = 512;  // 16 pages: the pages' minimum split of 512 tokens
constexpr int kDefaultSMs = 152;       // GB300: planned for when no device can be queried
constexpr int kTileKeys = 128;         // key tile of the tensor-core kernel

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// SM count of the current device, cached per device; kDefaultSMs when no
// device can be queried (a host without a GPU sizing workspaces).  The split
// choice and the workspace size depend on it, so a workspace sized with one
// device current fits the calls made with that device current.
int current_device_sms() {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return kDefaultSMs;
    }
    if (dev >= 0 && dev < kMaxDev) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        return kDefaultSMs;
    }
    if (dev >= 0 && dev < kMaxDev) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

// Key splits of the tile kernels: with at most two waves of CTAs the last
// wave can leave most SMs idle (every CTA of an unmasked or long causal row
// runs about as long as the others), so the keys are split to the count that
// minimises waves / splits, plus ~2 % of a CTA per split for the partial
// states and their merge, when that saves at least 10 %; splits keep >= 512
// keys.  More CTAs than that are balanced by the block scheduler.
int tile_splits(int64_t ctas, int max_keys, int num_splits, int sms) {
    if (num_splits > 0) return num_splits;
    int s = 1;
    if (ctas <= 2 * static_cast<int64_t>(sms)) {
        const int s_max = std::max(1, std::min(8, max_keys / 512));
        const double unsplit = static_cast<double>((ctas + sms - 1) / sms);
        double best = unsplit;
        for (int c = 2; c <= s_max; ++c) {
            const double waves = static_cast<double>((ctas * c + sms - 1) / sms);
            const double cost = waves / c + 0.02 * c;
            if (cost < best - 1e-9) {
                best = cost;
                s = c;
            }
        }
        if (best > 0.9 * unsplit) s = 1;
    }
    return s;
}


Plan plan_attention(int batch, int max_q_rows, int Hq, int Hkv, int D, int max_kv_len,
                    int num_splits, unsigned flags, int sms) {
    Plan pl;
    const int G = Hkv > 0 ? Hq / Hkv : 0;
    // tensor-core tiles for several rows per sequence, and for single-row
    // decode with a head group the decode kernel does not take (8 or 16 query
    // heads per K/V head: one token x G heads fills a tile held four times)
    const bool decode_kernel_takes = max_q_rows == 1 && pkv::decode_supported(D, G);
    if (!(flags & PKV_FLAG_SIMT_ONLY) && max_q_rows >= 1 && !decode_kernel_takes &&
        pkv::attn_tc_supported(D, G)) {
        // tensor-core tiles, one CTA per tile (two tiles when a sequence has
        // more rows than one holds), keys split as tile_splits chooses.
        pl.kernel = Kernel::kTile;
        const int tq = pkv::attn_tc_rows_per_tile(G);
        const int rows_per_cta = max_q_rows > tq ? 2 * tq : tq;
        const int tiles_x = (max_q_rows + rows_per_cta - 1) / rows_per_cta;
        const int64_t ctas = static_cast<int64_t>(tiles_x) * Hkv * batch;
        // stream-K (on request, PKV_FLAG_STREAM_K): one persistent CTA per SM,
        // each running one whole first-wave tile pair and then a contiguous
        // share of the remaining pairs' key tiles.  Not the default: on the
        // video step's 280 pairs (1.84 waves) it measured 0.323 ms against
        // 0.280 ms for this grid -- identical pairs run 129-155 us on
        // different SMs, which static shares cannot absorb and the grid's
        // second wave, scheduled as SMs free up, does; every share also
        // starts and ends a segment (Q reload, pipeline refill, the merge).
        const int64_t key_tiles = (static_cast<int64_t>(max_kv_len) + kTileKeys - 1) / kTileKeys;
        if (pkv::attn_tc_two_tile(max_q_rows, G) && num_splits == 0 && (flags & PKV_FLAG_STREAM_K) &&
            !(flags & PKV_FLAG_TILE_GRID) && sms <= 1023 && ctas * key_tiles < (1ll << 31) && key_tiles > 0) {
            pl.sk_ctas = sms;
            pl.sk_units = static_cast<int>(ctas);
            pl.sk_tiles_x = tiles_x;
            pl.splits = 1;
            pl.split_keys = static_cast<int>(key_tiles * kTileKeys);
            pl.ws_bytes = pkv::attn_tc_sk_bytes(pl.sk_units, pl.sk_ctas, D);
            return pl;
        }
        const int s = tile_splits(ctas, max_kv_len, num_splits, sms);
        const int per = (max_kv_len + s - 1) / std::max(s, 1);
        pl.split_keys = std::max(kTileKeys, (per + kTileKeys - 1) / kTileKeys * kTileKeys);
        pl.splits = std::max(1, (max_kv_len + pl.split_keys - 1) / pl.split_keys);
        if (pl.splits > 1) {
            const size_t states = static_cast<size_t>(batch) * max_q_rows * Hq * pl.splits;
            pl.ws_bytes = round_up(states * D * sizeof(float), 256) + round_up(states * sizeof(float), 256);
        }
        return pl;
    }
    if ((flags & PKV_FLAG_SIMT_ONLY) || max_q_rows != 1 || !pkv::decode_supported(D, G)) {
        pl.kernel = Kernel::kSimt;
        return pl;
    }
    pl.kernel = Kernel::kDecode;
    // Work units (split, K/V head, sequence) are handed out dynamically to the
    // persistent CTAs (3 per SM); each unit ends with a merge of its warps'
    // states, so units should be long, but numerous enough to balance ragged
    // lengths: aim for ~6 units per resident CTA at the host's length bound,
    // never below the pages' minimum split of 512 keys, and at least 1024 keys
    // while that still leaves one unit per resident CTA (short rows, e.g. the
    // private tails of shared-prefix rows, pay the per-unit cost otherwise).
    int keys = kDecodeSplitKeys;
    if (num_splits > 0) {
        const int per = (max_kv_len + num_splits - 1) / num_splits;
        keys = std::max(32, (per + 31) / 32 * 32);
    } else {
        const int64_t resident = 3 * static_cast<int64_t>(sms);
        const int64_t pairs = static_cast<int64_t>(batch) * Hkv;
        const int64_t target_units = 6 * resident;
        const int64_t per = (static_cast<int64_t>(max_kv_len) * pairs + target_units - 1) / target_units;
        const int64_t fill = (static_cast<int64_t>(max_kv_len) * pairs + resident - 1) / resident;
        const int64_t lo = std::max<int64_t>(kDecodeSplitKeys, std::min<int64_t>(1024, fill));
        keys = static_cast<int>((std::max<int64_t>(lo, per) + 31) / 32 * 32);
    }
    pl.split_keys = keys;
    pl.splits = std::max(1, (max_kv_len + keys - 1) / keys);
    // [scheduling: counters, unit order][partial outputs][partial LSEs]
    pl.ws_bytes = round_up(pkv::decode_sched_bytes(batch, Hkv, pl.splits), 256);
    if (pl.splits > 1) {
        const size_t states = static_cast<size_t>(batch) * max_q_rows * Hq * pl.splits;
        pl.ws_bytes += round_up(states * D * sizeof(float), 256) + round_up(states * sizeof(float), 256);
    }
    return pl;
}

}  // namespace

pkv_status pkv::report(pkv_status status, const char* message) {
    g_last_error = message;
    return status;
}

extern "C" {

const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    }
    return "PKV_UNKNOWN_STATUS";
}

const char* pkv_last_error(void) { return g_last_error.c_str(); }

pkv_status kv_scatter_slots(const void* k_src, const void* v_src, int64_t num_tokens,
                            int64_t num_src_rows, int num_kv_heads, int head_dim,
                            int64_t src_token_stride, int64_t src_head_stride,
                            const int64_t* slots, const int64_t* slots2, const int64_t* src_idx,
                            void* k_pool, void* v_pool, int64_t num_pages, int page_size,
                            int64_t page_stride, pkv_dtype dtype, unsigned flags, int32_t* err,
                            void* stream) {
    const int esz = elem_size(dtype);
    if (esz == 0) return fail(PKV_ERR_INVALID_ARG, "scatter: unknown dtype %d", (int)dtype);
    if (num_tokens < 0 || num_src_rows < 0 || num_kv_heads < 0 || head_dim < 0 || num_pages < 0)
        return fail(PKV_ERR_INVALID_ARG, "scatter: negative size");
    if (num_tokens == 0 || num_kv_heads == 0 || head_dim == 0) return ok();
    if (!k_src || !v_src || !slots || !k_pool || !v_pool)
        return fail(PKV_ERR_INVALID_ARG, "scatter: null pointer");
    if (page_size <= 0) return fail(PKV_ERR_INVALID_ARG, "scatter: page_size must be positive");
    if (page_stride < static_cast<int64_t>(page_size) * num_kv_heads * head_dim)
        return fail(PKV_ERR_INVALID_ARG, "scatter: page_stride %lld smaller than a page",
                    (long long)page_stride);
    if (src_token_stride < 0 || src_head_stride < 0)
        return fail(PKV_ERR_INVALID_ARG, "scatter: negative source stride");
    if (!src_idx && num_src_rows < num_tokens)
        return fail(PKV_ERR_INVALID_ARG, "scatter: %lld source rows for %lld tokens",
                    (long long)num_src_rows, (long long)num_tokens);
    if (!aligned(k_src, esz) || !aligned(v_src, esz) || !aligned(k_pool, esz) || !aligned(v_pool, esz))
        return fail(PKV_ERR_INVALID_ARG, "scatter: pointers not aligned to the element size");
    if ((flags & PKV_FLAG_CHECKED) && !err)
        return fail(PKV_ERR_INVALID_ARG, "scatter: checked mode needs an error flag");
    pkv::ScatterArgs a{k_src, v_src, num_tokens, num_src_rows, num_kv_heads, head_dim, esz,
                       src_token_stride, src_head_stride, slots, slots2, src_idx, k_pool, v_pool,
                       num_pages, page_size, page_stride, (flags & PKV_FLAG_CHECKED) != 0, err};
    return from_cuda(pkv::launch_scatter(a, static_cast<cudaStream_t>(stream)), "scatter launch");
}

size_t paged_attention_workspace_size(int batch, int max_q_rows, int num_q_heads,
                                      int num_kv_heads, int head_dim, int max_kv_len,
                                      int num_splits, unsigned flags) {
    if (batch <= 0 || max_q_rows <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_kv_len < 0)
        return 0;
    return plan_attention(batch, max_q_rows, num_q_heads, num_kv_heads, head_dim, max_kv_len,
                          num_splits, flags, current_device_sms())
        .ws_bytes;
}

pkv_status pkv_plan_attention(int batch, int max_q_rows, int num_q_heads, int num_kv_heads,
                              int head_dim, int max_kv_len, int num_splits, unsigned flags,
                              int num_sms, int* kernel, int* splits, int* split_keys,
                              size_t* workspace_bytes) {
    if (batch <= 0 || max_q_rows <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_kv_len < 0 ||
        num_splits < 0 || num_q_heads % num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "plan: sizes must be positive, heads a multiple of K/V heads");
    if (!kernel || !splits || !split_keys || !workspace_bytes)
        return fail(PKV_ERR_INVALID_ARG, "plan: null output pointer");
    const Plan pl = plan_attention(batch, max_q_rows, num_q_heads, num_kv_heads, head_dim, max_kv_len,
                                   num_splits, flags, num_sms > 0 ? num_sms : current_device_sms());
    *kernel = pl.kernel == Kernel::kDecode ? static_cast<int>(PKV_KERNEL_DECODE)
            : pl.kernel == Kernel::kTile && pl.sk_ctas > 0 ? static_cast<int>(PKV_KERNEL_TILE_STREAM_K)
            : pl.kernel == Kernel::kTile   ? static_cast<int>(PKV_KERNEL_TILE)
            : pl.kernel == Kernel::kSimt   ? static_cast<int>(PKV_KERNEL_SIMT)
                                           : static_cast<int>(PKV_KERNEL_NONE);
    *splits = pl.splits;
    *split_keys = pl.split_keys;
    *workspace_bytes = pl.ws_bytes;
    return ok();
}

pkv_status paged_attention(const void* q, int64_t q_token_stride, int64_t q_head_stride,
                           const void* k_pool, const void* v_pool, int64_t num_pages,
                           int page_size, int64_t page_stride, const int32_t* block_table,
                           int64_t block_table_stride, const int32_t* kv_lens,
                           const int32_t* q_indptr, const int32_t* q_real, int batch,
                           int max_q_rows, int max_kv_len, int num_q_heads, int num_kv_heads,
                           int head_dim, pkv_mask mask, int causal_block, float scale, void* out,
                           pkv_dtype out_dtype, float* lse, void* workspace,
                           size_t workspace_bytes, int num_splits, unsigned flags, int32_t* err,
                           void* stream) {
    if (batch < 0 || max_q_rows < 0 || max_kv_len < 0 || num_q_heads < 0 || num_kv_heads < 0 ||
        num_pages < 0 || num_splits < 0)
        return fail(PKV_ERR_INVALID_ARG, "attention: negative size");
    if (batch == 0 || max_q_rows == 0 || num_q_heads == 0) return ok();
    if (num_kv_heads == 0 || num_q_heads % num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "attention: %d query heads is not a multiple of %d K/V heads",
                    num_q_heads, num_kv_heads);
    if (!q || !k_pool || !v_pool || !block_table || !kv_lens || !q_indptr || !out)
        return fail(PKV_ERR_INVALID_ARG, "attention: null pointer");
    if (page_size != 32)
        return fail(PKV_ERR_UNSUPPORTED, "attention: page_size %d (only 32-token pages)", page_size);
    if (head_dim != 64 && head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "attention: head_dim %d (64 or 128)", head_dim);
    if (mask != PKV_MASK_NONE && mask != PKV_MASK_CAUSAL && mask != PKV_MASK_BLOCK_CAUSAL)
        return fail(PKV_ERR_INVALID_ARG, "attention: unknown mask %d", (int)mask);
    if (mask == PKV_MASK_BLOCK_CAUSAL && causal_block <= 0)
        return fail(PKV_ERR_INVALID_ARG, "attention: block-causal mask needs causal_block > 0");
    if (out_dtype != PKV_BF16 && out_dtype != PKV_F32)
        return fail(PKV_ERR_UNSUPPORTED, "attention: output dtype must be bf16 or f32");
    if (batch > 65535 || num_kv_heads > 65535)
        return fail(PKV_ERR_UNSUPPORTED, "attention: batch or K/V heads above 65535");
    if (page_stride < static_cast<int64_t>(page_size) * num_kv_heads * head_dim || page_stride % 8)
        return fail(PKV_ERR_INVALID_ARG,
                    "attention: page_stride %lld must cover a page and be a multiple of 8",
                    (long long)page_stride);
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || q_token_stride % 8 ||
        q_head_stride % 8 || q_token_stride < 0 || q_head_stride < 0)
        return fail(PKV_ERR_INVALID_ARG,
                    "attention: q / pools must be 16-byte aligned with strides multiple of 8");
    if (!aligned(out, 16) || (lse && !aligned(lse, 4)))
        return fail(PKV_ERR_INVALID_ARG, "attention: output must be 16-byte aligned");
    const int64_t pages_needed = (static_cast<int64_t>(max_kv_len) + page_size - 1) / page_size;
    if (block_table_stride < pages_needed)
        return fail(PKV_ERR_INVALID_ARG, "attention: block_table_stride %lld < %lld pages for max_kv_len",
                    (long long)block_table_stride, (long long)pages_needed);
    if ((flags & (PKV_FLAG_CHECKED | PKV_FLAG_TEST_WAIT_TIMEOUT)) && !err)
        return fail(PKV_ERR_INVALID_ARG, "attention: checked mode and the wait test need an error flag");

    const Plan pl = plan_attention(batch, max_q_rows, num_q_heads, num_kv_heads, head_dim,
                                   max_kv_len, num_splits, flags, current_device_sms());
    if (pl.ws_bytes > 0) {
        if (!workspace || workspace_bytes < pl.ws_bytes || !aligned(workspace, 256))
            return fail(PKV_ERR_WORKSPACE, "attention: workspace needs %zu bytes, 256-byte aligned",
                        pl.ws_bytes);
    }
    if ((flags & PKV_FLAG_TEST_WAIT_TIMEOUT) && pl.kernel != Kernel::kDecode)
        return fail(PKV_ERR_UNSUPPORTED, "attention: the wait test runs on the decode kernel only");

    pkv::AttnParams p{};
    p.q = q;
    p.q_token_stride = q_token_stride;
    p.q_head_stride = q_head_stride;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.num_pages = num_pages;
    p.page_stride = page_stride;
    p.block_table = block_table;
    p.block_table_stride = block_table_stride;
    p.kv_lens = kv_lens;
    p.q_indptr = q_indptr;
    p.q_real = q_real;
    p.batch = batch;
    p.max_q_rows = max_q_rows;
    p.max_kv_len = max_kv_len;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.mask = static_cast<int>(mask);
    p.causal_block = causal_block;
    const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    p.scale_log2 = sc * 1.4426950408889634f;
    p.out = out;
    p.out_f32 = out_dtype == PKV_F32;
    p.lse = lse;
    p.num_splits = pl.splits;
    p.split_keys = pl.split_keys;
    p.checked = (flags & PKV_FLAG_CHECKED) != 0;
    p.err = err;
    p.test_wait_timeout = (flags & PKV_FLAG_TEST_WAIT_TIMEOUT) != 0;
    if (pl.kernel == Kernel::kTile && static_cast<int64_t>(batch) * pl.splits > 65535)
        return fail(PKV_ERR_UNSUPPORTED, "attention: batch x key splits above 65535");
    if (pl.kernel == Kernel::kTile && pl.splits > 1) {
        const size_t states = static_cast<size_t>(batch) * max_q_rows * num_q_heads * pl.splits;
        p.ws_o = static_cast<float*>(workspace);
        p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                            round_up(states * head_dim * sizeof(float), 256));
    }
    if (pl.kernel == Kernel::kTile && pl.sk_ctas > 0) {
        // [unit offsets][fragment directory][fragment LSEs][fragment outputs]
        char* w = static_cast<char*>(workspace);
        p.sk_ctas = pl.sk_ctas;
        p.sk_units = pl.sk_units;
        p.sk_tiles_x = pl.sk_tiles_x;
        p.sk_dp = pl.sk_units >= pl.sk_ctas ? pl.sk_ctas : 0;
        p.sk_unit_off = reinterpret_cast<int*>(w);
        w += round_up((static_cast<size_t>(pl.sk_units) + 1) * sizeof(int), 256);
        p.sk_cta_off = reinterpret_cast<int*>(w);
        w += round_up((static_cast<size_t>(pl.sk_ctas) + 1) * sizeof(int), 256);
        p.sk_dir = reinterpret_cast<int4*>(w);
        w += round_up(2 * static_cast<size_t>(pl.sk_ctas) * 16, 256);
        p.sk_frag_lse = reinterpret_cast<float*>(w);
        w += round_up(2 * static_cast<size_t>(pl.sk_ctas) * 2 * 128 * sizeof(float), 256);
        p.sk_frag_o = reinterpret_cast<float*>(w);
    }
    if (pl.kernel == Kernel::kDecode) {
        char* w = static_cast<char*>(workspace);
        p.ws_counters = reinterpret_cast<int*>(w);
        w += round_up(pkv::decode_sched_bytes(batch, num_kv_heads, pl.splits), 256);
        if (pl.splits > 1) {
            const size_t states = static_cast<size_t>(batch) * max_q_rows * num_q_heads * pl.splits;
            p.ws_o = reinterpret_cast<float*>(w);
            p.ws_lse = reinterpret_cast<float*>(w + round_up(states * head_dim * sizeof(float), 256));
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (pl.kernel == Kernel::kSimt) return from_cuda(pkv::launch_attn_simt(p, s), "attention (simt)");

    CUtensorMap tk, tv;
    pkv_status st = make_pool_map(&tk, k_pool, head_dim, num_kv_heads, page_size, num_pages, page_stride);
    if (st != PKV_OK) return st;
    st = make_pool_map(&tv, v_pool, head_dim, num_kv_heads, page_size, num_pages, page_stride);
    if (st != PKV_OK) return st;
    if (pl.kernel == Kernel::kTile) {
        cudaError_t e = pkv::launch_attn_tc(p, nullptr, &tk, &tv, s);
        if (e != cudaSuccess) return from_cuda(e, "attention (tensor-core tiles)");
        if (pl.splits > 1) return from_cuda(pkv::launch_split_reduce(p, s), "attention (split reduce)");
        return ok();
    }
    return from_cuda(pkv::launch_decode(p, &tk, &tv, s), "attention (decode)");
}

namespace {
// Key splits of a grouped call: one CTA per (group, token tile, K/V head);
// the groups' count is known only on the device, so the host bound (every
// slot a group) sizes the choice, like plan_attention's tile rule.
Plan plan_grouped(int batch, int max_q_len, int max_group_tokens, int max_group_keys, int Hq, int Hkv,
                  int D, int num_splits, int sms) {
    Plan pl;
    pl.kernel = Kernel::kTile;
    const int G = Hkv > 0 ? Hq / Hkv : 1;
    const int tq = pkv::attn_tc_rows_per_tile(G);
    const int64_t ctas = static_cast<int64_t>((max_group_tokens + tq - 1) / tq) * Hkv * batch;
    const int s = tile_splits(ctas, max_group_keys, num_splits, sms);
    const int per = (max_group_keys + s - 1) / std::max(s, 1);
    pl.split_keys = std::max(kTileKeys, (per + kTileKeys - 1) / kTileKeys * kTileKeys);
    pl.splits = std::max(1, (max_group_keys + pl.split_keys - 1) / pl.split_keys);
    if (pl.splits > 1) {
        const size_t states = static_cast<size_t>(batch) * max_q_len * Hq * pl.splits;
        pl.ws_bytes = round_up(states * D * sizeof(float), 256) + round_up(states * sizeof(float), 256);
    }
    return pl;
}
}  // namespace

size_t shared_prefix_attention_workspace_size(int batch, int max_q_len, int max_group_tokens,
                                              int max_group_keys, int num_q_heads, int num_kv_heads,
                                              int head_dim, int num_splits) {
    if (batch <= 0 || max_q_len <= 0 || max_group_tokens <= 0 || num_kv_heads <= 0) return 0;
    return plan_grouped(batch, max_q_len, max_group_tokens, max_group_keys, num_q_heads, num_kv_heads,
                        head_dim, num_splits, current_device_sms())
        .ws_bytes;
}

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
                                   int32_t* err, void* stream) {
    if (batch < 0 || max_q_len < 0 || max_group_tokens < 0 || max_group_keys < 0 || num_q_heads < 0 ||
        num_kv_heads < 0 || num_pages < 0 || num_splits < 0)
        return fail(PKV_ERR_INVALID_ARG, "shared prefix: negative size");
    if (batch == 0 || max_q_len == 0 || max_group_tokens == 0 || num_q_heads == 0) return ok();
    if (num_kv_heads == 0 || num_q_heads % num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "shared prefix: %d query heads is not a multiple of %d K/V heads",
                    num_q_heads, num_kv_heads);
    if (!q || !k_pool || !v_pool || !group_rows || !run_lens || !group_indptr || !perm || !tail_start ||
        !tail_lens || !num_groups || !q_indptr || !out)
        return fail(PKV_ERR_INVALID_ARG, "shared prefix: null pointer");
    if (page_size != 32)
        return fail(PKV_ERR_UNSUPPORTED, "shared prefix: page_size %d (only 32-token pages)", page_size);
    if (!pkv::attn_tc_supported(head_dim, num_q_heads / num_kv_heads))
        return fail(PKV_ERR_UNSUPPORTED, "shared prefix: head_dim 64 or 128 and 1-64 grouped heads only");
    if (out_dtype != PKV_BF16 && out_dtype != PKV_F32)
        return fail(PKV_ERR_UNSUPPORTED, "shared prefix: output dtype must be bf16 or f32");
    if (batch > 65535 || num_kv_heads > 65535)
        return fail(PKV_ERR_UNSUPPORTED, "shared prefix: batch or K/V heads above 65535");
    if (page_stride < static_cast<int64_t>(page_size) * num_kv_heads * head_dim || page_stride % 8)
        return fail(PKV_ERR_INVALID_ARG, "shared prefix: page_stride must cover a page, multiple of 8");
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || q_token_stride % 8 ||
        q_head_stride % 8 || q_token_stride < 0 || q_head_stride < 0)
        return fail(PKV_ERR_INVALID_ARG, "shared prefix: q / pools 16-byte aligned, strides multiple of 8");
    if (!aligned(out, 16) || (lse && !aligned(lse, 4)))
        return fail(PKV_ERR_INVALID_ARG, "shared prefix: output must be 16-byte aligned");
    if (group_row_stride < (static_cast<int64_t>(max_group_keys) + 31) / 32)
        return fail(PKV_ERR_INVALID_ARG, "shared prefix: group_row_stride below max_group_keys / 32");
    const Plan pl = plan_grouped(batch, max_q_len, max_group_tokens, max_group_keys, num_q_heads,
                                 num_kv_heads, head_dim, num_splits, current_device_sms());
    if (pl.ws_bytes > 0 && (!workspace || workspace_bytes < pl.ws_bytes || !aligned(workspace, 256)))
        return fail(PKV_ERR_WORKSPACE, "shared prefix: workspace needs %zu bytes, 256-byte aligned",
                    pl.ws_bytes);
    if (static_cast<int64_t>(batch) * pl.splits > 65535)
        return fail(PKV_ERR_UNSUPPORTED, "shared prefix: batch x key splits above 65535");

    pkv::AttnParams p{};
    p.q = q;
    p.q_token_stride = q_token_stride;
    p.q_head_stride = q_head_stride;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.num_pages = num_pages;
    p.page_stride = page_stride;
    p.block_table = group_rows;
    p.block_table_stride = group_row_stride;
    p.q_indptr = q_indptr;
    p.batch = batch;
    p.max_q_rows = max_q_len;
    p.max_kv_len = max_group_keys;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.mask = PKV_MASK_NONE;
    const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    p.scale_log2 = sc * 1.4426950408889634f;
    p.out = out;
    p.out_f32 = out_dtype == PKV_F32;
    p.lse = lse;
    p.num_splits = pl.splits;
    p.split_keys = pl.split_keys;
    p.checked = (flags & PKV_FLAG_CHECKED) != 0;
    p.err = err;
    p.grp_run_lens = run_lens;
    p.grp_indptr = group_indptr;
    p.grp_perm = perm;
    p.grp_tail_start = tail_start;
    p.grp_tail_lens = tail_lens;
    p.grp_num_groups = num_groups;
    p.grp_max_tokens = max_group_tokens;
    if (pl.splits > 1) {
        const size_t states = static_cast<size_t>(batch) * max_q_len * num_q_heads * pl.splits;
        p.ws_o = static_cast<float*>(workspace);
        p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                            round_up(states * head_dim * sizeof(float), 256));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CUtensorMap tk, tv;
    pkv_status st = make_pool_map(&tk, k_pool, head_dim, num_kv_heads, page_size, num_pages, page_stride);
    if (st != PKV_OK) return st;
    st = make_pool_map(&tv, v_pool, head_dim, num_kv_heads, page_size, num_pages, page_stride);
    if (st != PKV_OK) return st;
    cudaError_t e = pkv::launch_attn_tc_grouped(p, &tk, &tv, s);
    if (e != cudaSuccess) return from_cuda(e, "shared prefix (grouped tiles)");
    if (pl.splits > 1) return from_cuda(pkv::launch_split_reduce(p, s), "shared prefix (split reduce)");
    return ok();
}

pkv_status merge_attn_states(const void* o_a, const float* lse_a, const void* o_b,
                             const float* lse_b, pkv_dtype in_dtype, int64_t rows, int num_heads,
                             int head_dim, void* o_out, pkv_dtype out_dtype, float* lse_out,
                             void* stream) {
    if (rows < 0 || num_heads < 0 || head_dim < 0)
        return fail(PKV_ERR_INVALID_ARG, "merge: negative size");
    if (rows == 0 || num_heads == 0 || head_dim == 0) return ok();
    if (!o_a || !lse_a || !o_b || !lse_b || !o_out)
        return fail(PKV_ERR_INVALID_ARG, "merge: null pointer");
    if ((in_dtype != PKV_BF16 && in_dtype != PKV_F32) || (out_dtype != PKV_BF16 && out_dtype != PKV_F32))
        return fail(PKV_ERR_UNSUPPORTED, "merge: dtypes must be bf16 or f32");
    if (head_dim % 4 || head_dim > 512)
        return fail(PKV_ERR_UNSUPPORTED, "merge: head_dim %d (a multiple of 4, at most 512)", head_dim);
    const size_t ia = in_dtype == PKV_F32 ? 16 : 8, oa = out_dtype == PKV_F32 ? 16 : 8;
    if (!aligned(o_a, ia) || !aligned(o_b, ia) || !aligned(o_out, oa) || !aligned(lse_a, 4) ||
        !aligned(lse_b, 4) || (lse_out && !aligned(lse_out, 4)))
        return fail(PKV_ERR_INVALID_ARG, "merge: misaligned pointer");
    return from_cuda(pkv::launch_merge(o_a, lse_a, o_b, lse_b, in_dtype == PKV_F32, rows, num_heads,
                                       head_dim, o_out, out_dtype == PKV_F32, lse_out,
                                       static_cast<cudaStream_t>(stream)),
                     "merge launch");
}

pkv_status rope_write_kv_paged(void* q, int64_t q_token_stride, int64_t q_head_stride,
                               int num_q_heads, const void* k_src, const void* v_src,
                               int64_t src_token_stride, int64_t src_head_stride,
                               int64_t num_tokens, int num_kv_heads, int head_dim,
                               const int64_t* positions, const float* cos_sin,
                               int64_t max_position, const int64_t* slots, void* k_pool,
                               void* v_pool, int64_t num_pages, int page_size,
                               int64_t page_stride, unsigned flags, int32_t* err, void* stream) {
    if (num_tokens < 0 || num_q_heads < 0 || num_kv_heads < 0 || head_dim < 0 || num_pages < 0 ||
        max_position < 0)
        return fail(PKV_ERR_INVALID_ARG, "rope: negative size");
    if (num_tokens == 0) return ok();
    if (!q || !k_src || !v_src || !positions || !cos_sin || !slots || !k_pool || !v_pool)
        return fail(PKV_ERR_INVALID_ARG, "rope: null pointer");
    if (head_dim <= 0 || head_dim % 16)
        return fail(PKV_ERR_UNSUPPORTED, "rope: head_dim %d (a multiple of 16)", head_dim);
    if (max_position == 0) return fail(PKV_ERR_INVALID_ARG, "rope: empty cos/sin table");
    if (page_size <= 0 || page_stride < static_cast<int64_t>(page_size) * num_kv_heads * head_dim ||
        page_stride % 8)
        return fail(PKV_ERR_INVALID_ARG, "rope: page_stride must cover a page, a multiple of 8");
    if (!aligned(q, 16) || !aligned(k_src, 16) || !aligned(v_src, 16) || !aligned(k_pool, 16) ||
        !aligned(v_pool, 16) || !aligned(cos_sin, 16) || q_token_stride % 8 || q_head_stride % 8 ||
        src_token_stride % 8 || src_head_stride % 8 || q_token_stride < 0 || q_head_stride < 0 ||
        src_token_stride < 0 || src_head_stride < 0)
        return fail(PKV_ERR_INVALID_ARG, "rope: 16-byte aligned pointers and strides multiple of 8");
    if ((flags & PKV_FLAG_CHECKED) && !err)
        return fail(PKV_ERR_INVALID_ARG, "rope: checked mode needs an error flag");
    pkv::RopeArgs a{q, q_token_stride, q_head_stride, num_q_heads, k_src, v_src, src_token_stride,
                    src_head_stride, num_tokens, num_kv_heads, head_dim, positions, cos_sin,
                    max_position, slots, k_pool, v_pool, num_pages, page_size, page_stride,
                    (flags & PKV_FLAG_CHECKED) != 0, err};
    return from_cuda(pkv::launch_rope_write(a, static_cast<cudaStream_t>(stream)), "rope launch");
}

pkv_status copy_kv_slots(void* k_pool, void* v_pool, int num_layers, int64_t layer_stride,
                         int64_t num_pages, int page_size, int64_t page_stride, int num_kv_heads,
                         int head_dim, pkv_dtype dtype, const int64_t* src_slots,
                         const int64_t* dst_slots, int64_t num_copies, unsigned flags,
                         int32_t* err, void* stream) {
    const int esz = elem_size(dtype);
    if (esz == 0) return fail(PKV_ERR_INVALID_ARG, "copy: unknown dtype %d", (int)dtype);
    if (num_copies < 0 || num_layers < 0 || num_pages < 0 || num_kv_heads < 0 || head_dim < 0)
        return fail(PKV_ERR_INVALID_ARG, "copy: negative size");
    if (num_copies == 0 || num_layers == 0 || num_kv_heads == 0 || head_dim == 0) return ok();
    if (!k_pool || !v_pool || !src_slots || !dst_slots)
        return fail(PKV_ERR_INVALID_ARG, "copy: null pointer");
    const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * esz;
    if (row_bytes % 16)
        return fail(PKV_ERR_UNSUPPORTED, "copy: a slot row must be a multiple of 16 bytes");
    if (page_size <= 0 || page_stride < static_cast<int64_t>(page_size) * num_kv_heads * head_dim ||
        (page_stride * esz) % 16)
        return fail(PKV_ERR_INVALID_ARG, "copy: page_stride must cover a page, 16-byte multiple");
    if (num_layers > 1 && (layer_stride < num_pages * page_stride || (layer_stride * esz) % 16))
        return fail(PKV_ERR_INVALID_ARG, "copy: layer_stride must cover a layer's pool, 16-byte multiple");
    if (num_layers > 65535) return fail(PKV_ERR_UNSUPPORTED, "copy: more than 65535 layers");
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16))
        return fail(PKV_ERR_INVALID_ARG, "copy: pools must be 16-byte aligned");
    if ((flags & PKV_FLAG_CHECKED) && !err)
        return fail(PKV_ERR_INVALID_ARG, "copy: checked mode needs an error flag");
    pkv::CopySlotsArgs a{k_pool, v_pool, num_layers, layer_stride, num_pages, page_size, page_stride,
                         num_kv_heads, head_dim, esz, src_slots, dst_slots, num_copies,
                         (flags & PKV_FLAG_CHECKED) != 0, err};
    return from_cuda(pkv::launch_copy_slots(a, static_cast<cudaStream_t>(stream)), "copy launch");
}

pkv_status causal_layout(const int32_t* table, int64_t num_logical_pages, const int64_t* committed,
                         int64_t pin_tokens, int64_t window_tokens, int num_staged, int block_size,
                         const int32_t* private_pages, int private_stride, int page_size,
                         int32_t* rows, int64_t row_stride, int32_t* kv_lens, int32_t* q_indptr,
                         int64_t* staged_slots, int64_t* staged_slots2, int64_t* committed_src,
                         int64_t* committed_dst, int64_t committed_capacity,
                         int64_t* current_src_idx, int64_t* current_dst, int64_t current_capacity,
                         int32_t* err, void* stream) {
    if (page_size != 32) return fail(PKV_ERR_UNSUPPORTED, "layout: page_size %d (32 only)", page_size);
    if (num_staged < 0 || block_size <= 0 || pin_tokens < 0 || window_tokens < 0 ||
        num_logical_pages < 0 || private_stride < 0 || row_stride < 0)
        return fail(PKV_ERR_INVALID_ARG, "layout: negative size or block_size < 1");
    if (num_staged == 0) return ok();
    const int64_t num_blocks = (static_cast<int64_t>(num_staged) + block_size - 1) / block_size;
    if (!table || !committed || !private_pages || !rows || !kv_lens || !q_indptr || !staged_slots ||
        !staged_slots2 || !committed_src || !committed_dst || !current_src_idx || !current_dst)
        return fail(PKV_ERR_INVALID_ARG, "layout: null pointer");
    if (row_stride < 1 || private_stride < 1)
        return fail(PKV_ERR_INVALID_ARG, "layout: row_stride and private_stride must be >= 1");
    if (committed_capacity < num_blocks * PKV_LAYOUT_COMMITTED_PER_BLOCK ||
        current_capacity < num_blocks * PKV_LAYOUT_CURRENT_PER_BLOCK)
        return fail(PKV_ERR_INVALID_ARG,
                    "layout: copy lists need %lld committed and %lld current entries for %lld blocks",
                    static_cast<long long>(num_blocks * PKV_LAYOUT_COMMITTED_PER_BLOCK),
                    static_cast<long long>(num_blocks * PKV_LAYOUT_CURRENT_PER_BLOCK),
                    static_cast<long long>(num_blocks));
    if (pin_tokens + window_tokens + block_size > 0x7fffffffLL)
        return fail(PKV_ERR_UNSUPPORTED, "layout: a row of more than 2^31 keys");
    if (num_blocks > 0x7fffffffLL) return fail(PKV_ERR_UNSUPPORTED, "layout: too many blocks");
    pkv::LayoutArgs a{table, num_logical_pages, committed, pin_tokens, window_tokens, num_staged,
                      block_size, static_cast<int>(num_blocks), private_pages, private_stride, rows,
                      row_stride, kv_lens, q_indptr, staged_slots, staged_slots2, committed_src,
                      committed_dst, current_src_idx, current_dst, err};
    return from_cuda(pkv::launch_causal_layout(a, static_cast<cudaStream_t>(stream)), "layout launch");
}

pkv_status plan_shared_prefix(const int32_t* block_table, int64_t block_table_stride,
                              const int32_t* kv_lens, const int32_t* q_indptr, int batch,
                              int max_pages, int32_t* group_rows, int64_t group_row_stride,
                              int32_t* run_lens, int32_t* group_indptr, int32_t* perm,
                              int32_t* group_of, int32_t* tail_start, int32_t* tail_lens,
                              int32_t* num_groups, int32_t* err, void* stream) {
    if (batch < 0 || max_pages < 0 || group_row_stride < 0)
        return fail(PKV_ERR_INVALID_ARG, "plan: negative size");
    if (batch == 0) return ok();
    if (batch > 1024) return fail(PKV_ERR_UNSUPPORTED, "plan: batch %d above 1024", batch);
    if (!block_table || !kv_lens || !q_indptr || !group_rows || !run_lens || !group_indptr || !perm ||
        !group_of || !tail_start || !tail_lens || !num_groups)
        return fail(PKV_ERR_INVALID_ARG, "plan: null pointer");
    if (block_table_stride < max_pages)
        return fail(PKV_ERR_INVALID_ARG, "plan: block_table_stride %lld < max_pages %d",
                    static_cast<long long>(block_table_stride), max_pages);
    if (group_row_stride < 1) return fail(PKV_ERR_INVALID_ARG, "plan: group_row_stride must be >= 1");
    pkv::PlanArgs a{block_table, block_table_stride, kv_lens, q_indptr, batch, max_pages, group_rows,
                    group_row_stride, run_lens, group_indptr, perm, group_of, tail_start, tail_lens,
                    num_groups, err};
    return from_cuda(pkv::launch_plan(a, static_cast<cudaStream_t>(stream)), "plan launch");
}

pkv_status rotate_rows(void* x, int64_t rows, int64_t cols, int64_t row_stride, int elem_size_b,
                       int64_t shift, void* stream) {
    if (rows < 0 || cols < 0) return fail(PKV_ERR_INVALID_ARG, "rotate: negative size");
    if (elem_size_b != 1 && elem_size_b != 2 && elem_size_b != 4 && elem_size_b != 8 &&
        elem_size_b != 16)
        return fail(PKV_ERR_UNSUPPORTED, "rotate: element size %d (1, 2, 4, 8 or 16)", elem_size_b);
    if (rows == 0 || cols <= 1) return ok();
    if (!x) return fail(PKV_ERR_INVALID_ARG, "rotate: null pointer");
    if (rows > 1 && row_stride < cols)
        return fail(PKV_ERR_INVALID_ARG, "rotate: row_stride %lld < cols %lld (rows overlap)",
                    (long long)row_stride, (long long)cols);
    if (!aligned(x, elem_size_b)) return fail(PKV_ERR_INVALID_ARG, "rotate: misaligned buffer");
    int64_t sh = shift % cols;
    if (sh < 0) sh += cols;
    if (sh == 0) return ok();
    // widest unit (up to 16 bytes) that divides every byte quantity involved
    const int64_t es = elem_size_b;
    int unit = 16;
    for (; unit > 1; unit >>= 1) {
        const bool fits = (cols * es) % unit == 0 && (sh * es) % unit == 0 &&
                          (rows == 1 || (row_stride * es) % unit == 0) && aligned(x, unit);
        if (fits) break;
    }
    const int64_t ucols = cols * es / unit, ushift = sh * es / unit;
    const int64_t ustride = rows == 1 ? ucols : row_stride * es / unit;
    return from_cuda(pkv::launch_rotate(x, rows, ucols, ustride, unit, ushift,
                                        static_cast<cudaStream_t>(stream)),
                     "rotate launch");
}

}  // extern "C"
