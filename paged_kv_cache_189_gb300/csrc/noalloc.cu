// noalloc.cu -- paged_attention_no_alloc: paged attention whose scratch memory
// is a fixed array owned by the library, for callers that cannot allocate.
//
// Some callers of this library have no way to hand it a workspace: code that
// enqueues work while a CUDA graph is being captured (a cudaMalloc there fails
// or breaks the capture), serving processes that fix their device memory at
// start-up and forbid allocator calls on the request path, and plugin-style
// hosts that pass only input and output pointers.  For them this entry point
// runs the same attention path as paged_attention, with its scratch (the
// split-KV partial outputs and the scheduling counters) taken from the
// file-scope device array below instead of a caller buffer.
//
// The array is PKV_NO_ALLOC_SCRATCH_BYTES large and lives on every GPU that
// loads the library until the process exits.  Its device address is looked up
// on the first call made with a device current, and again whenever that
// device's context has changed since (after cudaDeviceReset the module is
// loaded anew and the array may move); that first call should therefore
// happen before any stream capture.  All calls on a device share the array,
// so calls that may run at the same time on the GPU (different streams
// without ordering) race on it.  The counters that must start at zero are
// cleared by every call (as paged_attention does); the partial outputs are
// fully rewritten before they are read.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_scratch[PKV_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// cuCtxGetCurrent through the runtime's driver entry point (no link-time
// dependency on libcuda); null if the driver does not offer it.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Device address of the scratch array on the current device (host code may
// not use the symbol itself as a pointer).
pkv_status scratch_on_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return pkv::report(PKV_ERR_CUDA, "paged_attention_no_alloc: cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices)
        return pkv::report(PKV_ERR_UNSUPPORTED, "paged_attention_no_alloc: device index too large");
    // the context current on this thread (null before the runtime has made
    // one current; the lookup below does that)
    auto current_ctx = [] {
        CUcontext c = nullptr;
        if (auto fn = ctx_get_current_fn()) {
            if (fn(&c) != CUDA_SUCCESS) c = nullptr;
        }
        return c;
    };
    const CUcontext ctx = current_ctx();
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p) {
            char msg[160];
            snprintf(msg, sizeof(msg), "paged_attention_no_alloc: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
            return pkv::report(PKV_ERR_CUDA, msg);
        }
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_ctx();
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status paged_attention_no_alloc(
    const void* q, int64_t q_token_stride, int64_t q_head_stride, const void* k_pool,
    const void* v_pool, int64_t num_pages, int page_size, int64_t page_stride,
    const int32_t* block_table, int64_t block_table_stride, const int32_t* kv_lens,
    const int32_t* q_indptr, const int32_t* q_real, int batch, int max_q_rows, int max_kv_len,
    int num_q_heads, int num_kv_heads, int head_dim, pkv_mask mask, int causal_block, float scale,
    void* out, pkv_dtype out_dtype, float* lse, int num_splits, unsigned flags, int32_t* err,
    void* stream) {
    const size_t need = paged_attention_workspace_size(batch, max_q_rows, num_q_heads, num_kv_heads,
                                                       head_dim, max_kv_len, num_splits, flags);
    if (need > PKV_NO_ALLOC_SCRATCH_BYTES) {
        char msg[240];
        snprintf(msg, sizeof(msg),
                 "paged_attention_no_alloc: this call needs %zu bytes of scratch but the library's "
                 "fixed scratch holds %zu; use paged_attention with a workspace",
                 need, static_cast<size_t>(PKV_NO_ALLOC_SCRATCH_BYTES));
        return pkv::report(PKV_ERR_WORKSPACE, msg);
    }
    void* ws = nullptr;
    if (need > 0) {
        const pkv_status st = scratch_on_current_device(&ws);
        if (st != PKV_OK) return st;
    }
    return paged_attention(q, q_token_stride, q_head_stride, k_pool, v_pool, num_pages, page_size,
                           page_stride, block_table, block_table_stride, kv_lens, q_indptr, q_real,
                           batch, max_q_rows, max_kv_len, num_q_heads, num_kv_heads, head_dim, mask,
                           causal_block, scale, out, out_dtype, lse, ws,
                           need > 0 ? static_cast<size_t>(PKV_NO_ALLOC_SCRATCH_BYTES) : 0,
                           num_splits, flags, err, stream);
}
