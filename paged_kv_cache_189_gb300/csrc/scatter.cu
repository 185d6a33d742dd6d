// scatter.cu -- kv_scatter_slots: copy new K/V token rows into pool slots.
//
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Cache ("Chunk K/V write" bullet) and per-file notes on scatterKvSlots: one
// kernel reads every source row once, any token/head stride, one or two
// destination slots, optional source indices, vector-width dispatch.
//
// Design: a flat grid of threads, one per (token, K|V, head, vector) so that a
// warp moves 32 consecutive 16-byte vectors of one head row (coalesced reads of
// the source and writes of the slot); the vector width is the widest of
// 16/8/4/2 bytes that every pointer and stride allows.  Both destinations reuse
// the loaded vector, so the source is read once.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

template <typename Vec>
__global__ void __launch_bounds__(256) scatter_kernel(ScatterArgs a, int64_t vecs_per_head,
                                                      int64_t total) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int64_t c = idx % vecs_per_head;
    int64_t rest = idx / vecs_per_head;
    const int h = static_cast<int>(rest % a.num_kv_heads);
    rest /= a.num_kv_heads;
    const int which = static_cast<int>(rest & 1);  // 0 = K, 1 = V
    const int64_t t = rest >> 1;

    int64_t src = t;
    if (a.src_idx) {
        src = a.src_idx[t];
        if (a.checked && (src < 0 || src >= a.num_src_rows)) {
            if (which == 0 && h == 0 && c == 0) set_err(a.err, PKV_ERRBIT_SRC);
            return;
        }
    }
    const int64_t s1 = a.slots[t];
    const int64_t s2 = a.slots2 ? a.slots2[t] : -1;
    if (s1 < 0 && s2 < 0) return;

    const int esz = a.elem_size;
    const char* base = static_cast<const char*>(which ? a.v_src : a.k_src);
    const Vec v = *reinterpret_cast<const Vec*>(
        base + (src * a.src_token_stride + h * a.src_head_stride) * esz + c * sizeof(Vec));

    char* pool = static_cast<char*>(which ? a.v_pool : a.k_pool);
    const int64_t num_slots = a.num_pages * a.page_size;
    const int64_t row_elems = static_cast<int64_t>(a.num_kv_heads) * a.head_dim;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int64_t slot = k ? s2 : s1;
        if (slot < 0) continue;
        if (a.checked && slot >= num_slots) {
            if (which == 0 && h == 0 && c == 0) set_err(a.err, PKV_ERRBIT_SLOT);
            continue;
        }
        const int64_t page = slot / a.page_size;
        const int64_t off = slot - page * a.page_size;
        char* dst = pool + (page * a.page_stride + off * row_elems + static_cast<int64_t>(h) *
                                                                        a.head_dim) * esz +
                    c * sizeof(Vec);
        *reinterpret_cast<Vec*>(dst) = v;
    }
}

bool aligned(const void* p, int64_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

}  // namespace

cudaError_t launch_scatter(const ScatterArgs& a, cudaStream_t s) {
    const int esz = a.elem_size;
    const int64_t head_bytes = static_cast<int64_t>(a.head_dim) * esz;
    int vec = 16;
    for (; vec > esz; vec >>= 1) {
        const bool ok = head_bytes % vec == 0 && aligned(a.k_src, vec) && aligned(a.v_src, vec) &&
                        aligned(a.k_pool, vec) && aligned(a.v_pool, vec) &&
                        (a.src_token_stride * esz) % vec == 0 &&
                        (a.src_head_stride * esz) % vec == 0 && (a.page_stride * esz) % vec == 0;
        if (ok) break;
    }
    const int64_t vecs_per_head = head_bytes / vec;
    const int64_t total = a.num_tokens * 2 * a.num_kv_heads * vecs_per_head;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    switch (vec) {
        case 16: scatter_kernel<uint4><<<blocks, threads, 0, s>>>(a, vecs_per_head, total); break;
        case 8: scatter_kernel<uint2><<<blocks, threads, 0, s>>>(a, vecs_per_head, total); break;
        case 4: scatter_kernel<uint32_t><<<blocks, threads, 0, s>>>(a, vecs_per_head, total); break;
        default: scatter_kernel<uint16_t><<<blocks, threads, 0, s>>>(a, vecs_per_head, total); break;
    }
    return cudaGetLastError();
}

}  // namespace pkv
