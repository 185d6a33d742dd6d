// scatter.cu -- kv_scatter_slots: copy new K/V token rows into pool slots.
//
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Cache ("Chunk K/V write" bullet) and per-file notes on scatterKvSlots: one
// kernel reads every source row once, any token/head stride, one or two
// destination slots, optional source indices, vector-width dispatch.
//
// Design: one block per token; its threads stride over the token's K and V
// row in vectors (a warp moves 32 consecutive vectors of a head row: coalesced
// reads of the source and writes of the slot).  The vector width is the widest
// of 16/8/4/2 bytes that every pointer and stride allows.  Both destinations
// reuse the loaded vector, so the source is read once.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// One block per token: the block's threads stride over the token's K and V
// row vectors (2 x Hkv x D*esz/Vec of them), so all index arithmetic is 32-bit
// and the slot and source index are read once per token.
template <typename Vec>
__global__ void __launch_bounds__(256) scatter_kernel(ScatterArgs a, int vecs_per_head) {
    const int64_t t = blockIdx.x;
    int64_t src = t;
    if (a.src_idx) {
        src = a.src_idx[t];
        if (a.checked && (src < 0 || src >= a.num_src_rows)) {
            if (threadIdx.x == 0) set_err(a.err, PKV_ERRBIT_SRC);
            return;
        }
    }
    int64_t s1 = a.slots[t];
    int64_t s2 = a.slots2 ? a.slots2[t] : -1;
    const int64_t num_slots = a.num_pages * a.page_size;
    if (a.checked) {
        if (s1 >= num_slots || s2 >= num_slots) {
            if (threadIdx.x == 0) set_err(a.err, PKV_ERRBIT_SLOT);
            if (s1 >= num_slots) s1 = -1;
            if (s2 >= num_slots) s2 = -1;
        }
    }
    if (s1 < 0 && s2 < 0) return;
    const int esz = a.elem_size;
    const int64_t row_elems = static_cast<int64_t>(a.num_kv_heads) * a.head_dim;
    // addresses of the K rows at the two destinations (a skipped one points at slot 0)
    const int64_t u1 = s1 < 0 ? 0 : s1, u2 = s2 < 0 ? 0 : s2;
    const int64_t p1 = u1 / a.page_size, p2 = u2 / a.page_size;
    char* const d1k = static_cast<char*>(a.k_pool) +
                      (p1 * a.page_stride + (u1 - p1 * a.page_size) * row_elems) * esz;
    char* const d2k = static_cast<char*>(a.k_pool) +
                      (p2 * a.page_stride + (u2 - p2 * a.page_size) * row_elems) * esz;
    const int64_t kv_off = static_cast<char*>(a.v_pool) - static_cast<char*>(a.k_pool);
    const char* const srck = static_cast<const char*>(a.k_src) + src * a.src_token_stride * esz;
    const int64_t src_kv_off = static_cast<const char*>(a.v_src) - static_cast<const char*>(a.k_src);
    const int per_row = a.num_kv_heads * vecs_per_head;
    for (int i = threadIdx.x; i < 2 * per_row; i += blockDim.x) {
        const int which = i >= per_row;          // 0 = K, 1 = V
        const int j = i - which * per_row;
        const int h = j / vecs_per_head;
        const int c = j - h * vecs_per_head;
        const Vec v = *reinterpret_cast<const Vec*>(srck + which * src_kv_off +
                                                    static_cast<int64_t>(h) * a.src_head_stride * esz +
                                                    c * static_cast<int>(sizeof(Vec)));
        const int64_t dst_off = which * kv_off + static_cast<int64_t>(h) * a.head_dim * esz +
                                c * static_cast<int>(sizeof(Vec));
        if (s1 >= 0) *reinterpret_cast<Vec*>(d1k + dst_off) = v;
        if (s2 >= 0) *reinterpret_cast<Vec*>(d2k + dst_off) = v;
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
    const int vecs_per_head = static_cast<int>(head_bytes / vec);
    if (a.num_tokens == 0 || vecs_per_head == 0) return cudaSuccess;
    if (a.num_tokens > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int per_token = 2 * a.num_kv_heads * vecs_per_head;
    const int threads = per_token >= 256 ? 256 : ((per_token + 31) / 32) * 32;
    const dim3 grid(static_cast<unsigned>(a.num_tokens));
    switch (vec) {
        case 16: scatter_kernel<uint4><<<grid, threads, 0, s>>>(a, vecs_per_head); break;
        case 8: scatter_kernel<uint2><<<grid, threads, 0, s>>>(a, vecs_per_head); break;
        case 4: scatter_kernel<uint32_t><<<grid, threads, 0, s>>>(a, vecs_per_head); break;
        default: scatter_kernel<uint16_t><<<grid, threads, 0, s>>>(a, vecs_per_head); break;
    }
    return cudaGetLastError();
}

}  // namespace pkv
