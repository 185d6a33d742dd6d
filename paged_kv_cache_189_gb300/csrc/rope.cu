// rope.cu -- rope_write_kv_paged: rotary embedding of Q (in place) and K,
// with the rotated K and the V written into pool slots, in one launch; and
// copy_kv_slots: pool-to-pool copy of whole slot rows across layers.
//
// "Support shared-prefix attention for n-sample requests in FMHA", commit
// notes: RoPE and the K/V write are one kernel (Q rotated in place, the rotated
// K and the V written straight to the pool; NeoX RoPE, no or linear scaling;
// RoPE at the absolute positions, the write at the slot the table names).
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Cache and the per-file notes on causalLayout.cu: one pool-to-pool copy
// (copy_kv_slots_) fills the private pages at commit, across layers, K/V and
// heads, sentinel entries skipped.
//
// Both are HBM-bound copies with a little arithmetic: one block per token (per
// (copy, layer) for the slot copy), 16-byte vectors, fp32 rotation.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ void unpack8(const uint4 w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = bf16lo(u[j]);
        f[2 * j + 1] = bf16hi(u[j]);
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// Work of one token, in 16-byte items: Q rotations (Hq x D/16 pair chunks of
// 8 pairs), K rotations (Hkv x D/16), V copies (Hkv x D/8 vectors).
__global__ void __launch_bounds__(256) rope_write_kernel(RopeArgs a) {
    const int64_t t = blockIdx.x;
    const int D = a.head_dim, H2 = D / 2;
    const int chunks = D / 16;  // 8-pair chunks per head
    int64_t pos = a.positions[t];
    const bool pos_ok = pos >= 0 && pos < a.max_position;
    if (!pos_ok) {
        if (a.checked && threadIdx.x == 0) set_err(a.err, PKV_ERRBIT_LEN);
        pos = pos < 0 ? 0 : a.max_position - 1;  // stay inside the table
    }
    int64_t slot = a.slots[t];
    if (a.checked && slot >= a.num_pages * a.page_size) {
        if (threadIdx.x == 0) set_err(a.err, PKV_ERRBIT_SLOT);
        slot = -1;
    }
    const float* cs = a.cos_sin + pos * D;
    const int64_t page = slot >= 0 ? slot / a.page_size : 0;
    const int64_t row_elems = static_cast<int64_t>(a.num_kv_heads) * D;
    const int64_t dst_row = page * a.page_stride + (slot >= 0 ? slot - page * a.page_size : 0) * row_elems;
    const int nq = a.num_q_heads * chunks, nk = a.num_kv_heads * chunks, nv = a.num_kv_heads * (D / 8);
    for (int it = threadIdx.x; it < nq + nk + nv; it += blockDim.x) {
        if (it < nq + nk) {
            const bool is_q = it < nq;
            const int j = is_q ? it : it - nq;
            const int h = j / chunks, c = j - h * chunks;
            const __nv_bfloat16* src;
            if (is_q) {
                src = static_cast<const __nv_bfloat16*>(a.q) + t * a.q_token_stride + h * a.q_head_stride;
            } else {
                if (slot < 0) continue;
                src = static_cast<const __nv_bfloat16*>(a.k_src) + t * a.src_token_stride + h * a.src_head_stride;
            }
            float x1[8], x2[8], o1[8], o2[8];
            unpack8(*reinterpret_cast<const uint4*>(src + c * 8), x1);
            unpack8(*reinterpret_cast<const uint4*>(src + H2 + c * 8), x2);
            const float4 c0 = *reinterpret_cast<const float4*>(cs + c * 8);
            const float4 c1 = *reinterpret_cast<const float4*>(cs + c * 8 + 4);
            const float4 s0 = *reinterpret_cast<const float4*>(cs + H2 + c * 8);
            const float4 s1 = *reinterpret_cast<const float4*>(cs + H2 + c * 8 + 4);
            const float co[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            const float si[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                o1[e] = fmaf(x1[e], co[e], -x2[e] * si[e]);
                o2[e] = fmaf(x2[e], co[e], x1[e] * si[e]);
            }
            __nv_bfloat16* dst;
            if (is_q) {
                dst = static_cast<__nv_bfloat16*>(a.q) + t * a.q_token_stride + h * a.q_head_stride;
            } else {
                dst = static_cast<__nv_bfloat16*>(a.k_pool) + dst_row + static_cast<int64_t>(h) * D;
            }
            *reinterpret_cast<uint4*>(dst + c * 8) = pack8(o1);
            *reinterpret_cast<uint4*>(dst + H2 + c * 8) = pack8(o2);
        } else {
            if (slot < 0) continue;
            const int j = it - nq - nk;
            const int h = j / (D / 8), c = j - h * (D / 8);
            const uint4 v = *reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(a.v_src) + t * a.src_token_stride + h * a.src_head_stride + c * 8);
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.v_pool) + dst_row +
                                      static_cast<int64_t>(h) * D + c * 8) = v;
        }
    }
}

// One block per (copy entry, layer): the whole K and V slot rows.
__global__ void __launch_bounds__(256) copy_slots_kernel(CopySlotsArgs a, int vecs_per_row) {
    const int64_t e = blockIdx.x;
    const int64_t layer = blockIdx.y;
    const int64_t src = a.src_slots[e], dst = a.dst_slots[e];
    if (src < 0 || dst < 0) return;  // sentinel
    const int64_t num_slots = a.num_pages * a.page_size;
    if (a.checked && (src >= num_slots || dst >= num_slots)) {
        if (threadIdx.x == 0 && layer == 0) set_err(a.err, PKV_ERRBIT_SLOT);
        return;
    }
    const int64_t row_bytes = static_cast<int64_t>(a.num_kv_heads) * a.head_dim * a.elem_size;
    auto slot_off = [&](int64_t s) {
        const int64_t pg = s / a.page_size;
        return (layer * a.layer_stride + pg * a.page_stride) * a.elem_size + (s - pg * a.page_size) * row_bytes;
    };
    const int64_t so = slot_off(src), dof = slot_off(dst);
    for (int i = threadIdx.x; i < 2 * vecs_per_row; i += blockDim.x) {
        const bool is_v = i >= vecs_per_row;
        char* base = static_cast<char*>(is_v ? a.v_pool : a.k_pool);
        const int c = is_v ? i - vecs_per_row : i;
        *reinterpret_cast<uint4*>(base + dof + c * 16) = *reinterpret_cast<const uint4*>(base + so + c * 16);
    }
}

}  // namespace

cudaError_t launch_rope_write(const RopeArgs& a, cudaStream_t s) {
    if (a.num_tokens == 0) return cudaSuccess;
    if (a.num_tokens > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    rope_write_kernel<<<static_cast<unsigned>(a.num_tokens), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_copy_slots(const CopySlotsArgs& a, cudaStream_t s) {
    if (a.num_copies == 0 || a.num_layers == 0) return cudaSuccess;
    if (a.num_copies > 0x7fffffffLL || a.num_layers > 65535) return cudaErrorInvalidConfiguration;
    const int vecs = static_cast<int>(static_cast<int64_t>(a.num_kv_heads) * a.head_dim * a.elem_size / 16);
    const int threads = 2 * vecs >= 256 ? 256 : ((2 * vecs + 31) / 32) * 32;
    copy_slots_kernel<<<dim3(static_cast<unsigned>(a.num_copies), a.num_layers), threads, 0, s>>>(a, vecs);
    return cudaGetLastError();
}

}  // namespace pkv
