// attn_simt.cu -- generic paged attention, one warp per (query row, head).
//
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Attention and Cache (frame-causal blocks, real-token seq_len, padding rows
// return zero).  This kernel covers every mask, row count and head grouping
// with the plainest GPU schedule: each warp walks its row's visible keys
// through the block table, lanes split the head dimension, a shuffle
// reduction forms each score, and an fp32 online softmax accumulates the
// output.  It is the cross-check for the fast kernels (PKV_FLAG_SIMT_ONLY)
// and the path for shapes they do not cover; it is not tuned.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ int visible_keys(int i, int qreal, int kv_len, int mask, int cb) {
    if (i >= qreal) return 0;
    const int first_new = kv_len - qreal;
    if (mask == PKV_MASK_NONE) return kv_len;
    if (mask == PKV_MASK_CAUSAL) return first_new + i + 1;
    const int block_end = (i / cb + 1) * cb;
    return first_new + min(qreal, block_end);
}

template <int D>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnParams p) {
    constexpr int DPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z;
    const int i = blockIdx.x;
    const int h = blockIdx.y * 4 + warp;
    if (h >= p.num_q_heads) return;
    const int r0 = p.q_indptr[b];
    const int nrows = p.q_indptr[b + 1] - r0;
    if (i >= nrows) return;
    const int row = r0 + i;
    const int qreal = p.q_real ? p.q_real[b] : nrows;
    int kv_len = p.kv_lens[b];
    if (p.checked && lane == 0 && i == 0 && h == 0 &&
        (kv_len > p.max_kv_len || kv_len < 0 || nrows > p.max_q_rows || qreal > nrows))
        set_err(p.err, PKV_ERRBIT_LEN);
    kv_len = min(max(kv_len, 0), p.max_kv_len);
    const int nvis = max(0, min(kv_len, visible_keys(i, min(qreal, nrows), kv_len, p.mask,
                                                     max(p.causal_block, 1))));
    const int G = p.num_q_heads / p.num_kv_heads;
    const int kvh = h / G;

    float q[DPL];
    const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(p.q) +
                              static_cast<int64_t>(row) * p.q_token_stride +
                              static_cast<int64_t>(h) * p.q_head_stride + lane * DPL;
#pragma unroll
    for (int j = 0; j < DPL; ++j) q[j] = __bfloat162float(qp[j]) * p.scale_log2;

    const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.block_table_stride;
    const int64_t row_elems = static_cast<int64_t>(p.num_kv_heads) * D;
    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[j] = 0.f;
    for (int key = 0; key < nvis; ++key) {
        const int page = bt[key >> 5];
        if (p.checked && (page < 0 || page >= p.num_pages)) {
            if (lane == 0) set_err(p.err, PKV_ERRBIT_PAGE);
            continue;
        }
        const int64_t off = static_cast<int64_t>(page) * p.page_stride + (key & 31) * row_elems +
                            static_cast<int64_t>(kvh) * D + lane * DPL;
        const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(p.k_pool) + off;
        const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(p.v_pool) + off;
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) dot = fmaf(q[j], __bfloat162float(kp[j]), dot);
        const float s = warp_sum(dot);
        const float m_new = fmaxf(m, s);
        const float alpha = fast_exp2(m - m_new);
        const float pk = fast_exp2(s - m_new);
        l = l * alpha + pk;
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = fmaf(pk, __bfloat162float(vp[j]), o[j] * alpha);
        m = m_new;
    }
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    const int64_t st = static_cast<int64_t>(row) * p.num_q_heads + h;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
        const float v = o[j] * inv;
        if (p.out_f32) static_cast<float*>(p.out)[st * D + lane * DPL + j] = v;
        else static_cast<__nv_bfloat16*>(p.out)[st * D + lane * DPL + j] = __float2bfloat16_rn(v);
    }
    if (p.lse && lane == 0) p.lse[st] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_attn_simt(const AttnParams& p, cudaStream_t s) {
    dim3 grid(p.max_q_rows, (p.num_q_heads + 3) / 4, p.batch);
    if (p.head_dim == 128) attn_simt_kernel<128><<<grid, 128, 0, s>>>(p);
    else attn_simt_kernel<64><<<grid, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
