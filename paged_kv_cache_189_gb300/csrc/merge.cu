// merge.cu -- exact LSE merge of attention states.
//
// "Support shared-prefix attention for n-sample requests in FMHA", commit
// notes: the prefix attention and the private-tail attention each return an
// output and its LSE, and one merge kernel joins them (an empty run has LSE
// -inf); the split-KV merge runs one program per (token, block of heads).
//
// merge_kernel: two states, one warp per (row, head), vectorised loads.
// split_reduce_kernel: the n-way version that finishes a split-KV attention
// call, one warp per (row, head).
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ float4 load4(const void* base, int64_t idx, bool f32) {
    if (f32) return reinterpret_cast<const float4*>(base)[idx >> 2];
    const uint2 w = reinterpret_cast<const uint2*>(base)[idx >> 2];
    return make_float4(bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y));
}
__device__ __forceinline__ void store4(void* base, int64_t idx, bool f32, float4 v) {
    if (f32) {
        reinterpret_cast<float4*>(base)[idx >> 2] = v;
    } else {
        reinterpret_cast<uint2*>(base)[idx >> 2] =
            make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
}

// One warp per (row, head) state; lanes stride over the 4-element vectors.
// All lanes read the two LSEs before lane 0 writes lse_out, so lse_out may
// alias lse_a or lse_b; o_out may alias o_a or o_b (each element is read and
// written by the same thread).
__global__ void __launch_bounds__(256) merge_kernel(const void* o_a, const float* lse_a,
                                                    const void* o_b, const float* lse_b,
                                                    bool in_f32, int64_t states, int head_dim,
                                                    void* o_out, bool out_f32, float* lse_out) {
    const int64_t st = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (st >= states) return;
    const float la = lse_a[st], lb = lse_b[st];
    __syncwarp();
    const float m = fmaxf(la, lb);
    float ca = 0.f, cb = 0.f, lse = -INFINITY;
    if (m != -INFINITY) {
        const float wa = __expf(la - m), wb = __expf(lb - m);  // exp(-inf) = 0
        const float inv = 1.0f / (wa + wb);
        ca = wa * inv;
        cb = wb * inv;
        lse = m + __logf(wa + wb);
    }
    for (int v = lane; v < (head_dim >> 2); v += 32) {
        const int64_t e = st * head_dim + v * 4;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m != -INFINITY) {
            const float4 a = load4(o_a, e, in_f32), b = load4(o_b, e, in_f32);
            o = make_float4(ca * a.x + cb * b.x, ca * a.y + cb * b.y, ca * a.z + cb * b.z,
                            ca * a.w + cb * b.w);
        }
        store4(o_out, e, out_f32, o);
    }
    if (lse_out && lane == 0) lse_out[st] = lse;
}

// One warp per (row, head): merge the valid splits of that row.
template <int D>
__global__ void __launch_bounds__(256) split_reduce_kernel(AttnParams p) {
    constexpr int DPL = D / 32;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int H = p.num_q_heads;
    const int b = blockIdx.y;
    const int row_in_seq = warp / H;
    const int h = warp - row_in_seq * H;
    if (row_in_seq >= p.max_q_rows) return;
    const int r0 = p.q_indptr[b];
    const int nrows = p.q_indptr[b + 1] - r0;
    if (row_in_seq >= nrows) return;
    const int row = r0 + row_in_seq;
    if (row >= static_cast<int64_t>(p.batch) * p.max_q_rows) return;  // workspace bound
    int nsplit = p.num_splits;  // grouped mode: every split wrote a state for every token
    if (!p.grp_perm) {
        const int qreal = p.q_real ? p.q_real[b] : nrows;
        int kv_len = min(p.kv_lens[b], p.max_kv_len);
        if (row_in_seq >= qreal) kv_len = 0;
        // splits that hold keys of this row (the rows of one sequence share them)
        nsplit = min(p.num_splits, (kv_len + p.split_keys - 1) / p.split_keys);
    }
    const int64_t st = static_cast<int64_t>(row) * H + h;
    const float* lses = p.ws_lse + st * p.num_splits;
    float m = -INFINITY;
    for (int s = 0; s < nsplit; ++s) m = fmaxf(m, lses[s]);
    float acc[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
        for (int s = 0; s < nsplit; ++s) {
            const float w = __expf(lses[s] - m);
            wsum += w;
            const float* o = p.ws_o + (st * p.num_splits + s) * D + lane * DPL;
#pragma unroll
            for (int j = 0; j < DPL; ++j) acc[j] += w * o[j];
        }
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    const int64_t ob = st * D + lane * DPL;
    if (p.out_f32) {
        float* out = static_cast<float*>(p.out) + ob;
#pragma unroll
        for (int j = 0; j < DPL; ++j) out[j] = acc[j] * inv;
    } else {
        uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + ob);
#pragma unroll
        for (int j = 0; j < DPL; j += 2) out[j / 2] = pack_bf16x2(acc[j] * inv, acc[j + 1] * inv);
    }
    if (p.lse && lane == 0) p.lse[st] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b,
                         const float* lse_b, bool in_f32, int64_t rows, int num_heads,
                         int head_dim, void* o_out, bool out_f32, float* lse_out,
                         cudaStream_t s) {
    const int64_t states = rows * num_heads;
    const int64_t threads_total = states * 32;
    if (threads_total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (threads_total + threads - 1) / threads;
    merge_kernel<<<blocks, threads, 0, s>>>(o_a, lse_a, o_b, lse_b, in_f32, states, head_dim,
                                            o_out, out_f32, lse_out);
    return cudaGetLastError();
}

cudaError_t launch_split_reduce(const AttnParams& p, cudaStream_t s) {
    const int warps = p.max_q_rows * p.num_q_heads;
    const int threads = 256;
    dim3 grid((warps * 32 + threads - 1) / threads, p.batch);
    if (p.head_dim == 128) {
        split_reduce_kernel<128><<<grid, threads, 0, s>>>(p);
    } else {
        split_reduce_kernel<64><<<grid, threads, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace pkv
