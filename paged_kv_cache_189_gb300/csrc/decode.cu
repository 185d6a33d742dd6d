// decode.cu -- paged attention for one query row per sequence (decode).
//
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Attention (paged attention over 32-token pages through the block table,
// real-token seq_len, zeroed padding rows) and "Support shared-prefix attention
// for n-sample requests in FMHA", split-KV commit notes (when a batch cannot
// fill the GPU, cut every row's keys into chunks of at least 512 tokens,
// attend each chunk, then merge the chunk states by LSE).
//
// Decode is bound by HBM: every K/V byte is read once and used for Hq/Hkv
// query heads.  The GB300 design:
//  * grid (split, K/V head, sequence); a split is 512 keys = 16 pages; CTAs
//    whose split lies past the sequence's length exit at once, so the grid is
//    sized from the host bound max_kv_len and stays graph-capturable.
//  * one producer warp streams whole pages of one K/V head (32 x D of K and
//    of V, two TMA boxes per 128 columns with 128-byte swizzling) into a
//    4-stage shared-memory ring, completion on mbarriers.
//  * four consumer warps each own 8 of a page's 32 keys (rows 8w..8w+7) and
//    keep their own online-softmax state over their keys, so no cross-warp
//    synchronisation is needed per page; the four states are merged once at
//    the end.
//  * QK: lane = (key k of 4, segment s of 8); a segment is 16 (D=128) or 8
//    (D=64) dims whose query values live in registers for the whole call; the
//    segment-to-chunk assignment makes every 8-lane phase of a 16-byte shared
//    load hit 8 distinct bank groups under the swizzle.  Partial dots are
//    summed across the 8 segments with shuffles.
//  * PV: lane owns D/32 consecutive output dims for all G heads; the
//    probabilities are broadcast through a small shared buffer.
//  * fp32 accumulation, base-2 online softmax with the scale folded into q,
//    the running output rescaled only when the running maximum moves.
#include <cuda.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kPage = 32;
constexpr int kWarps = 4;       // consumer warps
constexpr int kStages = 4;      // pages in flight per CTA
constexpr int kThreads = (kWarps + 1) * 32;

template <int D, int G>
struct DecodeSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = kPage * D * 2;          // one page-head of K (or V)
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kPbufOff = kRingBytes;                // [warps][8 keys][G] f32
    static constexpr int kPbufBytes = kWarps * 8 * G * 4;
    static constexpr int kRedOff = kPbufOff + kPbufBytes;      // m, l: [warps][G] f32 each
    static constexpr int kRedBytes = 2 * kWarps * G * 4;
    static constexpr int kBarOff = (kRedOff + kRedBytes + 7) & ~7;
    static constexpr int kBytes = kBarOff + 2 * kStages * 8;
    static constexpr int kAlloc = kBytes + 1024;               // slack for 1024-byte alignment
    static_assert(kWarps * G * D * 4 <= kRingBytes, "output reduction reuses the ring");
};

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 3)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const AttnParams p) {
    using S = DecodeSmem<D, G>;
    constexpr int kSegDims = D / 8;   // query dims held per QK lane
    constexpr int kDPL = D / 32;      // output dims per PV lane
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
    uint64_t* empty = full + kStages;
    float* pbuf = reinterpret_cast<float*>(smem + S::kPbufOff);
    float* red_m = reinterpret_cast<float*>(smem + S::kRedOff);
    float* red_l = red_m + kWarps * G;
    float* red_o = reinterpret_cast<float*>(smem);  // reuses the ring after the main loop

    const int split = blockIdx.x;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int r0 = p.q_indptr[b];
    const int nrows = p.q_indptr[b + 1] - r0;
    if (nrows <= 0) return;
    const int qreal = p.q_real ? p.q_real[b] : nrows;
    int kv_len = p.kv_lens[b];
    if (p.checked && threadIdx.x == 0 && split == 0 && kvh == 0 &&
        (kv_len > p.max_kv_len || kv_len < 0 || nrows > 1))
        set_err(p.err, PKV_ERRBIT_LEN);
    kv_len = min(max(kv_len, 0), p.max_kv_len);
    if (qreal <= 0) kv_len = 0;  // a padding row attends nothing
    const int key_begin = split * p.split_keys;
    const int key_end = min(kv_len, key_begin + p.split_keys);
    const int Hq = p.num_q_heads;

    if (key_end <= key_begin) {
        // no keys here: with a single split this CTA owns the final output row
        if (p.num_splits == 1 && split == 0) {
            for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
                const int h = kvh * G + e / D;
                const int64_t o = (static_cast<int64_t>(r0) * Hq + h) * D + (e % D);
                if (p.out_f32) static_cast<float*>(p.out)[o] = 0.f;
                else static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(0.f);
                if (p.lse && (e % D) == 0) p.lse[static_cast<int64_t>(r0) * Hq + h] = -INFINITY;
            }
        }
        return;
    }
    const int npages = (key_end - key_begin + kPage - 1) / kPage;
    const int page0 = key_begin / kPage;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kWarps) {
        // ---------------- producer: one lane issues the page loads ----------
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.block_table_stride + page0;
            int issued = 0;
            for (int i = 0; i < npages; ++i) {
                const int st = i % kStages;
                if (i >= kStages && !mbar_wait(&empty[st], ((i / kStages) - 1) & 1)) {
                    set_err(p.err, PKV_ERRBIT_TIMEOUT);
                    break;
                }
                int phys = bt[i];
                if (p.checked && (phys < 0 || phys >= p.num_pages)) {
                    set_err(p.err, PKV_ERRBIT_PAGE);
                    phys = static_cast<int>(p.num_pages);  // out of the tensor: TMA fills zeros
                }
                uint8_t* kd = smem + st * S::kStageBytes;
                uint8_t* vd = kd + S::kTileBytes;
                mbar_arrive_expect_tx(&full[st], S::kStageBytes);
#pragma unroll
                for (int h = 0; h < S::kHalves; ++h) {
                    tma_load_4d(kd + h * 4096, &tm_k, &full[st], h * 64, kvh, 0, phys);
                    tma_load_4d(vd + h * 4096, &tm_v, &full[st], h * 64, kvh, 0, phys);
                }
                issued = i + 1;
            }
            // do not leave while copies into this CTA's shared memory are in flight
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(&full[i % kStages], (i / kStages) & 1);
        }
        return;
    }

    // ---------------- consumers ---------------------------------------------
    const int kk = lane >> 3;   // key within a pass of 4
    const int seg = lane & 7;   // QK segment
    // chunks (16 bytes = 8 dims) of a 128-column half that this segment reads
    const int half = (D == 128) ? (seg >> 2) : 0;
    const int c0 = (D == 128) ? ((seg & 3) + 4 * (seg >> 2)) : seg;
    const int c1 = c0 ^ 4;

    float q[G][kSegDims];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const __nv_bfloat16* qh = static_cast<const __nv_bfloat16*>(p.q) +
                                  static_cast<int64_t>(r0) * p.q_token_stride +
                                  static_cast<int64_t>(kvh * G + g) * p.q_head_stride +
                                  half * 64;
        const uint4 a = *reinterpret_cast<const uint4*>(qh + c0 * 8);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            q[g][2 * j] = bf16lo(wa[j]) * p.scale_log2;
            q[g][2 * j + 1] = bf16hi(wa[j]) * p.scale_log2;
        }
        if constexpr (D == 128) {
            const uint4 c = *reinterpret_cast<const uint4*>(qh + c1 * 8);
            const uint32_t wc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                q[g][8 + 2 * j] = bf16lo(wc[j]) * p.scale_log2;
                q[g][8 + 2 * j + 1] = bf16hi(wc[j]) * p.scale_log2;
            }
        }
    }

    float m[G], l[G], o[G][kDPL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int j = 0; j < kDPL; ++j) o[g][j] = 0.f;
    }
    float* pb = pbuf + warp * 8 * G;
    // PV addressing of this lane's output dims [lane*kDPL, lane*kDPL + kDPL)
    const int pv_half = (D == 128) ? (lane >> 4) : 0;
    const int pv_chunk = (D == 128) ? ((lane & 15) >> 1) : (lane >> 2);
    const int pv_byte = (D == 128) ? ((lane & 1) * 8) : ((lane & 3) * 4);

    bool ok = true;
    for (int i = 0; i < npages; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(&full[st], (i / kStages) & 1)) {
            if (lane == 0) set_err(p.err, PKV_ERRBIT_TIMEOUT);
            ok = false;
            break;
        }
        const uint8_t* K = smem + st * S::kStageBytes;
        const uint8_t* V = K + S::kTileBytes;
        const int key0 = key_begin + i * kPage;

        float s[2][G];
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int row = warp * 8 + pass * 4 + kk;
            float acc[G];
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] = 0.f;
            {
                const uint4 a = *reinterpret_cast<const uint4*>(K + half * 4096 + sw128_offset(row, c0));
                const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float k0 = bf16lo(w[j]), k1 = bf16hi(w[j]);
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] = fmaf(q[g][2 * j + 1], k1, fmaf(q[g][2 * j], k0, acc[g]));
                }
            }
            if constexpr (D == 128) {
                const uint4 a = *reinterpret_cast<const uint4*>(K + half * 4096 + sw128_offset(row, c1));
                const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float k0 = bf16lo(w[j]), k1 = bf16hi(w[j]);
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        acc[g] = fmaf(q[g][8 + 2 * j + 1], k1, fmaf(q[g][8 + 2 * j], k0, acc[g]));
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 1);
                acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 2);
                acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 4);
            }
            const bool valid = key0 + row < key_end;
#pragma unroll
            for (int g = 0; g < G; ++g) s[pass][g] = valid ? acc[g] : -INFINITY;
        }

        // online softmax over this warp's 8 keys of the page
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = fmaxf(s[0][g], s[1][g]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m[g], mx);
            float p0 = 0.f, p1 = 0.f;
            if (m_new != -INFINITY) {
                if (m_new != m[g]) {  // warp-uniform
                    const float alpha = fast_exp2(m[g] - m_new);
                    l[g] *= alpha;
#pragma unroll
                    for (int j = 0; j < kDPL; ++j) o[g][j] *= alpha;
                    m[g] = m_new;
                }
                p0 = fast_exp2(s[0][g] - m_new);
                p1 = fast_exp2(s[1][g] - m_new);
            }
            if (seg == 0) {
                l[g] += p0 + p1;
                pb[kk * G + g] = p0;
                pb[(4 + kk) * G + g] = p1;
            }
        }
        __syncwarp();

        // PV over the warp's valid keys of this page
        const int nvalid = min(8, key_end - (key0 + warp * 8));
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            if (k8 < nvalid) {
                const int row = warp * 8 + k8;
                float pg[G];
#pragma unroll
                for (int g = 0; g < G; ++g) pg[g] = pb[k8 * G + g];
                const uint8_t* vp = V + pv_half * 4096 + sw128_offset(row, pv_chunk) + pv_byte;
                float v[kDPL];
                if constexpr (kDPL == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(vp);
                    v[0] = bf16lo(w.x); v[1] = bf16hi(w.x);
                    v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
                    v[0] = bf16lo(w); v[1] = bf16hi(w);
                }
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int j = 0; j < kDPL; ++j) o[g][j] = fmaf(pg[g], v[j], o[g][j]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    (void)ok;

    // ---------------- merge the four warps' states ---------------------------
#pragma unroll
    for (int g = 0; g < G; ++g) l[g] = warp_sum(l[g]);
    // every consumer is past its last shared read of the ring once all have
    // arrived here; the producer only waits on barriers from now on.
    asm volatile("bar.sync 1, %0;" ::"r"(kWarps * 32) : "memory");
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            red_m[warp * G + g] = m[g];
            red_l[warp * G + g] = l[g];
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < kDPL; ++j) red_o[(warp * G + g) * D + lane * kDPL + j] = o[g][j];
    asm volatile("bar.sync 1, %0;" ::"r"(kWarps * 32) : "memory");

    const int S_ = p.num_splits;
    for (int e = threadIdx.x; e < G * D; e += kWarps * 32) {
        const int g = e / D, d = e - (e / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * G + g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = fast_exp2(red_m[w * G + g] - M);
                L = fmaf(f, red_l[w * G + g], L);
                O = fmaf(f, red_o[(w * G + g) * D + d], O);
            }
        }
        const float inv = L > 0.f ? 1.0f / L : 0.f;
        O *= inv;
        const float lse = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
        const int h = kvh * G + g;
        const int64_t st = static_cast<int64_t>(r0) * Hq + h;
        if (S_ == 1) {
            if (p.out_f32) static_cast<float*>(p.out)[st * D + d] = O;
            else static_cast<__nv_bfloat16*>(p.out)[st * D + d] = __float2bfloat16_rn(O);
            if (p.lse && d == 0) p.lse[st] = lse;
        } else if (r0 < static_cast<int64_t>(p.batch) * p.max_q_rows) {  // workspace bound
            p.ws_o[(st * S_ + split) * D + d] = O;
            if (d == 0) p.ws_lse[st * S_ + split] = lse;
        }
    }
}

template <int D, int G>
cudaError_t launch_dg(const AttnParams& p, const void* tk, const void* tv, cudaStream_t s) {
    using S = DecodeSmem<D, G>;
    auto kern = decode_kernel<D, G>;
    // per device context; cheap, and not a stream operation (safe under capture)
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         S::kAlloc);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    kern<<<grid, kThreads, S::kAlloc, s>>>(*static_cast<const CUtensorMap*>(tk),
                                           *static_cast<const CUtensorMap*>(tv), p);
    return cudaGetLastError();
}

}  // namespace

bool decode_supported(int head_dim, int group) {
    return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4);
}

cudaError_t launch_decode(const AttnParams& p, const void* tk, const void* tv, cudaStream_t s) {
    const int G = p.num_q_heads / p.num_kv_heads;
#define PKV_DEC(D_, G_) \
    if (p.head_dim == D_ && G == G_) return launch_dg<D_, G_>(p, tk, tv, s);
    PKV_DEC(128, 4) PKV_DEC(128, 2) PKV_DEC(128, 1)
    PKV_DEC(64, 4) PKV_DEC(64, 2) PKV_DEC(64, 1)
#undef PKV_DEC
    return cudaErrorInvalidValue;
}

}  // namespace pkv
