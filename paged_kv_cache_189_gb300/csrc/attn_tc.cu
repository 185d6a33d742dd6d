// attn_tc.cu -- paged attention for many query rows on the 5th-generation
// tensor cores (tcgen05 MMA, accumulators in tensor memory, TMA-fed).
//
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Attention and Cache (paged attention over per-block rows through the block
// table, 32-token pages, frame-causal blocks, a real-token count with padding
// rows returned as zeros), and "Support shared-prefix attention for n-sample
// requests in FMHA" (the group's rows attend the shared pages once and return
// output + LSE for the merge).  Prefill, block-causal and shared-prefix tiles
// are dense contractions: enough query rows share each K/V page.
//
// Two kernels: the one-tile kernel described next (sequences whose rows fit
// one tile, grouped shared-prefix tiles, rows held four times for few rows),
// and the two-tile kernel further down (two 128-row tiles per CTA sharing
// every K/V tile, for sequences with more rows).  Both issue their MMAs from
// one lane in batches of eight with the next K/V tile's barrier probed inside
// a batch.
//
// One-tile kernel: one CTA = one tile of 128 query rows packed as (token, grouped head): token
// t0 + r / G, query head kvh * G + r % G for tensor-memory lane r, so the G
// query heads that share a K/V head share every K/V load.  Keys are walked in
// tiles of 128 (four 32-token pages) within the CTA's key split.
//
// Roles (224 threads, one CTA per SM):
//  * warps 0-3 (softmax): load the Q tile into swizzled shared memory; for
//    each key tile read S = Q K^T from tensor memory (one row per thread),
//    mask, online softmax in base 2 with a lazily moved maximum, write P as
//    bf16 into shared memory in the MMA's K-major swizzled layout, rescale O
//    in tensor memory when the maximum moved; finally normalise O and store it.
//  * warp 4 lane 0 and warp 6 lane 0 (producers): TMA loads of K pages
//    (2-stage ring) and of V pages (3-stage ring: V of tile j + 3 can only
//    start once P.V of tile j finished, so the deeper ring goes to V), one
//    issuing thread per ring, 4 pages x 2 column halves per 128-key tile,
//    through the block table, whose entries for the next tile are read one
//    tile ahead; pages past the sequence are read out of bounds, which TMA
//    fills with zeros.
//  * warp 5 (MMA): allocates 512 tensor-memory columns (two S buffers and O),
//    issues S_{j+2} = Q K_{j+2}^T and O += P_j V_j with tcgen05.mma
//    (kind::f16, bf16 in, f32 accumulate, M = N = 128), and signals through
//    tcgen05.commit on mbarriers.
// Every mbarrier wait gives up after ~2 s (error bit, orderly exit).
#include <cuda.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kTileM = 128;             // query rows per tile (tensor-memory lanes)
constexpr int kTileN = 128;             // keys per tile
constexpr int kKStages = 2;
constexpr int kVStages = 3;
constexpr int kThreads = 224;
constexpr int kHalfBytes = kTileM * 128;           // 128 rows x 64 bf16 = 16 KiB
constexpr int kPBytes = 2 * kHalfBytes;            // P: 128 rows x 128 keys bf16 = 32 KiB
constexpr int kMaxGroup = 64;           // head groups the tiles take (2 tokens per pair at least)

// Head-dim dependent sizes: a Q, K or V tile is 128 rows of D bf16, stored as
// D / 64 column halves of 128-byte swizzled rows (one TMA box each).
template <int D>
struct TileDim {
    static_assert(D == 64 || D == 128, "head dim 64 or 128");
    static constexpr int kHalves = D / 64;
    static constexpr int kChunks = D / 8;        // 16-byte chunks of a row
    static constexpr int kTile = kHalves * kHalfBytes;
    // one-tile kernel: Q, K ring, V ring, P, barriers, tensor-memory slot, flags, exchange
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kTile;
    static constexpr int kVOff = kKOff + kKStages * kTile;
    static constexpr int kPOff = kVOff + kVStages * kTile;
    static constexpr int kBarOff = kPOff + kPBytes;
};
// barriers: q_ready, k_full[2], k_empty[2], v_full[3], v_empty[3], s_full[2], p_full, p_free,
// mma_done
constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 1;
template <int D>
struct OneTileSmem {
    static constexpr int kTmemSlotOff = TileDim<D>::kBarOff + kNumBars * 8;
    static constexpr int kFlagOff = kTmemSlotOff + 8;
    static constexpr int kXchOff = kFlagOff + 16;   // replicated rows: [2][4][32] maxima, [2][4][32] sums
    static constexpr int kBytes = kXchOff + 2 * 2 * 4 * 32 * 4;
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
};
constexpr uint32_t kTmemCols = 512;     // S0 [0,128), S1 [128,256), O [256,256 + D)
constexpr float kLazyRescale = 8.0f;    // move the running max only past 2^8 growth
constexpr int kOrderMaxBatch = 128;     // longest-first dispatch up to this batch (B^2 ranking)

// ---------------------------------------------------------------------------
// tcgen05 wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(slot)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// arrive on the mbarrier once all previously issued tcgen05 operations of this thread completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

#define PKV_R8(i) "=r"(v[i + 0]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), \
                  "=r"(v[i + 4]), "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])
// 32 consecutive 32-bit columns of this thread's lane; waits for completion
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
        : "r"(taddr) : "memory");
}
// 128 consecutive 32-bit columns (four 32-column loads, one wait)
__device__ __forceinline__ void tmem_load128(uint32_t taddr, uint32_t (&v)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%129];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
        "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95}, [%130];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, "
        "%111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, "
        "%126, %127}, [%131];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24), PKV_R8(32), PKV_R8(40), PKV_R8(48),
          PKV_R8(56), PKV_R8(64), PKV_R8(72), PKV_R8(80), PKV_R8(88), PKV_R8(96), PKV_R8(104),
          PKV_R8(112), PKV_R8(120)
        : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96) : "memory");
}
#undef PKV_R8
#define PKV_W8(i) "r"(v[i + 0]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), \
                  "r"(v[i + 4]), "r"(v[i + 5]), "r"(v[i + 6]), "r"(v[i + 7])
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;"
        ::"r"(taddr), PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24) : "memory");
}
// entries 0..63 of v to 64 consecutive columns (two 32-column stores); the caller waits
__device__ __forceinline__ void tmem_store64_nowait(uint32_t taddr, const uint32_t (&v)[128]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%33], "
        "{%34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, "
        "%50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65};"
        ::"r"(taddr), PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24), "r"(taddr + 32), PKV_W8(32), PKV_W8(40),
          PKV_W8(48), PKV_W8(56) : "memory");
}
#undef PKV_W8

// max of three values in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// acc += the two bf16 values of a packed pair, each widened exactly to f32
__device__ __forceinline__ void add_bf16x2(float2& acc, uint32_t pk) {
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\t"
        "add.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(acc.x), "+f"(acc.y) : "r"(pk));
}
// named barrier `id` over `count` threads that also returns the AND of `pred`
__device__ __forceinline__ bool bar_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r) : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count) : "memory");
    return r != 0;
}
__device__ __forceinline__ void bar_sync_n(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, start address, leading
// and stride byte offsets (all in 16-byte units), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, A K-major,
// B K-major or MN-major, M and N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ int visible_keys(int i, int qreal, int kv_len, int mask, int cb) {
    if (i >= qreal) return 0;
    const int first_new = kv_len - qreal;
    if (mask == PKV_MASK_NONE) return kv_len;
    if (mask == PKV_MASK_CAUSAL) return first_new + i + 1;
    const int block_end = (i / cb + 1) * cb;
    return first_new + min(qreal, block_end);
}

struct TileGeom {
    int b, kvh, split, r0, nrows, qreal, kv_len, t0, kb, key_hi, nt;
};

// The sequence at position `pos` when the batch is ordered by key count,
// longest first (ties by index; any count order gives a permutation).  Every
// thread of the block calls it; `scratch` holds 2 * batch + 1 ints of shared
// memory that nothing else uses yet.
__device__ int longest_first(const AttnParams& p, int pos, int* scratch) {
    const int B = p.batch;
    int* rank = scratch;
    int* keys = scratch + B + 1;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        rank[i] = 0;
        keys[i] = p.kv_lens[i];
    }
    __syncthreads();
    for (int pi = threadIdx.x; pi < B * B; pi += blockDim.x) {
        const int b = pi / B, o = pi - b * B;
        if (keys[o] > keys[b] || (keys[o] == keys[b] && o < b)) atomicAdd(&rank[b], 1);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < B; b += blockDim.x)
        if (rank[b] == pos) rank[B] = b;
    __syncthreads();
    return rank[B];
}

__device__ __forceinline__ TileGeom tile_geometry(const AttnParams& p, int TQ, int b) {
    TileGeom g;
    g.b = b;
    g.split = blockIdx.z - (blockIdx.z / p.num_splits) * p.num_splits;
    g.kvh = blockIdx.y;
    g.r0 = p.q_indptr[g.b];
    g.nrows = min(p.q_indptr[g.b + 1] - g.r0, p.max_q_rows);
    g.t0 = blockIdx.x * TQ;
    g.qreal = min(p.q_real ? p.q_real[g.b] : g.nrows, g.nrows);
    g.kv_len = min(max(p.kv_lens[g.b], 0), p.max_kv_len);
    g.kb = g.split * p.split_keys;
    const int ke = min(g.kv_len, g.kb + p.split_keys);
    // visibility is non-decreasing in the row, so the tile's last real row bounds it
    const int last = min(g.t0 + TQ, g.nrows) - 1;
    int lim = 0;
    if (g.t0 < g.qreal)
        lim = visible_keys(min(last, g.qreal - 1), g.qreal, g.kv_len, p.mask, max(p.causal_block, 1));
    g.key_hi = min(ke, lim);
    g.nt = g.key_hi > g.kb ? (g.key_hi - g.kb + kTileN - 1) / kTileN : 0;
    return g;
}

// Columns [32c, 32c + 32) of one row's normalised output (or split partial).
template <int D>
__device__ __forceinline__ void store_row_chunk(const AttnParams& p, const TileGeom& g, int row_in_seq,
                                                int h, int c, const uint32_t (&v)[32], float inv_l) {
    const int64_t st = static_cast<int64_t>(g.r0 + row_in_seq) * p.num_q_heads + h;
    float o[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(v[e]) * inv_l;
    if (p.num_splits == 1 && !p.out_f32) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + st * D + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf16x2(o[8 * q], o[8 * q + 1]), pack_bf16x2(o[8 * q + 2], o[8 * q + 3]),
                                pack_bf16x2(o[8 * q + 4], o[8 * q + 5]), pack_bf16x2(o[8 * q + 6], o[8 * q + 7]));
        return;
    }
    float* base;
    if (p.num_splits == 1) {
        base = static_cast<float*>(p.out) + st * D;
    } else {
        if (g.r0 + row_in_seq >= static_cast<int64_t>(p.batch) * p.max_q_rows) return;
        base = p.ws_o + (st * p.num_splits + g.split) * D;
    }
    float4* dst = reinterpret_cast<float4*>(base + c * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}
__device__ __forceinline__ void store_row_lse(const AttnParams& p, const TileGeom& g, int row_in_seq,
                                              int h, float lse) {
    const int64_t st = static_cast<int64_t>(g.r0 + row_in_seq) * p.num_q_heads + h;
    if (p.num_splits == 1) {
        if (p.lse) p.lse[st] = lse;
    } else if (g.r0 + row_in_seq < static_cast<int64_t>(p.batch) * p.max_q_rows) {
        p.ws_lse[st * p.num_splits + g.split] = lse;
    }
}

// ---------------------------------------------------------------------------
// Grouped mode: the rows of a tile are the query tokens of one shared-prefix
// group (its members in order, each member's tokens in order) x the G heads.
// ---------------------------------------------------------------------------
struct GroupRow {
    int tok;      // token index in q / out (-1: no such row)
    int a, b, c;  // visible keys of the group row: [0, a) u [b, c)
};

// Token t of group slot `grp` (its members grp_perm[first .. first + count)).
// Member m's tokens are its last keys: token i of ql sees the shared run and
// its tail up to its own position (causal inside the tail).
__device__ __forceinline__ GroupRow group_row(const AttnParams& p, int grp, int first, int count, int t) {
    GroupRow gr{-1, 0, 0, 0};
    int acc = 0;
    for (int k = 0; k < count; ++k) {
        const int m = p.grp_perm[first + k];
        const int q0 = p.q_indptr[m], ql = p.q_indptr[m + 1] - q0;
        if (t < acc + ql) {
            const int i = t - acc;
            gr.tok = q0 + i;
            gr.a = p.grp_run_lens[grp];
            gr.b = 32 * p.grp_tail_start[m];
            gr.c = gr.b + p.grp_tail_lens[m] - ql + i + 1;
            return gr;
        }
        acc += ql;
    }
    return gr;
}

// Group slot, split and token tile of this CTA; nrows = the group's tokens
// (0 for a slot past the number of groups).
__device__ __forceinline__ TileGeom group_geometry(const AttnParams& p, int TQ, int& first, int& count) {
    TileGeom g;
    g.b = blockIdx.z / p.num_splits;
    g.split = blockIdx.z - g.b * p.num_splits;
    g.kvh = blockIdx.y;
    g.r0 = 0;
    g.t0 = blockIdx.x * TQ;
    g.kb = g.split * p.split_keys;
    g.nrows = g.qreal = g.kv_len = g.key_hi = g.nt = 0;
    first = count = 0;
    if (g.b >= *p.grp_num_groups) return g;
    first = p.grp_indptr[g.b];
    count = p.grp_indptr[g.b + 1] - first;
    int T = 0;
    for (int k = 0; k < count; ++k) {
        const int m = p.grp_perm[first + k];
        T += p.q_indptr[m + 1] - p.q_indptr[m];
    }
    g.nrows = g.qreal = T;
    return g;
}

// GC: the head group when fixed at compile time (the common 1, 2, 4, 8, 16),
// 0 to read it from the call
template <int D, int GC, bool GRP, int REP>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const AttnParams p) {
    using TD = TileDim<D>;
    using SM = OneTileSmem<D>;
    constexpr int ND = kTileM / REP;  // distinct rows of the tile (each held REP times)
    const int G = GC > 0 ? GC : p.num_q_heads / p.num_kv_heads;
    const int TQ = ND / G;            // tokens of the tile; rows from TQ * G on hold none
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    TileGeom g;
    int grp_first = 0, grp_count = 0;
    if constexpr (!GRP) {
        int b = blockIdx.z / p.num_splits;
        if (p.order_by_keys) b = longest_first(p, b, reinterpret_cast<int*>(smem + TD::kKOff));
        g = tile_geometry(p, TQ, b);
        if (g.t0 >= g.nrows) return;  // tile past this sequence's rows (uniform)
    } else {
        g = group_geometry(p, TQ, grp_first, grp_count);
        if (g.t0 >= g.nrows) return;  // empty group slot, or tile past the group's tokens
        // the keys the tile's rows see end at the largest of their visible ends
        // (reduced in the flag area of shared memory, initialised further down)
        int* s_keyhi = reinterpret_cast<int*>(smem + SM::kFlagOff + 8);
        if (threadIdx.x == 0) *s_keyhi = 0;
        __syncthreads();
        if (threadIdx.x < TQ * G) {
            const GroupRow gr = group_row(p, g.b, grp_first, grp_count, g.t0 + threadIdx.x / G);
            if (gr.tok >= 0) atomicMax(s_keyhi, max(gr.a, gr.c));
        }
        __syncthreads();
        g.kv_len = *s_keyhi;
        g.key_hi = min(g.kv_len, g.kb + p.split_keys);
        g.nt = g.key_hi > g.kb ? (g.key_hi - g.kb + kTileN - 1) / kTileN : 0;
    }

    if (g.nt == 0) {
        // no visible key in this split for any row of the tile: empty states
        if (threadIdx.x < TQ * G) {
            const int r = threadIdx.x;
            int i = g.t0 + r / G;
            bool exists = i < g.nrows;
            if constexpr (GRP) {
                const GroupRow gr = group_row(p, g.b, grp_first, grp_count, i);
                i = gr.tok;
                exists = gr.tok >= 0;
            }
            if (exists) {
                uint32_t zero[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) zero[e] = 0u;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) store_row_chunk<D>(p, g, i, g.kvh * G + r % G, c, zero, 0.f);
                store_row_lse(p, g, i, g.kvh * G + r % G, -INFINITY);
            }
        }
        return;
    }
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzle needs 1024-byte aligned tiles
        if (threadIdx.x == 0) set_err(p.err, PKV_ERRBIT_TIMEOUT);
        return;
    }

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TD::kBarOff);
    uint64_t* q_ready = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + kKStages;
    uint64_t* v_full = k_empty + kKStages;
    uint64_t* v_empty = v_full + kVStages;
    uint64_t* s_full = v_empty + kVStages;
    uint64_t* p_full = s_full + 2;
    uint64_t* p_free = p_full + 1;
    uint64_t* mma_done = p_free + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kTmemSlotOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::kFlagOff);

    if (threadIdx.x == 0) {
        mbar_init(q_ready, kTileM);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(p_full, kTileM);
        mbar_init(p_free, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(smem);
    // grouped mode: the keys [g0, g1) of member k's last tail page past its tail
    // (seen by no row); members' tails follow each other in the group row, so
    // these gaps come in increasing key order
    auto member_gap = [&](int k, int& g0, int& g1) {
        const int m = p.grp_perm[grp_first + k];
        g0 = 32 * p.grp_tail_start[m] + p.grp_tail_lens[m];
        g1 = (g0 + 31) / 32 * 32;
    };

    // a completed phase passes at once; a wait that gives up marks the CTA
    // aborted, and later pending waits return at once
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (mbar_wait(bar, parity)) return true;
        *abort_flag = 1;
        set_err(p.err, PKV_ERRBIT_TIMEOUT);
        return false;
    };

    if (warp == 4 || warp == 6) {
        // ============================ producers =============================
        // Lane 0 of warp 4 streams the K tiles, lane 0 of warp 6 the V tiles,
        // each through its own ring, so one ring's copies are issued while the
        // other thread waits for a free stage.  Each reads the next tile's
        // block-table entries one tile ahead (before that wait), so a freed
        // stage is refilled without a dependent global read in between.
        if (lane == 0) {
            const bool is_k = warp == 4;
            const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
            prefetch_tmap(tm);
            const int stages = is_k ? kKStages : kVStages;
            uint8_t* ring = smem + (is_k ? TD::kKOff : TD::kVOff);
            uint64_t* full = is_k ? k_full : v_full;
            uint64_t* empty = is_k ? k_empty : v_empty;
            const int32_t* bt = p.block_table + static_cast<int64_t>(g.b) * p.block_table_stride;
            const int last_page = (g.kv_len + 31) / 32;  // pages at or past it are never read
            // the physical pages of key tile j (past the last page: the
            // out-of-range sentinel, which the copy fills with zeros)
            auto fetch_pages = [&](int j, int (&ph)[4]) {
#pragma unroll
                for (int pg = 0; pg < 4; ++pg) {
                    const int lp = (g.kb + j * kTileN) / 32 + pg;
                    ph[pg] = lp < last_page ? bt[lp] : static_cast<int>(p.num_pages);
                }
            };
            int next[4] = {0, 0, 0, 0};
            if (g.nt > 0) fetch_pages(0, next);
            int issued = 0;
            for (; issued < g.nt; ++issued) {
                const int s = issued % stages;
                const int cur[4] = {next[0], next[1], next[2], next[3]};
                if (issued + 1 < g.nt) fetch_pages(issued + 1, next);
                if (issued >= stages && !wait(&empty[s], ((issued / stages) - 1) & 1)) break;
                mbar_arrive_expect_tx(&full[s], TD::kTile);
#pragma unroll
                for (int pg = 0; pg < 4; ++pg) {
                    const int lp = (g.kb + issued * kTileN) / 32 + pg;
                    int phys = cur[pg];
                    if (p.checked && lp < last_page && (phys < 0 || phys >= p.num_pages)) {
                        set_err(p.err, PKV_ERRBIT_PAGE);
                        phys = static_cast<int>(p.num_pages);
                    }
#pragma unroll
                    for (int h = 0; h < TD::kHalves; ++h)
                        tma_load_4d(ring + s * TD::kTile + h * kHalfBytes + pg * 4096, tm, &full[s], h * 64, g.kvh,
                                    0, phys);
                }
            }
            // do not leave with copies into this CTA's shared memory in flight
            for (int j = max(0, issued - stages); j < issued; ++j) mbar_wait(&full[j % stages], (j / stages) & 1);
        }
    } else if (warp == 5) {
        // ============================== MMA ================================
        // As in the two-tile kernel: an MMA issue returns about when the
        // previous one is done, so the waits for K and V tiles sit inside a
        // batch (after its fourth MMA) and each batch builds its descriptors once.
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(kTileM, kTileN, false);  // K rows are K-major
            constexpr uint32_t kIdescO = idesc_bf16(kTileM, D, true);        // V rows are MN-major
            const uint32_t tmem_o = tmem + 256;
            const uint64_t dq = sdesc_sw128(sbase + TD::kQOff, 16, 1024);
            // A = P (K-major over keys): the same layout and offsets as Q
            const uint64_t dp = sdesc_sw128(sbase + TD::kPOff, 16, 1024);
            auto issue_s = [&](int j, auto&& mid) {
                const int s = j % kKStages;
                const uint64_t db = sdesc_sw128(sbase + TD::kKOff + s * TD::kTile, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                    umma_bf16(tmem + (j & 1) * 128, dq + off, db + off, kIdescS, kk > 0);
                    if (kk == 3) mid();
                }
                umma_commit(&s_full[j & 1]);
                umma_commit(&k_empty[s]);
            };
            const int nt = g.nt;
            // a tile's barrier is probed inside the batch before it; if its
            // copy has not landed, the batch goes on and the wait comes after
            bool ready = false;
            auto probe = [&](uint64_t* bar, uint32_t parity) {
                ready = mbar_test(bar, parity);
                if (ready) tc_fence_after();
            };
            auto settle = [&](uint64_t* bar, uint32_t parity) -> bool {
                if (ready) return true;
                if (!wait(bar, parity)) return false;
                tc_fence_after();
                return true;
            };
            bool ok = wait(q_ready, 0) && wait(&k_full[0], 0);
            if (ok) {
                tc_fence_after();
                issue_s(0, [&] {
                    if (nt > 1) probe(&k_full[1 % kKStages], (1 / kKStages) & 1);
                });
                if (nt > 1) {
                    ok = settle(&k_full[1 % kKStages], (1 / kKStages) & 1);
                    if (ok) issue_s(1, [&] { probe(&v_full[0], 0); });
                } else {
                    ready = false;
                }
                ok = ok && settle(&v_full[0], 0);
            }
            for (int j = 0; ok && j < nt; ++j) {
                // V_j was waited for inside an earlier batch
                if (!wait(p_full, j & 1)) break;
                tc_fence_after();
                const bool s_next = j + 2 < nt;
                const uint64_t bd = sdesc_sw128(sbase + TD::kVOff + (j % kVStages) * TD::kTile, kHalfBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < kTileN / 16; ++kk) {
                    // A = P (K-major over keys), B = V (rows = keys, columns = dims: MN-major);
                    // the two 64-column halves of V are LBO apart, 8-key groups SBO apart
                    const uint32_t offp = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                    umma_bf16(tmem_o, dp + offp, bd + ((kk * 16 * 128) >> 4), kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
                    if (kk == 3 && s_next) probe(&k_full[(j + 2) % kKStages], ((j + 2) / kKStages) & 1);
                }
                umma_commit(&v_empty[j % kVStages]);
                umma_commit(p_free);
                const bool v_next = j + 1 < nt;
                if (s_next) {
                    if (!settle(&k_full[(j + 2) % kKStages], ((j + 2) / kKStages) & 1)) break;
                    issue_s(j + 2, [&] {
                        if (v_next) probe(&v_full[(j + 1) % kVStages], ((j + 1) / kVStages) & 1);
                    });
                } else {
                    ready = false;
                }
                if (v_next && !settle(&v_full[(j + 1) % kVStages], ((j + 1) / kVStages) & 1)) break;
            }
            // nothing of this thread's still runs in the tensor pipe when the
            // CTA winds down (after a failed wait the last batch may be running)
            umma_commit(mma_done);
            if (!mbar_wait(mma_done, 0)) set_err(p.err, PKV_ERRBIT_TIMEOUT);
        }
    } else if (warp < 4) {
        // ============================ softmax ===============================
        if constexpr (REP == 1) {
            const int r = threadIdx.x;             // tile row = tensor-memory lane
            const int t = r / G, hg = r % G;
            const int h = g.kvh * G + hg;
            int i = g.t0 + t;                      // query row within the sequence (grouped: token)
            bool row_exists = t < TQ && i < g.nrows;
            int limit = 0;
            int vis_a = 0, vis_b = 0, vis_c = 0;   // grouped: visible keys [0, a) u [b, c)
            if constexpr (GRP) {
                const GroupRow gr = group_row(p, g.b, grp_first, grp_count, i);
                i = gr.tok;
                row_exists = t < TQ && gr.tok >= 0;
                vis_a = gr.a;
                vis_b = gr.b;
                vis_c = gr.c;
            } else {
                limit = row_exists ? visible_keys(i, g.qreal, g.kv_len, p.mask, max(p.causal_block, 1)) : 0;
            }
            // ---- Q tile -> swizzled shared memory (rows past the sequence: zeros)
            {
                const uint4* src = reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(p.q) + static_cast<int64_t>(g.r0 + i) * p.q_token_stride +
                    static_cast<int64_t>(h) * p.q_head_stride);
    #pragma unroll
                for (int c = 0; c < TD::kChunks; ++c) {
                    const uint4 v = row_exists ? src[c] : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(smem + TD::kQOff + (c >> 3) * kHalfBytes +
                                              sw128_offset(r, c & 7)) = v;
                }
                fence_proxy_async_smem();
                mbar_arrive(q_ready);
            }
            const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
            float m_used = -INFINITY;   // base-2 running maximum used for the exponentials
            float l = 0.f, l_b = 0.f;
            uint8_t* prow = smem + TD::kPOff;
            // warp-collective tensor-memory accesses follow every wait, so a wait
            // counts as passed only if it passed in every lane of the warp
            auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, wait(bar, parity));
            };
            // a warp none of whose rows sees a key (rows past the sequence, padding
            // rows) writes zero probabilities and skips the softmax arithmetic
            const bool warp_live = GRP || __any_sync(0xffffffffu, limit > 0);
            int gap_k = 0;  // grouped: the first member whose tail gap may still meet a key tile
            for (int j = 0; j < g.nt; ++j) {
                if (!wait_warp(&s_full[j & 1], (j >> 1) & 1)) break;
                tc_fence_after();
                uint32_t pk[kTileN / 2];
                float alpha = 1.f;
                bool live = warp_live;
                if constexpr (GRP) {
                    // grouped rows see the shared run and their own tail: per key tile
                    const int k0 = g.kb + j * kTileN;
                    live = __any_sync(0xffffffffu, row_exists && (k0 < vis_a || (k0 < vis_c && k0 + kTileN > vis_b)));
                }
                if (live) {
                    const int key0 = g.kb + j * kTileN;
                    uint32_t sv[kTileN];  // raw scores of this row (f32 bits)
                    tmem_load128(lane_addr + (j & 1) * 128, sv);
                    if constexpr (GRP) {
                        const int ta = vis_a - key0, tb = vis_b - key0, tc = vis_c - key0;
                        if (!row_exists || !(ta >= kTileN || (tb <= 0 && tc >= kTileN))) {
    #pragma unroll
                            for (int e = 0; e < kTileN; ++e)
                                sv[e] = row_exists && (e < ta || (e >= tb && e < tc)) ? sv[e]
                                                                                      : __float_as_uint(-INFINITY);
                        }
                    } else {
                        // keys at or past this row's visible limit are masked (diagonal tiles only)
                        const int nvis = limit - key0;
                        if (nvis < kTileN) {
    #pragma unroll
                            for (int e = 0; e < kTileN; ++e)
                                sv[e] = e < nvis ? sv[e] : __float_as_uint(-INFINITY);
                        }
                    }
                    // row maximum of the raw scores (the scale is positive)
                    float mx = __uint_as_float(sv[0]);
    #pragma unroll
                    for (int e = 1; e + 1 < kTileN; e += 2)
                        mx = fmax3(mx, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                    mx = fmaxf(mx, __uint_as_float(sv[kTileN - 1]));
                    mx *= p.scale_log2;
                    if (mx > m_used + kLazyRescale) {   // also true the first time a key is visible
                        alpha = fast_exp2(m_used - mx);  // 0 when m_used was -inf
                        m_used = mx;
                    }
                    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                    const float nm = m_used == -INFINITY ? 0.f : -m_used;
                    const float2 nm2 = make_float2(nm, nm);
                    float2 rs2 = make_float2(0.f, 0.f), rsb2 = make_float2(0.f, 0.f);
    #pragma unroll
                    for (int e = 0; e < kTileN; e += 2) {
                        // exponent argument s * scale - m for two keys in one packed FMA
                        const float2 xx = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                     sc2, nm2);
                        const float2 pp = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
                        pk[e / 2] = pack_bf16x2(pp.x, pp.y);
                        rs2 = __fadd2_rn(rs2, pp);
                        add_bf16x2(rsb2, pk[e / 2]);
                    }
                    // O is normalised by the sum of the bf16 probabilities the P.V product
                    // used (numerator and denominator carry the same rounding); the LSE
                    // uses the sum of the unrounded ones
                    l = l * alpha + (rs2.x + rs2.y);
                    l_b = l_b * alpha + (rsb2.x + rsb2.y);
                } else {
    #pragma unroll
                    for (int e = 0; e < kTileN / 2; ++e) pk[e] = 0u;
                }
                // P buffer and O are free once the previous P.V finished
                if (j > 0 && !wait_warp(p_free, (j - 1) & 1)) break;
                tc_fence_after();
                if (live && j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // O *= alpha for this row (warp-collective tensor-memory access)
    #pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tmem_load32(lane_addr + 256 + c * 32, v);
    #pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                                         make_float2(alpha, alpha));
                            v[e] = __float_as_uint(o2.x);
                            v[e + 1] = __float_as_uint(o2.y);
                        }
                        tmem_store32(lane_addr + 256 + c * 32, v);
                    }
                }
                const int key0 = g.kb + j * kTileN;
                // P row -> shared memory, K-major 128-byte swizzle, two 64-key halves
    #pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<uint4*>(prow + (c >> 3) * kHalfBytes + sw128_offset(r, c & 7)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                // V rows of keys past the sequence's length inside its last page hold
                // whatever the pool holds there; zero them so 0 * garbage cannot make NaN
                if (key0 + kTileN > g.kv_len && g.kv_len > key0) {
                    const int vs = j % kVStages;
                    if (!wait_warp(&v_full[vs], (j / kVStages) & 1)) break;
                    const int first = g.kv_len - key0;
                    const int last = min(kTileN, (first + 31) / 32 * 32);
                    uint8_t* vt = smem + TD::kVOff + vs * TD::kTile;
                    for (int idx = r; idx < (last - first) * TD::kChunks; idx += kTileM) {
                        const int row = first + idx / TD::kChunks, c = idx % TD::kChunks;
                        *reinterpret_cast<uint4*>(vt + (c >> 3) * kHalfBytes + sw128_offset(row, c & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                if constexpr (GRP) {
                    // the rest of each member's last tail page is seen by no row: zero
                    // those V rows too (same reason)
                    int g0, g1;
                    while (gap_k < grp_count) {  // gaps that end before this key tile
                        member_gap(gap_k, g0, g1);
                        if (g1 > key0) break;
                        ++gap_k;
                    }
                    bool any_gap = false;
                    for (int k = gap_k; k < grp_count; ++k) {
                        member_gap(k, g0, g1);
                        if (g0 >= key0 + kTileN) break;
                        if (g0 < g1) {
                            any_gap = true;
                            break;
                        }
                    }
                    if (any_gap) {
                        const int vs = j % kVStages;
                        if (!wait_warp(&v_full[vs], (j / kVStages) & 1)) break;
                        uint8_t* vt = smem + TD::kVOff + vs * TD::kTile;
                        for (int k = gap_k; k < grp_count; ++k) {
                            member_gap(k, g0, g1);
                            if (g0 >= key0 + kTileN) break;
                            const int lo = max(g0, key0) - key0, hi = min(g1, key0 + kTileN) - key0;
                            for (int idx = r; idx < (hi - lo) * TD::kChunks; idx += kTileM) {
                                const int row = lo + idx / TD::kChunks, c = idx % TD::kChunks;
                                *reinterpret_cast<uint4*>(vt + (c >> 3) * kHalfBytes + sw128_offset(row, c & 7)) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(p_full);
            }
            // ---- epilogue: O / l, 32 columns at a time
            const bool ok = wait_warp(p_free, (g.nt - 1) & 1);
            tc_fence_after();
            const bool any = l > 0.f && l_b > 0.f;
            const float inv_l = any ? 1.0f / l_b : 0.f;
    #pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_load32(lane_addr + 256 + c * 32, v);
                if (ok && row_exists) store_row_chunk<D>(p, g, i, h, c, v, inv_l);
            }
            if (ok && row_exists) store_row_lse(p, g, i, h, any ? (m_used + __log2f(l)) * kLn2 : -INFINITY);
        } else {
            // The tile's ND distinct rows are held REP times: lane r holds distinct row
            // dr = r % ND and, of every 128-key tile, the CW = 128 / REP key columns
            // [part * CW, part * CW + CW), part = r / ND.  Its P row is zero outside
            // them, so the REP copies of a row accumulate disjoint partial sums of O
            // (all with the same running maximum, exchanged every key tile) that the
            // epilogue adds.  REP = 1 is the plain one-row-per-lane tile.
            constexpr int CW = kTileN / REP;
            const int r = threadIdx.x;             // tensor-memory lane
            const int dr = r % ND, part = r / ND;
            const int t = dr / G, hg = dr % G;
            const int h = g.kvh * G + hg;
            int i = g.t0 + t;                      // query row within the sequence (grouped: token)
            bool row_exists = t < TQ && i < g.nrows;
            int limit = 0;
            int vis_a = 0, vis_b = 0, vis_c = 0;   // grouped: visible keys [0, a) u [b, c)
            if constexpr (GRP) {
                const GroupRow gr = group_row(p, g.b, grp_first, grp_count, i);
                i = gr.tok;
                row_exists = t < TQ && gr.tok >= 0;
                vis_a = gr.a;
                vis_b = gr.b;
                vis_c = gr.c;
            } else {
                limit = row_exists ? visible_keys(i, g.qreal, g.kv_len, p.mask, max(p.causal_block, 1)) : 0;
            }
            // ---- Q tile -> swizzled shared memory (rows past the sequence: zeros)
            {
                const uint4* src = reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(p.q) + static_cast<int64_t>(g.r0 + i) * p.q_token_stride +
                    static_cast<int64_t>(h) * p.q_head_stride);
    #pragma unroll
                for (int c = 0; c < TD::kChunks; ++c) {
                    const uint4 v = row_exists ? src[c] : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(smem + TD::kQOff + (c >> 3) * kHalfBytes +
                                              sw128_offset(r, c & 7)) = v;
                }
                fence_proxy_async_smem();
                mbar_arrive(q_ready);
            }
            const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
            float m_used = -INFINITY;   // base-2 running maximum used for the exponentials
            float l = 0.f, l_b = 0.f;
            uint8_t* prow = smem + TD::kPOff;
            float* xmax = reinterpret_cast<float*>(smem + SM::kXchOff);  // [key tile parity][part][dr]
            float* xsum = xmax + 2 * 4 * 32;                          // [l, l_b][part][dr]
            // warp-collective tensor-memory accesses follow every wait, so a wait
            // counts as passed only if it passed in every lane of the warp
            auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, wait(bar, parity));
            };
            // a warp none of whose rows sees a key (rows past the sequence, padding
            // rows) writes zero probabilities and skips the softmax arithmetic
            const bool warp_live = GRP || __any_sync(0xffffffffu, limit > 0);
            // this lane owns its P row; the chunks of the other copies' key columns
            // stay zero for the whole launch, so they are written once here
            if constexpr (REP > 1) {
    #pragma unroll
                for (int c = 0; c < 16; ++c)
                    if (c / (CW / 8) != part)
                        *reinterpret_cast<uint4*>(prow + (c >> 3) * kHalfBytes + sw128_offset(r, c & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
            }
            // with copies, the four warps exchange maxima every key tile; a failed
            // wait is carried to the next exchange, where all of them leave together
            bool ok_run = true;
            int gap_k = 0;  // grouped: the first member whose tail gap may still meet a key tile
            for (int j = 0; j < g.nt; ++j) {
                ok_run = ok_run && wait_warp(&s_full[j & 1], (j >> 1) & 1);
                if (REP == 1 && !ok_run) break;
                tc_fence_after();
                const int key0 = g.kb + j * kTileN;
                const int col0 = key0 + part * CW;  // first key of this lane's columns
                bool live = warp_live;
                if constexpr (GRP) {
                    // grouped rows see the shared run and their own tail: per key tile
                    live = __any_sync(0xffffffffu, row_exists && (key0 < vis_a || (key0 < vis_c && key0 + kTileN > vis_b)));
                }
                uint32_t pk[CW / 2];
                float alpha = 1.f;
                uint32_t sv[CW];  // raw scores of this row's columns (f32 bits)
                float mx = -INFINITY;
                if (ok_run && live) {
                    if constexpr (CW == kTileN) {
                        tmem_load128(lane_addr + (j & 1) * 128, sv);
                    } else {
    #pragma unroll
                        for (int c = 0; c < CW / 32; ++c) {
                            uint32_t v32[32];
                            tmem_load32(lane_addr + (j & 1) * 128 + part * CW + c * 32, v32);
    #pragma unroll
                            for (int e = 0; e < 32; ++e) sv[c * 32 + e] = v32[e];
                        }
                    }
                    if constexpr (GRP) {
                        const int ta = vis_a - col0, tb = vis_b - col0, tc = vis_c - col0;
                        if (!row_exists || !(ta >= CW || (tb <= 0 && tc >= CW))) {
    #pragma unroll
                            for (int e = 0; e < CW; ++e)
                                sv[e] = row_exists && (e < ta || (e >= tb && e < tc)) ? sv[e]
                                                                                      : __float_as_uint(-INFINITY);
                        }
                    } else {
                        // keys at or past this row's visible limit are masked (diagonal tiles only)
                        const int nvis = limit - col0;
                        if (nvis < CW) {
    #pragma unroll
                            for (int e = 0; e < CW; ++e)
                                sv[e] = e < nvis ? sv[e] : __float_as_uint(-INFINITY);
                        }
                    }
                    // row maximum of the raw scores (the scale is positive)
                    mx = __uint_as_float(sv[0]);
    #pragma unroll
                    for (int e = 1; e + 1 < CW; e += 2)
                        mx = fmax3(mx, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
                    mx = fmaxf(mx, __uint_as_float(sv[CW - 1]));
                }
                if constexpr (REP > 1) {
                    xmax[((j & 1) * REP + part) * ND + dr] = mx;
                    if (!bar_and(1, kTileM, ok_run)) break;
                    mx = -INFINITY;
    #pragma unroll
                    for (int q = 0; q < REP; ++q) mx = fmaxf(mx, xmax[((j & 1) * REP + q) * ND + dr]);
                }
                if (ok_run && live) {
                    mx *= p.scale_log2;
                    if (mx > m_used + kLazyRescale) {   // also true the first time a key is visible
                        alpha = fast_exp2(m_used - mx);  // 0 when m_used was -inf
                        m_used = mx;
                    }
                    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                    const float nm = m_used == -INFINITY ? 0.f : -m_used;
                    const float2 nm2 = make_float2(nm, nm);
                    float2 rs2 = make_float2(0.f, 0.f), rsb2 = make_float2(0.f, 0.f);
    #pragma unroll
                    for (int e = 0; e < CW; e += 2) {
                        // exponent argument s * scale - m for two keys in one packed FMA
                        const float2 xx = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                     sc2, nm2);
                        const float2 pp = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
                        pk[e / 2] = pack_bf16x2(pp.x, pp.y);
                        rs2 = __fadd2_rn(rs2, pp);
                        add_bf16x2(rsb2, pk[e / 2]);
                    }
                    // O is normalised by the sum of the bf16 probabilities the P.V product
                    // used (numerator and denominator carry the same rounding); the LSE
                    // uses the sum of the unrounded ones
                    l = l * alpha + (rs2.x + rs2.y);
                    l_b = l_b * alpha + (rsb2.x + rsb2.y);
                } else {
    #pragma unroll
                    for (int e = 0; e < CW / 2; ++e) pk[e] = 0u;
                }
                // P buffer and O are free once the previous P.V finished
                if (j > 0) ok_run = ok_run && wait_warp(p_free, (j - 1) & 1);
                if (REP == 1 && !ok_run) break;
                tc_fence_after();
                if (ok_run) {
                    if (live && j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                        // O *= alpha for this row (warp-collective tensor-memory access)
    #pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t v[32];
                            tmem_load32(lane_addr + 256 + c * 32, v);
    #pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                                             make_float2(alpha, alpha));
                                v[e] = __float_as_uint(o2.x);
                                v[e + 1] = __float_as_uint(o2.y);
                            }
                            tmem_store32(lane_addr + 256 + c * 32, v);
                        }
                    }
                    // P row -> shared memory, K-major 128-byte swizzle, two 64-key halves;
                    // 16-byte chunk c holds keys [8c, 8c + 8): this lane's chunks from pk
                    // (the others were zeroed before the key loop)
    #pragma unroll
                    for (int cc = 0; cc < CW / 8; ++cc) {
                        const int c = part * (CW / 8) + cc;
                        *reinterpret_cast<uint4*>(prow + (c >> 3) * kHalfBytes + sw128_offset(r, c & 7)) =
                            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                    }
                    // V rows of keys past the sequence's length inside its last page hold
                    // whatever the pool holds there; zero them so 0 * garbage cannot make NaN
                    if (key0 + kTileN > g.kv_len && g.kv_len > key0) {
                        const int vs = j % kVStages;
                        ok_run = ok_run && wait_warp(&v_full[vs], (j / kVStages) & 1);
                        if (REP == 1 && !ok_run) break;
                        if (ok_run) {
                            const int first = g.kv_len - key0;
                            const int last = min(kTileN, (first + 31) / 32 * 32);
                            uint8_t* vt = smem + TD::kVOff + vs * TD::kTile;
                            for (int idx = r; idx < (last - first) * TD::kChunks; idx += kTileM) {
                                const int row = first + idx / TD::kChunks, c = idx % TD::kChunks;
                                *reinterpret_cast<uint4*>(vt + (c >> 3) * kHalfBytes + sw128_offset(row, c & 7)) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                    }
                    if constexpr (GRP) {
                        // the rest of each member's last tail page is seen by no row: zero
                        // those V rows too (same reason)
                        int g0, g1;
                        while (gap_k < grp_count) {  // gaps that end before this key tile
                            member_gap(gap_k, g0, g1);
                            if (g1 > key0) break;
                            ++gap_k;
                        }
                        bool any_gap = false;
                        for (int k = gap_k; k < grp_count; ++k) {
                            member_gap(k, g0, g1);
                            if (g0 >= key0 + kTileN) break;
                            if (g0 < g1) {
                                any_gap = true;
                                break;
                            }
                        }
                        if (any_gap) {
                            const int vs = j % kVStages;
                            ok_run = ok_run && wait_warp(&v_full[vs], (j / kVStages) & 1);
                            if (REP == 1 && !ok_run) break;
                            uint8_t* vt = smem + TD::kVOff + vs * TD::kTile;
                            for (int k = gap_k; ok_run && k < grp_count; ++k) {
                                member_gap(k, g0, g1);
                                if (g0 >= key0 + kTileN) break;
                                const int lo = max(g0, key0) - key0, hi = min(g1, key0 + kTileN) - key0;
                                for (int idx = r; idx < (hi - lo) * TD::kChunks; idx += kTileM) {
                                    const int row = lo + idx / TD::kChunks, c = idx % TD::kChunks;
                                    *reinterpret_cast<uint4*>(vt + (c >> 3) * kHalfBytes + sw128_offset(row, c & 7)) =
                                        make_uint4(0u, 0u, 0u, 0u);
                                }
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(p_full);
                }
            }
            // ---- epilogue: O / l, 32 columns at a time
            const bool ok = ok_run && wait_warp(p_free, (g.nt - 1) & 1);
            tc_fence_after();
            if constexpr (REP == 1) {
                const bool any = l > 0.f && l_b > 0.f;
                const float inv_l = any ? 1.0f / l_b : 0.f;
    #pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_load32(lane_addr + 256 + c * 32, v);
                    if (ok && row_exists) store_row_chunk<D>(p, g, i, h, c, v, inv_l);
                }
                if (ok && row_exists) store_row_lse(p, g, i, h, any ? (m_used + __log2f(l)) * kLn2 : -INFINITY);
            } else {
                // the copies' partial sums: l and l_b through the exchange area, O rows
                // through the K ring (drained: every K tile was consumed by an S that
                // finished before the last P.V); float4 q of a row sits at slot
                // (q + dr) mod 32 so that a warp's stores spread over the banks
                float4* obuf = reinterpret_cast<float4*>(smem + TD::kKOff);
                constexpr int kRowF4 = D / 4;  // float4 of an O row
                xsum[(0 * REP + part) * ND + dr] = l;
                xsum[(1 * REP + part) * ND + dr] = l_b;
    #pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_load32(lane_addr + 256 + c * 32, v);
    #pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int q = c * 8 + k;
                        obuf[(part * ND + dr) * kRowF4 + ((q + dr) & (kRowF4 - 1))] =
                            make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                        __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
                    }
                }
                bar_sync_n(1, kTileM);
                float lt = 0.f, lbt = 0.f;
    #pragma unroll
                for (int q = 0; q < REP; ++q) {
                    lt += xsum[(0 * REP + q) * ND + dr];
                    lbt += xsum[(1 * REP + q) * ND + dr];
                }
                const bool any = lt > 0.f && lbt > 0.f;
                const float inv_l = any ? 1.0f / lbt : 0.f;
                // this lane adds up the copies' 32-column output chunks part,
                // part + REP, ... of its row
                for (int cc = part; cc < D / 32; cc += REP) {
                    uint32_t v[32];
    #pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int q = cc * 8 + k;
                        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
    #pragma unroll
                        for (int c2 = 0; c2 < REP; ++c2) {
                            const float4 b4 = obuf[(c2 * ND + dr) * kRowF4 + ((q + dr) & (kRowF4 - 1))];
                            a4.x += b4.x;
                            a4.y += b4.y;
                            a4.z += b4.z;
                            a4.w += b4.w;
                        }
                        v[4 * k] = __float_as_uint(a4.x);
                        v[4 * k + 1] = __float_as_uint(a4.y);
                        v[4 * k + 2] = __float_as_uint(a4.z);
                        v[4 * k + 3] = __float_as_uint(a4.w);
                    }
                    if (ok && row_exists) store_row_chunk<D>(p, g, i, h, cc, v, inv_l);
                }
                if (ok && row_exists && part == 0)
                    store_row_lse(p, g, i, h, any ? (m_used + __log2f(lt)) * kLn2 : -INFINITY);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

// barriers: q_ready, k_full[2], k_empty[2], v_full[3], v_empty[3], s_full[2], p_full[2], o_full[2],
// mma_done
constexpr int kNumBars2 = 1 + 2 * kKStages + 2 * kVStages + 7;

__device__ __forceinline__ void tmem_store_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// ===========================================================================
// Two query tiles per CTA (tile A = rows [0,128), tile B = rows [128,256) of
// the CTA's 2 x TQ tokens) sharing every K/V load.  While one tile's softmax
// runs, the tensor core works on the other tile, so the exponentials and the
// MMAs overlap.  P is written back into tensor memory over the tile's S
// columns (packed bf16 pairs) and the P.V product reads its A operand from
// tensor memory, which leaves shared memory for the two Q tiles and the K/V
// rings.  Tensor memory: S_A [0,128) O_A [128,256) S_B [256,384) O_B [384,512).
//
// Four softmax warps per tile, one thread per row: a thread reads its row's
// 128 scores of a key tile from tensor memory in one pass, keeps them in
// registers for the maximum and the exponentials, and writes the packed P
// (128 keys in columns [0,64) of the tile's S region) over them; no thread
// exchanges anything with another.  The 168 registers this takes (the row's
// scores among them) fit because the CTA has ten warps, at most three per SM
// sub-partition.  (Eight softmax warps per tile, each taking half a row with
// the maxima exchanged between the two, capped every thread at 96 registers
// and read the scores twice per key tile: 0.281 ms against 0.266 ms on the
// video step.)
// Roles (352 threads): warps 0-3 softmax A, warps 4-7 softmax B (quadrant
// warp & 3), warp 8 the K producer, warp 9 MMA, warp 10 the V producer.
// Every wait gives up after ~2 s.
// ===========================================================================
// 11 warps: 0-7 softmax (four per tile), 8 and 10 the TMA producers (K and
// V rings), 9 the MMA issuer.  Three warps per SM sub-partition at most, so
// each thread may hold 168 registers (the row's 128 scores among them)
constexpr int kThreads2 = 352;
constexpr int kProducerWarp2 = 8;
constexpr int kMmaWarp2 = 9;
constexpr int kVProducerWarp2 = 10;
constexpr int kRegs2 = 168;
template <int D>
struct TwoTileSmem {
    static constexpr int kTile = TileDim<D>::kTile;
    static constexpr int kQOff = 0;                          // Q_A, Q_B
    static constexpr int kKOff = kQOff + 2 * kTile;
    static constexpr int kVOff = kKOff + kKStages * kTile;
    static constexpr int kBarOff = kVOff + kVStages * kTile;
    static constexpr int kTmemSlotOff = kBarOff + kNumBars2 * 8;
    static constexpr int kFlagOff = kTmemSlotOff + 8;
    static constexpr int kBytes = kFlagOff + 16;
    static_assert(kBytes <= 227 * 1024, "shared memory per CTA");
};


// ---------------------------------------------------------------------------
// Work of the two-tile kernel.  A unit is one tile pair (2 x TQ tokens) of one
// sequence and K/V head, over the keys of one split; a segment is a range
// [j0, j1) of a unit's 128-key tiles.  With the one-CTA-per-tile grid every
// CTA runs one segment: its unit's whole key range.  The stream-K schedule
// (tile pairs of at most two waves) keeps one CTA per SM: while the units fill
// a whole wave, CTA c first runs unit c whole (the first wave, in grid order:
// the units that read the same K/V run together and share it in L2); the
// remaining units are shared out stream-K style, each CTA taking a contiguous
// range of their key tiles, sized so that every CTA's whole-unit work plus its
// share is the same.  Work is counted in key tiles: a unit whose rows fill
// only one tile costs about as much per key tile as a pair (its softmax chain,
// not the tensor pipe, sets the period; measured 0.96 of a pair's).
// ---------------------------------------------------------------------------
constexpr int kSkWeightPair = 1;
constexpr int kSkWeightOne = 1;
constexpr int kSkFragRows = 2 * kTileM;

struct Seg {
    TileGeom g;
    int u, j0, j1;
    bool two;
    bool shared;  // from the stream-K share (else a whole unit of the first wave)
};

// Geometry of the tile pair x of sequence b, K/V head kvh, key split `split`.
__device__ __forceinline__ TileGeom pair_geometry(const AttnParams& p, int TQ, int b, int kvh, int x,
                                                  int split) {
    TileGeom g;
    g.b = b;
    g.kvh = kvh;
    g.split = split;
    g.r0 = p.q_indptr[b];
    g.nrows = min(p.q_indptr[b + 1] - g.r0, p.max_q_rows);
    g.t0 = x * 2 * TQ;
    g.qreal = min(p.q_real ? p.q_real[b] : g.nrows, g.nrows);
    g.kv_len = min(max(p.kv_lens[b], 0), p.max_kv_len);
    g.kb = split * p.split_keys;
    const int ke = min(g.kv_len, g.kb + p.split_keys);
    // visibility is non-decreasing in the row, so the pair's last real row bounds it
    const int last = min(g.t0 + 2 * TQ, g.nrows) - 1;
    int lim = 0;
    if (g.t0 < g.qreal)
        lim = visible_keys(min(last, g.qreal - 1), g.qreal, g.kv_len, p.mask, max(p.causal_block, 1));
    g.key_hi = min(ke, lim);
    g.nt = g.key_hi > g.kb ? (g.key_hi - g.kb + kTileN - 1) / kTileN : 0;
    return g;
}

// Stream-K unit u: tile pairs fastest, then K/V heads, then sequences, so the
// units that read the same K/V run on neighbouring CTAs at about the same time.
__device__ __forceinline__ TileGeom sk_unit(const AttnParams& p, int TQ, int u) {
    const int x = u % p.sk_tiles_x;
    const int bh = u / p.sk_tiles_x;
    return pair_geometry(p, TQ, bh / p.num_kv_heads, bh % p.num_kv_heads, x, 0);
}

__device__ __forceinline__ int sk_weight(const TileGeom& g, int TQ) {
    return g.t0 + TQ < g.nrows ? kSkWeightPair : kSkWeightOne;
}

// The segments of one CTA, in order.  Every role of the CTA walks them itself.
template <bool SK>
struct SegIter {
    int u = 0, end_u = 0;  // stream-K: next shared unit (index among the shared ones)
    int a = 0, a1 = 0;     // this CTA's share [a, a1) of the shared units' weighted key tiles
    bool dp = false;       // the first-wave unit is still to come
    bool done = false;

    __device__ __forceinline__ void init(const AttnParams& p) {
        if constexpr (SK) {
            dp = p.sk_dp > 0;
            a = p.sk_cta_off[blockIdx.x];
            a1 = p.sk_cta_off[blockIdx.x + 1];
            end_u = p.sk_units - p.sk_dp;
            // the last shared unit that starts at or before a
            int lo = 0, hi = max(end_u - 1, 0);
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.sk_unit_off[mid] <= a) lo = mid;
                else hi = mid - 1;
            }
            u = lo;
        }
    }
    __device__ __forceinline__ bool next(const AttnParams& p, int TQ, Seg& s) {
        if constexpr (!SK) {
            if (done) return false;
            done = true;
            s.g = pair_geometry(p, TQ, blockIdx.z / p.num_splits, blockIdx.y, blockIdx.x,
                                blockIdx.z % p.num_splits);
            s.u = -1;
            s.j0 = 0;
            s.j1 = s.g.nt;
            s.two = s.g.t0 + TQ < s.g.nrows;
            s.shared = false;
            return s.g.t0 < s.g.nrows && s.g.nt > 0;
        } else {
            if (dp) {
                dp = false;
                s.g = sk_unit(p, TQ, blockIdx.x);
                s.u = blockIdx.x;
                s.j0 = 0;
                s.j1 = s.g.nt;
                s.two = s.g.t0 + TQ < s.g.nrows;
                s.shared = false;
                if (s.g.t0 < s.g.nrows && s.g.nt > 0) return true;
            }
            while (!done && a < a1 && u < end_u) {
                const int off = p.sk_unit_off[u];
                if (off >= a1) break;
                const int off1 = p.sk_unit_off[u + 1];
                const int cur = p.sk_dp + u++;
                if (off1 == off) continue;  // no key tile
                s.g = sk_unit(p, TQ, cur);
                const int w = sk_weight(s.g, TQ);
                s.u = cur;
                s.j0 = a > off ? (a - off + w - 1) / w : 0;
                s.j1 = min(s.g.nt, (a1 - off + w - 1) / w);
                s.two = s.g.t0 + TQ < s.g.nrows;
                s.shared = true;
                if (s.j1 > s.j0) return true;
            }
            done = true;
            return false;
        }
    }
};

// Zero output and LSE = -inf for the existing rows of a pair whose rows see no
// key.  Threads 0 .. 2 * kTileM - 1 each take one row.
template <int D>
__device__ __forceinline__ void zero_pair_rows(const AttnParams& p, const TileGeom& g, int G, int TQ) {
    if (threadIdx.x >= 2 * kTileM) return;
    const int x = threadIdx.x / kTileM, r = threadIdx.x % kTileM;
    const int i = g.t0 + x * TQ + r / G;
    if (r / G >= TQ || i >= g.nrows) return;
    uint32_t zero[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) zero[e] = 0u;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) store_row_chunk<D>(p, g, i, g.kvh * G + r % G, c, zero, 0.f);
    store_row_lse(p, g, i, g.kvh * G + r % G, -INFINITY);
}

template <int D, int GC, bool SK>
__global__ void __maxnreg__(kRegs2)
    attn_tc2_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const AttnParams p) {
    using TD = TileDim<D>;
    using SM = TwoTileSmem<D>;
    const int G = GC > 0 ? GC : p.num_q_heads / p.num_kv_heads;
    const int TQ = kTileM / G;  // tokens per tile; rows from TQ * G on hold none
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    SegIter<SK> it0;
    if constexpr (SK) {
        // launched behind the planner with programmatic serialisation: its unit
        // offsets are visible after this wait
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // this CTA's fragment slots hold nothing until a partial segment says so
        if (threadIdx.x < 2) p.sk_dir[blockIdx.x * 2 + threadIdx.x] = make_int4(-1, 0, 0, 0);
        // pairs with rows but no visible key: zero rows (units u = CTA mod grid)
        for (int u = blockIdx.x; u < p.sk_units; u += p.sk_ctas) {
            const TileGeom g = sk_unit(p, TQ, u);
            if (g.t0 < g.nrows && g.nt == 0) zero_pair_rows<D>(p, g, G, TQ);
        }
        it0.init(p);
    } else {
        const TileGeom g = pair_geometry(p, TQ, blockIdx.z / p.num_splits, blockIdx.y, blockIdx.x,
                                         blockIdx.z % p.num_splits);
        if (g.t0 >= g.nrows) return;  // uniform
        if (g.nt == 0) {
            zero_pair_rows<D>(p, g, G, TQ);
            return;
        }
    }
    {
        // a CTA without a segment leaves before any set-up (uniform)
        SegIter<SK> probe = it0;
        Seg s;
        if (!probe.next(p, TQ, s)) return;
    }
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) set_err(p.err, PKV_ERRBIT_TIMEOUT);
        return;
    }

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBarOff);
    uint64_t* q_ready = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + kKStages;
    uint64_t* v_full = k_empty + kKStages;
    uint64_t* v_empty = v_full + kVStages;
    uint64_t* s_full = v_empty + kVStages;  // [tile]
    uint64_t* p_full = s_full + 2;          // [tile]
    uint64_t* o_full = p_full + 2;          // [tile]
    uint64_t* mma_done = o_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kTmemSlotOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::kFlagOff);

    if (threadIdx.x == 0) {
        mbar_init(q_ready, 2 * kTileM);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);  // one elected arrive per softmax warp of the tile
            mbar_init(&o_full[x], 1);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp2) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(smem);

    // a completed phase passes at once; a pending one gives up early once
    // another thread of the CTA has timed out
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (mbar_wait(bar, parity)) return true;
        *abort_flag = 1;
        set_err(p.err, PKV_ERRBIT_TIMEOUT);
        return false;
    };

    if (warp == kProducerWarp2 || warp == kVProducerWarp2) {
        // ============================ producers =============================
        // Lane 0 of warp 8 streams the K tiles of every segment in order, lane
        // 0 of warp 10 the V tiles, each through its own ring running across
        // segment boundaries (n counts the tiles of all segments), so one
        // ring's copies are issued while the other thread waits for a free
        // stage.  Each reads the next tile's block-table entries one tile ahead.
        if (lane == 0) {
            const bool is_k = warp == kProducerWarp2;
            const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
            prefetch_tmap(tm);
            const int stages = is_k ? kKStages : kVStages;
            uint8_t* ring = smem + (is_k ? SM::kKOff : SM::kVOff);
            uint64_t* full = is_k ? k_full : v_full;
            uint64_t* empty = is_k ? k_empty : v_empty;
            SegIter<SK> it = it0;
            Seg sg;
            int n = 0;  // tiles issued
            bool alive = true;
            while (alive && it.next(p, TQ, sg)) {
                const TileGeom& g = sg.g;
                const int32_t* bt = p.block_table + static_cast<int64_t>(g.b) * p.block_table_stride;
                const int last_page = (g.kv_len + 31) / 32;
                auto fetch_pages = [&](int j, int (&ph)[4]) {
#pragma unroll
                    for (int pg = 0; pg < 4; ++pg) {
                        const int lp = (g.kb + j * kTileN) / 32 + pg;
                        ph[pg] = lp < last_page ? bt[lp] : static_cast<int>(p.num_pages);
                    }
                };
                int next[4] = {0, 0, 0, 0};
                if (sg.j0 < sg.j1) fetch_pages(sg.j0, next);
                for (int j = sg.j0; j < sg.j1; ++j) {
                    const int s = n % stages;
                    const int cur[4] = {next[0], next[1], next[2], next[3]};
                    if (j + 1 < sg.j1) fetch_pages(j + 1, next);
                    if (n >= stages && !wait(&empty[s], ((n / stages) - 1) & 1)) {
                        alive = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], TD::kTile);
#pragma unroll
                    for (int pg = 0; pg < 4; ++pg) {
                        const int lp = (g.kb + j * kTileN) / 32 + pg;
                        int phys = cur[pg];
                        if (p.checked && lp < last_page && (phys < 0 || phys >= p.num_pages)) {
                            set_err(p.err, PKV_ERRBIT_PAGE);
                            phys = static_cast<int>(p.num_pages);
                        }
#pragma unroll
                        for (int h = 0; h < TD::kHalves; ++h)
                            tma_load_4d(ring + s * TD::kTile + h * kHalfBytes + pg * 4096, tm, &full[s], h * 64,
                                        g.kvh, 0, phys);
                    }
                    ++n;
                }
            }
            // do not leave with copies into this CTA's shared memory in flight
            for (int j = max(0, n - stages); j < n; ++j) mbar_wait(&full[j % stages], (j / stages) & 1);
        }
    } else if (warp == kMmaWarp2) {
        // ============================== MMA ================================
        // An MMA issue returns about when the previous MMA is done, so the
        // pipe holds about one instruction: every wait and commit between two
        // batches leaves it idle.  The waits for K and V tiles (normally long
        // loaded) therefore sit inside a batch, after its fourth MMA, and each
        // batch builds its two descriptors once (the start address field takes
        // the offsets of its k-steps as plain additions).
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(kTileM, kTileN, false);
            constexpr uint32_t kIdescO = idesc_bf16(kTileM, D, true);
            auto nop = [] {};
            auto issue_s = [&](int x, int gt, auto&& mid) {
                const uint64_t da = sdesc_sw128(sbase + SM::kQOff + x * TD::kTile, 16, 1024);
                const uint64_t db = sdesc_sw128(sbase + SM::kKOff + (gt % kKStages) * TD::kTile, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
                    umma_bf16(tmem + x * 256, da + off, db + off, kIdescS, kk > 0);
                    if (kk == 3) mid();
                }
                umma_commit(&s_full[x]);
            };
            auto issue_pv = [&](int x, int gt, bool acc, auto&& mid) {
                const uint64_t bd = sdesc_sw128(sbase + SM::kVOff + (gt % kVStages) * TD::kTile, kHalfBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < kTileN / 16; ++kk) {
                    // A = P in tensor memory: the 128 keys packed in columns
                    // [0, 64); 16 keys = 8 columns per step
                    umma_bf16_ts(tmem + x * 256 + 128, tmem + x * 256 + kk * 8, bd + ((kk * 16 * 128) >> 4),
                                 kIdescO, (acc || kk > 0) ? 1u : 0u);
                    if (kk == 3) mid();
                }
            };
            // a tile's barrier is probed inside the batch before it; if its copy
            // has not landed, the batch goes on and the wait comes after
            bool ready = false;
            auto probe = [&](uint64_t* bar, uint32_t parity) {
                ready = mbar_test(bar, parity);
                if (ready) tc_fence_after();
            };
            auto settle = [&](uint64_t* bar, uint32_t parity) -> bool {
                if (ready) return true;
                if (!wait(bar, parity)) return false;
                tc_fence_after();
                return true;
            };
            SegIter<SK> it = it0;
            Seg sg;
            int gt = 0;          // K/V tiles consumed (ring position)
            int na = 0, nb = 0;  // P tiles of tile A / tile B consumed
            int qn = 0;          // segments (Q tiles loaded)
            bool ok = true;
            while (ok && it.next(p, TQ, sg)) {
                const bool two = sg.two;
                // the segment's Q tiles are in shared memory; its first S MMAs
                // follow every MMA of the previous segment in the pipe
                ok = wait(q_ready, qn & 1) && wait(&k_full[gt % kKStages], (gt / kKStages) & 1);
                ++qn;
                if (!ok) break;
                tc_fence_after();
                issue_s(0, gt, [&] { probe(&v_full[gt % kVStages], (gt / kVStages) & 1); });
                if (two) issue_s(1, gt, nop);
                umma_commit(&k_empty[gt % kKStages]);
                ok = settle(&v_full[gt % kVStages], (gt / kVStages) & 1);
                for (int j = sg.j0; ok && j < sg.j1; ++j, ++gt) {
                    // V(gt) has landed (settled at the end of the previous step)
                    const bool more = j + 1 < sg.j1;
                    if (!wait(&p_full[0], na & 1)) {
                        ok = false;
                        break;
                    }
                    ++na;
                    tc_fence_after();
                    issue_pv(0, gt, j > sg.j0, [&] {
                        if (more) probe(&k_full[(gt + 1) % kKStages], ((gt + 1) / kKStages) & 1);
                    });
                    if (more) {
                        if (!settle(&k_full[(gt + 1) % kKStages], ((gt + 1) / kKStages) & 1)) {
                            ok = false;
                            break;
                        }
                        issue_s(0, gt + 1, [&] {
                            probe(&v_full[(gt + 1) % kVStages], ((gt + 1) / kVStages) & 1);
                        });
                    } else {
                        umma_commit(&o_full[0]);
                    }
                    if (two) {
                        if (!wait(&p_full[1], nb & 1)) {
                            ok = false;
                            break;
                        }
                        ++nb;
                        tc_fence_after();
                        issue_pv(1, gt, j > sg.j0, nop);
                    }
                    umma_commit(&v_empty[gt % kVStages]);
                    if (more) {
                        if (two) issue_s(1, gt + 1, nop);
                        umma_commit(&k_empty[(gt + 1) % kKStages]);
                        if (!settle(&v_full[(gt + 1) % kVStages], ((gt + 1) / kVStages) & 1)) {
                            ok = false;
                            break;
                        }
                    } else if (two) {
                        umma_commit(&o_full[1]);
                    }
                }
            }
            // nothing of this thread's still runs in the tensor pipe when the
            // CTA winds down (after a failed wait the last batch may be running)
            umma_commit(mma_done);
            if (!mbar_wait(mma_done, 0)) set_err(p.err, PKV_ERRBIT_TIMEOUT);
        }
    } else if (warp < 8) {
        // ============================ softmax ===============================
        // warps 0-3: tile A, warps 4-7: tile B.  Each thread owns one row (its
        // lane of its warp's tensor-memory quadrant) and all 128 keys of every
        // key tile: the scores, their maximum and the probabilities stay in its
        // registers, with no exchange between threads.
        const int x = warp >> 2;               // tile
        const int r = (warp & 3) * 32 + lane;  // row in the tile = tensor-memory lane
        const int t = r / G, hg = r % G;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + x * 256;
        const uint32_t o_addr = lane_addr + 128;  // this row's O columns
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        SegIter<SK> it = it0;
        Seg sg;
        int gt = 0;     // K/V ring position of the segment's first tile
        int nit = 0;    // key tiles of this tile's rows processed (S / P phases)
        int nseg = 0;   // segments in which this tile had rows (O phases)
        int qn = 0;     // segments (Q phases)
        int slot = 0;   // shared segments of this CTA (fragment slot of a partial one)
        bool ok = true;
        while (ok && it.next(p, TQ, sg)) {
            const TileGeom& g = sg.g;
            const int i = g.t0 + x * TQ + t;
            const int h = g.kvh * G + hg;
            const bool row_exists = t < TQ && i < g.nrows;
            const int limit = row_exists ? visible_keys(i, g.qreal, g.kv_len, p.mask, max(p.causal_block, 1))
                                         : 0;
            {
                // the row's query into the swizzled Q tile.  The previous segment's
                // S MMAs have finished reading this Q tile (their S was consumed),
                // and its O was read before this arrive, ahead of the segment's
                // first P.V
                const uint4* src = reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(p.q) + static_cast<int64_t>(g.r0 + i) * p.q_token_stride +
                    static_cast<int64_t>(h) * p.q_head_stride);
                uint8_t* qt = smem + SM::kQOff + x * TD::kTile;
#pragma unroll
                for (int c = 0; c < TD::kChunks; ++c) {
                    const uint4 v = row_exists ? src[c] : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(qt + (c >> 3) * kHalfBytes + sw128_offset(r, c & 7)) = v;
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(q_ready);
            }
            const bool active = x == 0 || sg.two;  // no rows in tile B: nothing to do
            const int n_seg_tiles = sg.j1 - sg.j0;
            if (!active) {
                // one arrive per segment and thread: wait for this segment's
                // Q phase before arriving for the next one
                ok = wait(q_ready, qn & 1);
                ++qn;
                gt += n_seg_tiles;
                slot += sg.shared ? 1 : 0;
                continue;
            }
            ++qn;
            float m_used = -INFINITY;
            float l = 0.f, l_b = 0.f;
            const bool warp_live = __any_sync(0xffffffffu, limit > 0);
            for (int j = sg.j0; j < sg.j1; ++j, ++nit) {
                if (!__all_sync(0xffffffffu, wait(&s_full[x], nit & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int key0 = g.kb + j * kTileN;
                if (warp_live) {
                    uint32_t sv[kTileN];  // this row's scores (f32 bits), then its packed P
                    tmem_load128(lane_addr, sv);
                    const int nvis = limit - key0;  // keys past it are masked (diagonal tiles only)
                    if (__any_sync(0xffffffffu, nvis < kTileN)) {
#pragma unroll
                        for (int e = 0; e < kTileN; ++e) sv[e] = e < nvis ? sv[e] : __float_as_uint(-INFINITY);
                    }
                    float a[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) a[q] = __uint_as_float(sv[q]);
#pragma unroll
                    for (int e = 8; e < kTileN; e += 16) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            a[q] = fmax3(a[q], __uint_as_float(sv[e + q]), __uint_as_float(sv[e + 8 + q]));
                    }
                    const float mraw = fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
                    const float mx = mraw * p.scale_log2;
                    float alpha = 1.f;
                    if (mx > m_used + kLazyRescale) {   // also true the first time a key is visible
                        alpha = fast_exp2(m_used - mx);  // 0 when m_used was -inf
                        m_used = mx;
                    }
                    const float nm = m_used == -INFINITY ? 0.f : -m_used;
                    const float2 nm2 = make_float2(nm, nm);
                    float2 rs2 = make_float2(0.f, 0.f), rsb2 = make_float2(0.f, 0.f);
                    // probabilities packed in place: keys (2k, 2k + 1) land in sv[k]
                    // (k <= 2k: read before written); P over S columns [0, 64)
#pragma unroll
                    for (int k2 = 0; k2 < kTileN / 2; ++k2) {
                        const float2 xx = __ffma2_rn(
                            make_float2(__uint_as_float(sv[2 * k2]), __uint_as_float(sv[2 * k2 + 1])), sc2, nm2);
                        const float2 pp = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
                        sv[k2] = pack_bf16x2(pp.x, pp.y);
                        rs2 = __fadd2_rn(rs2, pp);
                        add_bf16x2(rsb2, sv[k2]);
                    }
                    tmem_store64_nowait(lane_addr, sv);
                    // O *= alpha for this row (before the next P.V, which follows
                    // this warp's arrive below)
                    if (j > sg.j0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t v[32];
                            tmem_load32(o_addr + c * 32, v);
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                                             make_float2(alpha, alpha));
                                v[e] = __float_as_uint(o2.x);
                                v[e + 1] = __float_as_uint(o2.y);
                            }
                            tmem_store32(o_addr + c * 32, v);
                        }
                    }
                    tmem_store_wait();
                    l = l * alpha + (rs2.x + rs2.y);
                    l_b = l_b * alpha + (rsb2.x + rsb2.y);
                } else {
                    uint32_t zero[kTileN];
#pragma unroll
                    for (int e = 0; e < kTileN / 2; ++e) zero[e] = 0u;
                    tmem_store64_nowait(lane_addr, zero);
                    tmem_store_wait();
                }
                // keys past the sequence's length inside its last page: zero their V rows
                if (x == 0 && key0 + kTileN > g.kv_len && g.kv_len > key0) {
                    const int gj = gt + (j - sg.j0);
                    const int vs = gj % kVStages;
                    if (__all_sync(0xffffffffu, wait(&v_full[vs], (gj / kVStages) & 1))) {
                        const int first = g.kv_len - key0;
                        const int lastr = min(kTileN, (first + 31) / 32 * 32);
                        uint8_t* vt = smem + SM::kVOff + vs * TD::kTile;
                        for (int idx = r; idx < (lastr - first) * TD::kChunks; idx += kTileM) {
                            const int row = first + idx / TD::kChunks, c16 = idx % TD::kChunks;
                            *reinterpret_cast<uint4*>(vt + (c16 >> 3) * kHalfBytes + sw128_offset(row, c16 & 7)) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[x]);
            }
            // ---- epilogue: O / l
            const bool ok_o = __all_sync(0xffffffffu, ok && wait(&o_full[x], nseg & 1));
            ++nseg;
            tc_fence_after();
            // a segment that is not its unit's whole key range leaves a partial
            // state in this CTA's fragment slot (the first or the last segment)
            const bool whole = sg.j0 == 0 && sg.j1 == g.nt;
            const int fslot = blockIdx.x * 2 + (slot == 0 ? 0 : 1);
            const bool any = l > 0.f && l_b > 0.f;
            const float inv_l = any ? 1.0f / l_b : 0.f;
            if (ok_o && row_exists) {
                const float lse = any ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
                if (whole) store_row_lse(p, g, i, h, lse);
                else p.sk_frag_lse[static_cast<int64_t>(fslot) * kSkFragRows + x * kTileM + r] = lse;
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_load32(o_addr + c * 32, v);
                if (ok_o && row_exists) {
                    if (whole) {
                        store_row_chunk<D>(p, g, i, h, c, v, inv_l);
                    } else {
                        float4* dst = reinterpret_cast<float4*>(
                            p.sk_frag_o + (static_cast<int64_t>(fslot) * kSkFragRows + x * kTileM + r) * D + c * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = make_float4(__uint_as_float(v[4 * q]) * inv_l, __uint_as_float(v[4 * q + 1]) * inv_l,
                                                 __uint_as_float(v[4 * q + 2]) * inv_l,
                                                 __uint_as_float(v[4 * q + 3]) * inv_l);
                    }
                }
            }
            if constexpr (SK) {
                if (!whole && ok_o && threadIdx.x == 0) p.sk_dir[fslot] = make_int4(sg.u, sg.j0, sg.j1, g.nt);
            }
            ok = ok && ok_o;
            gt += n_seg_tiles;
            slot += sg.shared ? 1 : 0;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp2) tmem_dealloc(tmem, kTmemCols);
}

// Block-wide exclusive prefix sum of one value per thread (blockDim 1024);
// returns the thread's exclusive sum and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_sum(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = (wid > 0 ? warp_tot[wid - 1] : 0) + incl - v;
    *total = warp_tot[31];
    __syncthreads();
    return before;
}

// Stream-K planner (one CTA of 1024 threads): the weighted key-tile offsets of
// the shared units and every CTA's share of them.  A CTA's share is what
// brings its work (its whole first-wave unit plus the share) to the average;
// shares are scaled to add up to the shared units' total.
__global__ void __launch_bounds__(1024) tc2_sk_plan_kernel(const AttnParams p) {
    const int TQ = kTileM / (p.num_q_heads / p.num_kv_heads);
    // the persistent launch may start its prologue now; it waits for this
    // grid's completion before it reads the offsets
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int warp_tot[32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    auto cost_of = [&](int u) {
        const TileGeom g = sk_unit(p, TQ, u);
        return g.t0 < g.nrows ? g.nt * sk_weight(g, TQ) : 0;
    };
    const int n_shared = p.sk_units - p.sk_dp;
    for (int base = 0; base < n_shared; base += 1024) {
        const int k = base + threadIdx.x;
        const int cost = k < n_shared ? cost_of(p.sk_dp + k) : 0;
        int tot;
        const int before = block_exclusive_sum(cost, warp_tot, &tot);
        if (k < n_shared) p.sk_unit_off[k] = carry + before;
        __syncthreads();
        if (threadIdx.x == 0) carry += tot;
        __syncthreads();
    }
    const int w_shared = carry;
    if (threadIdx.x == 0) p.sk_unit_off[n_shared] = w_shared;
    // shares: the first-wave unit of CTA c costs dp_c; the target is the mean
    // of all work per CTA
    const int c = threadIdx.x;
    const int dp_c = c < p.sk_dp ? cost_of(c) : 0;
    int dp_tot;
    block_exclusive_sum(c < p.sk_ctas ? dp_c : 0, warp_tot, &dp_tot);
    const int64_t target = (static_cast<int64_t>(dp_tot) + w_shared) / p.sk_ctas;
    const int want = c < p.sk_ctas ? static_cast<int>(target > dp_c ? target - dp_c : 0) : 0;
    int want_tot;
    const int want_before = block_exclusive_sum(want, warp_tot, &want_tot);
    if (c <= p.sk_ctas) {
        // (no CTA below the mean, from rounding: equal shares)
        const int64_t off = want_tot > 0 ? static_cast<int64_t>(want_before) * w_shared / want_tot
                                         : static_cast<int64_t>(c) * w_shared / p.sk_ctas;
        p.sk_cta_off[c] = c == p.sk_ctas ? w_shared : static_cast<int>(off);
    }
}

// Stream-K reduce: for every unit split between CTAs, the CTA slot holding the
// unit's first keys names the following CTAs' first slots that hold the rest,
// and their partial states are merged by LSE into the output.  Grid: (fragment
// slot, group of 8 fragment rows); one warp per row, every load of a row in
// flight at once.
constexpr int kSkReduceRows = 8;
template <int D>
__global__ void __launch_bounds__(32 * kSkReduceRows) tc2_sk_reduce_kernel(const AttnParams p) {
    const int G = p.num_q_heads / p.num_kv_heads;
    const int TQ = kTileM / G;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int4 d = p.sk_dir[blockIdx.x];
    if (d.x < 0 || d.y != 0) return;  // not partial, or not the unit's first keys
    // a unit spans at most every CTA plus one (the host keeps the grid under 1024)
    constexpr int kMaxFrag = 1024;
    __shared__ int frag[kMaxFrag];
    __shared__ int nfrag;
    if (threadIdx.x == 0) {
        int n = 0;
        frag[n++] = blockIdx.x;
        int covered = d.z;
        for (int c = blockIdx.x / 2 + 1; c < p.sk_ctas && covered < d.w && n < kMaxFrag; ++c) {
            const int4 e = p.sk_dir[c * 2];
            if (e.x != d.x) continue;  // a CTA without keys (empty share)
            if (e.y != covered) break;
            frag[n++] = c * 2;
            covered = e.z;
        }
        if (covered != d.w && blockIdx.y == 0) set_err(p.err, PKV_ERRBIT_TIMEOUT);  // never expected
        nfrag = n;
    }
    __syncthreads();
    const TileGeom g = sk_unit(p, TQ, d.x);
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.y * kSkReduceRows + (threadIdx.x >> 5);
    const int x = row / kTileM, r = row % kTileM;
    const int i = g.t0 + x * TQ + r / G;
    if (r / G >= TQ || i >= g.nrows) return;
    const int h = g.kvh * G + r % G;
    const int n = nfrag;
    // the fragments' LSEs, one per lane (more than 32 fragments: in rounds)
    float m = -INFINITY;
    for (int f0 = 0; f0 < n; f0 += 32) {
        const float lf = f0 + lane < n
                             ? __ldcg(p.sk_frag_lse + static_cast<int64_t>(frag[f0 + lane]) * kSkFragRows + row)
                             : -INFINITY;
        m = fmaxf(m, lf);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (m != -INFINITY) {
#pragma unroll 4
        for (int f = 0; f < n; ++f) {
            const int64_t fr = static_cast<int64_t>(frag[f]) * kSkFragRows + row;
            const float w = __expf(__ldcg(p.sk_frag_lse + fr) - m);
            const float4 o = lane < D / 4 ? __ldcg(reinterpret_cast<const float4*>(p.sk_frag_o + fr * D) + lane)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
            wsum += w;
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
        }
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    const int64_t st = static_cast<int64_t>(g.r0 + i) * p.num_q_heads + h;
    if (lane < D / 4) {
        if (p.out_f32) {
            reinterpret_cast<float4*>(static_cast<float*>(p.out) + st * D)[lane] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + st * D)[lane] =
                make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
        }
    }
    if (p.lse && lane == 0) p.lse[st] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
}

template <int D, int GC>
cudaError_t launch_g2(const AttnParams& p, const void* tk, const void* tv, cudaStream_t s) {
    const bool sk = p.sk_ctas > 0;
    // the stream-K schedule (on request) reads the group from the call
    auto kern = sk ? attn_tc2_kernel<D, 0, true> : attn_tc2_kernel<D, GC, false>;
    constexpr int kSmem = TwoTileSmem<D>::kBytes;
    // shared-memory opt-in: once per device and kernel
    static DeviceOnce opted[2];
    int dev = 0, done = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = opted[sk ? 1 : 0].get(dev, &done, [&](int, int* v) {
        *v = 1;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    });
    if (e != cudaSuccess) return e;
    const int TQ = kTileM / (p.num_q_heads / p.num_kv_heads);
    if (!sk) {
        dim3 grid((p.max_q_rows + 2 * TQ - 1) / (2 * TQ), p.num_kv_heads, p.batch * p.num_splits);
        kern<<<grid, kThreads2, kSmem, s>>>(*static_cast<const CUtensorMap*>(tk),
                                            *static_cast<const CUtensorMap*>(tv), p);
        return cudaGetLastError();
    }
    // planner, then the persistent launch and the reduce, each behind the
    // previous one with programmatic serialisation (its prologue overlaps)
    tc2_sk_plan_kernel<<<1, 1024, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.sk_ctas));
    cfg.blockDim = dim3(kThreads2);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, *static_cast<const CUtensorMap*>(tk),
                           *static_cast<const CUtensorMap*>(tv), p);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3(static_cast<unsigned>(2 * p.sk_ctas), kSkFragRows / kSkReduceRows);
    rcfg.blockDim = dim3(32 * kSkReduceRows);
    rcfg.stream = s;
    rcfg.attrs = attr;
    rcfg.numAttrs = 1;
    return cudaLaunchKernelEx(&rcfg, tc2_sk_reduce_kernel<D>, p);
}

// One-tile launches: when a tile's rows (query rows x grouped heads) fit in
// one 32-lane quadrant, they are held four times and each warp takes a
// quarter of every key tile's columns.
template <int D, int GC, bool GRP, int REP>
cudaError_t launch_one(const AttnParams& p, int rows, const void* tk, const void* tv, cudaStream_t s) {
    auto kern = attn_tc_kernel<D, GC, GRP, REP>;
    constexpr int kSmem = OneTileSmem<D>::kBytes;
    // shared-memory opt-in: once per device
    static DeviceOnce opted;
    int dev = 0, done = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = opted.get(dev, &done, [&](int, int* v) {
        *v = 1;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    });
    if (e != cudaSuccess) return e;
    const int TQ = kTileM / (p.num_q_heads / p.num_kv_heads * REP);
    dim3 grid((rows + TQ - 1) / TQ, p.num_kv_heads, p.batch * p.num_splits);
    // more than one wave of CTAs (one per SM) over a small batch: dispatch the
    // longest sequences first, so the last wave holds the shortest ones
    static DeviceOnce sm_count;
    int sms = 0;
    e = sm_count.get(dev, &sms, [](int d, int* v) {
        return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, d);
    });
    if (e != cudaSuccess) return e;
    AttnParams q = p;
    q.order_by_keys = !GRP && p.batch >= 2 && p.batch <= kOrderMaxBatch &&
                      static_cast<int64_t>(grid.x) * grid.y * grid.z > sms;
    kern<<<grid, kThreads, kSmem, s>>>(*static_cast<const CUtensorMap*>(tk),
                                       *static_cast<const CUtensorMap*>(tv), q);
    return cudaGetLastError();
}

template <int D, int GC, bool GRP>
cudaError_t launch_one_rep(const AttnParams& p, int rows, const void* tk, const void* tv, cudaStream_t s) {
    const int G = p.num_q_heads / p.num_kv_heads;
    if (rows * G <= kTileM / 4) return launch_one<D, GC, GRP, 4>(p, rows, tk, tv, s);
    return launch_one<D, GC, GRP, 1>(p, rows, tk, tv, s);
}

// head_dim 128: the common head groups fixed at compile time, any other read
// from the call; head_dim 64: read from the call
template <int D, bool GRP>
cudaError_t launch_one_g(const AttnParams& p, int rows, const void* tk, const void* tv, cudaStream_t s) {
    if constexpr (D == 128) {
        switch (p.num_q_heads / p.num_kv_heads) {
            case 1: return launch_one_rep<D, 1, GRP>(p, rows, tk, tv, s);
            case 2: return launch_one_rep<D, 2, GRP>(p, rows, tk, tv, s);
            case 4: return launch_one_rep<D, 4, GRP>(p, rows, tk, tv, s);
            case 8: return launch_one_rep<D, 8, GRP>(p, rows, tk, tv, s);
            case 16: return launch_one_rep<D, 16, GRP>(p, rows, tk, tv, s);
        }
    }
    return launch_one_rep<D, 0, GRP>(p, rows, tk, tv, s);
}

template <int D>
cudaError_t launch_two_g(const AttnParams& p, const void* tk, const void* tv, cudaStream_t s) {
    if constexpr (D == 128) {
        switch (p.num_q_heads / p.num_kv_heads) {
            case 1: return launch_g2<D, 1>(p, tk, tv, s);
            case 2: return launch_g2<D, 2>(p, tk, tv, s);
            case 4: return launch_g2<D, 4>(p, tk, tv, s);
            case 8: return launch_g2<D, 8>(p, tk, tv, s);
            case 16: return launch_g2<D, 16>(p, tk, tv, s);
        }
    }
    return launch_g2<D, 0>(p, tk, tv, s);
}

}  // namespace

bool attn_tc_supported(int head_dim, int group) {
    return (head_dim == 64 || head_dim == 128) && group >= 1 && group <= kMaxGroup;
}

int attn_tc_rows_per_tile(int group) { return kTileM / group; }

bool attn_tc_two_tile(int max_q_rows, int group) { return max_q_rows > kTileM / group; }

size_t attn_tc_sk_bytes(int units, int ctas, int head_dim) {
    auto r256 = [](size_t n) { return (n + 255) / 256 * 256; };
    return r256((static_cast<size_t>(units) + 1) * sizeof(int)) + r256((static_cast<size_t>(ctas) + 1) * sizeof(int)) +
           r256(2 * static_cast<size_t>(ctas) * 16) +
           r256(2 * static_cast<size_t>(ctas) * kSkFragRows * sizeof(float)) +
           r256(2 * static_cast<size_t>(ctas) * kSkFragRows * head_dim * sizeof(float));
}

cudaError_t launch_attn_tc_grouped(const AttnParams& p, const void* tk, const void* tv, cudaStream_t s) {
    if (p.head_dim == 128) return launch_one_g<128, true>(p, p.grp_max_tokens, tk, tv, s);
    if (p.head_dim == 64) return launch_one_g<64, true>(p, p.grp_max_tokens, tk, tv, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_tc(const AttnParams& p, const void*, const void* tk, const void* tv,
                           cudaStream_t s) {
    const int G = p.num_q_heads / p.num_kv_heads;
    const bool two = p.max_q_rows > kTileM / G;
    if (p.head_dim == 128)
        return two ? launch_two_g<128>(p, tk, tv, s) : launch_one_g<128, false>(p, p.max_q_rows, tk, tv, s);
    if (p.head_dim == 64)
        return two ? launch_two_g<64>(p, tk, tv, s) : launch_one_g<64, false>(p, p.max_q_rows, tk, tv, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
