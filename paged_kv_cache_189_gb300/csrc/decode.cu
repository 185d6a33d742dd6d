// decode.cu -- paged attention for one query row per sequence (decode).
//
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Attention (paged attention over 32-token pages through the block table,
// real-token seq_len, zeroed padding rows) and "Support shared-prefix attention
// for n-sample requests in FMHA", split-KV commit notes (cut every row's keys
// into chunks of at least 512 tokens, attend each chunk, merge the chunk
// states by LSE; a merge that walks every split per (token, heads)).
//
// Decode is bound by HBM: every K/V byte is read once and used for the
// G = Hq/Hkv query heads that share it.  The GB300 design:
//  * work unit = (split of split_keys keys, K/V head, sequence), handed out by
//    an atomic ticket, so the kernel is persistent (a few CTAs per SM) and
//    balances ragged lengths dynamically; the grid never depends on device
//    lengths, so a call is graph-capturable.  When the units outnumber the
//    CTAs, a one-CTA planning launch before it orders them: every full split
//    first (split-major, sequences with more full splits first), then each
//    sequence's partial last split, longest first, then the rows without keys
//    -- so the launch ends on the shortest units instead of leaving SMs idle
//    behind full-length ones.
//  * one producer lane per CTA fetches tickets, reads each ticket's unit from
//    the planned list, copies the unit's G query rows into shared memory with bulk
//    copies, and streams the unit's pages of one K/V head (32 x D of K and of
//    V, 64-column TMA boxes, 128-byte swizzle) into a 4-stage ring.  It runs
//    ahead across unit boundaries, so the ring stays full while the consumers
//    finish a unit.
//  * four consumer warps each own 8 of a page's 32 keys (rows 8w..8w+7) and
//    keep their own online softmax over those keys; their states are merged in
//    shared memory once per unit.
//  * QK: lane = (key of 4, segment of 8 x 16 dims); query values live in
//    registers for the whole unit; the segment-to-chunk assignment makes every
//    8-lane phase of a 16-byte shared load hit 8 distinct bank groups under
//    the swizzle; packed fp32x2 FMAs; partial dots summed with shuffles.
//  * PV: lane owns D/32 consecutive output dims for all G heads; the
//    probabilities are broadcast as duplicated pairs through shared memory so
//    the packed FMAs need no register moves.
//  * split merge fused in: each split writes its (O, LSE) partial, and the
//    last split of a (sequence, K/V head) to finish (an atomic count) merges
//    all of them into the output.  No second kernel.
//  * fp32 accumulation, base-2 online softmax with the scale folded into q,
//    output rescaled only when a warp's running maximum moves.
#include <cuda.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 4
#endif
#ifndef PKV_DECODE_MIN_BLOCKS
#define PKV_DECODE_MIN_BLOCKS 3
#endif

constexpr int kPage = 32;
constexpr int kWarps = 4;                      // consumer warps
constexpr int kStages = PKV_DECODE_STAGES;     // pages in flight per CTA
constexpr int kMinBlocks = PKV_DECODE_MIN_BLOCKS;  // CTAs per SM the sizes are chosen for
constexpr int kThreads = (kWarps + 1) * 32;
// PKV_FLAG_TEST_WAIT_TIMEOUT: the limit of the waits that are meant to run
// out (consumers on a barrier nothing completes; the producer's ring waits)
constexpr uint64_t kTestWaitNs = 20000;

struct UnitDesc {
    int b, kvh, split, key_begin, key_end, r0, nsplit, pad;
};

template <int D, int G>
struct DecodeSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = kPage * D * 2;          // one page-head of K (or V)
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kRedHeads = G < 2 ? G : 2;            // heads per output-merge round
    static constexpr int kQbufOff = kRingBytes;                // [2 slots][G][D] bf16
    static constexpr int kQbufBytes = 2 * G * D * 2;
    static constexpr int kRedOOff = kQbufOff + kQbufBytes;     // [warps][kRedHeads][D] f32
    static constexpr int kRedOBytes = kWarps * kRedHeads * D * 4;
    static constexpr int kPbufOff = kRedOOff + kRedOBytes;     // per warp: [8 keys][G] float2 + [G] alpha
    static constexpr int kPbufWarp = 8 * G * 8 + G * 4;
    static constexpr int kPbufBytes = kWarps * ((kPbufWarp + 15) & ~15);
    static constexpr int kRedMLOff = kPbufOff + kPbufBytes;    // m, l: [warps][G] f32
    static constexpr int kRedMLBytes = 2 * kWarps * G * 4;
    static constexpr int kDescOff = kRedMLOff + kRedMLBytes;   // 2 UnitDesc + flags
    static constexpr int kDescBytes = 2 * sizeof(UnitDesc) + 16;
    static constexpr int kBarOff = (kDescOff + kDescBytes + 7) & ~7;
    // full[kStages], empty[kStages], dfull[2], dempty[2], never (test hook)
    static constexpr int kBytes = kBarOff + (2 * kStages + 5) * 8;
    // 228 KiB of shared memory per SM, 1 KiB of it reserved per CTA
    static_assert(kBytes <= (228 / kMinBlocks - 1) * 1024, "CTAs per SM must fit in shared memory");
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// Scheduling region of the workspace: [0] unit ticket and [1 + b*Hkv + h]
// finished splits; the unit count; the sequences in full-split order; the unit
// list (split, b*Hkv + h) in ticket order.
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;
constexpr int kPlanMaxFull = 2047;  // full splits per sequence the planner orders
constexpr int kPlanBuckets = 1024;  // length buckets of the partial splits
constexpr int kPlanSmemSeqs = 4096; // sequences whose full-split order stays in shared memory

__host__ __device__ constexpr size_t align256(size_t n) { return (n + 255) / 256 * 256; }

struct Sched {
    int* counters;
    int* total;
    int* seq_at_pos;
    int2* list;
    __host__ __device__ static size_t counters_bytes(int B, int Hkv) {
        return align256((static_cast<size_t>(B) * Hkv + 1) * sizeof(int));
    }
    __host__ __device__ static size_t bytes(int B, int Hkv, int S) {
        return counters_bytes(B, Hkv) + 256 + align256(static_cast<size_t>(B) * sizeof(int)) +
               align256(static_cast<size_t>(B) * Hkv * (S > 0 ? S : 1) * sizeof(int2));
    }
    __host__ __device__ Sched(void* base, int B, int Hkv) {
        char* w = static_cast<char*>(base);
        counters = reinterpret_cast<int*>(w);
        w += counters_bytes(B, Hkv);
        total = reinterpret_cast<int*>(w);
        w += 256;
        seq_at_pos = reinterpret_cast<int*>(w);
        w += align256(static_cast<size_t>(B) * sizeof(int));
        list = reinterpret_cast<int2*>(w);
    }
};

// whether the planner can order the units of this call (else: split-major)
inline bool plan_fits(const AttnParams& p) { return p.max_kv_len / p.split_keys <= kPlanMaxFull; }

// The keys a decode row attends (0 for a padding row), or -1 for a sequence
// without rows; the same reading of the inputs as the producer's.
__device__ __forceinline__ int row_keys(const AttnParams& p, int b) {
    const int nrows = p.q_indptr[b + 1] - p.q_indptr[b];
    if (nrows <= 0) return -1;
    const int qreal = p.q_real ? p.q_real[b] : nrows;
    const int kv = min(max(p.kv_lens[b], 0), p.max_kv_len);
    return qreal <= 0 ? 0 : kv;
}

// In-place exclusive prefix sum of a[0, n), n <= 2 * kPlanThreads; returns the
// total.  All threads of the block call it.
__device__ int block_scan_exclusive(int* a, int n, int* warp_tot) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int i0 = 2 * t, i1 = 2 * t + 1;
    const int x0 = i0 < n ? a[i0] : 0, x1 = i1 < n ? a[i1] : 0;
    int v = x0 + x1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) warp_tot[w] = v;
    __syncthreads();
    if (w == 0) {
        int u = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, u, o);
            if (lane >= o) u += y;
        }
        warp_tot[lane] = u;  // inclusive over warps
    }
    __syncthreads();
    const int before = (w > 0 ? warp_tot[w - 1] : 0) + v - (x0 + x1);
    const int total = warp_tot[31];
    __syncthreads();
    if (i0 < n) a[i0] = before;
    if (i1 < n) a[i1] = before + x0;
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const AttnParams p) {
    __shared__ int cnt_f[kPlanMaxFull + 2];   // sequences per full-split count, then cursors
    __shared__ int gt_f[kPlanMaxFull + 2];    // sequences with more than s full splits
    __shared__ int cnt_r[kPlanBuckets];       // partial splits per length bucket, then cursors
    __shared__ int warp_tot[32];
    __shared__ int n_empty, e_cur;
    __shared__ int seq_smem[kPlanSmemSeqs];   // sequences in full-split order (small batches)
    // the decode launch behind this one may start its prologue now; it waits
    // for this grid's writes before reading any of them
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int B = p.batch, Hkv = p.num_kv_heads, SK = p.split_keys;
    const int nF = p.max_kv_len / SK + 1;     // full-split counts 0 .. nF - 1
    Sched sc(p.ws_counters, B, Hkv);
    int* seq_at_pos = B <= kPlanSmemSeqs ? seq_smem : sc.seq_at_pos;
    const int tid = threadIdx.x;
    int keys0 = -1;                           // row_keys of b = tid (the first pass's)
    for (int i = tid; i <= B * Hkv; i += kPlanThreads) sc.counters[i] = 0;
    for (int i = tid; i < nF + 1; i += kPlanThreads) cnt_f[i] = 0;
    for (int i = tid; i < kPlanBuckets; i += kPlanThreads) cnt_r[i] = 0;
    if (tid == 0) n_empty = e_cur = 0;
    __syncthreads();
    auto bucket_of = [&](int r) {  // longer partial splits in higher buckets
        return static_cast<int>((static_cast<int64_t>(r) * kPlanBuckets) / SK);
    };
    for (int b = tid, j = 0; b < B; b += kPlanThreads, ++j) {
        const int kv = row_keys(p, b);
        if (j == 0) keys0 = kv;
        if (kv < 0) continue;
        const int f = kv / SK, r = kv - f * SK;
        atomicAdd(&cnt_f[f], 1);
        if (r > 0) atomicAdd(&cnt_r[bucket_of(r)], 1);
        if (kv == 0) atomicAdd(&n_empty, 1);
    }
    __syncthreads();
    // sequences with more than s full splits: gt_f[s] = (all with f >= 1) - #{1 <= f <= s}
    cnt_f[0] = 0;  // sequences without a full split take no position
    __syncthreads();
    for (int i = tid; i < nF; i += kPlanThreads) gt_f[i] = cnt_f[i];
    __syncthreads();
    const int with_full = block_scan_exclusive(gt_f, nF, warp_tot);  // gt_f[s] = #{f < s}
    for (int i = tid; i < nF; i += kPlanThreads) {
        const int le = gt_f[i] + cnt_f[i];       // #{1 <= f <= s}
        gt_f[i] = with_full - le;                // #{f > s}
        cnt_f[i] = with_full - le;               // cursor: positions of f == s start here
    }
    __syncthreads();
    // unit index of the first full unit of split s: Hkv * sum_{t < s} gt_f[t]
    const int full_seq_splits = block_scan_exclusive(gt_f, nF, warp_tot);
    const int full_units = full_seq_splits * Hkv;
    // partial splits, longest bucket first: start of bucket k = #{buckets > k}
    const int partials = block_scan_exclusive(cnt_r, kPlanBuckets, warp_tot);  // #{< k}
    __syncthreads();
    for (int b = tid, j = 0; b < B; b += kPlanThreads, ++j) {
        const int kv = j == 0 ? keys0 : row_keys(p, b);
        if (kv < 0) continue;
        const int f = kv / SK, r = kv - f * SK;
        if (f > 0) seq_at_pos[atomicAdd(&cnt_f[f], 1)] = b;
        int at = -1, split = 0;
        if (r > 0) {
            // descending: the first slot of bucket k is partials - #{<= k}
            const int k = bucket_of(r);
            const int below = atomicAdd(&cnt_r[k], 1);  // #{< k} + rank in bucket
            at = full_units + (partials - 1 - below) * Hkv;
            split = f;
        } else if (kv == 0) {
            at = full_units + (partials + atomicAdd(&e_cur, 1)) * Hkv;
        }
        if (at >= 0)
            for (int h = 0; h < Hkv; ++h) sc.list[at + h] = make_int2(split, b * Hkv + h);
    }
    __syncthreads();
    // full units, split-major; split s holds the gt_f-count sequences of most full splits
    for (int u = tid; u < full_units; u += kPlanThreads) {
        int lo = 0, hi = nF - 1;  // last s with Hkv * gt_f[s] <= u (gt_f now holds the prefix)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gt_f[mid] * Hkv <= u) lo = mid; else hi = mid - 1;
        }
        const int idx = u - gt_f[lo] * Hkv;
        sc.list[u] = make_int2(lo, seq_at_pos[idx / Hkv] * Hkv + idx % Hkv);
    }
    if (tid == 0) *sc.total = full_units + (partials + n_empty) * Hkv;
}

// The same order for a small batch (B <= kSmallPlanSeqs sequences, fewer than
// kSmallPlanSplits full splits each), one thread per sequence and exact ranks
// instead of counting passes: four warps and three barriers instead of 32 warps
// and a dozen.  Sequence b with f full splits and a partial split of r keys:
//  * its full split s < f is unit Hkv * (P(s) + rank_f(b)) + h, where P(s) =
//    sum over all sequences of min(f, s) (the units of the splits before s) and
//    rank_f(b) = #{sequences with more full splits, or as many and a lower
//    index} -- exactly the sequences ahead of b among those with a split s;
//  * its partial split follows every full one, at rank_r(b) = #{sequences with
//    a longer partial split, or as long and a lower index};
//  * a row without keys (split 0, zeros) follows every partial split.
constexpr int kSmallPlanSeqs = 128;
constexpr int kSmallPlanSplits = 64;

__global__ void __launch_bounds__(kSmallPlanSeqs) decode_plan_small_kernel(const AttnParams p) {
    __shared__ int2 s_fr[kSmallPlanSeqs];        // (full splits, partial keys); f = -1: no rows
    __shared__ int s_cnt[kSmallPlanSplits];      // sequences per full-split count
    __shared__ int s_p[kSmallPlanSplits];        // P(s)
    __shared__ int s_tot[3];                     // full seq-splits, partial splits, empty rows
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int B = p.batch, Hkv = p.num_kv_heads, SK = p.split_keys;
    const int t = threadIdx.x;
    const Sched sc(p.ws_counters, B, Hkv);
    for (int i = t; i <= B * Hkv; i += kSmallPlanSeqs) sc.counters[i] = 0;
    if (t < kSmallPlanSplits) s_cnt[t] = 0;
    if (t < 3) s_tot[t] = 0;
    const int kv = t < B ? row_keys(p, t) : -1;
    const int f = kv > 0 ? kv / SK : 0;
    const int r = kv > 0 ? kv - f * SK : 0;
    s_fr[t] = make_int2(kv >= 0 ? f : -1, r);
    __syncthreads();
    if (kv >= 0) {
        atomicAdd(&s_cnt[f], 1);
        if (f > 0) atomicAdd(&s_tot[0], f);
        if (r > 0) atomicAdd(&s_tot[1], 1);
        if (kv == 0) atomicAdd(&s_tot[2], 1);
    }
    __syncthreads();
    if (t < kSmallPlanSplits) {
        int acc = 0;
        for (int v = 1; v < kSmallPlanSplits; ++v) acc += s_cnt[v] * min(v, t);
        s_p[t] = acc;
    }
    // ranks among the batch (ties by index)
    int rank_f = 0, rank_r = 0, rank_e = 0;
    for (int o = 0; o < B; ++o) {
        const int2 x = s_fr[o];
        rank_f += (x.x > f || (x.x == f && o < t)) ? 1 : 0;
        rank_r += (x.y > r || (x.y == r && o < t)) ? 1 : 0;
        rank_e += (x.x == 0 && x.y == 0 && o < t) ? 1 : 0;
    }
    __syncthreads();
    const int full_units = s_tot[0] * Hkv, partials = s_tot[1], empty = s_tot[2];
    if (kv >= 0) {
        // rank_e counted the earlier entries (0, 0): rows without keys
        // (sequences without rows carry f = -1)
        for (int s = 0; s < f; ++s) {
            const int u = Hkv * (s_p[s] + rank_f);
            for (int h = 0; h < Hkv; ++h) sc.list[u + h] = make_int2(s, t * Hkv + h);
        }
        int at = -1, split = 0;
        if (r > 0) {
            at = full_units + rank_r * Hkv;
            split = f;
        } else if (kv == 0) {
            at = full_units + (partials + rank_e) * Hkv;
        }
        if (at >= 0)
            for (int h = 0; h < Hkv; ++h) sc.list[at + h] = make_int2(split, t * Hkv + h);
    }
    if (t == 0) *sc.total = full_units + (partials + empty) * Hkv;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kWarps * 32) : "memory");
}

// Sum each of the G per-lane partial dots over the 8 lanes of a key group
// (lanes differing in bits 0..2) and leave one head's total per lane:
// a transpose-style butterfly (G=4: 4 shuffles instead of 12).  The head a
// lane ends with is head_of_lane<G>(seg).
template <int G>
__device__ __forceinline__ float reduce_heads(const float (&v)[G], int seg) {
    if constexpr (G == 4) {
        const bool hi = seg & 4;
        float k0 = hi ? v[2] : v[0], k1 = hi ? v[3] : v[1];
        const float s0 = hi ? v[0] : v[2], s1 = hi ? v[1] : v[3];
        k0 += __shfl_xor_sync(0xffffffffu, s0, 4);
        k1 += __shfl_xor_sync(0xffffffffu, s1, 4);
        const bool hi2 = seg & 2;
        float k = hi2 ? k1 : k0;
        const float sn = hi2 ? k0 : k1;
        k += __shfl_xor_sync(0xffffffffu, sn, 2);
        k += __shfl_xor_sync(0xffffffffu, k, 1);
        return k;
    } else if constexpr (G == 2) {
        const bool hi = seg & 4;
        float k = hi ? v[1] : v[0];
        const float sn = hi ? v[0] : v[1];
        k += __shfl_xor_sync(0xffffffffu, sn, 4);
        k += __shfl_xor_sync(0xffffffffu, k, 2);
        k += __shfl_xor_sync(0xffffffffu, k, 1);
        return k;
    } else {
        float k = v[0];
        k += __shfl_xor_sync(0xffffffffu, k, 4);
        k += __shfl_xor_sync(0xffffffffu, k, 2);
        k += __shfl_xor_sync(0xffffffffu, k, 1);
        return k;
    }
}
template <int G>
__device__ __forceinline__ int head_of_lane(int seg) {
    return G == 4 ? (seg >> 1) : (G == 2 ? (seg >> 2) : 0);
}

// Per-warp running state: the lane's own head (max, sum over this warp's
// keys) and the lane's output dims for every head.
template <int G, int DPL>
struct WarpState {
    float m, l;
    float2 o2[G][DPL / 2];
};

// One page for one consumer warp.  FULL: all 32 keys of the page are valid.
template <int D, int G, bool FULL>
__device__ __forceinline__ void decode_page(WarpState<G, D / 32>& ws, const float2 (&q2)[G][D / 16],
                                            const uint8_t* K, const uint8_t* V, float2* pb,
                                            float* alpha_buf, int warp, int kk, int seg, int lane,
                                            int nvalid_rows) {
    constexpr int kDPL = D / 32;
    const int half = (D == 128) ? (seg >> 2) : 0;
    const int c0 = (D == 128) ? ((seg & 3) + 4 * (seg >> 2)) : seg;
    const int hg = head_of_lane<G>(seg);
    const bool rep = (seg & (8 / G - 1)) == 0;  // one lane per (key, head) publishes

    float s[2];
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int row = warp * 8 + pass * 4 + kk;
        float2 acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
        {
            const uint4 a = *reinterpret_cast<const uint4*>(K + half * 4096 + sw128_offset(row, c0));
            const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 kv = make_float2(bf16lo(w[j]), bf16hi(w[j]));
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = __ffma2_rn(q2[g][j], kv, acc[g]);
            }
        }
        if constexpr (D == 128) {
            const uint4 a = *reinterpret_cast<const uint4*>(K + half * 4096 + sw128_offset(row, c0 ^ 4));
            const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 kv = make_float2(bf16lo(w[j]), bf16hi(w[j]));
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = __ffma2_rn(q2[g][4 + j], kv, acc[g]);
            }
        }
        float part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] = acc[g].x + acc[g].y;
        const float t = reduce_heads<G>(part, seg);
        s[pass] = (FULL || (pass * 4 + kk) < nvalid_rows) ? t : -INFINITY;
    }

    // online softmax of the lane's head over this warp's 8 keys
    float mx = fmaxf(s[0], s[1]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float m_new = fmaxf(ws.m, mx);
    float p0 = 0.f, p1 = 0.f, alpha = 1.f;
    if (m_new != -INFINITY) {
        alpha = fast_exp2(ws.m - m_new);  // 0 on the first keys, 1 if unchanged
        p0 = fast_exp2(s[0] - m_new);
        p1 = fast_exp2(s[1] - m_new);
        ws.m = m_new;
    }
    ws.l = ws.l * alpha + (rep ? p0 + p1 : 0.f);
    if (rep) {
        pb[kk * G + hg] = make_float2(p0, p0);
        pb[(4 + kk) * G + hg] = make_float2(p1, p1);
        if (kk == 0) alpha_buf[hg] = alpha;
    }
    __syncwarp();

    // rescale the output of any head whose maximum moved (warp-uniform test)
    float al[G];
#pragma unroll
    for (int g = 0; g < G; ++g) al[g] = alpha_buf[g];
    bool moved = false;
#pragma unroll
    for (int g = 0; g < G; ++g) moved |= al[g] != 1.f;
    if (moved) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int j = 0; j < kDPL / 2; ++j)
                ws.o2[g][j] = make_float2(ws.o2[g][j].x * al[g], ws.o2[g][j].y * al[g]);
    }

    // PV over the warp's keys of this page
    const int pv_half = (D == 128) ? (lane >> 4) : 0;
    const int pv_chunk = (D == 128) ? ((lane & 15) >> 1) : (lane >> 2);
    const int pv_byte = (D == 128) ? ((lane & 1) * 8) : ((lane & 3) * 4);
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8) {
        if (FULL || k8 < nvalid_rows) {
            const int row = warp * 8 + k8;
            const uint8_t* vp = V + pv_half * 4096 + sw128_offset(row, pv_chunk) + pv_byte;
            if constexpr (kDPL == 4) {
                const uint2 w = *reinterpret_cast<const uint2*>(vp);
                const float2 va = make_float2(bf16lo(w.x), bf16hi(w.x));
                const float2 vb = make_float2(bf16lo(w.y), bf16hi(w.y));
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float2 pp = pb[k8 * G + g];
                    ws.o2[g][0] = __ffma2_rn(pp, va, ws.o2[g][0]);
                    ws.o2[g][1] = __ffma2_rn(pp, vb, ws.o2[g][1]);
                }
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
                const float2 va = make_float2(bf16lo(w), bf16hi(w));
#pragma unroll
                for (int g = 0; g < G; ++g) ws.o2[g][0] = __ffma2_rn(pb[k8 * G + g], va, ws.o2[g][0]);
            }
        }
    }
    __syncwarp();
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const AttnParams p) {
    using S = DecodeSmem<D, G>;
    constexpr int kDPL = D / 32;      // output dims per PV lane
    // The dynamic shared window of a CTA starts 1024-byte aligned (no static
    // shared memory here), which the 128-byte TMA swizzle pattern relies on.
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
    uint64_t* empty = full + kStages;
    uint64_t* dfull = empty + kStages;   // [2] unit descriptor + its query rows landed
    uint64_t* dempty = dfull + 2;        // [2] consumers done with the descriptor slot
    uint64_t* never = dempty + 2;        // test hook: a barrier nothing completes
    UnitDesc* desc = reinterpret_cast<UnitDesc*>(smem + S::kDescOff);
    int* flags = reinterpret_cast<int*>(smem + S::kDescOff + 2 * sizeof(UnitDesc));
    float* red_o = reinterpret_cast<float*>(smem + S::kRedOOff);
    float* red_m = reinterpret_cast<float*>(smem + S::kRedMLOff);
    float* red_l = red_m + kWarps * G;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int Hq = p.num_q_heads;
    const int Hkv = p.num_kv_heads;
    const int SK = p.split_keys;
    const int S_ = p.num_splits;
    const int64_t rows_bound = static_cast<int64_t>(p.batch) * p.max_q_rows;

    if ((smem_u32(smem) & 1023u) != 0) {  // never expected; refuse rather than misread tiles
        if (threadIdx.x == 0) set_err(p.err, PKV_ERRBIT_TIMEOUT);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&dfull[s], 1);
            mbar_init(&dempty[s], kWarps);
        }
        mbar_init(never, 1);
        flags[0] = 0;  // "this CTA merges the splits of its unit"
        flags[1] = 0;  // set when a consumer wait gives up
        fence_mbar_init();
    }
    // launched behind the planner with programmatic serialisation: its unit
    // order and zeroed counters are visible after this wait
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();

    if (warp == kWarps) {
        // ====================== producer ======================================
        if (lane != 0) return;
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        const Sched sc(p.ws_counters, p.batch, Hkv);
        int* ticket = sc.counters;
        const int BH = p.batch * Hkv;
        const bool listed = p.planned;
        const int units = listed ? __ldcg(sc.total) : BH * S_;
        const uint64_t ring_limit = p.test_wait_timeout ? kTestWaitNs : 2000000000ull;
        int i = 0;  // pages issued so far (ring position)
        int published = 0;  // unit descriptors published (dfull phases armed)
        bool alive = true;
        for (int k = 0; alive; ++k) {
            UnitDesc d;
            d.b = -1;
            for (;;) {
                const int u = atomicAdd(ticket, 1);
                if (u >= units) break;
                int split, bh;
                if (listed) {
                    const int2 e = __ldcg(&sc.list[u]);
                    split = e.x;
                    bh = e.y;
                } else {
                    split = u / BH;
                    bh = u - split * BH;
                }
                const int b = bh / Hkv;
                const int r0 = p.q_indptr[b];
                const int nrows = p.q_indptr[b + 1] - r0;
                if (nrows <= 0) continue;
                const int qreal = p.q_real ? p.q_real[b] : nrows;
                int kv_len = p.kv_lens[b];
                if (p.checked && (kv_len > p.max_kv_len || kv_len < 0 || nrows > 1))
                    set_err(p.err, PKV_ERRBIT_LEN);
                kv_len = min(max(kv_len, 0), p.max_kv_len);
                if (qreal <= 0) kv_len = 0;  // a padding row attends nothing
                const int kb = split * SK;
                const int ke = min(kv_len, kb + SK);
                // a unit with keys, or split 0 of a row without keys (writes zeros)
                if (ke > kb || split == 0) {
                    d.b = b;
                    d.kvh = bh - b * Hkv;
                    d.split = split;
                    d.key_begin = kb;
                    d.key_end = max(ke, kb);
                    d.r0 = r0;
                    d.nsplit = (kv_len + SK - 1) / SK;
                    break;
                }
            }
            const int slot = k & 1;
            if (k >= 2 && !mbar_wait(&dempty[slot], ((k >> 1) - 1) & 1, ring_limit)) {
                set_err(p.err, PKV_ERRBIT_TIMEOUT);
                d.b = -1;  // tell the consumers to stop (they may time out too)
            }
            desc[slot] = d;
            if (d.b >= 0 && d.key_end > d.key_begin) {
                mbar_arrive_expect_tx(&dfull[slot], G * D * 2);
                const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                            static_cast<int64_t>(d.r0) * p.q_token_stride;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    bulk_load(smem + S::kQbufOff + (slot * G + g) * D * 2,
                              qrow + static_cast<int64_t>(d.kvh * G + g) * p.q_head_stride,
                              D * 2, &dfull[slot]);
            } else {
                mbar_arrive(&dfull[slot]);
            }
            published = k + 1;
            if (d.b < 0) break;
            const int npages = (d.key_end - d.key_begin + kPage - 1) / kPage;
            const int32_t* bt =
                p.block_table + static_cast<int64_t>(d.b) * p.block_table_stride + d.key_begin / kPage;
            for (int pi = 0; pi < npages; ++pi, ++i) {
                const int st = i % kStages;
                if (i >= kStages && !mbar_wait(&empty[st], ((i / kStages) - 1) & 1, ring_limit)) {
                    set_err(p.err, PKV_ERRBIT_TIMEOUT);
                    alive = false;
                    break;
                }
                int phys = bt[pi];
                if (p.checked && (phys < 0 || phys >= p.num_pages)) {
                    set_err(p.err, PKV_ERRBIT_PAGE);
                    phys = static_cast<int>(p.num_pages);  // outside the tensor: TMA fills zeros
                }
                uint8_t* kd = smem + st * S::kStageBytes;
                uint8_t* vd = kd + S::kTileBytes;
                mbar_arrive_expect_tx(&full[st], S::kStageBytes);
#pragma unroll
                for (int h = 0; h < S::kHalves; ++h) {
                    tma_load_4d(kd + h * 4096, &tm_k, &full[st], h * 64, d.kvh, 0, phys);
                    tma_load_4d(vd + h * 4096, &tm_v, &full[st], h * 64, d.kvh, 0, phys);
                }
            }
        }
        // do not leave while copies into this CTA's shared memory are in flight:
        // the last pages of the ring, and the query rows of the last two
        // descriptors (consumers that gave up never waited for them)
        for (int j = max(0, i - kStages); j < i; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1);
        for (int k = max(0, published - 2); k < published; ++k) mbar_wait(&dfull[k & 1], (k >> 1) & 1);
        return;
    }

    // ====================== consumers =========================================
    const int kk = lane >> 3;   // key within a pass of 4
    const int seg = lane & 7;   // QK segment
    const int half = (D == 128) ? (seg >> 2) : 0;
    const int c0 = (D == 128) ? ((seg & 3) + 4 * (seg >> 2)) : seg;
    const int hg = head_of_lane<G>(seg);
    const bool rep = (seg & (8 / G - 1)) == 0;
    float2* pb = reinterpret_cast<float2*>(smem + S::kPbufOff + warp * ((S::kPbufWarp + 15) & ~15));
    float* alpha_buf = reinterpret_cast<float*>(pb + 8 * G);

    int i = 0;  // pages consumed so far (ring position)
    for (int k = 0;; ++k) {
        const int slot = k & 1;
        if (!mbar_wait(&dfull[slot], (k >> 1) & 1)) {
            if (lane == 0) set_err(p.err, PKV_ERRBIT_TIMEOUT);
            break;
        }
        const UnitDesc d = desc[slot];
        if (d.b < 0) break;

        // query rows of the unit, pre-scaled into the base-2 domain
        float2 q2[G][D / 16];
        if (d.key_end > d.key_begin) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const __nv_bfloat16* qh =
                    reinterpret_cast<const __nv_bfloat16*>(smem + S::kQbufOff) + (slot * G + g) * D + half * 64;
                const uint4 a = *reinterpret_cast<const uint4*>(qh + c0 * 8);
                const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    q2[g][j] = make_float2(bf16lo(wa[j]) * p.scale_log2, bf16hi(wa[j]) * p.scale_log2);
                if constexpr (D == 128) {
                    const uint4 c = *reinterpret_cast<const uint4*>(qh + (c0 ^ 4) * 8);
                    const uint32_t wc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        q2[g][4 + j] =
                            make_float2(bf16lo(wc[j]) * p.scale_log2, bf16hi(wc[j]) * p.scale_log2);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[slot]);

        WarpState<G, kDPL> ws;
        ws.m = -INFINITY;
        ws.l = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int j = 0; j < kDPL / 2; ++j) ws.o2[g][j] = make_float2(0.f, 0.f);

        int npages = (d.key_end - d.key_begin + kPage - 1) / kPage;
        bool failed = false;
        if (p.test_wait_timeout && npages > 0 && !mbar_wait(never, 0, kTestWaitNs)) {
            // the test hook: a page wait that runs out, before the unit's first
            // page is consumed; the unit is abandoned as after a real timeout
            if (lane == 0) set_err(p.err, PKV_ERRBIT_TIMEOUT);
            failed = true;
            npages = 0;
        }
        for (int pi = 0; pi < npages; ++pi, ++i) {
            const int st = i % kStages;
            if (!mbar_wait(&full[st], (i / kStages) & 1)) {
                // give up on this unit but still take part in the barriers below,
                // so that every consumer warp leaves together
                if (lane == 0) set_err(p.err, PKV_ERRBIT_TIMEOUT);
                failed = true;
                break;
            }
            const uint8_t* K = smem + st * S::kStageBytes;
            const uint8_t* V = K + S::kTileBytes;
            const int key0 = d.key_begin + pi * kPage;
            if (key0 + kPage <= d.key_end) {
                decode_page<D, G, true>(ws, q2, K, V, pb, alpha_buf, warp, kk, seg, lane, 8);
            } else {
                const int nvalid_rows = min(8, d.key_end - (key0 + warp * 8));
                decode_page<D, G, false>(ws, q2, K, V, pb, alpha_buf, warp, kk, seg, lane, nvalid_rows);
            }
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        if (failed && lane == 0) flags[1] = 1;

        // ---------------- merge the four warps' states of this unit ---------
        // the lane's head sum over this warp's keys (rep lanes hold the terms)
        ws.l += __shfl_xor_sync(0xffffffffu, ws.l, 8);
        ws.l += __shfl_xor_sync(0xffffffffu, ws.l, 16);
        if (kk == 0 && rep) {
            red_m[warp * G + hg] = ws.m;
            red_l[warp * G + hg] = ws.l;
        }
        const int bh = d.b * Hkv + d.kvh;
        const bool partial = d.nsplit > 1;
        constexpr int RH = S::kRedHeads;
#pragma unroll
        for (int g0 = 0; g0 < G; g0 += RH) {
#pragma unroll
            for (int gg = 0; gg < RH; ++gg)
#pragma unroll
                for (int j = 0; j < kDPL / 2; ++j)
                    *reinterpret_cast<float2*>(&red_o[(warp * RH + gg) * D + lane * kDPL + 2 * j]) =
                        ws.o2[g0 + gg][j];
            consumer_sync();
            for (int e = threadIdx.x; e < RH * D; e += kWarps * 32) {
                const int gg = e / D, dd = e - (e / D) * D;
                const int g = g0 + gg;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * G + g]);
                float L = 0.f, O = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) {
                        const float f = fast_exp2(red_m[w * G + g] - M);
                        L = fmaf(f, red_l[w * G + g], L);
                        O = fmaf(f, red_o[(w * RH + gg) * D + dd], O);
                    }
                }
                O *= L > 0.f ? 1.0f / L : 0.f;
                const float lse = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
                const int64_t st = static_cast<int64_t>(d.r0) * Hq + d.kvh * G + g;
                if (!partial) {
                    if (p.out_f32) static_cast<float*>(p.out)[st * D + dd] = O;
                    else static_cast<__nv_bfloat16*>(p.out)[st * D + dd] = __float2bfloat16_rn(O);
                    if (p.lse && dd == 0) p.lse[st] = lse;
                } else if (d.r0 < rows_bound) {
                    p.ws_o[(st * S_ + d.split) * D + dd] = O;
                    if (dd == 0) p.ws_lse[st * S_ + d.split] = lse;
                }
            }
            consumer_sync();  // red_o is rewritten by the next round
        }
        if (partial && d.r0 < rows_bound) {
            // the last split of this (sequence, K/V head) to finish merges all
            __threadfence();
            consumer_sync();
            if (threadIdx.x == 0) {
                const int done = atomicAdd(&p.ws_counters[1 + bh], 1);
                const int last = done == d.nsplit - 1;
                if (last) atomicExch(&p.ws_counters[1 + bh], 0);
                flags[0] = last;
            }
            consumer_sync();
            if (flags[0]) {
                __threadfence();
                for (int e = threadIdx.x; e < G * D; e += kWarps * 32) {
                    const int g = e / D, dd = e - (e / D) * D;
                    const int64_t st = static_cast<int64_t>(d.r0) * Hq + d.kvh * G + g;
                    const float* lses = p.ws_lse + st * S_;
                    const float* os = p.ws_o + st * S_ * D + dd;
                    // the splits' states eight at a time, all loads in flight
                    // together, merged online (one chunk: max first, then sums)
                    float M = -INFINITY, L = 0.f, O = 0.f;
                    for (int sp0 = 0; sp0 < d.nsplit; sp0 += 8) {
                        float lv[8], ov[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const bool in = sp0 + u < d.nsplit;
                            lv[u] = in ? __ldcg(lses + sp0 + u) : -INFINITY;
                            ov[u] = in ? __ldcg(os + static_cast<int64_t>(sp0 + u) * D) : 0.f;
                        }
                        float mc = lv[0];
#pragma unroll
                        for (int u = 1; u < 8; ++u) mc = fmaxf(mc, lv[u]);
                        const float Mn = fmaxf(M, mc);
                        if (Mn != -INFINITY) {
                            const float c = __expf(M - Mn);  // 0 while nothing was merged
                            L *= c;
                            O *= c;
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const float w = __expf(lv[u] - Mn);
                                L += w;
                                O = fmaf(w, ov[u], O);
                            }
                            M = Mn;
                        }
                    }
                    O *= L > 0.f ? 1.0f / L : 0.f;
                    if (p.out_f32) static_cast<float*>(p.out)[st * D + dd] = O;
                    else static_cast<__nv_bfloat16*>(p.out)[st * D + dd] = __float2bfloat16_rn(O);
                    if (p.lse && dd == 0) p.lse[st] = L > 0.f ? M + __logf(L) : -INFINITY;
                }
            }
            consumer_sync();  // flags[0] is rewritten by the next unit
        }
        if (flags[1]) break;  // a wait timed out: every consumer warp stops here
    }
}

template <int D, int G>
cudaError_t launch_dg(const AttnParams& p_in, const void* tk, const void* tv, int dev, int sms,
                      cudaStream_t s) {
    using S = DecodeSmem<D, G>;
    auto kern = decode_kernel<D, G>;
    // shared-memory opt-in and occupancy: once per device
    static DeviceOnce occupancy;
    int per_sm = 0;
    cudaError_t e = occupancy.get(dev, &per_sm, [&](int, int* v) {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
        if (r != cudaSuccess) return r;
        int n = 0;
        r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, S::kBytes);
        *v = n > 0 ? n : 1;
        return r;
    });
    if (e != cudaSuccess) return e;
    const int64_t units = static_cast<int64_t>(p_in.batch) * p_in.num_kv_heads * p_in.num_splits;
    const int64_t grid = std::min<int64_t>(units, static_cast<int64_t>(std::max(per_sm, 1)) * sms);
    // the unit tickets and the per-(sequence, head) split counts start at zero.
    // With more units than CTAs the planner also orders the units (the tail
    // then runs on the shortest); otherwise every unit starts at once and a
    // plain reset is the shorter path
    AttnParams p = p_in;
    p.planned = units > grid && plan_fits(p);
    if (p.planned) {
        if (p.batch <= kSmallPlanSeqs && p.max_kv_len / p.split_keys < kSmallPlanSplits)
            decode_plan_small_kernel<<<1, kSmallPlanSeqs, 0, s>>>(p);
        else
            decode_plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
        e = cudaGetLastError();
    } else {
        e = cudaMemsetAsync(p.ws_counters, 0, Sched::counters_bytes(p.batch, p.num_kv_heads), s);
    }
    if (e != cudaSuccess) return e;
    // behind the planner: programmatic serialisation lets the launch and the
    // CTAs' prologue overlap the planner (the kernel waits for its writes)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = S::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.planned ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, *static_cast<const CUtensorMap*>(tk),
                              *static_cast<const CUtensorMap*>(tv), p);
}

}  // namespace

bool decode_supported(int head_dim, int group) {
    return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4);
}

size_t decode_sched_bytes(int batch, int num_kv_heads, int splits) {
    return Sched::bytes(batch, num_kv_heads, splits);
}

cudaError_t launch_decode(const AttnParams& p, const void* tk, const void* tv, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static DeviceOnce sm_count;
    e = sm_count.get(dev, &sms, [](int d, int* v) {
        return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, d);
    });
    if (e != cudaSuccess) return e;
    const int G = p.num_q_heads / p.num_kv_heads;
#define PKV_DEC(D_, G_) \
    if (p.head_dim == D_ && G == G_) return launch_dg<D_, G_>(p, tk, tv, dev, sms, s);
    PKV_DEC(128, 4) PKV_DEC(128, 2) PKV_DEC(128, 1)
    PKV_DEC(64, 4) PKV_DEC(64, 2) PKV_DEC(64, 1)
#undef PKV_DEC
    return cudaErrorInvalidValue;
}

}  // namespace pkv
