// layout.cu -- causal_layout: the per-block rows of a forward over exact
// windows, computed on the device at commit.
//
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Cache ("Exact window" bullet: a page table starts a key sequence only at a
// page boundary, so each causal block gets private pages at the end of its row
// holding the visible slots of the partly visible pages, then the block's own
// tokens; the commit bullet: a layout kernel reads the table and rewrites the
// per-block tensors on the device) and the review notes on committed_private /
// current_private.
//
// Geometry of block k (positions in the long sequence, page P = 32):
//   base = pin + committed, s = base + k * block_size, e = s + n (n its tokens),
//   window start ws = max(pin, s - window), visible = [0, pin) u [ws, e).
// A logical page is referenced directly when it is fully visible and ends at
// or before s.  Because the visible set is two intervals, those pages are at
// most two contiguous ranges and the remaining visible tokens (the private
// tokens, in logical order) at most three intervals:
//   ws == pin: pages [0, s/P) by reference; private [P*(s/P), e).
//   ws >  pin: pages [0, pin/P) and [ceil(ws/P), s/P) (if not empty);
//              private [P*(pin/P), pin) (fixed-region tail),
//              [ws, P*ceil(ws/P)) and [P*(s/P), e) -- or [ws, e) as one
//              interval when the second page range is empty.
// Private tokens ascend in position, so the committed ones (position < base)
// come first, then the earlier blocks' staged tokens, then the block's own:
// each list index is the private index minus the preceding kinds' counts.
//
// One CTA per block; everything is closed form, no search.  Bounds on every
// output are checked against the caller's strides and capacities.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kP = 32;
constexpr int kComPerBlock = 3 * (kP - 1);
constexpr int kCurPerBlock = 2 * (kP - 1);

__device__ __forceinline__ int64_t overlap(int64_t a0, int64_t a1, int64_t b0, int64_t b1) {
    const int64_t lo = a0 > b0 ? a0 : b0, hi = a1 < b1 ? a1 : b1;
    return hi > lo ? hi - lo : 0;
}

__global__ void __launch_bounds__(256) causal_layout_kernel(LayoutArgs a) {
    const int k = blockIdx.x;
    const int64_t F = a.pin, W = a.window;
    const int64_t committed = *a.committed;
    const int64_t base = F + (committed > 0 ? committed : 0);
    const int first = k * a.block_size;
    const int n = min(a.block_size, a.num_staged - first);
    const int64_t s = base + first, e = s + n;
    const int64_t ws = s - W > F ? s - W : F;

    // direct page ranges [0, r1) and [r2a, r2b); private intervals A, B, C
    int64_t r1, r2a = 0, r2b = 0;
    int64_t a0 = 0, a1 = 0, b0 = 0, b1 = 0, c0 = 0, c1 = 0;
    if (ws == F) {
        r1 = s / kP;
        c0 = r1 * kP;
        c1 = e;
    } else {
        r1 = F / kP;
        a0 = r1 * kP;
        a1 = F;
        const int64_t c = (ws + kP - 1) / kP, f = s / kP;
        if (c < f) {
            r2a = c;
            r2b = f;
            b0 = ws;
            b1 = c * kP;
            c0 = f * kP;
            c1 = e;
        } else {
            b0 = ws;
            b1 = e;
        }
    }
    const int64_t na = a1 - a0, nb = b1 - b0, nc = c1 - c0;
    const int64_t n_priv = na + nb + nc;
    const int64_t n_direct = r1 + (r2b - r2a);
    const int64_t n_com = overlap(a0, a1, 0, base) + overlap(b0, b1, 0, base) + overlap(c0, c1, 0, base);
    const int64_t n_cur = overlap(a0, a1, base, s) + overlap(b0, b1, base, s) + overlap(c0, c1, base, s);
    const int64_t priv_pages = (n_priv + kP - 1) / kP;
    const int32_t* priv = a.private_pages + static_cast<int64_t>(k) * a.private_stride;

    if (threadIdx.x == 0) {
        bool bad_len = priv_pages > a.private_stride || n_direct + priv_pages > a.row_stride ||
                       n_com > kComPerBlock || n_cur > kCurPerBlock;
        if (bad_len) set_err(a.err, PKV_ERRBIT_LEN);
        if ((e + kP - 1) / kP > a.num_logical_pages) set_err(a.err, PKV_ERRBIT_PAGE);
        a.kv_lens[k] = static_cast<int32_t>(n_direct * kP + n_priv);
        a.q_indptr[k] = first;
        if (k == 0) a.q_indptr[a.num_blocks] = a.num_staged;
    }
    auto slot_of = [&](int64_t p) -> int64_t {
        const int64_t lp = p / kP;
        if (lp >= a.num_logical_pages) return -1;
        return static_cast<int64_t>(a.table[lp]) * kP + (p - lp * kP);
    };

    // the row: direct pages, then private pages, then -1
    for (int64_t j = threadIdx.x; j < a.row_stride; j += blockDim.x) {
        int32_t v = -1;
        if (j < r1) {
            v = j < a.num_logical_pages ? a.table[j] : -1;
        } else if (j < n_direct) {
            const int64_t lp = r2a + (j - r1);
            v = lp < a.num_logical_pages ? a.table[lp] : -1;
        } else if (j - n_direct < priv_pages && j - n_direct < a.private_stride) {
            v = priv[j - n_direct];
        }
        a.rows[static_cast<int64_t>(k) * a.row_stride + j] = v;
    }
    // the private tokens
    for (int64_t i = threadIdx.x; i < n_priv; i += blockDim.x) {
        const int64_t p = i < na ? a0 + i : (i < na + nb ? b0 + (i - na) : c0 + (i - na - nb));
        const int64_t pg = i / kP;
        const int64_t dst = pg < a.private_stride ? static_cast<int64_t>(priv[pg]) * kP + (i - pg * kP) : -1;
        if (p < base) {
            if (i < kComPerBlock) {
                const int64_t src = slot_of(p);
                const int64_t at = static_cast<int64_t>(k) * kComPerBlock + i;
                a.com_src[at] = dst >= 0 ? src : -1;
                a.com_dst[at] = src >= 0 ? dst : -1;
            }
        } else if (p < s) {
            const int64_t c = i - n_com;
            if (c < kCurPerBlock) {
                const int64_t at = static_cast<int64_t>(k) * kCurPerBlock + c;
                a.cur_src[at] = dst >= 0 ? p - base : -1;
                a.cur_dst[at] = dst;
            }
        } else {
            a.staged_slots2[p - base] = dst;
        }
    }
    // sentinels after the block's entries
    for (int64_t c = n_com + threadIdx.x; c < kComPerBlock; c += blockDim.x) {
        a.com_src[static_cast<int64_t>(k) * kComPerBlock + c] = -1;
        a.com_dst[static_cast<int64_t>(k) * kComPerBlock + c] = -1;
    }
    for (int64_t c = n_cur + threadIdx.x; c < kCurPerBlock; c += blockDim.x) {
        a.cur_src[static_cast<int64_t>(k) * kCurPerBlock + c] = -1;
        a.cur_dst[static_cast<int64_t>(k) * kCurPerBlock + c] = -1;
    }
    // the block's own tokens: their own logical slots
    for (int t = threadIdx.x; t < n; t += blockDim.x) a.staged_slots[first + t] = slot_of(s + t);
}

}  // namespace

cudaError_t launch_causal_layout(const LayoutArgs& a, cudaStream_t s) {
    if (a.num_blocks == 0) return cudaSuccess;
    causal_layout_kernel<<<a.num_blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pkv
