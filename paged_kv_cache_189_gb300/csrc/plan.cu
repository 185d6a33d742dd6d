// plan.cu -- plan_shared_prefix: the shared-prefix grouping of a decode /
// verification batch, built on the device once per step.
//
// "Support shared-prefix attention for n-sample requests in FMHA", commit
// notes: rows whose K/V block tables start with identical pages are grouped;
// each group's shared pages are read once; once per step a device kernel
// builds each row's page table from its group's shared run onward (batch
// order) and its K/V length past the run; the grouping depends on every
// block-table entry it read (so it is rebuilt from the tables, never reused
// across steps).
//
// Rules (one thread per row, rows r = 0..B-1, pages of 32 tokens):
//  * committed pages c_r = (kv_len - q_len) / 32: whole pages before the row's
//    first new token;
//  * leader(r) = the first row r' <= r with c_r' >= 1 and the same first page
//    (r itself when c_r = 0): one group per leader, groups ordered by leader,
//    members by row index;
//  * shared run of a group of >= 2 rows = the longest run of leading pages
//    identical in every member, at most min c over the members; 0 for a row
//    alone;
//  * group row = the run, then each member's tail pages in member order; a
//    row's tail = its keys past the run.
// One CTA (B <= 1024) computes the grouping: the batch-wide ranks and offsets
// are block scans in shared memory, the leader search O(B^2 / threads) in
// shared memory, the common-prefix scan one warp per member row.
// A second kernel writes the group rows, one CTA per group slot.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kPP = 32;
constexpr int kMaxRows = 1024;

// exclusive prefix sum of every thread's v in thread order: shuffle scans
// inside each warp, then over the warps' totals (buf: 32 ints)
__device__ int block_exclusive_scan(int v, int* buf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) buf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (blockDim.x >> 5) ? buf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        buf[lane] = w;
    }
    __syncthreads();
    const int res = (warp > 0 ? buf[warp - 1] : 0) + x - v;
    __syncthreads();  // buf is reused by the next scan
    return res;
}

__global__ void __launch_bounds__(kMaxRows) plan_kernel(PlanArgs a) {
    __shared__ int s_cp[kMaxRows];      // committed pages
    __shared__ int s_first[kMaxRows];   // first page (valid when s_cp >= 1)
    __shared__ int s_leader[kMaxRows];
    __shared__ int s_run[kMaxRows];     // at leader index: shared run in pages
    __shared__ int s_size[kMaxRows];    // at leader index: members
    __shared__ int s_tp[kMaxRows];      // tail pages
    __shared__ int s_scan[kMaxRows];
    const int B = a.batch;
    const int r = threadIdx.x;
    const bool row = r < B;
    const int32_t* trow = a.block_table + static_cast<int64_t>(r) * a.block_table_stride;

    int kv = 0, cp = 0;
    if (row) {
        kv = max(a.kv_lens[r], 0);
        const int ql = max(a.q_indptr[r + 1] - a.q_indptr[r], 0);
        cp = max(kv - ql, 0) / kPP;
        if (cp > a.max_pages) {
            set_err(a.err, PKV_ERRBIT_LEN);
            cp = a.max_pages;
        }
        s_cp[r] = cp;
        s_first[r] = cp >= 1 ? trow[0] : -1;
        s_size[r] = 0;
    }
    __syncthreads();
    // leaders: one warp per row, its lanes test 32 earlier rows per step (ballot)
    const int warp = r >> 5, lane = r & 31, nwarps = blockDim.x >> 5;
    for (int rr = warp; rr < B; rr += nwarps) {
        int ld = rr;
        if (s_cp[rr] >= 1) {
            const int f = s_first[rr];
            for (int b0 = 0; b0 < rr; b0 += 32) {
                const int r2 = b0 + lane;
                const unsigned bal = __ballot_sync(0xffffffffu, r2 < rr && s_cp[r2] >= 1 && s_first[r2] == f);
                if (bal) {
                    ld = b0 + __ffs(bal) - 1;
                    break;
                }
            }
        }
        if (lane == 0) {
            s_leader[rr] = ld;
            atomicAdd(&s_size[ld], 1);
            if (ld == rr) s_run[rr] = s_cp[rr];
        }
    }
    __syncthreads();
    const int leader = row ? s_leader[r] : r;
    // shared run: every member lowers its leader's run to its own committed
    // pages and to the first page where its table differs from the leader's.
    // One warp per member row compares 32 pages per ballot, the loads of eight
    // steps in flight before any compare, and stops at the first difference (a
    // member's table usually differs from its leader's a few pages past the
    // shared prefix).  (Two rows per warp step, twice the loads in flight,
    // measured the same.)
    if (row && leader != r) atomicMin(&s_run[leader], cp);  // never past a member's new tokens
    for (int rr = warp; rr < B; rr += nwarps) {
        const int ld = s_leader[rr];
        if (ld == rr) continue;  // uniform in the warp
        const int n = min(s_cp[rr], s_cp[ld]);
        const int32_t* ta = a.block_table + static_cast<int64_t>(rr) * a.block_table_stride;
        const int32_t* tb = a.block_table + static_cast<int64_t>(ld) * a.block_table_stride;
        int first = n;
        for (int base = 0; base < n && first == n; base += 8 * 32) {
            int32_t va[8], vb[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int pg = base + k * 32 + lane;
                va[k] = pg < n ? ta[pg] : 0;
                vb[k] = pg < n ? tb[pg] : 0;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const unsigned diff = __ballot_sync(0xffffffffu, va[k] != vb[k]);
                if (diff != 0u && first == n) first = base + k * 32 + __ffs(static_cast<int>(diff)) - 1;
            }
        }
        if (lane == 0 && first < n) atomicMin(&s_run[ld], first);
    }
    __syncthreads();
    if (row && leader == r && s_size[r] < 2) s_run[r] = 0;
    __syncthreads();
    // tails
    int run = 0, tail_len = 0, tail_pages = 0, pos = 0;
    if (row) {
        run = s_run[leader];
        tail_len = kv - run * kPP;
        tail_pages = (tail_len + kPP - 1) / kPP;
        if (run + tail_pages > a.max_pages) {
            set_err(a.err, PKV_ERRBIT_LEN);
            tail_pages = max(a.max_pages - run, 0);
        }
        s_tp[r] = tail_pages;
    }
    __syncthreads();
    // position among the group's members and tail start: one warp per row sums
    // the earlier members' tail pages 32 rows per step
    __shared__ int s_pos[kMaxRows], s_tstart[kMaxRows];
    for (int rr = warp; rr < B; rr += nwarps) {
        const int ld = s_leader[rr];
        int cnt = 0, pages = 0;
        for (int b0 = 0; b0 < rr; b0 += 32) {
            const int r2 = b0 + lane;
            const bool same = r2 < rr && s_leader[r2] == ld;
            cnt += __popc(__ballot_sync(0xffffffffu, same));
            int v = same ? s_tp[r2] : 0;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            pages += v;
        }
        if (lane == 0) {
            s_pos[rr] = cnt;
            s_tstart[rr] = s_run[ld] + pages;
        }
    }
    __syncthreads();
    int tail_start = run;
    if (row) {
        pos = s_pos[r];
        tail_start = s_tstart[r];
    }
    // group index and offsets (scans over leader flags / sizes in row order)
    const bool is_leader = row && leader == r;
    // one scan of (leader flag << 16 | members): both sums stay below 2^11
    const int packed = block_exclusive_scan(is_leader ? (1 << 16) | s_size[r] : 0, s_scan);
    const int gidx_mine = packed >> 16;
    const int goff_mine = packed & 0xffff;
    // publish the leaders' values through shared memory
    __shared__ int s_gidx[kMaxRows];
    __shared__ int s_goff[kMaxRows];
    if (is_leader) {
        s_gidx[r] = gidx_mine;
        s_goff[r] = goff_mine;
    }
    __shared__ int s_ngroups;
    if (r == B - 1) {
        // number of groups = leaders among all rows
        s_ngroups = gidx_mine + (is_leader ? 1 : 0);
        *a.num_groups = s_ngroups;
    }
    __syncthreads();
    const int ngroups = s_ngroups;
    if (row) {
        const int g = s_gidx[leader];
        a.group_of[r] = g;
        a.perm[s_goff[leader] + pos] = r;
        a.tail_start[r] = tail_start;
        a.tail_lens[r] = tail_len;
        if (is_leader) {
            a.run_lens[g] = run * kPP;
            a.group_indptr[g] = s_goff[r];
        }
        if (tail_start + tail_pages > a.group_row_stride) set_err(a.err, PKV_ERRBIT_LEN);
    }
    // unused group slots; group_indptr[g] = B from the group count on
    for (int g = ngroups + r; g <= B; g += blockDim.x) {
        if (g < B) a.run_lens[g] = 0;
        a.group_indptr[g] = B;
    }
}

// One CTA per group slot: the slot's row (the run from its first member, every
// member's tail pages at its tail start, -1 after), written from the plan's
// outputs; a slot past the number of groups gets -1 throughout.
__global__ void __launch_bounds__(256) plan_rows_kernel(PlanArgs a) {
    const int g = blockIdx.x;
    const int64_t stride = a.group_row_stride;
    int32_t* grow = a.group_rows + static_cast<int64_t>(g) * stride;
    const int ngroups = *a.num_groups;
    // the group's members (row, tail start) in shared memory; then every entry of
    // the row is one independent load: the run from the first member, a tail
    // page from the member whose tail covers it, or -1
    __shared__ int s_m[kMaxRows], s_ts[kMaxRows];
    __shared__ int s_n, s_run, s_end;
    if (threadIdx.x == 0) {
        s_n = 0;
        s_run = 0;
        s_end = 0;
        if (g < ngroups) {
            const int first = a.group_indptr[g], last = a.group_indptr[g + 1];
            s_n = min(last - first, kMaxRows);
            s_run = a.run_lens[g] / kPP;
        }
    }
    __syncthreads();
    const int n = s_n, run = s_run;
    if (g < ngroups) {
        const int first = a.group_indptr[g];
        for (int k = threadIdx.x; k < n; k += blockDim.x) {
            const int m = a.perm[first + k];
            s_m[k] = m;
            s_ts[k] = a.tail_start[m];
            if (k == n - 1) {
                const int tp = min((a.tail_lens[m] + kPP - 1) / kPP, max(a.max_pages - run, 0));
                s_end = a.tail_start[m] + tp;
            }
        }
    }
    __syncthreads();
    const int64_t end = s_end < stride ? s_end : stride;
    const int32_t* lrow = n > 0 ? a.block_table + static_cast<int64_t>(s_m[0]) * a.block_table_stride : nullptr;
    for (int64_t p = threadIdx.x; p < stride; p += blockDim.x) {
        int32_t v = -1;
        if (p < run) {
            v = lrow[p];
        } else if (p < end) {
            int lo = 0, hi = n - 1;  // last member whose tail starts at or before p
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_ts[mid] <= p) lo = mid; else hi = mid - 1;
            }
            v = a.block_table[static_cast<int64_t>(s_m[lo]) * a.block_table_stride + run + (p - s_ts[lo])];
        }
        grow[p] = v;
    }
}

}  // namespace

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    plan_kernel<<<1, kMaxRows, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    plan_rows_kernel<<<a.batch, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pkv
