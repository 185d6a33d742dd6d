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
// Single CTA (B <= 1024): the batch-wide rank and offset computations are
// block scans in shared memory; the pairwise passes are O(B^2 / threads).
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kPP = 32;
constexpr int kMaxRows = 1024;

// exclusive prefix sum of v over the first n threads' values (n <= blockDim)
__device__ int block_exclusive_scan(int v, int* buf) {
    const int t = threadIdx.x;
    buf[t] = v;
    __syncthreads();
    for (int off = 1; off < blockDim.x; off <<= 1) {
        const int add = t >= off ? buf[t - off] : 0;
        __syncthreads();
        buf[t] += add;
        __syncthreads();
    }
    const int incl = buf[t];
    __syncthreads();
    return incl - v;
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
    // leaders
    int leader = r;
    if (row && cp >= 1) {
        const int f = s_first[r];
        for (int r2 = 0; r2 < r; ++r2) {
            if (s_cp[r2] >= 1 && s_first[r2] == f) {
                leader = r2;
                break;
            }
        }
    }
    if (row) {
        s_leader[r] = leader;
        atomicAdd(&s_size[leader], 1);
        if (leader == r) s_run[r] = cp;
    }
    __syncthreads();
    // shared run: every member lowers its leader's run to their common prefix
    if (row && leader != r) {
        const int32_t* lrow = a.block_table + static_cast<int64_t>(leader) * a.block_table_stride;
        const int lim = min(cp, s_cp[leader]);
        int p = 0;
        while (p < lim && trow[p] == lrow[p]) ++p;
        atomicMin(&s_run[leader], p);
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
    int tail_start = run;
    if (row) {
        for (int r2 = 0; r2 < r; ++r2) {
            if (s_leader[r2] == leader) {
                ++pos;
                tail_start += s_tp[r2];
            }
        }
    }
    // group index and offsets (scans over leader flags / sizes in row order)
    const bool is_leader = row && leader == r;
    const int gidx_mine = block_exclusive_scan(is_leader ? 1 : 0, s_scan);
    const int goff_mine = block_exclusive_scan(is_leader ? s_size[r] : 0, s_scan);
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
        int32_t* grow = a.group_rows + static_cast<int64_t>(g) * a.group_row_stride;
        if (is_leader) {
            a.run_lens[g] = run * kPP;
            a.group_indptr[g] = s_goff[r];
            for (int p = 0; p < run && p < a.group_row_stride; ++p) grow[p] = trow[p];
        }
        if (tail_start + tail_pages > a.group_row_stride) set_err(a.err, PKV_ERRBIT_LEN);
        for (int i = 0; i < tail_pages && tail_start + i < a.group_row_stride; ++i)
            grow[tail_start + i] = trow[run + i];
    }
    // unused group slots; group_indptr[g] = B from the group count on
    for (int g = ngroups + r; g <= B; g += blockDim.x) {
        if (g < B) a.run_lens[g] = 0;
        a.group_indptr[g] = B;
    }
    // the last member of each group knows where its group's pages end
    if (row) {
        bool last = true;
        for (int r2 = r + 1; r2 < B; ++r2) {
            if (s_leader[r2] == leader) {
                last = false;
                break;
            }
        }
        if (last) {
            int32_t* grow = a.group_rows + static_cast<int64_t>(s_gidx[leader]) * a.group_row_stride;
            for (int64_t p = tail_start + tail_pages; p < a.group_row_stride; ++p) grow[p] = -1;
        }
    }
    for (int64_t i = static_cast<int64_t>(ngroups) * a.group_row_stride + r;
         i < static_cast<int64_t>(B) * a.group_row_stride; i += blockDim.x)
        a.group_rows[i] = -1;
}

}  // namespace

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    plan_kernel<<<1, kMaxRows, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pkv
