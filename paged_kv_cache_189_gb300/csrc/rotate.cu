// rotate.cu -- rotate_rows: in-place left rotation of every row.
//
// "Paged causal K/V cache and cached attention for VisualGen", Description,
// Cache (eviction is an in-place rotation on the device) and per-file notes on
// rotateRows (element sizes, shifts, strided rows, no-op cases; the page's
// kernel uses three reversals).
//
// Two kernels, chosen on the host:
//  * cycle kernel: a left rotation by `shift` of `cols` elements splits into
//    g = gcd(cols, shift) independent cycles of length cols / g (position p
//    takes the value of p + shift).  One thread walks one cycle, loading
//    eight values ahead before storing, so every element is read once and
//    written once (the algorithmic 2x bytes) and consecutive threads touch
//    consecutive addresses.  Used when rows * g gives enough threads.
//  * reversal kernels: the three-reversal identity (reverse [0, shift) and
//    [shift, cols), then the whole row) in two launches; any g, twice the
//    traffic.  Used when the cycles are too few to fill the GPU.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

template <int U> struct UnitT;
template <> struct UnitT<1> { using T = uint8_t; };
template <> struct UnitT<2> { using T = uint16_t; };
template <> struct UnitT<4> { using T = uint32_t; };
template <> struct UnitT<8> { using T = uint2; };
template <> struct UnitT<16> { using T = uint4; };

constexpr int kAhead = 8;

template <int U>
__global__ void __launch_bounds__(256) rotate_cycles_kernel(char* x, int64_t rows, int64_t cols,
                                                            int64_t row_stride, int64_t shift,
                                                            int64_t g) {
    using T = typename UnitT<U>::T;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= g * rows) return;
    const int64_t r = idx / g;
    const int64_t start = idx - r * g;
    T* row = reinterpret_cast<T*>(x + r * row_stride * U);
    const int64_t len = cols / g;
    // positions p_k = (start + k * shift) mod cols; new[p_k] = old[p_{k+1}]
    const T first = row[start];
    int64_t pos = start;  // p_k, next to be stored
    int64_t k = 0;
    while (k < len - 1) {
        const int64_t left = len - 1 - k;
        const int n = left < kAhead ? static_cast<int>(left) : kAhead;
        T vals[kAhead];
        int64_t src[kAhead];
        int64_t p = pos;
#pragma unroll
        for (int i = 0; i < kAhead; ++i) {
            if (i < n) {
                p += shift;
                if (p >= cols) p -= cols;
                src[i] = p;
                vals[i] = row[p];
            }
        }
#pragma unroll
        for (int i = 0; i < kAhead; ++i) {
            if (i < n) {
                row[pos] = vals[i];
                pos = src[i];
            }
        }
        k += n;
    }
    row[pos] = first;
}

// Reverse [a0, a1) and, when b1 > b0, [b0, b1) of every row.
template <int U>
__global__ void __launch_bounds__(256) reverse_kernel(char* x, int64_t rows, int64_t row_stride,
                                                      int64_t a0, int64_t a1, int64_t b0,
                                                      int64_t b1) {
    using T = typename UnitT<U>::T;
    const int64_t half_a = (a1 - a0) / 2;
    const int64_t half_b = (b1 - b0) / 2;
    const int64_t per_row = half_a + half_b;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= per_row * rows) return;
    const int64_t r = idx / per_row;
    int64_t i = idx - r * per_row;
    T* row = reinterpret_cast<T*>(x + r * row_stride * U);
    int64_t lo, hi;
    if (i < half_a) {
        lo = a0 + i;
        hi = a1 - 1 - i;
    } else {
        i -= half_a;
        lo = b0 + i;
        hi = b1 - 1 - i;
    }
    const T t = row[lo];
    row[lo] = row[hi];
    row[hi] = t;
}

int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

template <int U>
cudaError_t run(void* x, int64_t rows, int64_t cols, int64_t row_stride, int64_t shift,
                cudaStream_t s) {
    char* p = static_cast<char*>(x);
    const int threads = 256;
    const int64_t g = gcd64(cols, shift);
    // enough independent cycles to keep HBM busy (each thread keeps 8 loads in flight)
    if (g * rows >= 16384) {
        const int64_t blocks = (g * rows + threads - 1) / threads;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        rotate_cycles_kernel<U><<<blocks, threads, 0, s>>>(p, rows, cols, row_stride, shift, g);
        return cudaGetLastError();
    }
    const int64_t n1 = (shift / 2 + (cols - shift) / 2) * rows;
    if (n1 > 0) {
        reverse_kernel<U><<<(n1 + threads - 1) / threads, threads, 0, s>>>(p, rows, row_stride, 0,
                                                                          shift, shift, cols);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int64_t n2 = (cols / 2) * rows;
    reverse_kernel<U><<<(n2 + threads - 1) / threads, threads, 0, s>>>(p, rows, row_stride, 0,
                                                                      cols, 0, 0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rotate(void* x, int64_t rows, int64_t cols, int64_t row_stride, int unit,
                          int64_t shift, cudaStream_t s) {
    switch (unit) {
        case 16: return run<16>(x, rows, cols, row_stride, shift, s);
        case 8: return run<8>(x, rows, cols, row_stride, shift, s);
        case 4: return run<4>(x, rows, cols, row_stride, shift, s);
        case 2: return run<2>(x, rows, cols, row_stride, shift, s);
        default: return run<1>(x, rows, cols, row_stride, shift, s);
    }
}

}  // namespace pkv
