// Device helpers shared by the kernel translation units.  Each unit that
// includes this header gets its own copy of the error word (one per CUDA
// module); lc_last_device_error reads and clears all of them.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "lc_internal.h"
#include "ptx.cuh"

namespace lc {

// First error recorded by this module's kernels since it was last read:
// bits 0-7 lc_status, 8-15 kernel class, 16-63 block index.
static __device__ unsigned long long g_error_word;

__device__ __forceinline__ void report_error(uint32_t status, uint32_t kernel_class) {
    const unsigned long long v = static_cast<unsigned long long>(status) |
                                 (static_cast<unsigned long long>(kernel_class) << 8) |
                                 (static_cast<unsigned long long>(blockIdx.x) << 16);
    atomicCAS(&g_error_word, 0ull, v);
}

// Host side: read this module's error word, clearing it when set.
static inline cudaError_t take_module_error(unsigned long long *v) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_error_word, sizeof(*v));
    if (e != cudaSuccess || *v == 0) return e;
    const unsigned long long zero = 0;
    return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
}

__host__ __device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv &f) {
    return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(n, f.m)) + n) >> f.s);
}

// Global stores of the copy kernels: with LC_STORE_CS = 1 (or CS = true for
// one call site) they carry the streaming cache hint (st.global.cs: the line
// is likely written once, evict it first).  Measured on GB300: the window
// sum gains 1.4 points of the copy peak with it (97.9 -> 99.3 %); the vector
// copy loses 1.2, the tile transpose moves -1.5 .. +2.3 by width, the other
// classes do not move.
#ifndef LC_STORE_CS
#define LC_STORE_CS 0
#endif
template <typename T, bool CS = (LC_STORE_CS != 0)>
__device__ __forceinline__ void store_out(void *p, const T &v) {
    if constexpr (CS)
        __stcs(reinterpret_cast<T *>(p), v);
    else
        *reinterpret_cast<T *>(p) = v;
}

template <int B> struct Word;
template <> struct Word<1> { using T = uint8_t; };
template <> struct Word<2> { using T = uint16_t; };
template <> struct Word<4> { using T = uint32_t; };
template <> struct Word<8> { using T = uint2; };
template <> struct Word<16> { using T = uint4; };

}  // namespace lc
