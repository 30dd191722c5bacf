// Window sum with a cooperative shared-memory fetch (MLC course "Ep7: GPU and
// Hardware Acceleration", section "Window Sum Example"):
//     b[i] = a[i] + a[i+1] + ... + a[i+window-1]   (float32, left to right).
//
// A CTA takes chunks of kStChunk outputs.  Copy in: the chunk's inputs plus
// the (window - 1)-element halo are fetched into shared memory by all threads
// with the [outer, threads, vec] split of "copy -> gmem_smem" (16-byte
// asynchronous copies when the base allows, a guarded 4-byte tail), into one
// of two buffers so that the next chunk's fetch overlaps this chunk's sums.
// Compute, windows of up to kStRegWindow: thread t produces outputs
// 4 (g T + t) .. + 3 of the chunk from two 16-byte shared reads (lanes read
// consecutive 16-byte words: conflict-free), every sum formed in registers in
// the page's order, and stores them as one 16-byte word when the output base
// allows.  Wider windows: thread t produces outputs t, t + T, ..., reading
// window consecutive shared words per output.  Each input word leaves HBM
// once.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

// Threads per CTA and outputs per thread per chunk (compile-time knobs so
// that variants can be measured).  Measured on GB300 on 2^28 outputs, window
// 3, 4096-output chunks: 1024 threads x 4 outputs 97.2 % of the copy peak,
// 512 x 8 95.2 %, 256 x 16 93.1 %, 128 x 32 93.1 %.
#ifndef LC_WIN_THREADS
#define LC_WIN_THREADS 1024
#endif
#ifndef LC_WIN_PER
#define LC_WIN_PER 4
#endif
constexpr int kStThreads = LC_WIN_THREADS;
constexpr int kStPer = LC_WIN_PER;                 // outputs per thread per chunk
constexpr int kStChunk = kStThreads * kStPer;      // outputs per chunk
constexpr int kStMaxWindow = LC_WINDOW_SUM_MAX;
constexpr int kStBuf = kStChunk + kStMaxWindow;    // floats per shared buffer
constexpr int kStRegWindow = 5;                    // widest window summed from registers
static_assert(kStPer % 4 == 0, "the register path forms four sums per group");

struct StencilArgs {
    const float *a;
    float *b;
    int64_t n;        // outputs
    int32_t window;
    int64_t n_chunks;
    bool vec_out;     // b is 16-byte aligned
};

// Issues this thread's share of chunk c's fetch into buffer `buf` and commits
// it as one cp.async group (empty group past the last chunk).
template <bool VEC>
__device__ __forceinline__ void fetch_chunk(const StencilArgs &p, int64_t c, uint32_t buf) {
    const int t = threadIdx.x;
    if (c < p.n_chunks) {
        const int64_t i0 = c * kStChunk;
        const int need = static_cast<int>(lmin(kStChunk + p.window - 1, p.n + p.window - 1 - i0));
        int done = 0;
        if (VEC) {
            const int nv = need / 4;
            for (int q = t; q < nv; q += kStThreads) ptx::cp_async16(buf + 16 * q, p.a + i0 + 4 * q);
            done = nv * 4;
        }
        for (int j = done + t; j < need; j += kStThreads) ptx::cp_async4(buf + 4 * j, p.a + i0 + j);
    }
    ptx::cp_async_commit();
}

// Outputs i0 + j .. i0 + j + 3 of a window of WIN (<= kStRegWindow) from the
// chunk's shared inputs cur[j .. j + 7].
template <int WIN>
__device__ __forceinline__ void sums4(const StencilArgs &p, const float *cur, int64_t i0, int j) {
    const float4 lo = *reinterpret_cast<const float4 *>(cur + j);
    const float4 hi = *reinterpret_cast<const float4 *>(cur + j + 4);
    const float x[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    float o[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        float acc = x[v];
#pragma unroll
        for (int k = 1; k < WIN; ++k) acc = __fadd_rn(acc, x[v + k]);
        o[v] = acc;
    }
    const int64_t i = i0 + j;
    if (p.vec_out && i + 4 <= p.n) {
        store_out<float4, true>(p.b + i, make_float4(o[0], o[1], o[2], o[3]));
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v)
            if (i + v < p.n) p.b[i + v] = o[v];
    }
}

// Chunks c = blockIdx.x + i * gridDim.x, double-buffered: chunk i+1's fetch
// is in flight while chunk i is summed.  WIN = 0: any window (per-output
// loop over shared words); WIN > 0: that window, from registers.
template <bool VEC, int WIN>
__global__ void __launch_bounds__(kStThreads) k_window_sum(const __grid_constant__ StencilArgs p) {
    __shared__ __align__(16) float s[2][kStBuf];
    const int t = threadIdx.x;
    const uint32_t buf0 = ptx::smem_addr(&s[0][0]), buf1 = ptx::smem_addr(&s[1][0]);
    int64_t c = blockIdx.x;
    fetch_chunk<VEC>(p, c, buf0);
    for (int it = 0; c < p.n_chunks; c += gridDim.x, ++it) {
        fetch_chunk<VEC>(p, c + gridDim.x, (it & 1) ? buf0 : buf1);
        ptx::cp_async_wait<1>();  // this thread's part of chunk c has landed
        __syncthreads();          // ... and everyone else's
        const float *cur = s[it & 1];
        const int64_t i0 = c * kStChunk;
        if constexpr (WIN > 0) {
#pragma unroll
            for (int g = 0; g < kStPer / 4; ++g) {
                const int j = 4 * (g * kStThreads + t);  // lanes read consecutive 16-byte words
                if (i0 + j < p.n) sums4<WIN>(p, cur, i0, j);
            }
        } else {
#pragma unroll 4
            for (int q = 0; q < kStPer; ++q) {
                const int j = q * kStThreads + t;  // lanes read consecutive words
                if (i0 + j < p.n) {
                    float acc = cur[j];
                    for (int k = 1; k < p.window; ++k) acc = __fadd_rn(acc, cur[j + k]);
                    p.b[i0 + j] = acc;
                }
            }
        }
        __syncthreads();  // the buffer just read is refilled at the next iteration's start
    }
    ptx::cp_async_wait<0>();
}

namespace {

template <bool VEC, int WIN>
int launch_window_sum(const StencilArgs &p, cudaStream_t cs) {
    const void *fn = reinterpret_cast<const void *>(&k_window_sum<VEC, WIN>);
    int sms, per;
    if (prepare(fn, kStThreads, 0, 0, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const unsigned grid = static_cast<unsigned>(lmin(p.n_chunks, int64_t(sms) * per));
    k_window_sum<VEC, WIN><<<grid, kStThreads, 0, cs>>>(p);
    return finish_launch();
}

template <bool VEC>
int launch_window_sum_v(const StencilArgs &p, cudaStream_t cs) {
    switch (p.window) {
        case 2: return launch_window_sum<VEC, 2>(p, cs);
        case 3: return launch_window_sum<VEC, 3>(p, cs);
        case 4: return launch_window_sum<VEC, 4>(p, cs);
        case 5: return launch_window_sum<VEC, 5>(p, cs);
        default: return launch_window_sum<VEC, 0>(p, cs);
    }
}

}  // namespace

}  // namespace lc

extern "C" int lc_window_sum_f32(const float *a, float *b, int64_t n_out, int32_t window, lc_stream_t stream) {
    using namespace lc;
    if (n_out < 0 || window < 1 || window > LC_WINDOW_SUM_MAX) return LC_ERR_SHAPE;
    if (n_out == 0) return LC_OK;
    if (!a || !b) return LC_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(a) % 4 || reinterpret_cast<uintptr_t>(b) % 4) return LC_ERR_ALIGN;
    const int64_t n_in = n_out + window - 1;
    if (n_in > (int64_t(1) << 60) / 4) return LC_ERR_OVERFLOW;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), a1 = a0 + uintptr_t(n_in) * 4;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b), b1 = b0 + uintptr_t(n_out) * 4;
    if (a0 < b1 && b0 < a1) return LC_ERR_OVERLAP;
    StencilArgs p{a, b, n_out, window, (n_out + kStChunk - 1) / kStChunk, b0 % 16 == 0};
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    return a0 % 16 == 0 ? launch_window_sum_v<true>(p, cs) : launch_window_sum_v<false>(p, cs);
}
