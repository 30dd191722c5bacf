// Window sum with a cooperative shared-memory fetch (MLC course "Ep7: GPU and
// Hardware Acceleration", section "Window Sum Example"):
//     b[i] = a[i] + a[i+1] + ... + a[i+window-1]   (float32, left to right).
//
// A CTA takes chunks of kStChunk outputs.  Copy in: the chunk's inputs plus
// the (window - 1)-element halo are fetched into shared memory by all threads
// with the [outer, threads, vec] split of "copy -> gmem_smem" (16-byte
// asynchronous copies when the base allows, a guarded 4-byte tail), into one
// of two buffers so that the next chunk's fetch overlaps this chunk's sums.
// Compute: thread t produces outputs t, t + T, ... of the chunk, reading
// window consecutive shared words (lanes read consecutive words:
// conflict-free) and storing 32 consecutive floats per warp.  Each input word
// leaves HBM once.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

constexpr int kStThreads = 256;
constexpr int kStPer = 16;                         // outputs per thread per chunk
constexpr int kStChunk = kStThreads * kStPer;      // outputs per chunk
constexpr int kStMaxWindow = LC_WINDOW_SUM_MAX;
constexpr int kStBuf = kStChunk + kStMaxWindow;    // floats per shared buffer

struct StencilArgs {
    const float *a;
    float *b;
    int64_t n;        // outputs
    int32_t window;
    int64_t n_chunks;
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

// Chunks c = blockIdx.x + i * gridDim.x, double-buffered: chunk i+1's fetch
// is in flight while chunk i is summed.
template <bool VEC>
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
#pragma unroll 4
        for (int q = 0; q < kStPer; ++q) {
            const int j = q * kStThreads + t;  // lanes read consecutive words
            if (i0 + j < p.n) {
                float acc = cur[j];
                for (int k = 1; k < p.window; ++k) acc = __fadd_rn(acc, cur[j + k]);
                p.b[i0 + j] = acc;
            }
        }
        __syncthreads();  // the buffer just read is refilled at the next iteration's start
    }
    ptx::cp_async_wait<0>();
}

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
    StencilArgs p{a, b, n_out, window, (n_out + kStChunk - 1) / kStChunk};
    const bool vec = a0 % 16 == 0;
    const void *fn = vec ? reinterpret_cast<const void *>(&k_window_sum<true>)
                         : reinterpret_cast<const void *>(&k_window_sum<false>);
    int sms, per;
    if (prepare(fn, kStThreads, 0, 0, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const unsigned grid = static_cast<unsigned>(lmin(p.n_chunks, int64_t(sms) * per));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (vec)
        k_window_sum<true><<<grid, kStThreads, 0, cs>>>(p);
    else
        k_window_sum<false><<<grid, kStThreads, 0, cs>>>(p);
    return finish_launch();
}
