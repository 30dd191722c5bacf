// Copy under a loop-layout override (TileLang tutorial "loop_mapping.py",
// module docstring: a loop_layout= annotation replaces the default plan).
//
// One CTA of T threads per tile (tiles spread over the grid).  Thread t owns
// the points the override maps to (t, 0), (t, 1), ..., (t, L - 1) and moves
// them in slot order, global -> registers -> global.  A point's row-major
// flat index in the tile is the thread's part (its thread digits, fixed per
// thread) plus the slot's part (its slot digits); the flat index is then
// unflattened over the tile's logical modes into a source and a destination
// offset.  When the override's innermost mode is a slot mode of stride 1,
// `vec` consecutive slots are consecutive points of one contiguous run and
// move as one vector.  Several vectors per thread are in flight.
//
// Split path: when the loop's mixed radix and the tile's logical radix nest
// (one divisibility chain of suffix products), the thread digits and the
// slot digits fall on disjoint digits of the common refinement, on which
// both offsets are affine, so offset(thread part + slot part) =
// offset(thread part) + offset(slot part).  Each thread then computes its own
// offsets once, and each CTA tabulates the slot vectors' offsets once in
// shared memory (every lane of a warp reads the same entry: a broadcast); a
// vector costs one shared load and two adds instead of two digit decodes.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

// Vectors in flight per thread and slot vectors per shared offset table
// (compile-time knobs so that variants can be measured).
#ifndef LC_LOOP_UNROLL
#define LC_LOOP_UNROLL 4
#endif
#ifndef LC_LOOP_TABLE
#define LC_LOOP_TABLE 2048
#endif
constexpr int kLoopUnroll = LC_LOOP_UNROLL;
constexpr int kLoopTable = LC_LOOP_TABLE;  // 8 bytes per entry

struct LoopArgs {
    const uint8_t *src;  // word 0 of tile 0
    uint8_t *dst;
    int64_t sts, dts;  // tile strides, bytes
    int64_t n_tiles;
    int32_t n;  // logical modes of a tile, outermost first
    uint32_t e32[kMaxModes];
    FastDiv fd[kMaxModes];
    int64_t e64[kMaxModes];
    int64_t sb[kMaxModes], db[kMaxModes];  // strides, bytes
    int32_t nt, ns;                        // thread digits, slot digits (ascending stride)
    uint32_t te[LC_MAX_RANK];
    FastDiv tfd[LC_MAX_RANK];
    int64_t tw[LC_MAX_RANK];  // row-major weight of each thread digit
    uint32_t se32[LC_MAX_RANK];
    FastDiv sfd[LC_MAX_RANK];
    int64_t se64[LC_MAX_RANK];
    int64_t sw[LC_MAX_RANK];  // weight per unit of each digit of the VECTOR index
    int64_t N, L, nvec;       // points per tile, slots per thread, vectors per thread
    int32_t vec;
    int64_t *trace;
};

// Flat-index part of vector q of a thread: q's digits over the slot modes
// (the stride-1 digit counted in vectors), each times its weight.
template <bool WIDE>
__device__ __forceinline__ int64_t slot_flat(const LoopArgs &a, int64_t q) {
    int64_t f = 0;
    if (!WIDE) {
        uint32_t r = static_cast<uint32_t>(q);
        for (int i = 0; i < a.ns; ++i) {
            const uint32_t r2 = fast_div(r, a.sfd[i]);
            f += static_cast<int64_t>(r - r2 * a.se32[i]) * a.sw[i];
            r = r2;
        }
    } else {
        for (int i = 0; i < a.ns; ++i) {
            const int64_t q2 = q / a.se64[i];
            f += (q - q2 * a.se64[i]) * a.sw[i];
            q = q2;
        }
    }
    return f;
}

// Byte offsets of flat index `flat` of a tile, unflattened over the logical
// modes (last fastest).
template <bool WIDE>
__device__ __forceinline__ void point_offsets(const LoopArgs &a, int64_t flat, int64_t &so, int64_t &dof) {
    so = 0;
    dof = 0;
    if (!WIDE) {
        uint32_t r = static_cast<uint32_t>(flat);
        for (int i = a.n - 1; i >= 0; --i) {
            const uint32_t r2 = fast_div(r, a.fd[i]);
            const int64_t c = r - r2 * a.e32[i];
            so += c * a.sb[i];
            dof += c * a.db[i];
            r = r2;
        }
    } else {
        for (int i = a.n - 1; i >= 0; --i) {
            const int64_t r2 = flat / a.e64[i];
            const int64_t c = flat - r2 * a.e64[i];
            so += c * a.sb[i];
            dof += c * a.db[i];
            flat = r2;
        }
    }
}

// trace[tile * N + flat + j] = t * L + slot + j for the vector's points.
__device__ __forceinline__ void trace_vector(const LoopArgs &a, int64_t tile, int64_t flat, uint32_t t,
                                             int64_t q) {
    const int64_t base = tile * a.N + flat;
    const int64_t slot = static_cast<int64_t>(t) * a.L + q * a.vec;
    for (int j = 0; j < a.vec; ++j) a.trace[base + j] = slot + j;
}

template <int VB, bool WIDE, bool SPLIT>
__global__ void __launch_bounds__(LC_LOOP_MAX_THREADS) k_loop_copy(const __grid_constant__ LoopArgs a) {
    using T = typename Word<VB>::T;
    const uint32_t t = threadIdx.x;
    int64_t tflat = 0;  // this thread's part of every flat index
    {
        uint32_t r = t;
        for (int i = 0; i < a.nt; ++i) {
            const uint32_t r2 = fast_div(r, a.tfd[i]);
            tflat += static_cast<int64_t>(r - r2 * a.te[i]) * a.tw[i];
            r = r2;
        }
    }
    if constexpr (SPLIT) {
        __shared__ int2 tab[kLoopTable];  // (source, destination) byte offsets of slot vectors
        int64_t tso, tdo;
        point_offsets<WIDE>(a, tflat, tso, tdo);
        for (int64_t cb = 0; cb < a.nvec; cb += kLoopTable) {
            const int n = static_cast<int>(lmin(kLoopTable, a.nvec - cb));
            __syncthreads();  // the previous chunk's table is no longer read
            for (int i = t; i < n; i += blockDim.x) {
                int64_t so, dof;
                point_offsets<WIDE>(a, slot_flat<WIDE>(a, cb + i), so, dof);
                tab[i] = make_int2(static_cast<int>(so), static_cast<int>(dof));
            }
            __syncthreads();
            for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
                const uint8_t *src = a.src + tile * a.sts + tso;
                uint8_t *dst = a.dst + tile * a.dts + tdo;
                for (int i0 = 0; i0 < n; i0 += kLoopUnroll) {
                    T v[kLoopUnroll];
                    int2 o[kLoopUnroll];
#pragma unroll
                    for (int u = 0; u < kLoopUnroll; ++u) {
                        if (i0 + u < n) {
                            o[u] = tab[i0 + u];
                            v[u] = *reinterpret_cast<const T *>(src + o[u].x);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kLoopUnroll; ++u) {
                        if (i0 + u >= n) continue;
                        store_out<T>(dst + o[u].y, v[u]);
                        if (a.trace) trace_vector(a, tile, tflat + slot_flat<WIDE>(a, cb + i0 + u), t, cb + i0 + u);
                    }
                }
            }
        }
        return;
    }
    for (int64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x) {
        const uint8_t *src = a.src + tile * a.sts;
        uint8_t *dst = a.dst + tile * a.dts;
        for (int64_t q0 = 0; q0 < a.nvec; q0 += kLoopUnroll) {
            T v[kLoopUnroll];
            int64_t dofs[kLoopUnroll], flats[kLoopUnroll];
#pragma unroll
            for (int u = 0; u < kLoopUnroll; ++u) {
                dofs[u] = -1;
                flats[u] = 0;
                if (q0 + u < a.nvec) {
                    const int64_t flat = tflat + slot_flat<WIDE>(a, q0 + u);
                    int64_t so, dof;
                    point_offsets<WIDE>(a, flat, so, dof);
                    v[u] = *reinterpret_cast<const T *>(src + so);
                    dofs[u] = dof;
                    flats[u] = flat;
                }
            }
#pragma unroll
            for (int u = 0; u < kLoopUnroll; ++u) {
                if (dofs[u] < 0) continue;
                store_out<T>(dst + dofs[u], v[u]);
                if (a.trace) trace_vector(a, tile, flats[u], t, q0 + u);
            }
        }
    }
}

namespace {

template <int VB, bool WIDE, bool SPLIT>
int launch_loop_t(const LoopArgs &a, int threads, cudaStream_t stream) {
    const void *fn = reinterpret_cast<const void *>(&k_loop_copy<VB, WIDE, SPLIT>);
    int sms, per;
    if (prepare(fn, threads, 0, 0, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t grid = lmin(a.n_tiles, int64_t(sms) * (per > 0 ? per : 1));
    k_loop_copy<VB, WIDE, SPLIT><<<static_cast<unsigned>(grid), threads, 0, stream>>>(a);
    return finish_launch();
}

// The split path needs tile spans below 2^31 bytes, so never WIDE.
template <bool WIDE, bool SPLIT>
int launch_loop_w(int vb, const LoopArgs &a, int threads, cudaStream_t s) {
    switch (vb) {
        case 1: return launch_loop_t<1, WIDE, SPLIT>(a, threads, s);
        case 2: return launch_loop_t<2, WIDE, SPLIT>(a, threads, s);
        case 4: return launch_loop_t<4, WIDE, SPLIT>(a, threads, s);
        case 8: return launch_loop_t<8, WIDE, SPLIT>(a, threads, s);
        case 16: return launch_loop_t<16, WIDE, SPLIT>(a, threads, s);
    }
    return LC_ERR_UNSUPPORTED;
}

}  // namespace

int launch_loop(const LoopPlan &lp, const uint8_t *src, uint8_t *dst, int64_t *trace, cudaStream_t stream) {
    LoopArgs a{};
    a.src = src + lp.src_off * lp.w;
    a.dst = dst + lp.dst_off * lp.w;
    a.sts = lp.sts * lp.w;
    a.dts = lp.dts * lp.w;
    a.n_tiles = lp.n_tiles;
    const bool wide = lp.N >= (int64_t(1) << 32);
    a.n = lp.logical.n;
    for (int i = 0; i < a.n; ++i) {
        const Mode &m = lp.logical.m[i];
        a.e64[i] = m.e;
        a.sb[i] = m.s * lp.w;
        a.db[i] = m.d * lp.w;
        if (!wide) {
            a.e32[i] = static_cast<uint32_t>(m.e);
            a.fd[i] = make_fastdiv(a.e32[i]);
        }
    }
    a.nt = lp.nt;
    for (int i = 0; i < lp.nt; ++i) {
        a.te[i] = static_cast<uint32_t>(lp.td[i].e);  // T <= LC_LOOP_MAX_THREADS
        a.tfd[i] = make_fastdiv(a.te[i]);
        a.tw[i] = lp.td[i].weight;
    }
    // slot digits of the vector index: the stride-1 digit (the innermost
    // mode when vec > 1) counts vectors, so its extent shrinks by vec and its
    // weight grows by vec
    a.ns = lp.ns;
    for (int i = 0; i < lp.ns; ++i) {
        int64_t e = lp.sd[i].e, wgt = lp.sd[i].weight;
        if (i == 0 && lp.vec > 1) {
            e /= lp.vec;
            wgt *= lp.vec;
        }
        a.se64[i] = e;
        a.sw[i] = wgt;
        if (!wide) {
            a.se32[i] = static_cast<uint32_t>(e);
            a.sfd[i] = make_fastdiv(a.se32[i]);
        }
    }
    a.N = lp.N;
    a.L = lp.L;
    a.vec = lp.vec;
    a.nvec = lp.L / lp.vec;
    a.trace = trace;
    const int vb = lp.vec * lp.w;
    const int threads = static_cast<int>(lp.T);
    if (wide) return launch_loop_w<true, false>(vb, a, threads, stream);
    return lp.split ? launch_loop_w<false, true>(vb, a, threads, stream)
                    : launch_loop_w<false, false>(vb, a, threads, stream);
}

}  // namespace lc

extern "C" int lc_layout_copy_loop(const void *src, const lc_tile_layout *src_layout, void *dst,
                                   const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles,
                                   const lc_loop_layout *loop, int64_t *trace, lc_stream_t stream) {
    using namespace lc;
    PtrInfo ptr;
    ptr.src = reinterpret_cast<uintptr_t>(src);
    ptr.dst = reinterpret_cast<uintptr_t>(dst);
    ptr.check = true;
    LoopPlan lp;
    const int st = make_loop_plan(src_layout, dst_layout, elem_bytes, n_tiles, loop, ptr, &lp);
    if (st) return st;
    if (lp.n_tiles == 0 || lp.N == 0) return LC_OK;
    if (trace && reinterpret_cast<uintptr_t>(trace) % alignof(int64_t)) return LC_ERR_ALIGN;
    return launch_loop(lp, static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst), trace,
                       reinterpret_cast<cudaStream_t>(stream));
}
