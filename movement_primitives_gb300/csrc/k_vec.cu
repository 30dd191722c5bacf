// [outer, threads, vec] vector copy (Apache TVM docs "copy -> gmem_smem",
// section "Algorithm"; TileLang tutorial "loop_mapping.py" default partition).
//
// The destination-ordered modes are split into a run contiguous on both sides
// (1 word when there is none) and outer modes.  The run is cut into vectors
// of the widest of 16/8/4/2/1 bytes that keeps every per-thread pointer
// aligned; each thread moves whole vectors, global -> registers -> global.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

// Threads per CTA, vectors in flight per thread and the resident-CTA bound
// (compile-time knobs so that variants can be measured).  On GB300, with
// 512 MiB per side: 1024 threads x 4 vectors reached 88.5 % of the copy peak
// on a bf16 (0,2,1,3) permute with 64-byte runs against 86.3 % for
// 256 x 12, and gained 26 % on 16-byte runs and 6-10 % on strided gathers;
// 1024 x 2, 1024 x 6, 768 x 4, 512 x 4 and 1024 x 4 held to 32 registers
// (two CTAs per SM) were all slower.
#ifndef LC_VEC_THREADS
#define LC_VEC_THREADS 1024
#endif
#ifndef LC_VEC_UNROLL
#define LC_VEC_UNROLL 4
#endif
#ifndef LC_VEC_MIN_BLOCKS
#define LC_VEC_MIN_BLOCKS 1
#endif
constexpr int kVecThreads = LC_VEC_THREADS;
constexpr int kVecUnroll = LC_VEC_UNROLL;  // vectors in flight per thread

struct VecArgs {
    const uint8_t *src;  // address of source word offset 0
    uint8_t *dst;        // address of destination word offset 0
    int32_t n;           // outer modes, outermost first
    uint32_t e32[kMaxModes];
    FastDiv fd[kMaxModes];
    int64_t e64[kMaxModes];
    int64_t sb[kMaxModes], db[kMaxModes];  // strides in BYTES
    uint32_t run_vecs;                     // vectors per contiguous run
    FastDiv run_fd;
    int64_t run_vecs64;
    int64_t nvec;      // vectors in the whole copy
    int64_t n_blocks;  // blocks of kVecUnroll * kVecThreads vectors
};

// Byte offsets of vector g: g = run index * run_vecs + position in the run,
// the run index unflattened row-major over the outer modes.
template <int VB, bool WIDE>
__device__ __forceinline__ void vec_offsets(const VecArgs &a, int64_t g, int64_t &so, int64_t &dof) {
    if (!WIDE) {
        const uint32_t gg = static_cast<uint32_t>(g);
        uint32_t q = fast_div(gg, a.run_fd);
        so = static_cast<int64_t>(gg - q * a.run_vecs) * VB;
        dof = so;
        for (int i = a.n - 1; i >= 0; --i) {
            const uint32_t q2 = fast_div(q, a.fd[i]);
            const int64_t c = q - q2 * a.e32[i];
            so += c * a.sb[i];
            dof += c * a.db[i];
            q = q2;
        }
    } else {
        int64_t q = g / a.run_vecs64;
        so = (g - q * a.run_vecs64) * VB;
        dof = so;
        for (int i = a.n - 1; i >= 0; --i) {
            const int64_t q2 = q / a.e64[i];
            const int64_t c = q - q2 * a.e64[i];
            so += c * a.sb[i];
            dof += c * a.db[i];
            q = q2;
        }
    }
}

// Block blk owns vectors [blk * U * T, (blk + 1) * U * T); within it round f,
// thread tid moves vector f * T + tid (access_idx = f * T + tid: thread =
// access_idx % T, slot = access_idx / T).  All U loads are issued before the
// U stores so that each thread keeps U vectors in flight.  Tails are guarded.
template <int VB, bool WIDE>
__global__ void __launch_bounds__(kVecThreads, LC_VEC_MIN_BLOCKS) k_vec_copy(const __grid_constant__ VecArgs a) {
    using T = typename Word<VB>::T;
    for (int64_t blk = blockIdx.x; blk < a.n_blocks; blk += gridDim.x) {
        const int64_t base = blk * (kVecUnroll * kVecThreads) + threadIdx.x;
        T v[kVecUnroll];
        int64_t dofs[kVecUnroll];
#pragma unroll
        for (int f = 0; f < kVecUnroll; ++f) {
            const int64_t g = base + int64_t(f) * kVecThreads;
            dofs[f] = -1;
            if (g < a.nvec) {
                int64_t so, dof;
                vec_offsets<VB, WIDE>(a, g, so, dof);
                v[f] = __ldg(reinterpret_cast<const T *>(a.src + so));
                dofs[f] = dof;
            }
        }
#pragma unroll
        for (int f = 0; f < kVecUnroll; ++f)
            if (dofs[f] >= 0) store_out<T>(a.dst + dofs[f], v[f]);
    }
}

namespace {

template <int VB, bool WIDE>
int launch_vec_t(const VecArgs &a, cudaStream_t stream) {
    const void *fn = reinterpret_cast<const void *>(&k_vec_copy<VB, WIDE>);
    int sms, per;
    if (prepare(fn, kVecThreads, 0, 0, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t grid = lmin(a.n_blocks, int64_t(sms) * per);
    k_vec_copy<VB, WIDE><<<static_cast<unsigned>(grid), kVecThreads, 0, stream>>>(a);
    return finish_launch();
}

template <bool WIDE>
int launch_vec_w(int vb, const VecArgs &a, cudaStream_t s) {
    switch (vb) {
        case 1: return launch_vec_t<1, WIDE>(a, s);
        case 2: return launch_vec_t<2, WIDE>(a, s);
        case 4: return launch_vec_t<4, WIDE>(a, s);
        case 8: return launch_vec_t<8, WIDE>(a, s);
        case 16: return launch_vec_t<16, WIDE>(a, s);
    }
    return LC_ERR_UNSUPPORTED;
}

}  // namespace

int launch_vec(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    VecArgs a{};
    a.src = src + p.src_off * p.w;
    a.dst = dst + p.dst_off * p.w;
    const VecPlan &vp = p.vec;
    a.n = vp.outer.n;
    int64_t runs = 1;
    bool wide = false;
    for (int i = 0; i < vp.outer.n; ++i) {
        const Mode &m = vp.outer.m[i];
        a.e64[i] = m.e;
        a.sb[i] = m.s * p.w;
        a.db[i] = m.d * p.w;
        runs *= m.e;
        if (m.e >= (int64_t(1) << 32)) {
            wide = true;
        } else {
            a.e32[i] = static_cast<uint32_t>(m.e);
            a.fd[i] = make_fastdiv(a.e32[i]);
        }
    }
    a.run_vecs64 = vp.run / vp.vec;
    a.nvec = runs * a.run_vecs64;
    if (a.nvec >= (int64_t(1) << 32) || a.run_vecs64 >= (int64_t(1) << 32)) wide = true;
    if (!wide) {
        a.run_vecs = static_cast<uint32_t>(a.run_vecs64);
        a.run_fd = make_fastdiv(a.run_vecs);
    }
    a.n_blocks = (a.nvec + kVecUnroll * kVecThreads - 1) / (kVecUnroll * kVecThreads);
    const int vb = vp.vec * p.w;
    return wide ? launch_vec_w<true>(vb, a, stream) : launch_vec_w<false>(vb, a, stream);
}

}  // namespace lc
