// Warp-shuffle permute: transposes of V x V word blocks (V = 16 / w) moved
// through registers and warp shuffles, with no shared memory at all.
//
// The shape it takes is the scale-factor transpose of Apache TVM docs
// "permute_layout" ("Demonstration program": a (4, 32) fp32 block stored
// with strides (32, 1) and written with strides (1, 4)) and its mirror: of
// the two modes that are contiguous on one side each, one spans exactly one
// 16-byte chunk (V words) and the other a multiple of V words.  Every
// 16-byte chunk of the source then holds one row of a V x V block and every
// 16-byte chunk of the destination one column of it, so a group of V lanes
// loads the block's V chunks with one 16-byte load each, transposes it in
// registers across the group ("permute_layout", section "Algorithm": the
// register-staged phases, here with the words travelling between lanes by
// __shfl_xor_sync instead of through a shared buffer), and stores V chunks
// with one 16-byte store each.  Both phases are warp-wide accesses to whole
// 16-byte chunks, coalesced on both sides; nothing is staged in shared
// memory, so there is nothing to bank-conflict.
//
// The V x V transpose is a butterfly: for d = V/2, ..., 1, lanes a and a ^ d
// swap the elements whose index differs from their own row in bit d (lane a
// with bit d set sends its elements with bit d clear and receives the
// partner's elements with bit d set, and the other way round).  Where an
// element distance d spans whole 4-byte registers this moves registers;
// below 4 bytes it moves the masked bytes of each register.
#include <cuda_runtime.h>

#include <type_traits>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

// Geometry measured on GB300 on the 2^20-tile scale-factor permute (1 GiB a
// side): CTAs of 512 threads, one per SM by registers (16 warps), 8 chunks
// in flight per lane, 2 contiguous rounds per warp group, loads that skip L1
// and streaming stores: 99.3-99.4 % of the copy peak.  Without the store
// hint 96.9 %; without the L1 hint as well 94.9 %; 24-32 warps per SM
// (256-thread CTAs, 64-80 registers) 86 %; 4 chunks per lane 87-91 %.
#ifndef LC_SHFL_THREADS
#define LC_SHFL_THREADS 512
#endif
// Resident CTAs per SM the kernel is compiled for (caps registers).
#ifndef LC_SHFL_MIN_BLOCKS
#define LC_SHFL_MIN_BLOCKS 1
#endif
// 16-byte chunks each lane keeps in flight.
#ifndef LC_SHFL_U
#define LC_SHFL_U 8
#endif
// Rounds of U chunks per lane over one contiguous group of blocks before the
// warp moves on to its next group.
#ifndef LC_SHFL_ROUNDS
#define LC_SHFL_ROUNDS 2
#endif
// Source loads: 0 through L1 (ld.global.nc), 1 skipping L1 allocation
// (L1::no_allocate), 2 the same with a 256-byte L2 prefetch hint.
#ifndef LC_SHFL_LOAD_NA
#define LC_SHFL_LOAD_NA 1
#endif
// 1: destination stores with the streaming hint (st.global.cs).
#ifndef LC_SHFL_STORE_CS
#define LC_SHFL_STORE_CS 1
#endif

__device__ __forceinline__ uint4 shfl_load(const void *p) {
    uint4 v;
#if LC_SHFL_LOAD_NA == 2
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#elif LC_SHFL_LOAD_NA == 1
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#else
    v = __ldg(reinterpret_cast<const uint4 *>(p));
#endif
    return v;
}

__device__ __forceinline__ void shfl_store(void *p, uint4 v) {
#if LC_SHFL_STORE_CS
    __stcs(reinterpret_cast<uint4 *>(p), v);
#else
    *reinterpret_cast<uint4 *>(p) = v;
#endif
}

struct ShflArgs {
    const uint8_t *src;  // address of word offset 0 of tile 0 on each side
    uint8_t *dst;
    // byte offset of lane a's chunk of block k of a batch entry:
    //   source a * sa + k * sk, destination a * da + k * dk
    int64_t sa, sk, da, dk;
    uint32_t kb;      // blocks per batch entry
    FastDiv kb_fd;
    uint32_t n_blocks;  // batch entries * kb (< 2^31)
    int32_t nb;         // batch modes, outermost first (byte strides)
    uint32_t be[kMaxModes];
    FastDiv bfd[kMaxModes];
    int64_t bs[kMaxModes], bd[kMaxModes];
};

// Byte offsets of lane a's chunk of block blk on both sides: blk = b * kb + k
// with b the batch entry (row-major over the batch modes; the outermost mode
// needs no division).  NARROW: every offset fits 32 bits.
template <bool NARROW>
struct ShflOff {
    using T = typename std::conditional<NARROW, uint32_t, int64_t>::type;
};

template <bool NARROW>
__device__ __forceinline__ void shfl_offsets(const ShflArgs &a, uint32_t blk, int ai,
                                             typename ShflOff<NARROW>::T &so,
                                             typename ShflOff<NARROW>::T &dof) {
    using T = typename ShflOff<NARROW>::T;
    uint32_t b = fast_div(blk, a.kb_fd);
    const T k = static_cast<T>(blk - b * a.kb);
    so = static_cast<T>(ai) * static_cast<T>(a.sa) + k * static_cast<T>(a.sk);
    dof = static_cast<T>(ai) * static_cast<T>(a.da) + k * static_cast<T>(a.dk);
    for (int i = a.nb - 1; i > 0; --i) {
        const uint32_t q = fast_div(b, a.bfd[i]);
        const T c = static_cast<T>(b - q * a.be[i]);
        so += c * static_cast<T>(a.bs[i]);
        dof += c * static_cast<T>(a.bd[i]);
        b = q;
    }
    if (a.nb > 0) {
        so += static_cast<T>(b) * static_cast<T>(a.bs[0]);
        dof += static_cast<T>(b) * static_cast<T>(a.bd[0]);
    }
}

// Transpose of the V x V block of w-byte words held by the V lanes of a group,
// each lane holding its row as 16 bytes in four registers (word q of the row
// at bytes q*w .. q*w + w - 1).  Afterwards lane a holds column a.  `ai` is
// the lane's index in its group; all 32 lanes must call it together.
template <int W>
__device__ __forceinline__ void group_transpose(uint32_t (&v)[4], int ai) {
    constexpr int V = 16 / W;
#pragma unroll
    for (int d = V / 2; d >= 1; d >>= 1) {
        const bool hi = (ai & d) != 0;
        const int bd = d * W;  // byte distance of the swapped words
        if (bd >= 4) {
            const int rd = bd / 4;  // register distance
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (r & rd) continue;
                const uint32_t send = hi ? v[r] : v[r | rd];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, d);
                if (hi)
                    v[r] = recv;
                else
                    v[r | rd] = recv;
            }
        } else {
            // bytes of the words whose index has bit d clear
            const uint32_t clear = (bd == 2) ? 0x0000ffffu : 0x00ff00ffu;
            const uint32_t set = ~clear;
            const int sh = 8 * bd;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t send = hi ? (v[r] << sh) : (v[r] >> sh);
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, d);
                v[r] = hi ? ((v[r] & set) | (recv & clear)) : ((v[r] & clear) | (recv & set));
            }
        }
    }
}

// Each warp takes U * G consecutive blocks per round (G = 32 / V groups of V
// lanes, one block per group per chunk slot): lane (g, a) of slot u moves
// chunk a of block base + u * G + g.  All loads of a round are issued before
// the first transpose, all stores after the last; the destination offsets
// are formed again at the stores so that only the data stays live across the
// loads.
template <int W, bool NARROW>
__global__ void __launch_bounds__(LC_SHFL_THREADS, LC_SHFL_MIN_BLOCKS) k_warp_shuffle(const __grid_constant__ ShflArgs a) {
    using T = typename ShflOff<NARROW>::T;
    constexpr int V = 16 / W, G = 32 / V, U = LC_SHFL_U;
    const int lane = threadIdx.x & 31;
    const int g = lane / V, ai = lane % V;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
    constexpr uint32_t R = LC_SHFL_ROUNDS;
    for (uint32_t group = warp * (R * U * G); group < a.n_blocks; group += n_warps * (R * U * G))
#pragma unroll 1
    for (uint32_t base = group + g; base - g < a.n_blocks && base - g < group + R * U * G; base += U * G) {
        uint32_t v[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t blk = base + u * G;
            v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0;
            if (blk < a.n_blocks) {
                T so, dof;
                shfl_offsets<NARROW>(a, blk, ai, so, dof);
                const uint4 x = shfl_load(a.src + so);
                v[u][0] = x.x;
                v[u][1] = x.y;
                v[u][2] = x.z;
                v[u][3] = x.w;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) group_transpose<W>(v[u], ai);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t blk = base + u * G;
            if (blk < a.n_blocks) {
                T so, dof;
                shfl_offsets<NARROW>(a, blk, ai, so, dof);
                shfl_store(a.dst + dof, make_uint4(v[u][0], v[u][1], v[u][2], v[u][3]));
            }
        }
    }
}

template <int W>
static int launch_shuffle_w(const ShflArgs &a, bool narrow, cudaStream_t stream) {
    const void *fn = narrow ? reinterpret_cast<const void *>(&k_warp_shuffle<W, true>)
                            : reinterpret_cast<const void *>(&k_warp_shuffle<W, false>);
    int sms, per;
    if (prepare(fn, LC_SHFL_THREADS, 0, 0, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    constexpr int V = 16 / W, G = 32 / V;
    constexpr int64_t per_warp = int64_t(LC_SHFL_ROUNDS) * LC_SHFL_U * G;
    const int64_t warps_needed = (int64_t(a.n_blocks) + per_warp - 1) / per_warp;
    const int64_t blocks_needed = (warps_needed + LC_SHFL_THREADS / 32 - 1) / (LC_SHFL_THREADS / 32);
    const unsigned grid = static_cast<unsigned>(lmin(blocks_needed, int64_t(sms) * per));
    if (narrow)
        k_warp_shuffle<W, true><<<grid, LC_SHFL_THREADS, 0, stream>>>(a);
    else
        k_warp_shuffle<W, false><<<grid, LC_SHFL_THREADS, 0, stream>>>(a);
    return finish_launch();
}

int launch_shuffle(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    const ShflPlan &sp = p.shfl;
    ShflArgs a{};
    const int64_t w = p.w;
    a.src = src + p.src_off * w;
    a.dst = dst + p.dst_off * w;
    a.sa = sp.sa * w;
    a.sk = sp.sk * w;
    a.da = sp.da * w;
    a.dk = sp.dk * w;
    a.kb = static_cast<uint32_t>(sp.kb);
    a.kb_fd = make_fastdiv(a.kb);
    a.n_blocks = static_cast<uint32_t>(sp.n_blocks);
    a.nb = sp.batch.n;
    for (int i = 0; i < sp.batch.n; ++i) {
        a.be[i] = static_cast<uint32_t>(sp.batch.m[i].e);
        a.bfd[i] = make_fastdiv(a.be[i]);
        a.bs[i] = sp.batch.m[i].s * w;
        a.bd[i] = sp.batch.m[i].d * w;
    }
    // every byte offset the kernel forms is at most the span each side reaches
    const bool narrow = p.src_hi - p.src_off * w < (int64_t(1) << 32) && p.dst_hi - p.dst_off * w < (int64_t(1) << 32);
    switch (p.w) {
        case 1: return launch_shuffle_w<1>(a, narrow, stream);
        case 2: return launch_shuffle_w<2>(a, narrow, stream);
        case 4: return launch_shuffle_w<4>(a, narrow, stream);
        case 8: return launch_shuffle_w<8>(a, narrow, stream);
    }
    return LC_ERR_UNSUPPORTED;
}

}  // namespace lc
