// Warp register-staged permute of dense units (Apache TVM docs
// "permute_layout", section "Algorithm"), staged through shared memory with
// the [outer, threads, vec] global <-> shared copy of "copy -> gmem_smem".
//
// A unit is a dense block of U = 32 * P words on both sides.  Each warp
// stages whole units in its own shared-memory slot with 16-byte coalesced
// loads, permutes each unit in place through registers under the per-lane
// XOR swizzle chosen by the host bank simulator, and writes the slot out
// with 16-byte coalesced stores.  Nothing waits on another warp.
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

constexpr int kWarpThreads = 256;
constexpr int kWarpsPerBlock = kWarpThreads / 32;
constexpr int kWarpSlotMax = 16 * 1024;  // the planner's units are at most 16 KiB

// Bytes of whole units staged per warp slot (at least one unit).
#ifndef LC_WARP_SLOT
#define LC_WARP_SLOT 4096
#endif
// Resident CTAs per SM the kernel is compiled for (caps registers).
#ifndef LC_WARP_MIN_BLOCKS
#define LC_WARP_MIN_BLOCKS 1
#endif

struct WarpArgs {
    const uint8_t *src;  // address of source word offset 0
    uint8_t *dst;
    int32_t un;  // unit modes, logical order (words)
    int32_t ue[kMaxModes], us[kMaxModes], ud[kMaxModes];
    int32_t P, shift, mask;
    uint32_t unit_bytes;
    int32_t nb;  // batch modes (BYTES strides), outermost first
    int64_t be[kMaxModes], bs[kMaxModes], bd[kMaxModes];
    FastDiv bfd[kMaxModes];  // batch extents, for 32-bit unit indices
    int32_t narrow;           // n_units < 2^32: unit indices use FastDiv
    FastDiv cpu_fd;           // 16-byte chunks per unit
    int32_t contig;           // units packed back to back on both sides
    int64_t n_units, units_per_stage;
    uint32_t stage_bytes;  // one warp slot
};

// Byte offsets of flat unit index u (row-major over the batch modes) on the
// source (str = bs) or destination (str = bd) side.
__device__ __forceinline__ int64_t unit_offset(const WarpArgs &a, int64_t u, const int64_t *str) {
    int64_t off = 0;
    if (a.narrow) {
        uint32_t q = static_cast<uint32_t>(u);
        for (int i = a.nb - 1; i >= 0; --i) {
            const uint32_t q2 = fast_div(q, a.bfd[i]);
            off += static_cast<int64_t>(q - q2 * a.bfd[i].d) * str[i];
            q = q2;
        }
    } else {
        for (int i = a.nb - 1; i >= 0; --i) {
            off += (u % a.be[i]) * str[i];
            u /= a.be[i];
        }
    }
    return off;
}

constexpr int kChunksInFlight = 8;  // 16-byte chunks each lane keeps in flight

// Per-lane byte offsets, inside one unit, of the P words lane `lane` stages:
// step r holds iteration j = r ^ ((lane >> shift) & mask), i.e. the logical
// index unflatten(lane + 32 j) over the unit's extents (last mode fastest).
template <int W, int PMAX>
__device__ __forceinline__ void lane_offsets(const WarpArgs &a, int lane, int32_t (&soff)[PMAX],
                                             int32_t (&doff)[PMAX]) {
#pragma unroll
    for (int r = 0; r < PMAX; ++r) {
        int32_t flat = lane + 32 * (r ^ ((lane >> a.shift) & a.mask)), so = 0, dof = 0;
        for (int i = a.un - 1; i >= 0; --i) {
            const int32_t c = flat % a.ue[i];
            flat /= a.ue[i];
            so += c * a.us[i];
            dof += c * a.ud[i];
        }
        soff[r] = so * W;
        doff[r] = dof * W;
    }
}

// Each warp owns a private shared-memory slot of G = units_per_stage units and
// loops over groups of G consecutive units:
//   in    the group's 16-byte chunks f = lane + 32 k are loaded (all loads
//         issued before any shared store) and stored to the slot: the
//         copy -> gmem_smem split [outer, threads = 32, vec = 16 bytes];
//   P4    the two register-staged phases on every unit of the slot, in place;
//   out   the slot's chunks leave with 16-byte stores to the destination.
// Only __syncwarp orders the phases; warps never wait for each other.
// CONTIG: the units are packed back to back on both sides (one batch mode of
// stride U), so a group is one contiguous byte range on each side and a chunk
// address is base + 16 f; otherwise each chunk finds its unit by division.
template <int W, int PMAX, bool CONTIG>
__global__ void __launch_bounds__(kWarpThreads, LC_WARP_MIN_BLOCKS) k_warp_permute(const __grid_constant__ WarpArgs a) {
    using T = typename Word<W>::T;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t soff[PMAX], doff[PMAX];
    lane_offsets<W, PMAX>(a, lane, soff, doff);
    uint8_t *slot = smem + static_cast<size_t>(warp) * a.stage_bytes;
    const uint32_t cpu = a.unit_bytes / 16;  // chunks per unit
    const int64_t n_groups = (a.n_units + a.units_per_stage - 1) / a.units_per_stage;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp; g < n_groups; g += warps) {
        const int64_t first = g * a.units_per_stage;
        const int cnt = static_cast<int>(lmin(a.units_per_stage, a.n_units - first));
        const int nchunks = cnt * static_cast<int>(cpu);
        const uint8_t *sg = a.src + first * a.unit_bytes;
        uint8_t *dg = a.dst + first * a.unit_bytes;
        for (int base = 0; base < nchunks; base += 32 * kChunksInFlight) {
            uint4 v[kChunksInFlight];
#pragma unroll
            for (int k = 0; k < kChunksInFlight; ++k) {
                const int f = base + lane + 32 * k;
                if (f < nchunks) {
                    const uint8_t *p;
                    if constexpr (CONTIG) {
                        p = sg + 16 * f;
                    } else {
                        const uint32_t u = fast_div(static_cast<uint32_t>(f), a.cpu_fd);
                        p = a.src + unit_offset(a, first + u, a.bs) + 16 * (f - u * cpu);
                    }
                    v[k] = __ldg(reinterpret_cast<const uint4 *>(p));
                }
            }
#pragma unroll
            for (int k = 0; k < kChunksInFlight; ++k) {
                const int f = base + lane + 32 * k;
                if (f < nchunks) *reinterpret_cast<uint4 *>(slot + 16 * f) = v[k];
            }
        }
        __syncwarp();
        for (int u = 0; u < cnt; ++u) {
            uint8_t *ub = slot + static_cast<size_t>(u) * a.unit_bytes;
            T regs[PMAX];
#pragma unroll
            for (int r = 0; r < PMAX; ++r)
                if (r < a.P) regs[r] = *reinterpret_cast<const T *>(ub + soff[r]);
            __syncwarp();
#pragma unroll
            for (int r = 0; r < PMAX; ++r)
                if (r < a.P) *reinterpret_cast<T *>(ub + doff[r]) = regs[r];
            __syncwarp();
        }
        for (int f = lane; f < nchunks; f += 32) {
            uint8_t *p;
            if constexpr (CONTIG) {
                p = dg + 16 * f;
            } else {
                const uint32_t u = fast_div(static_cast<uint32_t>(f), a.cpu_fd);
                p = a.dst + unit_offset(a, first + u, a.bd) + 16 * (f - u * cpu);
            }
            *reinterpret_cast<uint4 *>(p) = *reinterpret_cast<const uint4 *>(slot + 16 * f);
        }
        __syncwarp();
    }
}

namespace {

template <int W, int PMAX>
int launch_warp_t(const WarpArgs &a, cudaStream_t stream) {
    const void *fn = a.contig ? reinterpret_cast<const void *>(&k_warp_permute<W, PMAX, true>)
                              : reinterpret_cast<const void *>(&k_warp_permute<W, PMAX, false>);
    const int smem = kWarpsPerBlock * static_cast<int>(a.stage_bytes);
    int sms, per;
    if (prepare(fn, kWarpThreads, smem, kWarpsPerBlock * kWarpSlotMax, &sms, &per) != cudaSuccess)
        return LC_ERR_CUDA;
    const int64_t groups = (a.n_units + a.units_per_stage - 1) / a.units_per_stage;
    const int64_t grid = lmin((groups + kWarpsPerBlock - 1) / kWarpsPerBlock, int64_t(sms) * per);
    if (a.contig)
        k_warp_permute<W, PMAX, true><<<static_cast<unsigned>(grid), kWarpThreads, smem, stream>>>(a);
    else
        k_warp_permute<W, PMAX, false><<<static_cast<unsigned>(grid), kWarpThreads, smem, stream>>>(a);
    return finish_launch();
}

template <int W>
int launch_warp_w(int P, const WarpArgs &a, cudaStream_t s) {
    if (P <= 4) return launch_warp_t<W, 4>(a, s);
    if (P <= 8) return launch_warp_t<W, 8>(a, s);
    return launch_warp_t<W, 32>(a, s);
}

}  // namespace

int launch_warp(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    const WarpPlan &wp = p.warp;
    WarpArgs a{};
    a.src = src + p.src_off * p.w;
    a.dst = dst + p.dst_off * p.w;
    a.un = wp.unit.n;
    for (int i = 0; i < wp.unit.n; ++i) {
        a.ue[i] = static_cast<int32_t>(wp.unit.m[i].e);
        a.us[i] = static_cast<int32_t>(wp.unit.m[i].s);
        a.ud[i] = static_cast<int32_t>(wp.unit.m[i].d);
    }
    a.P = wp.P;
    a.shift = wp.shift;
    a.mask = wp.mask;
    a.unit_bytes = static_cast<uint32_t>(wp.U * p.w);
    a.nb = wp.batch.n;
    for (int i = 0; i < wp.batch.n; ++i) {
        a.be[i] = wp.batch.m[i].e;
        a.bs[i] = wp.batch.m[i].s * p.w;
        a.bd[i] = wp.batch.m[i].d * p.w;
    }
    a.narrow = wp.n_units < (int64_t(1) << 32);
    a.cpu_fd = make_fastdiv(a.unit_bytes / 16);
    a.contig = wp.batch.n == 0 ||
               (wp.batch.n == 1 && a.bs[0] == int64_t(a.unit_bytes) && a.bd[0] == int64_t(a.unit_bytes));
    if (a.narrow)
        for (int i = 0; i < wp.batch.n; ++i) a.bfd[i] = make_fastdiv(static_cast<uint32_t>(wp.batch.m[i].e));
    a.n_units = wp.n_units;
    a.units_per_stage = lmin(wp.n_units, std::max<int64_t>(1, LC_WARP_SLOT / (wp.U * p.w)));
    a.stage_bytes = static_cast<uint32_t>((a.units_per_stage * a.unit_bytes + 127) / 128 * 128);
    if (a.stage_bytes > static_cast<uint32_t>(kWarpSlotMax)) return LC_ERR_UNSUPPORTED;
    switch (p.w) {
        case 1: return launch_warp_w<1>(wp.P, a, stream);
        case 2: return launch_warp_w<2>(wp.P, a, stream);
        case 4: return launch_warp_w<4>(wp.P, a, stream);
        case 8: return launch_warp_w<8>(wp.P, a, stream);
        case 16: return launch_warp_w<16>(wp.P, a, stream);
    }
    return LC_ERR_UNSUPPORTED;
}

}  // namespace lc
