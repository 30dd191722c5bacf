// Warp permute kernels and their launch templates, shared by the per-width
// translation units k_warp_w{1,2,4,8,16}.cu (split so that the widths
// compile in parallel).  Internal header.
// Warp register-staged permute of dense units (Apache TVM docs
// "permute_layout", section "Algorithm"), staged through shared memory with
// the [outer, threads, vec] global <-> shared copy of "copy -> gmem_smem".
//
// A unit is a dense block of U = 32 * P words on both sides.  Each warp
// stages whole units in its own shared-memory slot with 16-byte coalesced
// loads, permutes each unit in place through registers under the per-lane
// XOR swizzle chosen by the host bank simulator, and writes the slot out
// with 16-byte coalesced stores.  Nothing waits on another warp.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "launch.h"
#include "layout_copy_device.cuh"

namespace lc {

constexpr int kWarpThreads = 256;
constexpr int kWarpsPerBlock = kWarpThreads / 32;
constexpr int kWarpSlotMax = 16 * 1024;  // the planner's units are at most 16 KiB

// Warp geometry measured on GB300 on the 2^20-tile scale-factor permute:
// 8 KiB slots, 4 chunks in flight per lane and 3 resident CTAs per SM move
// 98.3 % of the copy peak; 4 KiB slots with 8 chunks per lane at 2 CTAs per
// SM reached 93.2 %, 16 chunks per lane (1 CTA per SM) 46 %, 2 KiB slots 93 %.
// Bytes of whole units staged per warp slot (at least one unit).
#ifndef LC_WARP_SLOT
#define LC_WARP_SLOT 8192
#endif
// Resident CTAs per SM the kernel is compiled for (caps registers).
#ifndef LC_WARP_MIN_BLOCKS
#define LC_WARP_MIN_BLOCKS 3
#endif

struct WarpArgs {
    const uint8_t *src;  // address of source word offset 0
    uint8_t *dst;
    lc_warp_unit unit;  // unit modes (logical order, words), P, XOR swizzle
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

#ifndef LC_WARP_CHUNKS
#define LC_WARP_CHUNKS 4
#endif
// 1: slot loads skip L1 allocation (ld.global.nc.L1::no_allocate).
#ifndef LC_WARP_LOAD_NA
#define LC_WARP_LOAD_NA 0
#endif

__device__ __forceinline__ uint4 warp_slot_load(const void *p) {
#if LC_WARP_LOAD_NA
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
#else
    return __ldg(reinterpret_cast<const uint4 *>(p));
#endif
}
constexpr int kChunksInFlight = LC_WARP_CHUNKS;  // 16-byte chunks each lane keeps in flight

// Each warp owns a private shared-memory slot of G = units_per_stage units and
// loops over groups of G consecutive units:
//   in    the group's 16-byte chunks f = lane + 32 k are loaded (all loads
//         issued before any shared store) and stored to the slot: the
//         copy -> gmem_smem split [outer, threads = 32, vec = 16 bytes];
//   P4    the two register-staged phases on every unit of the slot, in place
//         (lc_device::warp_unit_permute, the shared-buffer op of the ABI);
//   out   the slot's chunks leave with 16-byte stores to the destination.
// Only __syncwarp orders the phases; warps never wait for each other.
// CONTIG: the units are packed back to back on both sides (one batch mode of
// stride U), so a group is one contiguous byte range on each side and a chunk
// address is base + 16 f; otherwise each chunk finds its unit by division.
template <int W, int PMAX, bool CONTIG>
__global__ void __launch_bounds__(kWarpThreads, LC_WARP_MIN_BLOCKS) k_warp_permute(const __grid_constant__ WarpArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t soff[PMAX], doff[PMAX];
    lc_device::warp_unit_offsets<W, PMAX>(a.unit, lane, soff, doff);
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
                    v[k] = warp_slot_load(p);
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
            lc_device::warp_unit_permute<W, PMAX>(ub, ub, a.unit.P, soff, doff);
        }
        for (int f = lane; f < nchunks; f += 32) {
            uint8_t *p;
            if constexpr (CONTIG) {
                p = dg + 16 * f;
            } else {
                const uint32_t u = fast_div(static_cast<uint32_t>(f), a.cpu_fd);
                p = a.dst + unit_offset(a, first + u, a.bd) + 16 * (f - u * cpu);
            }
            store_out<uint4>(p, *reinterpret_cast<const uint4 *>(slot + 16 * f));
        }
        __syncwarp();
    }
}

// lc_warp_unit_run: P4's op between two shared-memory buffers.  Each unit is
// handled by one warp, which stages up to kUnitMaxPerWarp units at a time:
// it copies each unit's source buffer into shared buffer A (and the
// destination buffer into B unless in place or unless the permute writes
// every word of B, i.e. the destination image is the whole buffer), permutes
// A -> B or A -> A with
// lc_device::warp_unit_permute, and copies the destination buffer out.
constexpr int kUnitWarps = 4;

// Units staged per warp at a time: as many as fit 2 KiB of each buffer kind,
// at most 8, so that a lane keeps several 16-byte chunks in flight.
constexpr uint32_t kUnitStageBytes = 2048;
constexpr int kUnitMaxPerWarp = 8;

struct UnitArgs {
    const uint8_t *src;
    uint8_t *dst;
    lc_warp_unit unit;
    int64_t n_units;
    uint32_t sbytes, dbytes;  // bytes of one source / destination buffer
    uint32_t buf;             // shared bytes per buffer (16-byte multiple)
    int32_t in_place;
    int32_t dst_dense;        // the permute writes every word of B: B is not read in
    int32_t upw;              // units staged per warp at a time
    int32_t chunked;          // sbytes and dbytes are 16-byte multiples
    FastDiv schunks, dchunks;  // 16-byte chunks per source / destination buffer
};

// Byte copy by one warp: 16-byte words when both ends and the size allow.
__device__ __forceinline__ void warp_copy(uint8_t *d, const uint8_t *s, uint32_t n, int lane) {
    if (((reinterpret_cast<uintptr_t>(d) | reinterpret_cast<uintptr_t>(s) | n) & 15) == 0) {
        for (uint32_t f = lane; f < n / 16; f += 32)
            reinterpret_cast<uint4 *>(d)[f] = reinterpret_cast<const uint4 *>(s)[f];
    } else {
        for (uint32_t f = lane; f < n; f += 32) d[f] = s[f];
    }
}

// Buffers of `cnt` units, `bytes` each back to back in global memory, into
// (to_shared) or out of their shared buffers, unit u's at slot + u * pitch:
// 16-byte chunks, kChunksInFlight per lane loaded before any is stored.
template <bool TO_SHARED>
__device__ __forceinline__ void unit_chunks(uint8_t *slot, uint32_t pitch, uint8_t *g, uint32_t bytes,
                                            const FastDiv &per, int cnt, int lane) {
    const int n = cnt * static_cast<int>(bytes / 16);
    for (int base = 0; base < n; base += 32 * kChunksInFlight) {
        uint4 v[kChunksInFlight];
        uint8_t *to[kChunksInFlight];
#pragma unroll
        for (int k = 0; k < kChunksInFlight; ++k) {
            const int f = base + lane + 32 * k;
            to[k] = nullptr;
            if (f < n) {
                const uint32_t u = fast_div(static_cast<uint32_t>(f), per);
                uint8_t *sh = slot + u * pitch + 16 * (f - u * per.d);
                uint8_t *gl = g + 16 * static_cast<int64_t>(f);
                v[k] = *reinterpret_cast<const uint4 *>(TO_SHARED ? gl : sh);
                to[k] = TO_SHARED ? sh : gl;
            }
        }
#pragma unroll
        for (int k = 0; k < kChunksInFlight; ++k)
            if (to[k]) *reinterpret_cast<uint4 *>(to[k]) = v[k];
    }
}

template <int W, int PMAX>
__global__ void __launch_bounds__(kUnitWarps * 32) k_warp_unit_shared(const __grid_constant__ UnitArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // unit u of this warp's stage: A = slot + u * 2 buf, B = A + buf
    uint8_t *const slot = smem + static_cast<size_t>(warp) * a.upw * 2 * a.buf;
    const uint32_t pitch = 2 * a.buf;
    int32_t soff[PMAX], doff[PMAX];
    lc_device::warp_unit_offsets<W, PMAX>(a.unit, lane, soff, doff);
    const int64_t n_groups = (a.n_units + a.upw - 1) / a.upw;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * kUnitWarps + warp; g < n_groups;
         g += static_cast<int64_t>(gridDim.x) * kUnitWarps) {
        const int64_t first = g * a.upw;
        const int cnt = static_cast<int>(lmin(a.upw, a.n_units - first));
        uint8_t *const sg = const_cast<uint8_t *>(a.src) + first * a.sbytes;
        uint8_t *const dg = a.dst + first * a.dbytes;
        if (a.chunked) {
            unit_chunks<true>(slot, pitch, sg, a.sbytes, a.schunks, cnt, lane);
            if (!a.in_place && !a.dst_dense)
                unit_chunks<true>(slot + a.buf, pitch, dg, a.dbytes, a.dchunks, cnt, lane);
        } else {
            for (int u = 0; u < cnt; ++u) {
                warp_copy(slot + u * pitch, sg + static_cast<int64_t>(u) * a.sbytes, a.sbytes, lane);
                if (!a.in_place && !a.dst_dense)
                    warp_copy(slot + u * pitch + a.buf, dg + static_cast<int64_t>(u) * a.dbytes, a.dbytes, lane);
            }
        }
        __syncwarp();
        const uint32_t out = a.in_place ? 0 : a.buf;  // offset of the permuted buffer in a unit's slot
        for (int u = 0; u < cnt; ++u)
            lc_device::warp_unit_permute<W, PMAX>(slot + u * pitch + out, slot + u * pitch, a.unit.P, soff, doff);
        if (a.chunked) {
            unit_chunks<false>(slot + out, pitch, dg, a.dbytes, a.dchunks, cnt, lane);
        } else {
            for (int u = 0; u < cnt; ++u)
                warp_copy(dg + static_cast<int64_t>(u) * a.dbytes, slot + u * pitch + out, a.dbytes, lane);
        }
        __syncwarp();
    }
}

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

template <int W, int PMAX>
int launch_unit_t(const UnitArgs &a, cudaStream_t stream) {
    const void *fn = reinterpret_cast<const void *>(&k_warp_unit_shared<W, PMAX>);
    const int smem = kUnitWarps * a.upw * 2 * static_cast<int>(a.buf);
    int sms, per;
    if (prepare(fn, kUnitWarps * 32, smem, kUnitWarps * 2 * LC_WARP_UNIT_MAX_BYTES, &sms, &per) != cudaSuccess)
        return LC_ERR_CUDA;
    const int64_t groups = (a.n_units + a.upw - 1) / a.upw;
    const int64_t grid = lmin((groups + kUnitWarps - 1) / kUnitWarps, int64_t(sms) * std::max(per, 1));
    k_warp_unit_shared<W, PMAX><<<static_cast<unsigned>(grid), kUnitWarps * 32, smem, stream>>>(a);
    return finish_launch();
}

template <int W>
int launch_unit_w(const UnitArgs &a, cudaStream_t s) {
    if (a.unit.P <= 4) return launch_unit_t<W, 4>(a, s);
    if (a.unit.P <= 8) return launch_unit_t<W, 8>(a, s);
    return launch_unit_t<W, 32>(a, s);
}

template <int W>
int launch_warp_w(int P, const WarpArgs &a, cudaStream_t s) {
    if (P <= 4) return launch_warp_t<W, 4>(a, s);
    if (P <= 8) return launch_warp_t<W, 8>(a, s);
    return launch_warp_t<W, 32>(a, s);
}

// Per-width launchers, one translation unit each.
#define LC_WARP_WIDTH_LAUNCHERS(W)                                                  \
    int launch_warp_width##W(int P, const WarpArgs &a, cudaStream_t s);           \
    int launch_unit_width##W(const UnitArgs &a, cudaStream_t s);
LC_WARP_WIDTH_LAUNCHERS(1)
LC_WARP_WIDTH_LAUNCHERS(2)
LC_WARP_WIDTH_LAUNCHERS(4)
LC_WARP_WIDTH_LAUNCHERS(8)
LC_WARP_WIDTH_LAUNCHERS(16)

}  // namespace lc
