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

#include "bulk_store.cuh"
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
// The same for the nested form of units past 8 words a lane.
#ifndef LC_WARP_MIN_BLOCKS_NESTED
#define LC_WARP_MIN_BLOCKS_NESTED 3
#endif
// 8-byte words in the nested form: 32 words a lane are 64 registers of words
// alone.  Measured on a batch of 32 x 32 of them (8 KiB units, no bulk
// prefetch): 2 CTAs per SM with 8 chunks a lane in flight 76.6 % of the copy
// peak, against 61.7 % at 3 CTAs and 4 chunks and 70.9 % at 2 CTAs and 4.
#ifndef LC_WARP_MIN_BLOCKS_W8_NESTED
#define LC_WARP_MIN_BLOCKS_W8_NESTED 2
#endif
#ifndef LC_WARP_CHUNKS_W8_NESTED
#define LC_WARP_CHUNKS_W8_NESTED 8
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
    int32_t nested;           // 32 lies on the unit's suffix-product chain
    int32_t async;            // contiguous units, two slots a warp filled by bulk copies
    int64_t n_units, units_per_stage;
    uint32_t stage_bytes;  // one warp slot
    uint64_t timeout_ns;   // limit of each bounded barrier wait
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
// 1: contiguous units of more than 8 words a lane and at most
// LC_WARP_ASYNC_SLOT bytes take k_warp_permute_async (two slots a warp of
// LC_WARP_ASYNC_SLOT bytes).
#ifndef LC_WARP_ASYNC
#define LC_WARP_ASYNC 1
#endif
#ifndef LC_WARP_ASYNC_SLOT
#define LC_WARP_ASYNC_SLOT 4096
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

// The unit's offsets when 32 lies on the divisibility chain of its suffix
// products: the logical index lane + 32 j splits into disjoint lane digits
// and j digits, so the offset of step r on either side is this lane's own
// part plus the j part of j = r ^ sw, which lane j holds.  These are the
// offsets lc_device::warp_unit_offsets stores, 2 P registers a lane; here
// they are formed where each is used, from four registers and a shuffle, so
// that P = 32 (a 32 x 32 tile of words per unit) fits without spilling.
struct NestedLane {
    int32_t ls, ld;  // this lane's digits: offsets of index `lane`
    int32_t js, jd;  // offsets of index 32 * lane (read by other lanes as the j part)
    int32_t sw;      // the lane's XOR swizzle (lane >> shift) & mask
};

__device__ __forceinline__ NestedLane nested_lane(const lc_warp_unit &u, int lane) {
    NestedLane l;
    lc_device::unit_point(u, lane, l.ls, l.ld);
    lc_device::unit_point(u, lane < u.P ? 32 * lane : 0, l.js, l.jd);
    l.sw = (lane >> u.shift) & u.mask;
    return l;
}

// The two register-staged phases of lc_device::warp_unit_permute on one
// unit (the same words in the same order), offsets taken from NestedLane.
template <int W, int PMAX>
__device__ __forceinline__ void unit_permute_nested(uint8_t *d, const uint8_t *s, int P, const NestedLane &l) {
    using T = typename lc_device::unit_word<W>::type;
    T regs[PMAX];
#pragma unroll
    for (int r = 0; r < PMAX; ++r) {
        if (r < P) {  // P is the same on every lane: the shuffle sees the whole warp
            const int32_t js = __shfl_sync(0xffffffffu, l.js, (r ^ l.sw) & 31);
            regs[r] = *reinterpret_cast<const T *>(s + (l.ls + js) * W);
        }
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < PMAX; ++r) {
        if (r < P) {
            const int32_t jd = __shfl_sync(0xffffffffu, l.jd, (r ^ l.sw) & 31);
            *reinterpret_cast<T *>(d + (l.ld + jd) * W) = regs[r];
        }
    }
    __syncwarp();
}

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
// NESTED: the unit's offsets come from NestedLane (32 on its suffix chain).
template <int W, int PMAX, bool CONTIG, bool NESTED>
__global__ void __launch_bounds__(kWarpThreads, !NESTED ? LC_WARP_MIN_BLOCKS
                                                : W == 8 ? LC_WARP_MIN_BLOCKS_W8_NESTED
                                                         : LC_WARP_MIN_BLOCKS_NESTED)
    k_warp_permute(const __grid_constant__ WarpArgs a) {
    constexpr int CH = NESTED && W == 8 ? LC_WARP_CHUNKS_W8_NESTED : kChunksInFlight;  // chunks a lane in flight
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NOFF = NESTED ? 1 : PMAX;
    int32_t soff[NOFF], doff[NOFF];
    NestedLane nl{};
    if constexpr (NESTED)
        nl = nested_lane(a.unit, lane);
    else
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
        for (int base = 0; base < nchunks; base += 32 * CH) {
            uint4 v[CH];
#pragma unroll
            for (int k = 0; k < CH; ++k) {
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
            for (int k = 0; k < CH; ++k) {
                const int f = base + lane + 32 * k;
                if (f < nchunks) *reinterpret_cast<uint4 *>(slot + 16 * f) = v[k];
            }
        }
        __syncwarp();
        for (int u = 0; u < cnt; ++u) {
            uint8_t *ub = slot + static_cast<size_t>(u) * a.unit_bytes;
            if constexpr (NESTED)
                unit_permute_nested<W, PMAX>(ub, ub, a.unit.P, nl);
            else
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

// One-dimensional bulk copy global -> shared (no tensor map, PTX ISA
// cp.async.bulk): `bytes` (a multiple of 16) from a 16-byte aligned global
// address into this CTA's shared memory, completing `bytes` of transaction
// count on the mbarrier at `bar`.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst_smem, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst_smem), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// The permute of contiguous units with each warp's loads running one group
// ahead: a warp owns two slots; while it permutes and stores group g from
// one, a one-dimensional bulk copy (issued by lane 0, completing on that
// slot's mbarrier) fills the other with group g + (warps in the grid).  The
// loaded bytes travel without registers, so a lane's load latency hides
// behind its own permute and stores instead of only behind other warps.
// A slot is refilled once the warp's stores from it have read it (its
// __syncwarp); a proxy fence orders those generic accesses before the copy.
// Every wait is bounded: on a timeout the kernel records LC_ERR_TIMEOUT,
// waits (bounded) for the copies it started and returns.
// Shared layout: 8 bytes of mbarrier per slot (16 per warp, 128 bytes), then
// the slots, 2 per warp, stage_bytes each.
template <int W, int PMAX, bool NESTED>
__global__ void __launch_bounds__(kWarpThreads, NESTED ? LC_WARP_MIN_BLOCKS_NESTED : LC_WARP_MIN_BLOCKS)
    k_warp_permute_async(const __grid_constant__ WarpArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NOFF = NESTED ? 1 : PMAX;
    int32_t soff[NOFF], doff[NOFF];
    NestedLane nl{};
    if constexpr (NESTED)
        nl = nested_lane(a.unit, lane);
    else
        lc_device::warp_unit_offsets<W, PMAX>(a.unit, lane, soff, doff);
    const uint32_t bar = ptx::smem_addr(smem) + 16u * static_cast<uint32_t>(warp);  // slot b's at bar + 8 b
    uint8_t *const slots = smem + 128 + static_cast<size_t>(warp) * 2 * a.stage_bytes;
    const int64_t n_groups = (a.n_units + a.units_per_stage - 1) / a.units_per_stage;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
    if (g0 >= n_groups) return;
    if (lane == 0) {
        ptx::mbar_init(bar, 1);
        ptx::mbar_init(bar + 8, 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();
    auto group_bytes = [&](int64_t g) {
        return static_cast<uint32_t>(lmin(a.units_per_stage, a.n_units - g * a.units_per_stage) * a.unit_bytes);
    };
    auto issue = [&](int64_t g, int b) {  // lane 0 only
        const uint32_t bytes = group_bytes(g);
        ptx::mbar_arrive_expect_tx(bar + 8 * b, bytes);
        bulk_load_1d(ptx::smem_addr(slots + static_cast<size_t>(b) * a.stage_bytes),
                          a.src + g * a.units_per_stage * a.unit_bytes, bytes, bar + 8 * b);
    };
    if (lane == 0) issue(g0, 0);
    int i = 0;
    for (int64_t g = g0; g < n_groups; g += warps, ++i) {
        const int b = i & 1;
        const int64_t gn = g + warps;
        if (lane == 0 && gn < n_groups) {
            bulk::fence_proxy_async_smem();
            issue(gn, b ^ 1);
        }
        const uint32_t parity = static_cast<uint32_t>(i >> 1) & 1u;  // slot b's (i >> 1)-th fill
        const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(bar + 8 * b, parity, a.timeout_ns));
        if (!ok) {
            if (lane == 0) {
                report_error(LC_ERR_TIMEOUT, LC_KERNEL_WARP_PERMUTE);
                ptx::mbar_wait_bounded(bar + 8 * b, parity, a.timeout_ns);
                if (gn < n_groups)  // the copy into the other slot, started above
                    ptx::mbar_wait_bounded(bar + 8 * (b ^ 1), static_cast<uint32_t>((i + 1) >> 1) & 1u,
                                           a.timeout_ns);
            }
            __syncwarp();
            return;
        }
        uint8_t *const slot = slots + static_cast<size_t>(b) * a.stage_bytes;
        const int cnt = static_cast<int>(group_bytes(g) / a.unit_bytes);
        for (int u = 0; u < cnt; ++u) {
            uint8_t *ub = slot + static_cast<size_t>(u) * a.unit_bytes;
            if constexpr (NESTED)
                unit_permute_nested<W, PMAX>(ub, ub, a.unit.P, nl);
            else
                lc_device::warp_unit_permute<W, PMAX>(ub, ub, a.unit.P, soff, doff);
        }
        uint8_t *const dg = a.dst + g * a.units_per_stage * a.unit_bytes;
        const int nchunks = static_cast<int>(group_bytes(g) / 16);
        for (int f = lane; f < nchunks; f += 32)
            store_out<uint4>(dg + 16 * f, *reinterpret_cast<const uint4 *>(slot + 16 * f));
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

template <int W, int PMAX, bool NESTED>
int launch_warp_t(const WarpArgs &a, cudaStream_t stream) {
    if constexpr (PMAX > 8) {
        if (a.async) {
            const void *fn = reinterpret_cast<const void *>(&k_warp_permute_async<W, PMAX, NESTED>);
            const int smem = 128 + 2 * kWarpsPerBlock * static_cast<int>(a.stage_bytes);
            int sms, per;
            if (prepare(fn, kWarpThreads, smem, 128 + kWarpsPerBlock * kWarpSlotMax, &sms, &per) != cudaSuccess)
                return LC_ERR_CUDA;
            const int64_t groups = (a.n_units + a.units_per_stage - 1) / a.units_per_stage;
            const int64_t grid = lmin((groups + kWarpsPerBlock - 1) / kWarpsPerBlock, int64_t(sms) * per);
            k_warp_permute_async<W, PMAX, NESTED><<<static_cast<unsigned>(grid), kWarpThreads, smem, stream>>>(a);
            return finish_launch();
        }
    }  // the async instances exist only for PMAX = 32
    const void *fn = a.contig ? reinterpret_cast<const void *>(&k_warp_permute<W, PMAX, true, NESTED>)
                              : reinterpret_cast<const void *>(&k_warp_permute<W, PMAX, false, NESTED>);
    const int smem = kWarpsPerBlock * static_cast<int>(a.stage_bytes);
    int sms, per;
    if (prepare(fn, kWarpThreads, smem, kWarpsPerBlock * kWarpSlotMax, &sms, &per) != cudaSuccess)
        return LC_ERR_CUDA;
    const int64_t groups = (a.n_units + a.units_per_stage - 1) / a.units_per_stage;
    const int64_t grid = lmin((groups + kWarpsPerBlock - 1) / kWarpsPerBlock, int64_t(sms) * per);
    if (a.contig)
        k_warp_permute<W, PMAX, true, NESTED><<<static_cast<unsigned>(grid), kWarpThreads, smem, stream>>>(a);
    else
        k_warp_permute<W, PMAX, false, NESTED><<<static_cast<unsigned>(grid), kWarpThreads, smem, stream>>>(a);
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

// Up to P = 8 the stored offsets fit in registers (no spills at 3 CTAs per
// SM); past it they spilled (972 bytes of local loads a thread at P = 32),
// so nesting units form them as they go.
template <int W>
int launch_warp_w(int P, const WarpArgs &a, cudaStream_t s) {
    if (P <= 4) return launch_warp_t<W, 4, false>(a, s);
    if (P <= 8) return launch_warp_t<W, 8, false>(a, s);
    if (a.nested) return launch_warp_t<W, 32, true>(a, s);
    return launch_warp_t<W, 32, false>(a, s);
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
