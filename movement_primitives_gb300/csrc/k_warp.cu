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
#include "layout_copy_device.cuh"

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

constexpr int kChunksInFlight = 8;  // 16-byte chunks each lane keeps in flight

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
            *reinterpret_cast<uint4 *>(p) = *reinterpret_cast<const uint4 *>(slot + 16 * f);
        }
        __syncwarp();
    }
}

// lc_warp_unit_run: P4's op between two shared-memory buffers, one warp per
// unit.  The warp copies the unit's source buffer into shared buffer A (and
// the destination buffer into B unless in place), permutes A -> B or A -> A
// with lc_device::warp_unit_permute, and copies the destination buffer out.
constexpr int kUnitWarps = 4;

struct UnitArgs {
    const uint8_t *src;
    uint8_t *dst;
    lc_warp_unit unit;
    int64_t n_units;
    uint32_t sbytes, dbytes;  // bytes of one source / destination buffer
    uint32_t buf;             // shared bytes per buffer (16-byte multiple)
    int32_t in_place;
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

template <int W, int PMAX>
__global__ void __launch_bounds__(kUnitWarps * 32) k_warp_unit_shared(const __grid_constant__ UnitArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *A = smem + static_cast<size_t>(warp) * 2 * a.buf;
    uint8_t *B = A + a.buf;
    int32_t soff[PMAX], doff[PMAX];
    lc_device::warp_unit_offsets<W, PMAX>(a.unit, lane, soff, doff);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kUnitWarps + warp; i < a.n_units;
         i += static_cast<int64_t>(gridDim.x) * kUnitWarps) {
        warp_copy(A, a.src + i * a.sbytes, a.sbytes, lane);
        if (!a.in_place) warp_copy(B, a.dst + i * a.dbytes, a.dbytes, lane);
        __syncwarp();
        uint8_t *out = a.in_place ? A : B;
        lc_device::warp_unit_permute<W, PMAX>(out, A, a.unit.P, soff, doff);
        warp_copy(a.dst + i * a.dbytes, out, a.dbytes, lane);
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

template <int W, int PMAX>
int launch_unit_t(const UnitArgs &a, cudaStream_t stream) {
    const void *fn = reinterpret_cast<const void *>(&k_warp_unit_shared<W, PMAX>);
    const int smem = kUnitWarps * 2 * static_cast<int>(a.buf);
    int sms, per;
    if (prepare(fn, kUnitWarps * 32, smem, kUnitWarps * 2 * LC_WARP_UNIT_MAX_BYTES, &sms, &per) != cudaSuccess)
        return LC_ERR_CUDA;
    const int64_t grid = lmin((a.n_units + kUnitWarps - 1) / kUnitWarps, int64_t(sms) * std::max(per, 1));
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

}  // namespace

int launch_warp(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    const WarpPlan &wp = p.warp;
    WarpArgs a{};
    a.src = src + p.src_off * p.w;
    a.dst = dst + p.dst_off * p.w;
    if (wp.unit.n > LC_MAX_RANK) return LC_ERR_UNSUPPORTED;  // the planner keeps it below
    a.unit.n_modes = wp.unit.n;
    for (int i = 0; i < wp.unit.n; ++i) {
        a.unit.extent[i] = static_cast<int32_t>(wp.unit.m[i].e);
        a.unit.src_stride[i] = static_cast<int32_t>(wp.unit.m[i].s);
        a.unit.dst_stride[i] = static_cast<int32_t>(wp.unit.m[i].d);
    }
    a.unit.P = wp.P;
    a.unit.k = wp.k;
    a.unit.shift = wp.shift;
    a.unit.mask = wp.mask;
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

// A caller-supplied plan is checked in full, so that every offset the kernel
// forms stays inside its buffer: extents and strides consistent with P and
// the cosizes, and the XOR keeping j below P.
static bool unit_is_consistent(const lc_warp_unit &u) {
    if (u.n_modes < 1 || u.n_modes > LC_MAX_RANK || u.P < 1 || u.P > LC_WARP_UNIT_MAX_P) return false;
    int64_t total = 1, scos = 1, dcos = 1;
    for (int i = 0; i < u.n_modes; ++i) {
        if (u.extent[i] < 1 || u.src_stride[i] < 0 || u.dst_stride[i] < 0) return false;
        total *= u.extent[i];
        scos += int64_t(u.extent[i] - 1) * u.src_stride[i];
        dcos += int64_t(u.extent[i] - 1) * u.dst_stride[i];
    }
    if (total != int64_t(32) * u.P || scos != u.src_cosize || dcos != u.dst_cosize) return false;
    if (u.k < 0 || u.k > 5 || u.mask != (1 << u.k) - 1 || u.shift < 0 || u.shift > 31) return false;
    if (u.mask >= u.P || (u.mask && (u.P & (u.P - 1)))) return false;  // j = r ^ (.. & mask) < P
    return true;
}

extern "C" int lc_warp_unit_run(const void *src, void *dst, const lc_warp_unit *unit, int32_t elem_bytes,
                                int64_t n_units, int32_t in_place, lc_stream_t stream) {
    using namespace lc;
    if (!unit) return LC_ERR_NULL;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8 && elem_bytes != 16)
        return LC_ERR_ELEM_BYTES;
    if (n_units < 0 || !unit_is_consistent(*unit)) return LC_ERR_SHAPE;
    if (n_units == 0) return LC_OK;
    if (!src || !dst) return LC_ERR_NULL;
    const int64_t sb = int64_t(unit->src_cosize) * elem_bytes, db = int64_t(unit->dst_cosize) * elem_bytes;
    if (sb > LC_WARP_UNIT_MAX_BYTES || db > LC_WARP_UNIT_MAX_BYTES) return LC_ERR_SHAPE;
    if (in_place && unit->src_cosize < unit->dst_cosize) return LC_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16) return LC_ERR_ALIGN;
    if (n_units > (int64_t(1) << 62) / std::max(sb, db)) return LC_ERR_OVERFLOW;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), s1 = s0 + uintptr_t(n_units * sb);
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst), d1 = d0 + uintptr_t(n_units * db);
    if (s0 < d1 && d0 < s1) return LC_ERR_OVERLAP;
    UnitArgs a{};
    a.src = static_cast<const uint8_t *>(src);
    a.dst = static_cast<uint8_t *>(dst);
    a.unit = *unit;
    a.n_units = n_units;
    a.sbytes = static_cast<uint32_t>(sb);
    a.dbytes = static_cast<uint32_t>(db);
    a.buf = static_cast<uint32_t>((std::max(sb, db) + 15) / 16 * 16);
    a.in_place = in_place ? 1 : 0;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    switch (elem_bytes) {
        case 1: return launch_unit_w<1>(a, cs);
        case 2: return launch_unit_w<2>(a, cs);
        case 4: return launch_unit_w<4>(a, cs);
        case 8: return launch_unit_w<8>(a, cs);
        default: return launch_unit_w<16>(a, cs);
    }
}
