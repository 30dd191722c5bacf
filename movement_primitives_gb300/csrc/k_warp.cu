// Warp register-staged permute of bulk-copied units (Apache TVM docs
// "permute_layout", section "Algorithm").
//
// A unit is a dense block of U = 32 * P words on both sides.  Units are
// bulk-copied global -> shared (several per stage, contiguous ones merged into
// one copy), each warp permutes one unit in place through registers with the
// per-lane XOR swizzle chosen by the host bank simulator, then writes the
// unit out with 16-byte coalesced stores.
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

constexpr int kWarpThreads = 256;
constexpr int kWarpStages = 4;
constexpr int kWarpStageMax = 16 * 1024;  // the planner stages at most 16 KiB of units
constexpr int kWarpMaxSmem = 128 + kWarpStages * kWarpStageMax;

// 1: every copy of the warp permute on the load/store units (no TMA);
// 0: TMA bulk loads into a CTA-wide shared-memory ring.
#ifndef LC_WARP_LSU
#define LC_WARP_LSU 1
#endif
// Units staged per warp slot (LSU) or per ring stage (TMA), in bytes.
#ifndef LC_WARP_LSU_SLOT
#define LC_WARP_LSU_SLOT 4096
#endif
// Resident CTAs per SM the LSU kernel is compiled for (caps registers).
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
    int64_t n_units, units_per_stage, n_chunks;
    uint32_t stage_bytes;
    uint64_t timeout_ns;
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
__device__ __forceinline__ int64_t unit_dst_offset(const WarpArgs &a, int64_t u) { return unit_offset(a, u, a.bd); }

// Walks the units of chunk c (consecutive flat unit indices), merging units
// that are contiguous on the chosen side into one bulk copy, and hands each
// copy to `emit(byte_offset, bytes, smem_offset)`.
template <typename Emit>
__device__ __forceinline__ void walk_chunk(const WarpArgs &a, int64_t c, bool src_side, Emit emit) {
    const int64_t first = c * a.units_per_stage;
    const int64_t cnt = lmin(a.units_per_stage, a.n_units - first);
    const int64_t *str = src_side ? a.bs : a.bd;
    int64_t idx[kMaxModes];
    int64_t rest = first, off = 0;
    for (int i = a.nb - 1; i >= 0; --i) {
        idx[i] = rest % a.be[i];
        rest /= a.be[i];
        off += idx[i] * str[i];
    }
    int64_t run_off = off;
    uint32_t run_len = a.unit_bytes, smem_off = 0;
    for (int64_t u = 1; u < cnt; ++u) {
        for (int i = a.nb - 1; i >= 0; --i) {  // advance the unit odometer
            off += str[i];
            if (++idx[i] < a.be[i]) break;
            off -= idx[i] * str[i];
            idx[i] = 0;
        }
        if (off == run_off + run_len) {
            run_len += a.unit_bytes;
        } else {
            emit(run_off, run_len, smem_off);
            smem_off += run_len;
            run_off = off;
            run_len = a.unit_bytes;
        }
    }
    emit(run_off, run_len, smem_off);
}

__device__ __forceinline__ void warp_issue_load(const WarpArgs &a, int64_t c, uint32_t stage, uint32_t bar) {
    const int64_t cnt = lmin(a.units_per_stage, a.n_units - c * a.units_per_stage);
    ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(cnt * a.unit_bytes));
    walk_chunk(a, c, true, [&](int64_t off, uint32_t bytes, uint32_t soff) {
        ptx::bulk_g2s(stage + soff, a.src + off, bytes, bar);
    });
}

// One CTA streams chunks c = blockIdx.x + i * gridDim.x through a ring of
// kWarpStages shared-memory stages.  Thread 0 keeps the ring full of bulk
// loads (units contiguous in the source merged into one copy).  Each warp
// takes whole units of the landed stage:
//   phase 1  lane, step r reads the word of iteration j = r ^ ((lane >> shift)
//            & mask) through the source layout into regs[r]; __syncwarp;
//   phase 2  writes regs[r] through the destination layout, in place (the
//            barrier between the phases makes the aliasing safe, and a dense
//            destination image lands exactly on the unit); __syncwarp;
//   out      the unit, now in destination order, leaves with 16-byte
//            coalesced stores (the copy -> gmem_smem [outer, threads, vec]
//            split with vec = 16 bytes).
// A CTA barrier then frees the stage and thread 0 refills it.
template <int W, int PMAX>
__global__ void __launch_bounds__(kWarpThreads) k_warp_permute(const __grid_constant__ WarpArgs a) {
    using T = typename Word<W>::T;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *stages = smem + 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;

    // per-lane byte offsets of the P staged words inside one unit
    int32_t soff[PMAX], doff[PMAX];
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

    const int64_t n_local =
        a.n_chunks > blockIdx.x ? (a.n_chunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t bar0 = ptx::smem_addr(bars), stage0 = ptx::smem_addr(stages);
    if (tid == 0) {
        for (int s = 0; s < kWarpStages; ++s) ptx::mbar_init(bar0 + 8 * s, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int64_t i = 0; i < lmin(kWarpStages, n_local); ++i)
            warp_issue_load(a, blockIdx.x + i * gridDim.x, stage0 + i * a.stage_bytes, bar0 + 8 * i);

    const int chunks16 = static_cast<int>(a.unit_bytes / 16);
    for (int64_t i = 0; i < n_local; ++i) {
        const int s = static_cast<int>(i % kWarpStages);
        const uint32_t parity = static_cast<uint32_t>((i / kWarpStages) & 1);
        const int64_t c = blockIdx.x + i * gridDim.x;
        const bool ok = ptx::mbar_wait_bounded(bar0 + 8 * s, parity, a.timeout_ns);
        if (ok) {
            const int64_t first = c * a.units_per_stage;
            const int cnt = static_cast<int>(lmin(a.units_per_stage, a.n_units - first));
            uint8_t *st = stages + static_cast<size_t>(s) * a.stage_bytes;
            for (int u = warp; u < cnt; u += nwarps) {
                uint8_t *ub = st + static_cast<size_t>(u) * a.unit_bytes;
                T regs[PMAX];
#pragma unroll
                for (int r = 0; r < PMAX; ++r)
                    if (r < a.P) regs[r] = *reinterpret_cast<const T *>(ub + soff[r]);
                __syncwarp();
#pragma unroll
                for (int r = 0; r < PMAX; ++r)
                    if (r < a.P) *reinterpret_cast<T *>(ub + doff[r]) = regs[r];
                __syncwarp();
                uint8_t *dunit = a.dst + unit_dst_offset(a, first + u);
                for (int q = lane; q < chunks16; q += 32)
                    *reinterpret_cast<uint4 *>(dunit + 16 * q) = *reinterpret_cast<const uint4 *>(ub + 16 * q);
            }
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                report_error(LC_ERR_TIMEOUT, LC_KERNEL_WARP_PERMUTE);
                for (int64_t q = i; q < lmin(i + kWarpStages, n_local); ++q)
                    ptx::mbar_wait_bounded(bar0 + 8 * (q % kWarpStages),
                                           static_cast<uint32_t>((q / kWarpStages) & 1), a.timeout_ns);
            }
            return;
        }
        if (tid == 0 && i + kWarpStages < n_local)
            warp_issue_load(a, blockIdx.x + (i + kWarpStages) * gridDim.x, stage0 + s * a.stage_bytes,
                            bar0 + 8 * s);
    }
}


// ----------------------------------------------------------------------------
// the same permute with every copy on the load/store units
// ----------------------------------------------------------------------------

constexpr int kLsuMaxChunks = 8;  // 16-byte chunks each lane keeps in flight

// Per-lane byte offsets of the P words, as in k_warp_permute.
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
__global__ void __launch_bounds__(kWarpThreads, LC_WARP_MIN_BLOCKS) k_warp_permute_lsu(const __grid_constant__ WarpArgs a) {
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
        for (int base = 0; base < nchunks; base += 32 * kLsuMaxChunks) {
            uint4 v[kLsuMaxChunks];
#pragma unroll
            for (int k = 0; k < kLsuMaxChunks; ++k) {
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
            for (int k = 0; k < kLsuMaxChunks; ++k) {
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
int launch_warp_t(const WarpArgs &a, int smem, cudaStream_t stream) {
#if LC_WARP_LSU
    (void)smem;
    const void *fn = a.contig ? reinterpret_cast<const void *>(&k_warp_permute_lsu<W, PMAX, true>)
                              : reinterpret_cast<const void *>(&k_warp_permute_lsu<W, PMAX, false>);
    const int lsmem = (kWarpThreads / 32) * static_cast<int>(a.stage_bytes);
    int sms, per;
    if (prepare(fn, kWarpThreads, lsmem, (kWarpThreads / 32) * kWarpStageMax, &sms, &per) != cudaSuccess)
        return LC_ERR_CUDA;
    const int64_t groups = (a.n_units + a.units_per_stage - 1) / a.units_per_stage;
    const int64_t grid = lmin((groups + kWarpThreads / 32 - 1) / (kWarpThreads / 32), int64_t(sms) * per);
    if (a.contig)
        k_warp_permute_lsu<W, PMAX, true><<<static_cast<unsigned>(grid), kWarpThreads, lsmem, stream>>>(a);
    else
        k_warp_permute_lsu<W, PMAX, false><<<static_cast<unsigned>(grid), kWarpThreads, lsmem, stream>>>(a);
#else
    const void *fn = reinterpret_cast<const void *>(&k_warp_permute<W, PMAX>);
    int sms, per;
    if (prepare(fn, kWarpThreads, smem, kWarpMaxSmem, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t grid = lmin(a.n_chunks, int64_t(sms) * per);
    k_warp_permute<W, PMAX><<<static_cast<unsigned>(grid), kWarpThreads, smem, stream>>>(a);
#endif
    return finish_launch();
}

template <int W>
int launch_warp_w(int P, const WarpArgs &a, int smem, cudaStream_t s) {
    if (P <= 4) return launch_warp_t<W, 4>(a, smem, s);
    if (P <= 8) return launch_warp_t<W, 8>(a, smem, s);
    return launch_warp_t<W, 32>(a, smem, s);
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
    a.units_per_stage = wp.units_per_stage;
#if LC_WARP_LSU
    a.units_per_stage = lmin(wp.n_units, std::max<int64_t>(1, LC_WARP_LSU_SLOT / (wp.U * p.w)));
#endif
    a.n_chunks = (wp.n_units + wp.units_per_stage - 1) / wp.units_per_stage;
    a.stage_bytes = static_cast<uint32_t>((a.units_per_stage * a.unit_bytes + 127) / 128 * 128);
    if (a.stage_bytes > static_cast<uint32_t>(kWarpStageMax)) return LC_ERR_UNSUPPORTED;
    a.timeout_ns = wait_limit_ns();
    const int smem = 128 + kWarpStages * static_cast<int>(a.stage_bytes);
    switch (p.w) {
        case 1: return launch_warp_w<1>(wp.P, a, smem, stream);
        case 2: return launch_warp_w<2>(wp.P, a, smem, stream);
        case 4: return launch_warp_w<4>(wp.P, a, smem, stream);
        case 8: return launch_warp_w<8>(wp.P, a, smem, stream);
        case 16: return launch_warp_w<16>(wp.P, a, smem, stream);
    }
    return LC_ERR_UNSUPPORTED;
}

cudaError_t take_error_warp(unsigned long long *v) { return take_module_error(v); }

}  // namespace lc
