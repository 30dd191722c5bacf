// Warp register-staged permute of dense units (Apache TVM docs
// "permute_layout", section "Algorithm"), staged through shared memory with
// the [outer, threads, vec] global <-> shared copy of "copy -> gmem_smem".
//
// A unit is a dense block of U = 32 * P words on both sides.  Each warp
// stages whole units in its own shared-memory slot with 16-byte coalesced
// loads, permutes each unit in place through registers under the per-lane
// XOR swizzle chosen by the host bank simulator, and writes the slot out
// with 16-byte coalesced stores.  Nothing waits on another warp.
//
// This unit holds the host launchers (plan -> arguments) and the C-ABI
// entry point of the shared-buffer op; the kernels live in k_warp.cuh and
// are instantiated per word width in k_warp_w{1,2,4,8,16}.cu.
#include <cuda_runtime.h>

#include <algorithm>

#include "k_warp.cuh"

namespace lc {

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
    int64_t suffix = 1;  // the device's nesting test (lc_device::warp_unit_offsets)
    a.nested = 1;
    for (int i = wp.unit.n - 1; i >= 0; --i) {
        suffix *= wp.unit.m[i].e;
        a.nested &= (suffix % 32 == 0 || 32 % suffix == 0) ? 1 : 0;
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
    a.timeout_ns = wait_limit_ns();
    // Bulk-copy prefetch for contiguous units past 8 words a lane, up to one
    // slot: measured on batches of 32 x 32 transposes, 67 -> 91 % of the
    // copy peak (4-byte words), 41 -> 67 (2), 28 -> 41 (1); units of 8 words
    // and less lose with it (4 x 32 fp32 units 98.6 -> 92.4 %), and 8 KiB
    // units (two slots of them leave one CTA per SM) gain nothing.
    a.async = LC_WARP_ASYNC && a.contig && wp.P > 8 && a.unit_bytes <= LC_WARP_ASYNC_SLOT;
    const int64_t slot = a.async ? LC_WARP_ASYNC_SLOT : LC_WARP_SLOT;
    a.units_per_stage = lmin(wp.n_units, std::max<int64_t>(1, slot / (wp.U * p.w)));
    a.stage_bytes = static_cast<uint32_t>((a.units_per_stage * a.unit_bytes + 127) / 128 * 128);
    if (a.stage_bytes > static_cast<uint32_t>(a.async ? kWarpSlotMax / 2 : kWarpSlotMax)) return LC_ERR_UNSUPPORTED;
    switch (p.w) {
        case 1: return launch_warp_width1(wp.P, a, stream);
        case 2: return launch_warp_width2(wp.P, a, stream);
        case 4: return launch_warp_width4(wp.P, a, stream);
        case 8: return launch_warp_width8(wp.P, a, stream);
        case 16: return launch_warp_width16(wp.P, a, stream);
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

// The destination modes, sorted by stride, read 1, e_a, e_a e_b, ...: the
// image is exactly [0, 32 P) words, every word of the buffer written once.
static bool dst_modes_dense(const lc_warp_unit &u) {
    std::pair<int32_t, int32_t> m[LC_MAX_RANK];
    int n = 0;
    for (int i = 0; i < u.n_modes; ++i)
        if (u.extent[i] > 1) m[n++] = {u.dst_stride[i], u.extent[i]};
    std::sort(m, m + n);
    int64_t expect = 1;
    for (int i = 0; i < n; ++i) {
        if (m[i].first != expect) return false;
        expect *= m[i].second;
    }
    return expect == u.dst_cosize;
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
    a.upw = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(kUnitMaxPerWarp, kUnitStageBytes / a.buf)));
    a.chunked = sb % 16 == 0 && db % 16 == 0;
    if (a.chunked) {
        a.schunks = make_fastdiv(static_cast<uint32_t>(sb / 16));
        a.dchunks = make_fastdiv(static_cast<uint32_t>(db / 16));
    }
    a.in_place = in_place ? 1 : 0;
    a.dst_dense = dst_modes_dense(*unit) ? 1 : 0;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    switch (elem_bytes) {
        case 1: return launch_unit_width1(a, cs);
        case 2: return launch_unit_width2(a, cs);
        case 4: return launch_unit_width4(a, cs);
        case 8: return launch_unit_width8(a, cs);
        default: return launch_unit_width16(a, cs);
    }
}
