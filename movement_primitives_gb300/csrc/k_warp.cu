// Warp register-staged permute of bulk-copied units (Apache TVM docs
// "permute_layout", section "Algorithm").
//
// A unit is a dense block of U = 32 * P words on both sides.  Units are
// bulk-copied global -> shared (several per stage, contiguous ones merged into
// one copy), each warp permutes one unit in place through registers with the
// per-lane XOR swizzle chosen by the host bank simulator, and the stage is
// bulk-copied back.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

constexpr int kWarpThreads = 256;
constexpr int kWarpStages = 4;
constexpr int kWarpStageMax = 16 * 1024;  // the planner stages at most 16 KiB of units
constexpr int kWarpMaxSmem = 128 + kWarpStages * kWarpStageMax;

struct WarpArgs {
    const uint8_t *src;  // address of source word offset 0
    uint8_t *dst;
    int32_t un;  // unit modes, logical order (words)
    int32_t ue[kMaxModes], us[kMaxModes], ud[kMaxModes];
    int32_t P, shift, mask;
    uint32_t unit_bytes;
    int32_t nb;  // batch modes (BYTES strides), outermost first
    int64_t be[kMaxModes], bs[kMaxModes], bd[kMaxModes];
    int64_t n_units, units_per_stage, n_chunks;
    uint32_t stage_bytes;
    uint64_t timeout_ns;
};

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

__device__ __forceinline__ void warp_issue_store(const WarpArgs &a, int64_t c, uint32_t stage) {
    walk_chunk(a, c, false, [&](int64_t off, uint32_t bytes, uint32_t soff) {
        ptx::bulk_s2g(a.dst + off, stage + soff, bytes);
    });
    ptx::bulk_commit();
}

// One CTA streams chunks c = blockIdx.x + i * gridDim.x through a ring of
// kWarpStages shared-memory stages.  Thread 0 keeps kWarpStages - 1 bulk
// loads ahead; after the warps permute a stage in place, thread 0 bulk-stores
// it and refills the stage whose store was issued one iteration earlier, once
// that store has finished reading shared memory.
//
// Permute of one unit by one warp (the page's two phases): lane, step r reads
// the word of iteration j = r ^ ((lane >> shift) & mask) through the source
// layout into regs[r]; __syncwarp; writes regs[r] through the destination
// layout.  The unit is permuted in place: the barrier between the phases makes
// the aliasing safe, and a dense destination image lands exactly on the unit.
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
        for (int64_t i = 0; i < lmin(kWarpStages - 1, n_local); ++i)
            warp_issue_load(a, blockIdx.x + i * gridDim.x, stage0 + i * a.stage_bytes, bar0 + 8 * i);

    for (int64_t i = 0; i < n_local; ++i) {
        const int s = static_cast<int>(i % kWarpStages);
        const uint32_t parity = static_cast<uint32_t>((i / kWarpStages) & 1);
        const int64_t c = blockIdx.x + i * gridDim.x;
        const bool ok = ptx::mbar_wait_bounded(bar0 + 8 * s, parity, a.timeout_ns);
        if (ok) {
            const int cnt = static_cast<int>(lmin(a.units_per_stage, a.n_units - c * a.units_per_stage));
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
            }
            ptx::fence_proxy_async_smem();
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                report_error(LC_ERR_TIMEOUT, LC_KERNEL_WARP_PERMUTE);
                for (int64_t q = i; q < lmin(i + kWarpStages - 1, n_local); ++q)
                    ptx::mbar_wait_bounded(bar0 + 8 * (q % kWarpStages),
                                           static_cast<uint32_t>((q / kWarpStages) & 1), a.timeout_ns);
                ptx::bulk_wait_all();
            }
            return;
        }
        if (tid == 0) {
            warp_issue_store(a, c, stage0 + s * a.stage_bytes);
            const int64_t nxt = i + kWarpStages - 1;
            if (nxt < n_local) {
                ptx::bulk_wait_read<1>();  // the store issued last iteration has read its stage
                const int ns = static_cast<int>(nxt % kWarpStages);
                warp_issue_load(a, blockIdx.x + nxt * gridDim.x, stage0 + ns * a.stage_bytes, bar0 + 8 * ns);
            }
        }
    }
    if (tid == 0) ptx::bulk_wait_all();
}

namespace {

template <int W, int PMAX>
int launch_warp_t(const WarpArgs &a, int smem, cudaStream_t stream) {
    const void *fn = reinterpret_cast<const void *>(&k_warp_permute<W, PMAX>);
    int sms, per;
    if (prepare(fn, kWarpThreads, smem, kWarpMaxSmem, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t grid = lmin(a.n_chunks, int64_t(sms) * per);
    k_warp_permute<W, PMAX><<<static_cast<unsigned>(grid), kWarpThreads, smem, stream>>>(a);
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
    a.n_units = wp.n_units;
    a.units_per_stage = wp.units_per_stage;
    a.n_chunks = (wp.n_units + wp.units_per_stage - 1) / wp.units_per_stage;
    a.stage_bytes = static_cast<uint32_t>((wp.units_per_stage * a.unit_bytes + 127) / 128 * 128);
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
