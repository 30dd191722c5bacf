// TMA tensor copy: layouts whose innermost mode is contiguous on both sides
// (axis permutes that keep the last axis, row gathers, strided slices).
//
// The destination-ordered modes, innermost first, are the dimensions of two
// tensor maps over the same logical index: one with the source strides, one
// with the destination strides.  A tile (box) takes whole inner modes up to
// about 16 KiB.  One thread per CTA drives the copy engine: a TMA tensor load
// brings tile i into a ring stage ("copy -> gmem_smem": the global -> shared
// copy, here issued as one tensor copy instead of an [outer, threads, vec]
// loop), the stage's mbarrier completes it, and a TMA tensor store writes the
// same box through the destination map (the store phase's "TMA store").  No
// thread touches a word; the ring keeps S - 1 loads and the stores in flight.
// Boxes reaching past the tensor are zero-filled on load and clipped on store.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "device_common.cuh"
#include "launch.h"
#include "tensor_map.h"
#include "bulk_store.cuh"

namespace lc {

constexpr int kTmaStages = LC_TMA_STAGES;
constexpr int kTmaThreads = 32;  // one warp; lane 0 issues every copy

struct TmaCopyArgs {
    int32_t rank;       // tensor dimensions, 2..5
    int32_t box[5];     // box extent per dimension (TMA elements)
    FastDiv tiles[5];   // tiles per dimension
    uint32_t n_tiles;
    uint32_t tile_bytes;    // bytes one box moves
    uint32_t stage_stride;  // tile_bytes rounded up to 128 (stage alignment)
    uint64_t timeout_ns;
};

namespace {

__device__ __forceinline__ void tile_coords(const TmaCopyArgs &a, uint32_t t, int32_t (&c)[5]) {
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        if (k < a.rank) {
            const uint32_t q = fast_div(t, a.tiles[k]);
            c[k] = static_cast<int32_t>((t - q * a.tiles[k].d) * static_cast<uint32_t>(a.box[k]));
            t = q;
        } else {
            c[k] = 0;
        }
    }
}

__device__ __forceinline__ void tma_load(const void *tmap, int rank, const int32_t (&c)[5], uint32_t dst,
                                         uint32_t bar) {
    switch (rank) {
        case 2: ptx::tma_load_2d(dst, tmap, c[0], c[1], bar); break;
        case 3: ptx::tma_load_3d(dst, tmap, c[0], c[1], c[2], bar); break;
        case 4: ptx::tma_load_4d(dst, tmap, c[0], c[1], c[2], c[3], bar); break;
        default: ptx::tma_load_5d(dst, tmap, c[0], c[1], c[2], c[3], c[4], bar); break;
    }
}

}  // namespace

// CTA b copies tiles b, b + G, b + 2G, ... (G = gridDim.x).
__global__ void __launch_bounds__(kTmaThreads)
    k_tma_copy(const __grid_constant__ CUtensorMap src_map, const __grid_constant__ CUtensorMap dst_map,
               const __grid_constant__ TmaCopyArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    if (threadIdx.x != 0) return;
    const uint32_t bar0 = ptx::smem_addr(smem), buf0 = ptx::smem_addr(smem + 128);
    const uint32_t n_local = a.n_tiles > blockIdx.x ? (a.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    ptx::prefetch_tensormap(&src_map);
    ptx::prefetch_tensormap(&dst_map);
    for (int s = 0; s < kTmaStages; ++s) ptx::mbar_init(bar0 + 8 * s, 1);
    ptx::fence_mbar_init();

    auto issue_load = [&](uint32_t i) {
        const uint32_t s = i % kTmaStages;
        int32_t c[5];
        tile_coords(a, blockIdx.x + i * gridDim.x, c);
        ptx::mbar_arrive_expect_tx(bar0 + 8 * s, a.tile_bytes);
        tma_load(&src_map, a.rank, c, buf0 + s * a.stage_stride, bar0 + 8 * s);
    };
    uint32_t issued = 0;
    for (; issued < n_local && issued < uint32_t(kTmaStages); ++issued) issue_load(issued);

    for (uint32_t i = 0; i < n_local; ++i) {
        const uint32_t s = i % kTmaStages;
        if (!ptx::mbar_wait_bounded(bar0 + 8 * s, (i / kTmaStages) & 1, a.timeout_ns)) {
            report_error(LC_ERR_TIMEOUT, LC_KERNEL_TMA_COPY);
            bulk::wait_all();  // stores already issued
            for (uint32_t q = i; q < issued; ++q)  // loads that may still land in this CTA's ring
                ptx::mbar_wait_bounded(bar0 + 8 * (q % kTmaStages), (q / kTmaStages) & 1, a.timeout_ns);
            return;
        }
        bulk::fence_proxy_async_smem();
        int32_t c[5];
        tile_coords(a, blockIdx.x + i * gridDim.x, c);
        bulk::tma_store(&dst_map, a.rank, c, buf0 + s * a.stage_stride);
        bulk::commit();
        // refill the stage of tile i - 1 once its store has read it
        if (i >= 1 && issued < n_local) {
            bulk::wait_read<1>();
            issue_load(issued++);
        }
    }
    bulk::wait_all();
}

int launch_tma_copy(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    const TmaPlan &tp = p.tma;
    const ModeList &sl = p.sorted;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return LC_ERR_CUDA;
    const int w = p.w;
    const int mult = w == 16 ? 2 : 1;  // 16-byte words travel as two 8-byte elements
    const int eb = w / mult;
    CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (eb == 2) dt = CU_TENSOR_MAP_DATA_TYPE_UINT16;
    else if (eb == 4) dt = CU_TENSOR_MAP_DATA_TYPE_UINT32;
    else if (eb == 8) dt = CU_TENSOR_MAP_DATA_TYPE_UINT64;
    cuuint64_t dims[5], sstr[4], dstr[4];
    cuuint32_t box[5], estr[5];
    TmaCopyArgs a{};
    a.rank = tp.rank;
    uint64_t n_tiles = 1;
    for (int k = 0; k < tp.rank; ++k) {
        const Mode &m = sl.m[sl.n - 1 - k];
        dims[k] = static_cast<cuuint64_t>(m.e * (k == 0 ? mult : 1));
        if (k > 0) {
            sstr[k - 1] = static_cast<cuuint64_t>(m.s * w);
            dstr[k - 1] = static_cast<cuuint64_t>(m.d * w);
        }
        box[k] = static_cast<cuuint32_t>(tp.box[k]);
        estr[k] = 1;
        a.box[k] = tp.box[k];
        const uint64_t t = (dims[k] + box[k] - 1) / box[k];
        a.tiles[k] = make_fastdiv(static_cast<uint32_t>(t));
        n_tiles *= t;
    }
    if (n_tiles >= (uint64_t(1) << 32)) return LC_ERR_UNSUPPORTED;  // the planner keeps it below
    a.n_tiles = static_cast<uint32_t>(n_tiles);
    a.tile_bytes = static_cast<uint32_t>(tp.stage_bytes);
    a.stage_stride = (a.tile_bytes + 127u) / 128u * 128u;
    a.timeout_ns = wait_limit_ns();

    CUtensorMap smap, dmap;
    std::memset(&smap, 0, sizeof(smap));
    std::memset(&dmap, 0, sizeof(dmap));
    void *sbase = const_cast<uint8_t *>(src + p.src_off * w);
    void *dbase = dst + p.dst_off * w;
    const cuuint32_t r = static_cast<cuuint32_t>(tp.rank);
    if (enc(&smap, dt, r, sbase, dims, sstr, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&dmap, dt, r, dbase, dims, dstr, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return LC_ERR_UNSUPPORTED;  // the driver refused this tensor shape

    const int smem = 128 + kTmaStages * static_cast<int>(a.stage_stride);
    const void *fn = reinterpret_cast<const void *>(&k_tma_copy);
    int sms, per;
    if (prepare(fn, kTmaThreads, smem, 227 * 1024, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t grid = lmin(a.n_tiles, int64_t(sms) * per);
    k_tma_copy<<<static_cast<unsigned>(grid), kTmaThreads, smem, stream>>>(smap, dmap, a);
    return finish_launch();
}

cudaError_t take_error_tma_copy(unsigned long long *v) { return take_module_error(v); }

}  // namespace lc
