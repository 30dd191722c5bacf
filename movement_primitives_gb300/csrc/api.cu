// ABI entry points that launch work, the launch helpers shared by the kernel
// translation units, and the failure-path check kernel.
#include <cuda_runtime.h>

#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

// One thread waits on a shared-memory barrier that nothing arrives at; the
// bounded wait gives up after limit_ns and records LC_ERR_TIMEOUT.
__global__ void k_wait_timeout(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait_bounded(b, 0, limit_ns)) report_error(LC_ERR_TIMEOUT, 0xff);
}

uint64_t wait_limit_ns() {
    static const uint64_t v = [] {
        const char *e = std::getenv("LC_WAIT_TIMEOUT_NS");
        const long long x = e ? std::atoll(e) : 0;
        return x > 0 ? static_cast<uint64_t>(x) : uint64_t(2000000000);  // 2 s
    }();
    return v;
}

namespace {
std::mutex g_mu;
std::map<std::tuple<const void *, int, int, int>, int> g_occ;  // (fn, dev, threads, smem) -> blocks/SM
std::map<std::pair<const void *, int>, int> g_attr;             // (fn, dev) -> opted-in smem
std::map<int, int> g_sms;
}  // namespace

cudaError_t prepare(const void *fn, int threads, int smem, int attr_smem, int *sms, int *per_sm) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sms.find(dev);
    if (it == g_sms.end()) {
        int n = 0;
        if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        it = g_sms.emplace(dev, n).first;
    }
    *sms = it->second;
    const auto akey = std::make_pair(fn, dev);
    if (g_attr.find(akey) == g_attr.end()) {
        if (attr_smem > 48 * 1024 &&
            (e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, attr_smem)) != cudaSuccess)
            return e;
        g_attr.emplace(akey, attr_smem);
    }
    const auto key = std::make_tuple(fn, dev, threads, smem);
    auto jt = g_occ.find(key);
    if (jt == g_occ.end()) {
        int nb = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem)) != cudaSuccess) return e;
        jt = g_occ.emplace(key, nb < 1 ? 1 : nb).first;
    }
    *per_sm = jt->second;
    return cudaSuccess;
}

int launch_plan(const Plan &p, const uint8_t *s, uint8_t *d, cudaStream_t cs, bool fallback) {
    switch (p.kernel) {
        case LC_KERNEL_VEC_COPY: return launch_vec(p, s, d, cs);
        case LC_KERNEL_WARP_PERMUTE: return launch_warp(p, s, d, cs);
        case LC_KERNEL_WARP_SHUFFLE: return launch_shuffle(p, s, d, cs);
        case LC_KERNEL_SMEM_STAGED: return launch_staged(p, s, d, cs);
        case LC_KERNEL_SMEM_TRANSPOSE: return launch_smem(p, s, d, cs);
        case LC_KERNEL_TMA_COPY: {
            const int r = launch_tma_copy(p, s, d, cs);
            if (r != LC_ERR_UNSUPPORTED || !fallback) return r;
            return launch_vec(p, s, d, cs);  // the driver refused a tensor map: same copy, vector path
        }
        case LC_KERNEL_TILE_TRANSPOSE: {
            const int r = launch_tile(p, s, d, cs);
            if (r != LC_ERR_UNSUPPORTED || !fallback) return r;
            Plan q = p;  // the driver refused the tensor map: same tiles, shared-memory path
            q.smem_swz = choose_smem_swizzle(p.w);
            return launch_smem(q, s, d, cs);
        }
    }
    return LC_ERR_UNSUPPORTED;
}

}  // namespace lc

extern "C" int lc_layout_copy_ex(const void *src, const lc_tile_layout *src_layout, void *dst,
                                 const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles,
                                 int32_t kernel, lc_stream_t stream) {
    lc::Plan p;
    lc::PtrInfo ptr;
    ptr.src = reinterpret_cast<uintptr_t>(src);
    ptr.dst = reinterpret_cast<uintptr_t>(dst);
    ptr.check = true;
    const int st = lc::make_plan(src_layout, dst_layout, elem_bytes, n_tiles, kernel, ptr, &p);
    if (st) return st;
    if (p.total == 0) return LC_OK;
    // an automatic choice never declines a valid copy
    return lc::launch_plan(p, static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst),
                           reinterpret_cast<cudaStream_t>(stream), kernel == LC_KERNEL_AUTO);
}

namespace {

// Device address of byte `lo` of the range [base + lo, base + hi) if both of
// its ends are memory the device can address and the device sees the range
// contiguously; 0 otherwise.
uintptr_t device_view(const void *base, int64_t lo, int64_t hi) {
    const uint8_t *b = static_cast<const uint8_t *>(base);
    cudaPointerAttributes first{}, last{};
    if (cudaPointerGetAttributes(&first, b + lo) != cudaSuccess ||
        cudaPointerGetAttributes(&last, b + hi - 1) != cudaSuccess) {
        cudaGetLastError();  // a failed lookup leaves no sticky error behind
        return 0;
    }
    if (first.type == cudaMemoryTypeUnregistered || last.type == cudaMemoryTypeUnregistered ||
        !first.devicePointer || !last.devicePointer)
        return 0;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(first.devicePointer);
    const uintptr_t d1 = reinterpret_cast<uintptr_t>(last.devicePointer);
    if (d1 < d0 || d1 - d0 != uintptr_t(hi - 1 - lo)) return 0;
    return d0;
}

}  // namespace

extern "C" int lc_layout_copy_mapped(const void *src_host, const lc_tile_layout *src_layout, void *dst_host,
                                     const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles,
                                     lc_stream_t stream) {
    {  // two device buffers: the ordinary copy, TMA classes included
        cudaPointerAttributes as{}, ad{};
        const bool devs = src_host && dst_host && cudaPointerGetAttributes(&as, src_host) == cudaSuccess &&
                          cudaPointerGetAttributes(&ad, dst_host) == cudaSuccess &&
                          as.type == cudaMemoryTypeDevice && ad.type == cudaMemoryTypeDevice;
        cudaGetLastError();
        if (devs)
            return lc_layout_copy_ex(src_host, src_layout, dst_host, dst_layout, elem_bytes, n_tiles, LC_KERNEL_AUTO,
                                     stream);
    }
    lc::Plan p;
    lc::PtrInfo ptr;
    ptr.src = reinterpret_cast<uintptr_t>(src_host);
    ptr.dst = reinterpret_cast<uintptr_t>(dst_host);
    ptr.check = true;
    ptr.no_tma = true;
    const int st = lc::make_plan(src_layout, dst_layout, elem_bytes, n_tiles, LC_KERNEL_AUTO, ptr, &p);
    if (st) return st;
    if (p.total == 0) return LC_OK;
    const uintptr_t s0 = device_view(src_host, p.src_lo, p.src_hi);
    const uintptr_t d0 = device_view(dst_host, p.dst_lo, p.dst_hi);
    if (!s0 || !d0) return LC_ERR_NOT_MAPPED;
    // the device addresses keep the host addresses' alignment (mappings are page-granular)
    const uint8_t *s = reinterpret_cast<const uint8_t *>(s0 - uintptr_t(p.src_lo));
    uint8_t *d = reinterpret_cast<uint8_t *>(d0 - uintptr_t(p.dst_lo));
    if ((reinterpret_cast<uintptr_t>(s) ^ ptr.src) & 255 || (reinterpret_cast<uintptr_t>(d) ^ ptr.dst) & 255)
        return LC_ERR_NOT_MAPPED;
    return lc::launch_plan(p, s, d, reinterpret_cast<cudaStream_t>(stream), true);
}

extern "C" int lc_layout_copy(const void *src, const lc_tile_layout *src_layout, void *dst,
                              const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles,
                              lc_stream_t stream) {
    return lc_layout_copy_ex(src, src_layout, dst, dst_layout, elem_bytes, n_tiles, LC_KERNEL_AUTO, stream);
}

extern "C" int lc_last_device_error(lc_stream_t stream, uint64_t *detail) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LC_ERR_CUDA;
    unsigned long long words[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    cudaError_t (*const take[8])(unsigned long long *) = {
        lc::take_module_error, lc::take_error_tile, lc::take_error_tma_copy, lc::take_error_warp1,
        lc::take_error_warp2,  lc::take_error_warp4, lc::take_error_warp8, lc::take_error_warp16};
    for (int i = 0; i < 8; ++i)
        if (take[i](&words[i]) != cudaSuccess) return LC_ERR_CUDA;
    unsigned long long v = 0;
    for (unsigned long long w : words)
        if (!v && w) v = w;
    if (detail) *detail = v;
    return static_cast<int>(v & 0xff);
}

extern "C" int lc_debug_wait_timeout(int64_t timeout_ns, lc_stream_t stream) {
    if (timeout_ns < 1000) timeout_ns = 1000;
    if (timeout_ns > 1000000000) timeout_ns = 1000000000;
    lc::k_wait_timeout<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(timeout_ns));
    return cudaGetLastError() == cudaSuccess ? LC_OK : LC_ERR_CUDA;
}

extern "C" const char *lc_status_string(int32_t status) {
    switch (status) {
        case LC_OK: return "ok";
        case LC_ERR_NULL: return "a required pointer is NULL";
        case LC_ERR_RANK: return "rank outside 1..8";
        case LC_ERR_SHAPE: return "negative extent or tile count, or element count not a multiple of the warp";
        case LC_ERR_EXTENT_MISMATCH: return "non-unit extents of source and destination differ";
        case LC_ERR_ELEM_BYTES: return "element size not in {1,2,4,8,16}";
        case LC_ERR_BAD_STRIDE:
            return "negative stride or offset, zero destination stride, or a loop-layout mode feeding both or "
                   "neither of thread and slot";
        case LC_ERR_NOT_INJECTIVE: return "destination layout maps two logical indices to one offset";
        case LC_ERR_OVERLAP: return "source and destination byte ranges overlap";
        case LC_ERR_ALIGN: return "pointer not aligned to the element size";
        case LC_ERR_NO_SWIZZLE: return "no XOR swizzle makes both phases bank-conflict-free";
        case LC_ERR_CUDA: return "CUDA runtime error";
        case LC_ERR_TIMEOUT: return "a bounded device wait gave up";
        case LC_ERR_UNSUPPORTED: return "the requested kernel class cannot perform this copy";
        case LC_ERR_OVERFLOW: return "an offset does not fit in 63 bits";
        case LC_ERR_STAGING: return "the staging buffer is too small";
        case LC_ERR_LOOP_LAYOUT: return "the loop layout is not an exact partition of the tile (or has over 1024 threads)";
        case LC_ERR_UNDECIDED:
            return "the destination could not be shown one-to-one (no stride split settles it, too many words to "
                   "enumerate)";
        case LC_ERR_NOT_MAPPED: return "a byte range is not memory the device can address";
    }
    return "unknown status";
}

extern "C" const char *lc_kernel_name(int32_t kernel) {
    switch (kernel) {
        case LC_KERNEL_AUTO: return "auto";
        case LC_KERNEL_VEC_COPY: return "vec_copy";
        case LC_KERNEL_WARP_PERMUTE: return "warp_permute";
        case LC_KERNEL_TILE_TRANSPOSE: return "tile_transpose";
        case LC_KERNEL_SMEM_TRANSPOSE: return "smem_transpose";
        case LC_KERNEL_TMA_COPY: return "tma_copy";
        case LC_KERNEL_WARP_SHUFFLE: return "warp_shuffle";
        case LC_KERNEL_SMEM_STAGED: return "smem_staged";
    }
    return "unknown";
}
