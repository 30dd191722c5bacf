// The host-buffer copy for callers that cannot allocate device memory.
//
// lc_layout_copy_host needs a device staging buffer from its caller.  Some
// callers cannot provide one: a plugin inside an application whose allocator
// owns all device memory, code that must not call cudaMalloc because it can
// synchronise the whole device, or code about to be captured into a CUDA
// graph, where cudaMalloc is not allowed.  This entry point stages through a
// fixed buffer that lives in the library itself: a file-scope device array of
// LC_STATIC_STAGING_BYTES that every GPU loading the library keeps until the
// process exits.  No call allocates or frees anything.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress (it may load this module
// onto the device) and caches it; make that first call before any stream
// capture.  The array is shared by every call and keeps the previous call's
// bytes; nothing in it needs to start at zero, because every chunk's source
// span is uploaded before the permute reads it and the permute writes the
// whole destination image (a destination with holes has its span uploaded
// first).  Calls that overlap on the GPU (e.g. on two streams) race on the
// array: serialise them.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "launch.h"

namespace lc {
namespace {

static __device__ __align__(256) unsigned char g_static_staging[LC_STATIC_STAGING_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
unsigned char *g_static_ptr[kMaxDevices] = {nullptr};

// Device address of the staging array on the current device (looked up once).
int static_staging(unsigned char **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_staging) != cudaSuccess || !p) return LC_ERR_CUDA;
        g_static_ptr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_static_ptr[dev];
    return LC_OK;
}

int64_t cosize(const lc_tile_layout &l) {
    int64_t c = 1;
    for (int k = 0; k < l.rank; ++k) {
        if (l.shape[k] == 0) return 0;
        c += (l.shape[k] - 1) * l.stride[k];
    }
    return c;
}

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

}  // namespace
}  // namespace lc

extern "C" int lc_layout_copy_host_static(const void *src_host, const lc_tile_layout *src_layout,
                                          void *dst_host, const lc_tile_layout *dst_layout,
                                          int32_t elem_bytes, int64_t n_tiles, lc_stream_t stream) {
    using namespace lc;
    if (!src_layout || !dst_layout) return LC_ERR_NULL;
    Plan whole;
    PtrInfo none;
    int st = make_plan(src_layout, dst_layout, elem_bytes, n_tiles, LC_KERNEL_AUTO, none, &whole);
    if (st) return st;
    if (whole.total == 0) return LC_OK;
    if (!src_host || !dst_host) return LC_ERR_NULL;
    {
        const uintptr_t s0 = reinterpret_cast<uintptr_t>(src_host) + uintptr_t(whole.src_lo);
        const uintptr_t s1 = reinterpret_cast<uintptr_t>(src_host) + uintptr_t(whole.src_hi);
        const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst_host) + uintptr_t(whole.dst_lo);
        const uintptr_t d1 = reinterpret_cast<uintptr_t>(dst_host) + uintptr_t(whole.dst_hi);
        if (s0 < d1 && d0 < s1) return LC_ERR_OVERLAP;
    }

    const int64_t w = elem_bytes;
    const int64_t scos = cosize(*src_layout), dcos = cosize(*dst_layout);
    const int64_t sts = src_layout->tile_stride ? src_layout->tile_stride : scos;
    const int64_t dts = dst_layout->tile_stride ? dst_layout->tile_stride : dcos;
    int64_t dwords = 1;
    for (int k = 0; k < dst_layout->rank; ++k) dwords *= dst_layout->shape[k];
    const bool dst_dense = dwords == dcos && (n_tiles == 1 || dts == dcos);
    // Byte spans of `t` tiles starting at tile 0 (chunks have the same spans).
    auto src_span = [&](int64_t t) { return (src_layout->offset + (t - 1) * sts + scos) * w - src_layout->offset * w; };
    auto dst_span = [&](int64_t t) { return (dst_layout->offset + (t - 1) * dts + dcos) * w - dst_layout->offset * w; };
    auto need = [&](int64_t t) { return round256(src_span(t)) + round256(dst_span(t)); };

    // Largest chunk of tiles whose spans fit the array; chunks need disjoint
    // destination spans, otherwise the whole copy must fit at once.
    int64_t chunk = n_tiles;
    if (need(chunk) > LC_STATIC_STAGING_BYTES) {
        if (n_tiles == 1 || dts < dcos || need(1) > LC_STATIC_STAGING_BYTES) return LC_ERR_STAGING;
        int64_t lo = 1, hi = n_tiles;  // need(lo) fits, need(hi) does not
        while (hi - lo > 1) {
            const int64_t mid = lo + (hi - lo) / 2;
            (need(mid) <= LC_STATIC_STAGING_BYTES ? lo : hi) = mid;
        }
        chunk = lo;
    }
    unsigned char *stage = nullptr;
    if ((st = static_staging(&stage))) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t *sh = static_cast<const uint8_t *>(src_host);
    uint8_t *dh = static_cast<uint8_t *>(dst_host);
    for (int64_t t0 = 0; t0 < n_tiles; t0 += chunk) {
        const int64_t t1 = std::min(n_tiles, t0 + chunk);
        const int64_t s_lo = (src_layout->offset + t0 * sts) * w, s_len = src_span(t1 - t0);
        const int64_t d_lo = (dst_layout->offset + t0 * dts) * w, d_len = dst_span(t1 - t0);
        uint8_t *s_dev = stage;
        uint8_t *d_dev = stage + round256(s_len);
        if (cudaMemcpyAsync(s_dev, sh + s_lo, size_t(s_len), cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return LC_ERR_CUDA;
        if (!dst_dense && cudaMemcpyAsync(d_dev, dh + d_lo, size_t(d_len), cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return LC_ERR_CUDA;
        lc_tile_layout sl = *src_layout, dl = *dst_layout;  // chunk spans start at the chunk's first tile
        sl.offset = 0;
        dl.offset = 0;
        sl.tile_stride = sts;
        dl.tile_stride = dts;
        Plan p;
        PtrInfo ptr;
        ptr.src = reinterpret_cast<uintptr_t>(s_dev);
        ptr.dst = reinterpret_cast<uintptr_t>(d_dev);
        ptr.check = true;
        if ((st = make_plan(&sl, &dl, elem_bytes, t1 - t0, LC_KERNEL_AUTO, ptr, &p))) return st;
        if ((st = launch_plan(p, s_dev, d_dev, cs, true))) return st;
        if (cudaMemcpyAsync(dh + d_lo, d_dev, size_t(d_len), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
            return LC_ERR_CUDA;
    }
    return LC_OK;
}
