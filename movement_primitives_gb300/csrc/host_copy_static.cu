// The host-buffer copy for callers that cannot allocate device memory.
//
// lc_layout_copy_host needs a device staging buffer from its caller.  Some
// callers cannot provide one: a plugin inside an application whose allocator
// owns all device memory and hands none out, or code that must not call
// cudaMalloc because cudaMalloc can synchronise the whole device and stall
// work that other threads have queued.  This entry point stages through a
// fixed buffer that lives in the library itself: a file-scope device array of
// LC_STATIC_STAGING_BYTES that every GPU loading the library keeps until the
// process exits.  No call allocates or frees anything.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress (it may load this module
// onto the device) and keeps it for that device; it does so before checking
// anything else, so any call, even one that is refused, completes the set-up.
// That first call must not itself run inside a stream capture.  The address
// is kept for the life of the process: after cudaDeviceReset on a device,
// this entry point must not be called on that device again.  The array is shared by
// every call and keeps the previous call's bytes; nothing in it needs to
// start at zero, because every chunk's source span is uploaded before the
// permute reads it and the permute writes the whole destination image (a
// destination with holes has its span uploaded first).  Calls that overlap on
// the GPU (e.g. on two streams) race on the array: serialise them.
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

}  // namespace
}  // namespace lc

extern "C" int lc_layout_copy_host_static(const void *src_host, const lc_tile_layout *src_layout,
                                          void *dst_host, const lc_tile_layout *dst_layout,
                                          int32_t elem_bytes, int64_t n_tiles, lc_stream_t stream) {
    using namespace lc;
    if (!src_layout || !dst_layout) return LC_ERR_NULL;
    unsigned char *stage = nullptr;
    int st = static_staging(&stage);  // the set-up, before any early return
    if (st) return st;
    Plan whole;
    PtrInfo none;
    st = make_plan(src_layout, dst_layout, elem_bytes, n_tiles, LC_KERNEL_AUTO, none, &whole);
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

    const HostSides hs = host_sides(*src_layout, *dst_layout, elem_bytes, n_tiles);
    // Largest chunk of tiles whose spans fit the array; chunks need disjoint
    // destination spans, otherwise the whole copy must fit at once.
    int64_t chunk = n_tiles;
    if (hs.slot_bytes(chunk) > LC_STATIC_STAGING_BYTES) {
        if (n_tiles == 1 || hs.dts < hs.dcos || hs.slot_bytes(1) > LC_STATIC_STAGING_BYTES) return LC_ERR_STAGING;
        int64_t lo = 1, hi = n_tiles;  // slot_bytes(lo) fits, slot_bytes(hi) does not
        while (hi - lo > 1) {
            const int64_t mid = lo + (hi - lo) / 2;
            (hs.slot_bytes(mid) <= LC_STATIC_STAGING_BYTES ? lo : hi) = mid;
        }
        chunk = lo;
    }
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t *sh = static_cast<const uint8_t *>(src_host);
    uint8_t *dh = static_cast<uint8_t *>(dst_host);
    for (int64_t t0 = 0; t0 < n_tiles; t0 += chunk) {
        const int64_t t1 = std::min(n_tiles, t0 + chunk);
        const HostSpan s = hs.src(t0, t1), d = hs.dst(t0, t1);
        uint8_t *s_dev = stage;
        uint8_t *d_dev = stage + round256(s.hi - s.lo);
        if (cudaMemcpyAsync(s_dev, sh + s.lo, size_t(s.hi - s.lo), cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return LC_ERR_CUDA;
        if (!hs.dst_dense &&
            cudaMemcpyAsync(d_dev, dh + d.lo, size_t(d.hi - d.lo), cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return LC_ERR_CUDA;
        lc_tile_layout sl = *src_layout, dl = *dst_layout;  // chunk spans start at the chunk's first tile
        sl.offset = 0;
        dl.offset = 0;
        sl.tile_stride = hs.sts;
        dl.tile_stride = hs.dts;
        Plan p;
        PtrInfo ptr;
        ptr.src = reinterpret_cast<uintptr_t>(s_dev);
        ptr.dst = reinterpret_cast<uintptr_t>(d_dev);
        ptr.check = true;
        if ((st = make_plan(&sl, &dl, elem_bytes, t1 - t0, LC_KERNEL_AUTO, ptr, &p))) return st;
        if ((st = launch_plan(p, s_dev, d_dev, cs, true))) return st;
        if (cudaMemcpyAsync(dh + d.lo, d_dev, size_t(d.hi - d.lo), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
            return LC_ERR_CUDA;
    }
    return LC_OK;
}
