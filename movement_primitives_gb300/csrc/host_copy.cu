// Host-buffer entry point: the layout copy between two host buffers, with the
// transfers pipelined over chunks of tiles through a caller-provided device
// staging buffer.  Chunk c moves host -> device on a copy stream, is permuted
// on the caller's stream, and moves device -> host on a second copy stream;
// three staging slots let chunk c+1's upload and chunk c-1's download run
// while chunk c is permuted, with one chunk of slack.  Chunks hold about LC_HOST_CHUNK_BYTES of source, so
// the pipeline's fill (the first upload) and drain (the last download), which
// run without the other direction, stay a small part of the call.  Events
// order the three streams; everything joins back into the caller's stream
// before the call returns.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>

#include "launch.h"

namespace lc {
namespace {

// Staging slots and source bytes per chunk (compile-time knobs so that
// variants can be measured).  Measured on GB300 on a 1 GiB permute: two
// slots leave the upload stream idle while chunk c-2's download waits for
// its permute (310 GB/s at best); below about 32 MiB per chunk the per-chunk
// cost of the copies and event hops (about 13 us) dominates; three slots of
// 32-64 MiB reach 318-320 GB/s.
#ifndef LC_HOST_SLOTS
#define LC_HOST_SLOTS 3
#endif
#ifndef LC_HOST_CHUNK_BYTES
#define LC_HOST_CHUNK_BYTES (48ll << 20)
#endif
constexpr int kSlots = LC_HOST_SLOTS;
constexpr int64_t kChunkBytes = LC_HOST_CHUNK_BYTES;
constexpr int64_t kMaxChunks = 1024;

// Tiles per chunk: about kChunkBytes of source span (tile stride sts words of
// w bytes), at least one tile, at most kMaxChunks chunks.
int64_t default_chunk(int64_t n_tiles, int64_t sts, int64_t w) {
    const int64_t tile_bytes = std::max<int64_t>(1, sts * w);
    int64_t c = std::max<int64_t>(1, kChunkBytes / tile_bytes);
    c = std::max(c, (n_tiles + kMaxChunks - 1) / kMaxChunks);
    return std::min(c, n_tiles);
}

struct DeviceStreams {
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t uploaded[kSlots], permuted[kSlots], downloaded[kSlots];
};

std::mutex g_streams_mu;
std::map<int, DeviceStreams> g_streams;

// Two non-blocking copy streams and their events, created once per device.
cudaError_t device_streams(DeviceStreams **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_streams_mu);
    auto it = g_streams.find(dev);
    if (it == g_streams.end()) {
        DeviceStreams ds;
        if ((e = cudaStreamCreateWithFlags(&ds.up, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&ds.down, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&ds.start, cudaEventDisableTiming)) != cudaSuccess) return e;
        for (int s = 0; s < kSlots; ++s) {
            const unsigned f = cudaEventDisableTiming;
            if ((e = cudaEventCreateWithFlags(&ds.uploaded[s], f)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&ds.permuted[s], f)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&ds.downloaded[s], f)) != cudaSuccess) return e;
        }
        it = g_streams.emplace(dev, ds).first;
    }
    *out = &it->second;
    return cudaSuccess;
}

}  // namespace
}  // namespace lc

extern "C" int lc_layout_copy_host(const void *src_host, const lc_tile_layout *src_layout, void *dst_host,
                                   const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles,
                                   void *staging, int64_t staging_bytes, lc_stream_t stream) {
    using namespace lc;
    if (!src_layout || !dst_layout) return LC_ERR_NULL;
    // validate the layouts once (plan of the whole copy, pointers aside)
    Plan whole;
    PtrInfo none;
    int st = make_plan(src_layout, dst_layout, elem_bytes, n_tiles, LC_KERNEL_AUTO, none, &whole);
    if (st) return st;
    if (whole.total == 0) return LC_OK;
    if (!src_host || !dst_host || !staging) return LC_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(staging) % 256) return LC_ERR_ALIGN;
    {
        const uintptr_t s0 = reinterpret_cast<uintptr_t>(src_host) + uintptr_t(whole.src_lo);
        const uintptr_t s1 = reinterpret_cast<uintptr_t>(src_host) + uintptr_t(whole.src_hi);
        const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst_host) + uintptr_t(whole.dst_lo);
        const uintptr_t d1 = reinterpret_cast<uintptr_t>(dst_host) + uintptr_t(whole.dst_hi);
        if (s0 < d1 && d0 < s1) return LC_ERR_OVERLAP;
    }

    const HostSides hs = host_sides(*src_layout, *dst_layout, elem_bytes, n_tiles);
    const int64_t w = hs.w, scos = hs.scos, dcos = hs.dcos, sts = hs.sts, dts = hs.dts;
    // Chunks need disjoint destination spans; otherwise the copy is one chunk.
    const bool chunkable = n_tiles > 1 && dts >= dcos && sts >= 0;
    // Unless the destination image covers its span exactly, the span is
    // staged in first so that bytes outside the image keep their values.
    const bool dst_dense = hs.dst_dense;
    auto slot_bytes = [&](int64_t tiles) { return hs.slot_bytes(tiles); };
    int64_t chunk = n_tiles;
    int slots = 1;
    if (chunkable) {
        chunk = default_chunk(n_tiles, std::max<int64_t>(sts, scos), w);
        while (chunk > 1 && kSlots * slot_bytes(chunk) > staging_bytes) chunk = (chunk + 1) / 2;
        slots = kSlots;
        if (kSlots * slot_bytes(chunk) > staging_bytes) {
            chunk = n_tiles;  // not even two one-tile slots: try a single pass
            slots = 1;
        }
    }
    if (slots * slot_bytes(chunk) > staging_bytes) return LC_ERR_STAGING;
    const int64_t slot_size = slot_bytes(chunk);
    DeviceStreams *ds = nullptr;
    if (device_streams(&ds) != cudaSuccess) return LC_ERR_CUDA;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *stage = static_cast<uint8_t *>(staging);
    const uint8_t *sh = static_cast<const uint8_t *>(src_host);
    uint8_t *dh = static_cast<uint8_t *>(dst_host);

    // the copy streams start after everything already queued on the caller's stream
    if (cudaEventRecord(ds->start, cs) != cudaSuccess) return LC_ERR_CUDA;
    if (cudaStreamWaitEvent(ds->up, ds->start, 0) != cudaSuccess) return LC_ERR_CUDA;
    if (cudaStreamWaitEvent(ds->down, ds->start, 0) != cudaSuccess) return LC_ERR_CUDA;

    int64_t c = 0;
    for (int64_t t0 = 0; t0 < n_tiles; t0 += chunk, ++c) {
        const int64_t t1 = std::min(n_tiles, t0 + chunk);
        const int b = static_cast<int>(c % slots);
        const HostSpan s = hs.src(t0, t1);
        const HostSpan d = hs.dst(t0, t1);
        uint8_t *s_dev = stage + b * slot_size;
        uint8_t *d_dev = s_dev + round256(s.hi - s.lo);
        // upload once the slot's previous permute has read it
        if (c >= slots && cudaStreamWaitEvent(ds->up, ds->permuted[b], 0) != cudaSuccess) return LC_ERR_CUDA;
        if (c >= slots && cudaStreamWaitEvent(ds->up, ds->downloaded[b], 0) != cudaSuccess) return LC_ERR_CUDA;
        if (cudaMemcpyAsync(s_dev, sh + s.lo, size_t(s.hi - s.lo), cudaMemcpyHostToDevice, ds->up) != cudaSuccess)
            return LC_ERR_CUDA;
        if (!dst_dense &&
            cudaMemcpyAsync(d_dev, dh + d.lo, size_t(d.hi - d.lo), cudaMemcpyHostToDevice, ds->up) != cudaSuccess)
            return LC_ERR_CUDA;
        if (cudaEventRecord(ds->uploaded[b], ds->up) != cudaSuccess) return LC_ERR_CUDA;
        // permute the chunk: the same layouts; each staging copy starts exactly
        // at the chunk's first tile, so both bases are 0
        lc_tile_layout sl = *src_layout, dl = *dst_layout;
        sl.offset = 0;
        dl.offset = 0;
        sl.tile_stride = sts;
        dl.tile_stride = dts;
        if (cudaStreamWaitEvent(cs, ds->uploaded[b], 0) != cudaSuccess) return LC_ERR_CUDA;
        Plan p;
        PtrInfo ptr;
        ptr.src = reinterpret_cast<uintptr_t>(s_dev);
        ptr.dst = reinterpret_cast<uintptr_t>(d_dev);
        ptr.check = true;
        st = make_plan(&sl, &dl, elem_bytes, t1 - t0, LC_KERNEL_AUTO, ptr, &p);
        if (st) return st;
        if ((st = launch_plan(p, s_dev, d_dev, cs, true))) return st;
        if (cudaEventRecord(ds->permuted[b], cs) != cudaSuccess) return LC_ERR_CUDA;
        // download once permuted
        if (cudaStreamWaitEvent(ds->down, ds->permuted[b], 0) != cudaSuccess) return LC_ERR_CUDA;
        if (cudaMemcpyAsync(dh + d.lo, d_dev, size_t(d.hi - d.lo), cudaMemcpyDeviceToHost, ds->down) != cudaSuccess)
            return LC_ERR_CUDA;
        if (cudaEventRecord(ds->downloaded[b], ds->down) != cudaSuccess) return LC_ERR_CUDA;
    }
    // the caller's stream resumes after the last download
    for (int b = 0; b < slots && b < c; ++b)
        if (cudaStreamWaitEvent(cs, ds->downloaded[b], 0) != cudaSuccess) return LC_ERR_CUDA;
    return LC_OK;
}

extern "C" int64_t lc_host_staging_bytes(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout,
                                         int32_t elem_bytes, int64_t n_tiles) {
    using namespace lc;
    if (!src_layout || !dst_layout || n_tiles <= 0) return 0;
    const HostSides hs = host_sides(*src_layout, *dst_layout, elem_bytes, n_tiles);
    if (n_tiles > 1 && hs.dts >= hs.dcos)
        return kSlots * hs.slot_bytes(default_chunk(n_tiles, std::max<int64_t>(hs.sts, hs.scos), hs.w));
    return hs.slot_bytes(n_tiles);
}
