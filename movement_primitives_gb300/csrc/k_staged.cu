// Staged tile copy: the demonstration program of Apache TVM docs "copy ->
// gmem_smem" (a tile copied global -> shared, a CTA barrier, shared ->
// global) as a copy between two layouts.  One CTA stages one tile at a time:
// copy 1 moves the tile into a shared buffer holding its logical box
// row-major, the source layout driving the [outer, threads, vec] order;
// copy 2 moves it out, the destination layout driving.  Both copies are
// lc_device::gmem_smem_copy with their own partitions (guarded when the
// thread count does not divide the tile), through one shared-memory XOR
// swizzle chosen so that both copies' shared accesses are as free of bank
// conflicts as the simulator finds.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <string>

#include "device_common.cuh"
#include "launch.h"
#include "layout_copy_device.cuh"

// 0: the library's choice of shared swizzle is none (a variant for measuring
// what the swizzle buys).
#ifndef LC_STAGED_SWIZZLE
#define LC_STAGED_SWIZZLE 1
#endif

namespace lc {
namespace {

struct StagedArgs {
    const uint8_t *src;
    uint8_t *dst;
    lc_gmem_smem in, out;  // copy 1 (global = source), copy 2 (global = destination)
    int64_t sts, dts;      // tile strides, bytes
    int64_t n_tiles, N;
    int64_t *trace_in, *trace_out;
};

template <int W>
__global__ void __launch_bounds__(1024) k_staged(const __grid_constant__ StagedArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
        lc_device::gmem_smem_copy<W>(a.in, const_cast<uint8_t *>(a.src) + t * a.sts, smem, threadIdx.x, true,
                                     a.trace_in ? a.trace_in + t * a.N : nullptr);
        __syncthreads();
        lc_device::gmem_smem_copy<W>(a.out, a.dst + t * a.dts, smem, threadIdx.x, false,
                                     a.trace_out ? a.trace_out + t * a.N : nullptr);
        __syncthreads();
    }
}

// Shared byte addresses of one warp's accesses (lanes tid0 .. tid0 + 31 in
// round f) of a planned copy, through the swizzle; -1 for guarded lanes.
void warp_shared_addrs(const lc_gmem_smem &p, int64_t f, int tid0, int64_t *addr) {
    for (int l = 0; l < 32; ++l) {
        const int64_t first = (f * p.threads + tid0 + l) * p.vec;
        if (tid0 + l >= p.threads || first >= p.total) { addr[l] = -1; continue; }
        int64_t rest = first, s = p.s_offset;
        for (int i = p.n_modes - 1; i >= 0; --i) {
            s += (rest % p.extent[i]) * p.s_stride[i];
            rest /= p.extent[i];
        }
        const uint64_t o = uint64_t(s) * uint64_t(p.elem_bytes);
        const lc_smem_swizzle &z = p.swizzle;
        addr[l] = int64_t(o ^ (((o >> z.row_log2) & ((uint64_t(1) << z.bits) - 1)) << z.chunk_log2));
    }
}

// Worst bank degree over (up to) the first 64 warp accesses of a copy.
int copy_degree(const lc_gmem_smem &p) {
    int worst = 0, seen = 0;
    for (int64_t f = 0; f < p.outer && seen < 64; ++f)
        for (int t0 = 0; t0 < p.threads && seen < 64; t0 += 32, ++seen) {
            int64_t addr[32];
            warp_shared_addrs(p, f, t0, addr);
            int64_t live[32];
            int n = 0;
            for (int l = 0; l < 32; ++l)
                if (addr[l] >= 0) live[n++] = addr[l];
            for (int l = n; l < 32; ++l) live[l] = live[0];  // idle lanes repeat a live address
            if (n) worst = std::max(worst, access_degree_vec(live, p.vec * p.elem_bytes));
        }
    return worst;
}

std::mutex g_swz_mu;
std::map<std::string, lc_smem_swizzle> g_swz;  // layouts, width, threads -> chosen swizzle

}  // namespace

// Swizzle for a staged tile: among the candidates with the widest vectors
// (the sum of the two copies' vector widths: global access width decides
// more than shared bank degree -- on 65536 32 x 32 fp32 transposes a swizzle
// of 4-byte chunks took the shared load wavefronts from 68.9 M to 2.2 M but
// capped copy 1 at one word per access and ran at 543 against 362 us), the
// one whose worse copy has the lowest bank degree, then the simplest.
int choose_staged_swizzle(const lc_tile_layout &s, const lc_tile_layout &d, const lc_tile_layout &sh, int w,
                          int threads, lc_smem_swizzle *out) {
    std::string key;
    auto put = [&key](const void *p, size_t n) { key.append(static_cast<const char *>(p), n); };
    for (const lc_tile_layout *l : {&s, &d, &sh}) {  // field by field: the struct has padding
        put(&l->rank, sizeof(l->rank));
        put(l->shape, sizeof(int64_t) * size_t(l->rank));
        put(l->stride, sizeof(int64_t) * size_t(l->rank));
        put(&l->offset, sizeof(l->offset));
    }
    put(&w, sizeof(w));
    put(&threads, sizeof(threads));
    {
        std::lock_guard<std::mutex> lk(g_swz_mu);
        auto it = g_swz.find(key);
        if (it != g_swz.end()) { *out = it->second; return LC_OK; }
    }
    int best_deg = 1 << 30, best_vec = -1;
    lc_smem_swizzle best{0, 0, 0};
    int c0 = 0;
    while ((1 << c0) < std::max(w, 4)) ++c0;
    for (int bits = 0; bits <= 5; ++bits)
        for (int c = bits ? c0 : 0; c <= (bits ? 4 : 0); ++c)
            for (int r = bits ? c + bits : 0; r <= (bits ? 12 : 0); ++r) {
                const lc_smem_swizzle z{bits, c, r};
                lc_gmem_smem pi, po;
                if (lc_gmem_smem_plan(&s, &sh, w, threads, &z, &pi) != LC_OK) continue;
                if (lc_gmem_smem_plan(&d, &sh, w, threads, &z, &po) != LC_OK) continue;
                const int deg = std::max(copy_degree(pi), copy_degree(po));
                const int vec = pi.vec + po.vec;
                if (vec > best_vec || (vec == best_vec && deg < best_deg)) {
                    best_deg = deg;
                    best_vec = vec;
                    best = z;
                }
            }
    if (best_vec < 0) return LC_ERR_SHAPE;
    std::lock_guard<std::mutex> lk(g_swz_mu);
    if (g_swz.size() > 256) g_swz.clear();
    g_swz[key] = best;
    *out = best;
    return LC_OK;
}

}  // namespace lc

namespace lc {

// The launch behind lc_layout_copy_staged and the LC_KERNEL_SMEM_STAGED
// class; layouts, pointers and counts already validated.
int launch_staged_layouts(const void *src, const lc_tile_layout *src_layout, void *dst,
                          const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles, int32_t threads,
                          const lc_smem_swizzle *swizzle, int64_t *trace_in, int64_t *trace_out,
                          cudaStream_t cs) {
    PtrInfo ptr;
    ptr.src = reinterpret_cast<uintptr_t>(src);
    ptr.dst = reinterpret_cast<uintptr_t>(dst);
    int st = LC_OK;
    const int64_t w = elem_bytes;
    int64_t N = 1;
    for (int k = 0; k < src_layout->rank; ++k) N *= src_layout->shape[k];
    if (N * w > LC_STAGED_MAX_BYTES) return LC_ERR_SHAPE;
    // the shared tile: the logical box row-major
    lc_tile_layout sh{};
    sh.rank = src_layout->rank;
    int64_t acc = 1;
    for (int k = sh.rank - 1; k >= 0; --k) {
        sh.shape[k] = src_layout->shape[k];
        sh.stride[k] = acc;
        acc *= std::max<int64_t>(1, src_layout->shape[k]);
    }
    lc_smem_swizzle z{0, 0, 0};
    if (swizzle) z = *swizzle;
    else if (LC_STAGED_SWIZZLE &&
             (st = choose_staged_swizzle(*src_layout, *dst_layout, sh, elem_bytes, threads, &z)))
        return st;
    StagedArgs a{};
    if ((st = lc_gmem_smem_plan(src_layout, &sh, elem_bytes, threads, &z, &a.in))) return st;
    if ((st = lc_gmem_smem_plan(dst_layout, &sh, elem_bytes, threads, &z, &a.out))) return st;
    // Tile strides and base pointers must keep every vector aligned; a
    // vector wider than that is narrowed to single elements.
    const int64_t sts = (src_layout->tile_stride ? src_layout->tile_stride : cosize_of(*src_layout)) * w;
    const int64_t dts = (dst_layout->tile_stride ? dst_layout->tile_stride : cosize_of(*dst_layout)) * w;
    auto aligned = [&](uintptr_t p, int64_t ts, int64_t vb) {
        return p % uintptr_t(vb) == 0 && (n_tiles == 1 || ts % vb == 0);
    };
    if (!aligned(ptr.src, sts, a.in.vec * w)) {
        a.in.vec = 1;
        a.in.outer = (a.in.total + threads - 1) / threads;
        a.in.guarded = a.in.total % threads != 0;
    }
    if (!aligned(ptr.dst, dts, a.out.vec * w)) {
        a.out.vec = 1;
        a.out.outer = (a.out.total + threads - 1) / threads;
        a.out.guarded = a.out.total % threads != 0;
    }
    a.src = static_cast<const uint8_t *>(src);
    a.dst = static_cast<uint8_t *>(dst);
    a.sts = sts;
    a.dts = dts;
    a.n_tiles = n_tiles;
    a.N = N;
    a.trace_in = trace_in;
    a.trace_out = trace_out;
    // the swizzle only rewrites bits below chunk_log2 + bits: round the buffer
    // up to that span so that every stored offset stays inside it
    const int64_t span = std::max<int64_t>(z.bits ? (int64_t(1) << (z.chunk_log2 + z.bits)) : 16, 128);
    const int64_t smem_bytes = (N * w + span - 1) / span * span;
    if (smem_bytes > LC_STAGED_MAX_BYTES + 4096) return LC_ERR_SHAPE;  // a swizzle spanning past the tile budget
    const int smem = static_cast<int>(smem_bytes);
    const void *fn = nullptr;
    switch (elem_bytes) {
        case 1: fn = reinterpret_cast<const void *>(&k_staged<1>); break;
        case 2: fn = reinterpret_cast<const void *>(&k_staged<2>); break;
        case 4: fn = reinterpret_cast<const void *>(&k_staged<4>); break;
        case 8: fn = reinterpret_cast<const void *>(&k_staged<8>); break;
        default: fn = reinterpret_cast<const void *>(&k_staged<16>); break;
    }
    int sms, per;
    if (prepare(fn, threads, smem, LC_STAGED_MAX_BYTES + 4096, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const unsigned grid = static_cast<unsigned>(lmin(n_tiles, int64_t(sms) * per));
    switch (elem_bytes) {
        case 1: k_staged<1><<<grid, threads, smem, cs>>>(a); break;
        case 2: k_staged<2><<<grid, threads, smem, cs>>>(a); break;
        case 4: k_staged<4><<<grid, threads, smem, cs>>>(a); break;
        case 8: k_staged<8><<<grid, threads, smem, cs>>>(a); break;
        default: k_staged<16><<<grid, threads, smem, cs>>>(a); break;
    }
    return finish_launch();
}

int launch_staged(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    return launch_staged_layouts(src, &p.src_l, dst, &p.dst_l, p.w, p.n_tiles, kStagedThreads, nullptr, nullptr,
                                 nullptr, stream);
}

}  // namespace lc

extern "C" int lc_layout_copy_staged(const void *src, const lc_tile_layout *src_layout, void *dst,
                                     const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles,
                                     int32_t threads, const lc_smem_swizzle *swizzle, int64_t *trace_in,
                                     int64_t *trace_out, lc_stream_t stream) {
    using namespace lc;
    if (!src_layout || !dst_layout) return LC_ERR_NULL;
    if (threads < 32 || threads > 1024 || threads % 32) return LC_ERR_SHAPE;
    Plan p;
    PtrInfo ptr;
    ptr.src = reinterpret_cast<uintptr_t>(src);
    ptr.dst = reinterpret_cast<uintptr_t>(dst);
    ptr.check = true;
    const int st = make_plan(src_layout, dst_layout, elem_bytes, n_tiles, LC_KERNEL_SMEM_STAGED, ptr, &p);
    if (st) return st == LC_ERR_UNSUPPORTED ? LC_ERR_SHAPE : st;  // validation; no overlap is accepted
    if (p.total == 0) return LC_OK;
    return launch_staged_layouts(src, src_layout, dst, dst_layout, elem_bytes, n_tiles, threads, swizzle, trace_in,
                                 trace_out, reinterpret_cast<cudaStream_t>(stream));
}
