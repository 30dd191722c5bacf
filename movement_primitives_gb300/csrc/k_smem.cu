// Shared-memory tile transpose for any alignment: the two global <-> shared
// copies of Apache TVM docs "copy -> gmem_smem" around a swizzled shared tile.
//
// A CTA moves square tiles, 64 x 64 words for words of up to 4 bytes and
// 32 x 32 for 8- and 16-byte words (X = the destination's contiguous mode,
// Y = the source's).  Copy 1 (global -> shared): thread t, round f takes
// flat index f * T + t of the tile in source order (y fastest), so a warp
// reads 32 consecutive source words, and every thread issues all its loads
// before its shared stores.  Copy 2 (shared -> global): the same split in
// destination order (x fastest), so a warp writes 32 consecutive destination
// words.  The shared tile is row-major [x][y] with the column swizzled,
//     y' = y ^ (((x >> shift) & mask) * granule),
// a swizzled shared layout as the page describes ("routes s_off through the
// swizzle", which caps the vector to one word here); the host bank simulator
// picks (shift, mask) so that both copies are conflict-free.  Words move one
// at a time, so no alignment beyond the word size is needed; tiles on the
// ragged edge are guarded (the TileLang loop partition's guard).
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

constexpr int kSmemThreads = 256;

template <int W> struct SmemCfg {
    static constexpr int TILE = smem_tile_words(W);
    static constexpr int ROUNDS = TILE * TILE / kSmemThreads;
};

struct SmemArgs {
    const uint8_t *src;  // address of source word offset 0
    uint8_t *dst;
    int64_t eX, eY;      // extents
    int64_t sX, dY;      // source stride of X, destination stride of Y (bytes)
    int32_t nb;          // batch modes, outermost first (bytes strides)
    int64_t be[kMaxModes], bs[kMaxModes], bd[kMaxModes];
    int64_t tiles_x, tiles_y, n_tiles;
    int32_t shift, mask, granule;
};

// Tile ti -> source / destination bases and the tile's origin and extent.
struct TileRef {
    const uint8_t *s;
    uint8_t *d;
    int64_t x0, y0;
    int nx, ny;
};

template <int TILE>
__device__ __forceinline__ TileRef tile_ref(const SmemArgs &a, int64_t ti) {
    const int64_t ty = ti % a.tiles_y, rest = ti / a.tiles_y;  // Y-block fastest
    const int64_t tx = rest % a.tiles_x;
    int64_t b = rest / a.tiles_x;
    TileRef r{a.src, a.dst, tx * TILE, ty * TILE, 0, 0};
    for (int k = a.nb - 1; k >= 0; --k) {
        const int64_t c = b % a.be[k];
        b /= a.be[k];
        r.s += c * a.bs[k];
        r.d += c * a.bd[k];
    }
    r.nx = static_cast<int>(lmin(TILE, a.eX - r.x0));
    r.ny = static_cast<int>(lmin(TILE, a.eY - r.y0));
    return r;
}

// Copy 1's global half: this thread's words of tile r, all loads issued.
template <int W, int TILE, int ROUNDS, typename T>
__device__ __forceinline__ void tile_load(const SmemArgs &a, const TileRef &r, T (&v)[ROUNDS]) {
#pragma unroll
    for (int f = 0; f < ROUNDS; ++f) {
        const int flat = f * kSmemThreads + threadIdx.x;
        const int x = flat / TILE, y = flat % TILE;
        if (x < r.nx && y < r.ny) v[f] = *reinterpret_cast<const T *>(r.s + (r.x0 + x) * a.sX + (r.y0 + y) * W);
    }
}

// The CTA walks tiles ti = blockIdx.x + i * gridDim.x.  Tile i+1's loads are
// issued before tile i's shared -> global copy, so loads stay in flight
// while the previous tile drains.
template <int W>
__global__ void __launch_bounds__(kSmemThreads) k_smem_transpose(const __grid_constant__ SmemArgs a) {
    using T = typename Word<W>::T;
    constexpr int kSmemTile = SmemCfg<W>::TILE;
    constexpr int kRounds = SmemCfg<W>::ROUNDS;
    __shared__ __align__(16) T tile[kSmemTile][kSmemTile];
    const int t = threadIdx.x;
    int64_t ti = blockIdx.x;
    if (ti >= a.n_tiles) return;
    TileRef r = tile_ref<kSmemTile>(a, ti);
    T v[kRounds];
    tile_load<W, kSmemTile, kRounds>(a, r, v);
    for (; ti < a.n_tiles; ti += gridDim.x) {
        // copy 1's shared half: source order into the swizzled tile
#pragma unroll
        for (int f = 0; f < kRounds; ++f) {
            const int flat = f * kSmemThreads + t;
            const int x = flat / kSmemTile, y = flat % kSmemTile;
            if (x < r.nx && y < r.ny) tile[x][y ^ (((x >> a.shift) & a.mask) * a.granule)] = v[f];
        }
        __syncthreads();
        const TileRef cur = r;
        if (ti + gridDim.x < a.n_tiles) {  // next tile's loads, in flight during copy 2
            r = tile_ref<kSmemTile>(a, ti + gridDim.x);
            tile_load<W, kSmemTile, kRounds>(a, r, v);
        }
        // copy 2: shared -> global, destination order
#pragma unroll
        for (int f = 0; f < kRounds; ++f) {
            const int flat = f * kSmemThreads + t;
            const int y = flat / kSmemTile, x = flat % kSmemTile;
            if (x < cur.nx && y < cur.ny) {
                const int ys = y ^ (((x >> a.shift) & a.mask) * a.granule);
                *reinterpret_cast<T *>(cur.d + (cur.y0 + y) * a.dY + (cur.x0 + x) * W) = tile[x][ys];
            }
        }
        __syncthreads();
    }
}

namespace {

template <int W>
int launch_smem_t(const SmemArgs &a, cudaStream_t stream) {
    const void *fn = reinterpret_cast<const void *>(&k_smem_transpose<W>);
    int sms, per;
    if (prepare(fn, kSmemThreads, 0, 0, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t grid = lmin(a.n_tiles, int64_t(sms) * per);
    k_smem_transpose<W><<<static_cast<unsigned>(grid), kSmemThreads, 0, stream>>>(a);
    return finish_launch();
}

}  // namespace

int launch_smem(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    const TilePlan &tp = p.tile;
    const int w = p.w;
    SmemArgs a{};
    a.src = src + p.src_off * w;
    a.dst = dst + p.dst_off * w;
    a.eX = tp.X.e;
    a.eY = tp.Y.e;
    a.sX = tp.X.s * w;
    a.dY = tp.Y.d * w;
    a.nb = tp.batch.n;
    int64_t nbatch = 1;
    for (int i = 0; i < tp.batch.n; ++i) {
        a.be[i] = tp.batch.m[i].e;
        a.bs[i] = tp.batch.m[i].s * w;
        a.bd[i] = tp.batch.m[i].d * w;
        nbatch *= tp.batch.m[i].e;
    }
    const int tile = smem_tile_words(w);
    a.tiles_x = (tp.X.e + tile - 1) / tile;
    a.tiles_y = (tp.Y.e + tile - 1) / tile;
    a.n_tiles = a.tiles_x * a.tiles_y * nbatch;
    a.shift = p.smem_swz.shift;
    a.mask = p.smem_swz.mask;
    a.granule = p.smem_swz.granule;
    switch (w) {
        case 1: return launch_smem_t<1>(a, stream);
        case 2: return launch_smem_t<2>(a, stream);
        case 4: return launch_smem_t<4>(a, stream);
        case 8: return launch_smem_t<8>(a, stream);
        case 16: return launch_smem_t<16>(a, stream);
    }
    return LC_ERR_UNSUPPORTED;
}

}  // namespace lc
