// Shared-memory tile transpose for any alignment: the two global <-> shared
// copies of Apache TVM docs "copy -> gmem_smem" around a swizzled shared tile.
//
// A CTA moves square tiles, 64 x 64 words for words of up to 8 bytes and
// 32 x 32 for 16-byte words (X = the destination's contiguous mode,
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
//
// Address arithmetic per word is a constant-stride step.  With STEP = T / TILE
// rows per round, thread t always has column ly = t % TILE and first row
// lx = t / TILE < STEP, and round f adds STEP * f to the row.  The row's bits
// and lx's bits are disjoint, so the swizzle splits into a per-thread part and
// a per-round constant: sw(lx + STEP f) = sw(lx) ^ sw(STEP f) (shift, mask and
// the power-of-two granule all distribute over XOR).  Global addresses advance
// by STEP source (destination) rows per round; the tile's origin is decoded
// once per tile with invariant-divisor division.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "launch.h"

namespace lc {

constexpr int kSmemThreads = 256;

// Resident CTAs per SM the register allocation must allow (compile-time knobs
// so that variants can be measured).  Measured on GB300 on an 8191 x 8193
// transpose: fewer registers than these make the compiler split each thread's
// loads into dependent batches, which costs more than the extra CTAs gain.
#ifndef LC_SMEM_MIN_BLOCKS_W1
#define LC_SMEM_MIN_BLOCKS_W1 4
#endif
#ifndef LC_SMEM_MIN_BLOCKS_W2
#define LC_SMEM_MIN_BLOCKS_W2 3
#endif
#ifndef LC_SMEM_MIN_BLOCKS_W4
#define LC_SMEM_MIN_BLOCKS_W4 3
#endif
#ifndef LC_SMEM_MIN_BLOCKS_WIDE
#define LC_SMEM_MIN_BLOCKS_WIDE 2
#endif

template <int W> struct SmemCfg {
    static constexpr int MIN_BLOCKS = W == 1 ? LC_SMEM_MIN_BLOCKS_W1 : W == 2 ? LC_SMEM_MIN_BLOCKS_W2
                                    : W == 4 ? LC_SMEM_MIN_BLOCKS_W4 : LC_SMEM_MIN_BLOCKS_WIDE;
    static constexpr int TILE = smem_tile_words(W);
    static constexpr int ROUNDS = TILE * TILE / kSmemThreads;
    static constexpr int STEP = kSmemThreads / TILE;  // rows per round
};

struct SmemArgs {
    const uint8_t *src;  // address of source word offset 0
    uint8_t *dst;
    int64_t eX, eY;      // extents
    int64_t sX, dY;      // source stride of X, destination stride of Y (bytes)
    int32_t nb;          // batch modes, outermost first (byte strides)
    int64_t bs[kMaxModes], bd[kMaxModes];
    FastDiv be[kMaxModes];  // batch extents
    FastDiv tiles_x, tiles_y;
    uint32_t n_tiles;
    int32_t shift, mask, granule;
};

// Tile ti -> source / destination addresses of its origin, and its extent.
struct TileRef {
    const uint8_t *s;
    uint8_t *d;
    int nx, ny;
};

template <int TILE>
__device__ __forceinline__ TileRef tile_ref(const SmemArgs &a, uint32_t ti, int W) {
    const uint32_t rest = fast_div(ti, a.tiles_y);  // Y-block fastest
    const uint32_t ty = ti - rest * a.tiles_y.d;
    uint32_t b = fast_div(rest, a.tiles_x);
    const uint32_t tx = rest - b * a.tiles_x.d;
    const int64_t x0 = int64_t(tx) * TILE, y0 = int64_t(ty) * TILE;
    TileRef r{a.src + x0 * a.sX + y0 * W, a.dst + y0 * a.dY + x0 * W, 0, 0};
    for (int k = a.nb - 1; k >= 0; --k) {
        const uint32_t q = fast_div(b, a.be[k]);
        const uint32_t c = b - q * a.be[k].d;
        b = q;
        r.s += int64_t(c) * a.bs[k];
        r.d += int64_t(c) * a.bd[k];
    }
    r.nx = static_cast<int>(lmin(TILE, a.eX - x0));
    r.ny = static_cast<int>(lmin(TILE, a.eY - y0));
    return r;
}

// Copy 1's global half: this thread's words of tile r (rows lx + STEP f,
// column ly), all loads issued before any is used.
template <int W, bool FULL, typename T, int ROUNDS>
__device__ __forceinline__ void tile_load(const SmemArgs &a, const TileRef &r, int lx, int ly, T (&v)[ROUNDS]) {
    constexpr int STEP = SmemCfg<W>::STEP;
    const uint8_t *p = r.s + lx * a.sX + ly * W;
    const int64_t step = STEP * a.sX;
    if (FULL) {
#pragma unroll
        for (int f = 0; f < ROUNDS; ++f, p += step) v[f] = *reinterpret_cast<const T *>(p);
    } else if (ly < r.ny) {
#pragma unroll
        for (int f = 0; f < ROUNDS; ++f, p += step)
            if (lx + STEP * f < r.nx) v[f] = *reinterpret_cast<const T *>(p);
    }
}

// The CTA walks tiles ti = blockIdx.x + i * gridDim.x.  Tile i+1's loads are
// issued before tile i's shared -> global copy, so loads stay in flight
// while the previous tile drains.
template <int W>
__global__ void __launch_bounds__(kSmemThreads, SmemCfg<W>::MIN_BLOCKS) k_smem_transpose(const __grid_constant__ SmemArgs a) {
    using T = typename Word<W>::T;
    constexpr int TILE = SmemCfg<W>::TILE;
    constexpr int ROUNDS = SmemCfg<W>::ROUNDS;
    constexpr int STEP = SmemCfg<W>::STEP;
    __shared__ __align__(16) uint8_t tile[TILE * TILE * W];
    const int t = threadIdx.x;
    const int lx = t / TILE, ly = t % TILE;
    const int shift = a.shift, mask = a.mask, g = a.granule;
    // copy 1: row lx + STEP f, column ly ^ sw(lx) ^ sw(STEP f)
    uint8_t *const wrow = tile + lx * TILE * W;
    const int c1 = ly ^ (((lx >> shift) & mask) * g);
    // copy 2: row ly, column (lx + STEP f) ^ sw(ly) = c2 ^ STEP f
    const uint8_t *const rrow = tile + ly * TILE * W;
    const int c2 = lx ^ (((ly >> shift) & mask) * g);

    uint32_t ti = blockIdx.x;
    if (ti >= a.n_tiles) return;
    TileRef r = tile_ref<TILE>(a, ti, W);
    bool full = r.nx == TILE && r.ny == TILE;
    T v[ROUNDS];
    if (full)
        tile_load<W, true>(a, r, lx, ly, v);
    else
        tile_load<W, false>(a, r, lx, ly, v);
    for (; ti < a.n_tiles; ti += gridDim.x) {
        // copy 1's shared half (cells outside a ragged tile are written but
        // never read back)
#pragma unroll
        for (int f = 0; f < ROUNDS; ++f) {
            const int col = c1 ^ ((((STEP * f) >> shift) & mask) * g);
            *reinterpret_cast<T *>(wrow + (STEP * f * TILE + col) * W) = v[f];
        }
        __syncthreads();
        const TileRef cur = r;
        const bool cur_full = full;
        if (ti + gridDim.x < a.n_tiles) {  // next tile's loads, in flight during copy 2
            r = tile_ref<TILE>(a, ti + gridDim.x, W);
            full = r.nx == TILE && r.ny == TILE;
            if (full)
                tile_load<W, true>(a, r, lx, ly, v);
            else
                tile_load<W, false>(a, r, lx, ly, v);
        }
        // copy 2: shared -> global, destination order (row lx + STEP f, column ly)
        uint8_t *q = cur.d + lx * a.dY + ly * W;
        const int64_t step = STEP * a.dY;
        if (cur_full) {
#pragma unroll
            for (int f = 0; f < ROUNDS; ++f, q += step)
                *reinterpret_cast<T *>(q) = *reinterpret_cast<const T *>(rrow + (c2 ^ (STEP * f)) * W);
        } else if (ly < cur.nx) {
#pragma unroll
            for (int f = 0; f < ROUNDS; ++f, q += step)
                if (lx + STEP * f < cur.ny)
                    *reinterpret_cast<T *>(q) = *reinterpret_cast<const T *>(rrow + (c2 ^ (STEP * f)) * W);
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
        a.be[i] = make_fastdiv(static_cast<uint32_t>(tp.batch.m[i].e));
        a.bs[i] = tp.batch.m[i].s * w;
        a.bd[i] = tp.batch.m[i].d * w;
        nbatch *= tp.batch.m[i].e;
    }
    const int tile = smem_tile_words(w);
    const int64_t tx = (tp.X.e + tile - 1) / tile, ty = (tp.Y.e + tile - 1) / tile;
    const int64_t n_tiles = tx * ty * nbatch;
    if (n_tiles >= (int64_t(1) << 31)) return LC_ERR_UNSUPPORTED;  // the planner keeps it below
    a.tiles_x = make_fastdiv(static_cast<uint32_t>(tx));
    a.tiles_y = make_fastdiv(static_cast<uint32_t>(ty));
    a.n_tiles = static_cast<uint32_t>(n_tiles);
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
