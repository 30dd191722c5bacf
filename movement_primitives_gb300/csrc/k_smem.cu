// Shared-memory tile transpose for any alignment: the two global <-> shared
// copies of Apache TVM docs "copy -> gmem_smem" around a swizzled shared tile.
//
// X is the destination's contiguous mode, Y the source's.  A tile is TX
// source rows (x) by TYW words (y) (smem_geometry).  Row x of a tile is
// staged as RB bytes of aligned C-byte chunks (C = 4 bytes for words of up to
// 4 bytes, else the word size) starting at the chunk boundary at or below its
// word (x, y0); the bytes between that boundary and the word are the row's
// lead-in (0 .. C - w).  So rows of any alignment move in aligned chunks, and
// one- and two-byte words travel four bytes per load.
//
// Copy 1 (global -> shared): thread t loads chunk k = t % NC of rows
// t / NC + ROWS1 * g into registers, all loads issued before any is used,
// and stores chunk k of row x in slot k ^ ((x >> shift) & mask) of the row --
// the swizzled shared layout the page routes its shared offsets through; the
// host bank simulator picks (shift, mask) so that the chunk stores and the
// column reads of copy 2 are conflict-free.  Interior tiles whose rows lie
// inside the source's byte span load every chunk of every row; other tiles
// load only chunks that hold needed words, and a chunk that reaches outside
// the span is gathered byte by byte, so no byte outside the span is read.
//
// Copy 2 (shared -> global) is the [outer, threads, vec] split in destination
// order with vec = one word: thread t writes word x = t % TX of rows
// y0 + t / TX + STEP2 * f, a warp storing 32 consecutive destination words.
// Tiles on the ragged edge are guarded (the TileLang loop partition's guard).
//
// Addresses advance by constant strides per round, and the swizzle splits
// into a per-thread part and a per-round constant: the bits of the thread's
// first row and of the round's row offset are disjoint, and shift, mask and
// XOR distribute over them.  The CTA walks tiles blockIdx.x + i * gridDim.x
// (X-blocks fastest);
// tile i+1's loads are issued before tile i's copy 2, so they stay in flight
// while the previous tile drains.
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
    static constexpr SmemGeo G = smem_geometry(W);
    static constexpr int C = G.C, RB = G.RB, TX = G.TX, TYW = G.TYW;
    static constexpr int NC = RB / C;                // chunks per row
    static constexpr int ROWS1 = kSmemThreads / NC;  // rows per copy-1 round
    static constexpr int ROUNDS1 = TX / ROWS1;
    static constexpr int STEP2 = kSmemThreads / TX;  // rows of y per copy-2 round
    static constexpr int ROUNDS2 = TYW / STEP2;
    static_assert(kSmemThreads % NC == 0 && TX % ROWS1 == 0 && TYW % STEP2 == 0, "whole rounds");
    static_assert(C >= W && C % W == 0 && (C - W) + TYW * W <= RB, "a row holds its lead-in and TYW words");
};

struct SmemArgs {
    const uint8_t *src;  // address of source word offset 0
    uint8_t *dst;
    uintptr_t lo, hi;    // the source's byte span: only [lo, hi) is read
    int64_t eX, eY;      // extents
    int64_t sX, dY;      // source stride of X, destination stride of Y (bytes)
    int32_t nb;          // batch modes, outermost first (byte strides)
    int64_t bs[kMaxModes], bd[kMaxModes];
    FastDiv be[kMaxModes];  // batch extents
    FastDiv tiles_x, tiles_y;
    uint32_t n_tiles;
    int32_t shift, mask;
};

// Tile ti -> addresses of its word (x0, y0) on both sides, its extent, and
// whether it is whole (full extent, every staged chunk inside the span).
struct TileRef {
    uintptr_t s;
    uint8_t *d;
    int nx, ny;
    bool whole;
};

// Tile visiting order: 1 = X-block (destination row segment) fastest, so
// that tiles sharing the partly written 32-byte sectors at the ends of each
// destination row segment run close together; 0 = Y-block fastest.  Odd
// destination strides leave such sectors at both ends of every segment; with
// the X-block fastest they are completed in L2 before they leave it.
// Measured on GB300 (8191 x 8193): 1-, 2-, 4-, 8-byte words 36 -> 48 %,
// 49 -> 70 %, 77 -> 85 %, 90 -> 95 % of the copy peak against Y-block fastest.
#ifndef LC_SMEM_X_FASTEST
#define LC_SMEM_X_FASTEST 1
#endif

template <int W>
__device__ __forceinline__ TileRef tile_ref(const SmemArgs &a, uint32_t ti) {
    using G = SmemCfg<W>;
#if LC_SMEM_X_FASTEST
    const uint32_t rest = fast_div(ti, a.tiles_x);
    const uint32_t tx = ti - rest * a.tiles_x.d;
    uint32_t b = fast_div(rest, a.tiles_y);
    const uint32_t ty = rest - b * a.tiles_y.d;
#else
    const uint32_t rest = fast_div(ti, a.tiles_y);  // Y-block fastest
    const uint32_t ty = ti - rest * a.tiles_y.d;
    uint32_t b = fast_div(rest, a.tiles_x);
    const uint32_t tx = rest - b * a.tiles_x.d;
#endif
    const int64_t x0 = int64_t(tx) * G::TX, y0 = int64_t(ty) * G::TYW;
    const uint8_t *s = a.src + x0 * a.sX + y0 * W;
    uint8_t *d = a.dst + y0 * a.dY + x0 * W;
    for (int k = a.nb - 1; k >= 0; --k) {
        const uint32_t q = fast_div(b, a.be[k]);
        const uint32_t c = b - q * a.be[k].d;
        b = q;
        s += int64_t(c) * a.bs[k];
        d += int64_t(c) * a.bd[k];
    }
    TileRef r{reinterpret_cast<uintptr_t>(s), d, static_cast<int>(lmin(G::TX, a.eX - x0)),
              static_cast<int>(lmin(G::TYW, a.eY - y0)), false};
    r.whole = r.nx == G::TX && r.ny == G::TYW;
    if constexpr (G::C > W) {
        constexpr uintptr_t kAlign = ~uintptr_t(G::C - 1);
        const uintptr_t first = r.s & kAlign;
        const uintptr_t last = ((r.s + uintptr_t((G::TX - 1) * a.sX)) & kAlign) + G::RB;
        r.whole = r.whole && first >= a.lo && last <= a.hi;
    }
    return r;
}

// The four bytes of the chunk at c that lie inside [lo, hi), zero elsewhere.
__device__ __forceinline__ uint32_t gather_chunk(const SmemArgs &a, uintptr_t c) {
    uint32_t u = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b)
        if (c + b >= a.lo && c + b < a.hi) u |= uint32_t(*reinterpret_cast<const uint8_t *>(c + b)) << (8 * b);
    return u;
}

// Copy 1's global half: chunk k of this thread's rows xr + ROWS1 * g.
template <int W, bool WHOLE, typename CW, int ROUNDS>
__device__ __forceinline__ void load_chunks(const SmemArgs &a, const TileRef &r, int k, int xr, CW (&v)[ROUNDS]) {
    using G = SmemCfg<W>;
    constexpr int C = G::C;
    uintptr_t A = r.s + uintptr_t(xr * a.sX);  // word (x, y0) of the row
    const uintptr_t step = uintptr_t(G::ROWS1 * a.sX);
#pragma unroll
    for (int g = 0; g < ROUNDS; ++g, A += step) {
        const uintptr_t c = (C > W ? (A & ~uintptr_t(C - 1)) : A) + uintptr_t(k) * C;
        if (WHOLE) {
            v[g] = *reinterpret_cast<const CW *>(c);
        } else if (xr + G::ROWS1 * g < r.nx && c < A + uintptr_t(r.ny) * W && c + C > A) {
            if constexpr (C > W) {
                if (c >= a.lo && c + C <= a.hi)
                    v[g] = *reinterpret_cast<const CW *>(c);
                else
                    v[g] = gather_chunk(a, c);
            } else {
                v[g] = *reinterpret_cast<const CW *>(c);
            }
        }
    }
}

// Copy 2: thread t writes word x = t % TX of rows y0 + t / TX + STEP2 * f.
template <int W, bool FULL>
__device__ __forceinline__ void copy_out(const SmemArgs &a, const TileRef &r, const uint8_t *row, int x, int ly,
                                         int swc) {
    using G = SmemCfg<W>;
    using T = typename Word<W>::T;
    if (!FULL && x >= r.nx) return;
    const int lead = G::C > W ? static_cast<int>((r.s + uintptr_t(x * a.sX)) & (G::C - 1)) : 0;
    const int p0 = lead + ly * W;  // byte of word (x, y0 + ly) in the staged row
    uint8_t *q = r.d + ly * a.dY + x * W;
    const int64_t step = int64_t(G::STEP2) * a.dY;
#pragma unroll
    for (int f = 0; f < G::ROUNDS2; ++f, q += step)
        if (FULL || ly + G::STEP2 * f < r.ny)
            store_out<T>(q, *reinterpret_cast<const T *>(row + ((p0 + G::STEP2 * W * f) ^ swc)));
}

template <int W>
__global__ void __launch_bounds__(kSmemThreads, SmemCfg<W>::MIN_BLOCKS)
    k_smem_transpose(const __grid_constant__ SmemArgs a) {
    using G = SmemCfg<W>;
    using CW = typename Word<G::C>::T;
    __shared__ __align__(16) uint8_t tile[G::TX * G::RB];
    const int t = threadIdx.x;
    const int shift = a.shift, mask = a.mask;
    // copy 1: chunk k of rows xr + ROWS1 g, slot k ^ sw(xr) ^ sw(ROWS1 g)
    const int k = t % G::NC, xr = t / G::NC;
    const int slot0 = k ^ ((xr >> shift) & mask);
    uint8_t *const wrow = tile + xr * G::RB;
    // copy 2: word x of the staged rows, chunk slots XORed with sw(x)
    const int x2 = t % G::TX, ly = t / G::TX;
    const uint8_t *const rrow = tile + x2 * G::RB;
    const int swc = ((x2 >> shift) & mask) * G::C;

    uint32_t ti = blockIdx.x;
    if (ti >= a.n_tiles) return;
    TileRef r = tile_ref<W>(a, ti);
    CW v[G::ROUNDS1];
    if (r.whole)
        load_chunks<W, true>(a, r, k, xr, v);
    else
        load_chunks<W, false>(a, r, k, xr, v);
    for (; ti < a.n_tiles; ti += gridDim.x) {
        // copy 1's shared half (slots of chunks that were not loaded are
        // written but never read back)
#pragma unroll
        for (int g = 0; g < G::ROUNDS1; ++g) {
            const int slot = slot0 ^ (((G::ROWS1 * g) >> shift) & mask);
            *reinterpret_cast<CW *>(wrow + G::ROWS1 * g * G::RB + slot * G::C) = v[g];
        }
        __syncthreads();
        const TileRef cur = r;
        if (ti + gridDim.x < a.n_tiles) {  // next tile's loads, in flight during copy 2
            r = tile_ref<W>(a, ti + gridDim.x);
            if (r.whole)
                load_chunks<W, true>(a, r, k, xr, v);
            else
                load_chunks<W, false>(a, r, k, xr, v);
        }
        if (cur.nx == G::TX && cur.ny == G::TYW)
            copy_out<W, true>(a, cur, rrow, x2, ly, swc);
        else
            copy_out<W, false>(a, cur, rrow, x2, ly, swc);
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
    const SmemGeo g = smem_geometry(w);
    SmemArgs a{};
    a.src = src + p.src_off * w;
    a.dst = dst + p.dst_off * w;
    a.lo = reinterpret_cast<uintptr_t>(src) + uintptr_t(p.src_lo);
    a.hi = reinterpret_cast<uintptr_t>(src) + uintptr_t(p.src_hi);
    a.eX = tp.X.e;
    a.eY = tp.Y.e;
    a.sX = tp.X.s * w;
    a.dY = tp.Y.d * w;
    a.nb = tp.batch.n;
    int64_t nbatch = 1;
    for (int i = 0; i < tp.batch.n; ++i) {
        if (tp.batch.m[i].e >= (int64_t(1) << 31)) return LC_ERR_UNSUPPORTED;
        a.be[i] = make_fastdiv(static_cast<uint32_t>(tp.batch.m[i].e));
        a.bs[i] = tp.batch.m[i].s * w;
        a.bd[i] = tp.batch.m[i].d * w;
        nbatch *= tp.batch.m[i].e;
    }
    const int64_t tx = (tp.X.e + g.TX - 1) / g.TX, ty = (tp.Y.e + g.TYW - 1) / g.TYW;
    if (tx >= (int64_t(1) << 31) || ty >= (int64_t(1) << 31)) return LC_ERR_UNSUPPORTED;
    const int64_t n_tiles = tx * ty * nbatch;
    if (n_tiles >= (int64_t(1) << 31)) return LC_ERR_UNSUPPORTED;  // the planner keeps it below
    a.tiles_x = make_fastdiv(static_cast<uint32_t>(tx));
    a.tiles_y = make_fastdiv(static_cast<uint32_t>(ty));
    a.n_tiles = static_cast<uint32_t>(n_tiles);
    a.shift = p.smem_swz.shift;
    a.mask = p.smem_swz.mask;
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
