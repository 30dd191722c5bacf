// TMA tile transpose: tensor tiles in a shared-memory ring (mbarrier
// pipelined; 128- or 256-byte box rows), 16-byte shared reads, in-register
// transpose of the sub-16-byte words, 16-byte coalesced global stores.
//
// X is the mode contiguous in the destination, Y the one contiguous in the
// source; up to three batch modes ride along as extra tensor dimensions.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "device_common.cuh"
#include "launch.h"
#include "tensor_map.h"
#include "bulk_store.cuh"

namespace lc {

// Per-width tile geometry, measured on GB300 (A/B on one box, L2 flushed
// between launches): rows per TMA box, ring depth, and the visiting order.
// Every value is a compile-time knob so that variants can be measured.
#ifndef LC_TILE_ROWS_W1
#define LC_TILE_ROWS_W1 256
#endif
#ifndef LC_TILE_ROWS_W2
#define LC_TILE_ROWS_W2 256
#endif
#ifndef LC_TILE_ROWS_W4
#define LC_TILE_ROWS_W4 256
#endif
#ifndef LC_TILE_ROWS_W8
#define LC_TILE_ROWS_W8 128
#endif
#ifndef LC_TILE_ROWS_W16
#define LC_TILE_ROWS_W16 128
#endif
#ifndef LC_TILE_STAGES_W1
#define LC_TILE_STAGES_W1 2
#endif
#ifndef LC_TILE_STAGES_WIDE
#define LC_TILE_STAGES_WIDE 4
#endif
// 1: tiles visited Y-block (source column block) fastest, so CTAs running at
// the same time read neighbouring box-row segments of the same source rows;
// 0: X-block fastest.
#ifndef LC_TILE_Y_FASTEST
#define LC_TILE_Y_FASTEST 1
#endif
// 1: one thread waits on a stage's barrier and the CTA synchronises after it;
// 0: every thread waits on the barrier itself.
#ifndef LC_TILE_POLL_ONE
#define LC_TILE_POLL_ONE 0
#endif

// Bytes per TMA box row (128 or 256) and ring stages per width, measured on
// GB300: 256-byte rows with 3 stages move the 16384^2 bf16 transpose at
// 91.8 % (128-byte rows, 4 stages: 90.1 %) and the 8192^2 eight-byte one at
// 93.2 % (92.4 %); 1-byte words lose with them (61 % against 68 %), 4-byte
// words slightly (83.7 % against 84.6 %).
#ifndef LC_TILE_BOXB_W2
#define LC_TILE_BOXB_W2 256
#endif
#ifndef LC_TILE_BOXB_W8
#define LC_TILE_BOXB_W8 256
#endif
#ifndef LC_TILE_BOXB_OTHER
#define LC_TILE_BOXB_OTHER 128
#endif
#ifndef LC_TILE_STAGES_W2
#define LC_TILE_STAGES_W2 3
#endif
#ifndef LC_TILE_STAGES_W8
#define LC_TILE_STAGES_W8 3
#endif

// Shorter boxes for copies of at most LC_TILE_SHORT_MAX_BYTES a side, 1-,
// 2- and 4-byte words: measured on GB300 (L2 flushed by a read between
// launches), 128-row boxes move the 8192^2 transposes at 85 % (2-byte words,
// against 79 % with 256 rows) and 90 % (4-byte, against 85 %), while the
// 16384^2 2-byte transpose (512 MiB a side) drops from 91-92 % to 85-87 %.
#ifndef LC_TILE_SHORT_ROWS
#define LC_TILE_SHORT_ROWS 128
#endif
#ifndef LC_TILE_SHORT_MAX_BYTES
#define LC_TILE_SHORT_MAX_BYTES (256ll << 20)
#endif

#ifndef LC_TILE_BOXB_W1
#define LC_TILE_BOXB_W1 LC_TILE_BOXB_OTHER
#endif

// Box rows for 4-byte words on the short boxes when line stores are off:
// 256 bytes measured 90.5 % against 86.1 % with 128 (8192^2, 128-row boxes,
// 4 stages).
#ifndef LC_TILE_BOXB_W4_SHORT
#define LC_TILE_BOXB_W4_SHORT 256
#endif

// 1: on the short boxes of 1-, 2- and 4-byte words, micro-blocks are handed
// out so that one warp store writes whole 128-byte lines (8 row groups x 4
// chunks per warp: 4 destination rows x 128 bytes), over boxes of 128-byte
// rows; 0 (and everywhere else): 8 chunks x 4 row groups (8 destination rows
// x 64 bytes).  Measured on GB300 (8192^2 transposes, TMA ring, L2 flushed by
// a read): 1-byte words 86.7 % of the copy peak against 74.8-75.4 %, 2-byte
// 95.2-95.3 % against 87.5-87.9 %, 4-byte 90.8-91.1 % against 90.7-90.9 %;
// on 8- and 16-byte words (86.2 against 93.6 %, 85.2 against 92.4 %) and on
// the 16384^2 2-byte transpose (82.3 against 91.1-91.4 %) line stores lose.
#ifndef LC_TILE_LINE_STORES
#define LC_TILE_LINE_STORES 1
#endif
// 1: with line stores, the boxes land in shared memory under the TMA 128-byte
// swizzle (16-byte chunk k of row y at chunk k ^ (y & 7)), which makes the
// shared reads conflict-free (without it, two row groups of a quarter warp
// read the same banks: 93.6-94.0 % instead of 95.3 % for 2-byte words).
#ifndef LC_TILE_SWIZZLE
#define LC_TILE_SWIZZLE 1
#endif

// Threads per CTA at most (each takes one micro-block per round).  Measured
// on GB300 against 256: 512 for the 256-row boxes of 2-byte words (16384^2:
// 91.9 % against 91.1-91.4 %; 8-byte words lose 5 points with 512, 16-byte
// words 7), 128 for 16-byte words (8192^2: 93.2-93.3 % against 92.4-92.5 %;
// 4-, 8- and 2-byte words lose 0.7-1.4 points with 128).
#ifndef LC_TILE_MAX_THREADS
#define LC_TILE_MAX_THREADS 256
#endif
#ifndef LC_TILE_MAX_THREADS_W2_TALL
#define LC_TILE_MAX_THREADS_W2_TALL 512
#endif
#ifndef LC_TILE_MAX_THREADS_W16
#define LC_TILE_MAX_THREADS_W16 128
#endif

template <int W, bool SHORT = false> struct TileCfg {
    static constexpr bool LINES = LC_TILE_LINE_STORES != 0 && SHORT && W <= 4;
    static constexpr int BOXB = LINES    ? 128
                              : W == 1   ? LC_TILE_BOXB_W1
                              : W == 2   ? LC_TILE_BOXB_W2
                              : W == 4   ? (SHORT ? LC_TILE_BOXB_W4_SHORT : LC_TILE_BOXB_OTHER)
                              : W == 8   ? LC_TILE_BOXB_W8
                                         : LC_TILE_BOXB_OTHER;  // bytes per box row
    static constexpr int CPR = BOXB / 16;      // 16-byte chunks per box row
    static constexpr int V = 16 / W;           // words per 16-byte chunk
    static constexpr int TY = BOXB / W;        // words per box row
    static constexpr int R = SHORT ? LC_TILE_SHORT_ROWS
                           : W == 1 ? LC_TILE_ROWS_W1 : W == 2 ? LC_TILE_ROWS_W2 : W == 4 ? LC_TILE_ROWS_W4
                           : W == 8 ? LC_TILE_ROWS_W8 : LC_TILE_ROWS_W16;  // source rows per tile
    static constexpr int S = W == 1 ? LC_TILE_STAGES_W1 : W == 2 ? LC_TILE_STAGES_W2
                           : W == 8 ? LC_TILE_STAGES_W8 : LC_TILE_STAGES_WIDE;  // ring stages
    static constexpr int TILE_BYTES = BOXB * R;
    static constexpr int MB = CPR * R / V;        // V-row x 16-byte micro-blocks
    static constexpr int MAXT = W == 2 && !SHORT ? LC_TILE_MAX_THREADS_W2_TALL
                              : W == 16           ? LC_TILE_MAX_THREADS_W16
                                                  : LC_TILE_MAX_THREADS;
    static constexpr int NT = MB < MAXT ? MB : MAXT;  // at most one micro-block each per round
    static constexpr bool SWZ = LINES && LC_TILE_SWIZZLE != 0;
    // barriers in the first 128 bytes; a swizzled ring starts on a 1024-byte boundary
    static constexpr int SMEM = 128 + S * TILE_BYTES + (SWZ ? 1024 : 0);
    static_assert(R <= 256 && R % V == 0, "TMA boxes hold at most 256 rows, whole micro-blocks");
    static_assert(!LINES || ((R / V) % 8 == 0 && CPR % 4 == 0), "line stores: octets of row groups, chunk quads");
    static_assert((BOXB == 128 || BOXB == 256) && SMEM <= 227 * 1024, "box rows of 128 or 256 bytes, ring fits");
};

struct TileArgs {
    uint8_t *dst;    // address of destination word offset 0
    int64_t eX, eY;  // X contiguous in dst, Y contiguous in src (words)
    int64_t dY;      // destination stride of Y (bytes)
    int32_t nb;      // batch modes (<= 3), outermost first
    int64_t be[3], bd[3];
    int64_t tiles_x, tiles_y, n_tiles;
    // n_tiles < 2^32: tile and batch indices are split by 32-bit invariant
    // divisors instead of 64-bit division
    int32_t narrow;
    FastDiv ftx, fty, fbe[3];
    uint64_t timeout_ns;
};

// One-byte words, word t of the 16 input rows -> output rows 4t .. 4t + 3:
// 4 x 4 byte blocks, rows 4p .. 4p + 3 giving word p of each output row.
__device__ __forceinline__ void transpose_bytes_word(const uint32_t (&in)[16][4], int t, uint32_t (&o0)[4],
                                                     uint32_t (&o1)[4], uint32_t (&o2)[4], uint32_t (&o3)[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t A = in[4 * p][t], B = in[4 * p + 1][t];
        const uint32_t C = in[4 * p + 2][t], D = in[4 * p + 3][t];
        const uint32_t ab_lo = __byte_perm(A, B, 0x5140), ab_hi = __byte_perm(A, B, 0x7362);
        const uint32_t cd_lo = __byte_perm(C, D, 0x5140), cd_hi = __byte_perm(C, D, 0x7362);
        o0[p] = __byte_perm(ab_lo, cd_lo, 0x5410);
        o1[p] = __byte_perm(ab_lo, cd_lo, 0x7632);
        o2[p] = __byte_perm(ab_hi, cd_hi, 0x5410);
        o3[p] = __byte_perm(ab_hi, cd_hi, 0x7632);
    }
}

// V rows of one 16-byte column chunk -> V destination chunks: out[q] holds
// word q of every input row (a V x V transpose of W-byte words in registers;
// the 2-byte and 1-byte cases use byte permutes).
template <int W>
__device__ __forceinline__ void transpose_chunk(const uint32_t (&in)[16 / W][4], uint32_t (&out)[16 / W][4]) {
    if constexpr (W == 16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) out[0][k] = in[0][k];
    } else if constexpr (W == 8) {
        out[0][0] = in[0][0]; out[0][1] = in[0][1]; out[0][2] = in[1][0]; out[0][3] = in[1][1];
        out[1][0] = in[0][2]; out[1][1] = in[0][3]; out[1][2] = in[1][2]; out[1][3] = in[1][3];
    } else if constexpr (W == 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) out[q][i] = in[i][q];
    } else if constexpr (W == 2) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int p = 0; p < 4; ++p)
                out[q][p] = __byte_perm(in[2 * p][q >> 1], in[2 * p + 1][q >> 1], (q & 1) ? 0x7632 : 0x5410);
    } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) transpose_bytes_word(in, t, out[4 * t], out[4 * t + 1], out[4 * t + 2], out[4 * t + 3]);
    }
}

// Stores words [0, n) of a 16-byte chunk (the ragged right edge); the word
// index is a compile-time constant in every unrolled step, so the chunk stays
// in registers.
template <int W>
__device__ __forceinline__ void store_partial(uint8_t *p, const uint32_t (&v)[4], int n) {
    constexpr int V = 16 / W;
#pragma unroll
    for (int k = 0; k < V; ++k) {
        if (k >= n) break;
        if constexpr (W == 1) p[k] = static_cast<uint8_t>(v[k >> 2] >> (8 * (k & 3)));
        else if constexpr (W == 2) reinterpret_cast<uint16_t *>(p)[k] = static_cast<uint16_t>(v[k >> 1] >> (16 * (k & 1)));
        else if constexpr (W == 4) reinterpret_cast<uint32_t *>(p)[k] = v[k];
        else if constexpr (W == 8) reinterpret_cast<uint2 *>(p)[k] = make_uint2(v[2 * k], v[2 * k + 1]);
    }
}

// Tile index -> (tx, ty, flat batch index).
template <typename A>
__device__ __forceinline__ void tile_coords(const A &a, int64_t t, int64_t &tx, int64_t &ty, int64_t &b) {
    if (a.narrow) {
        const uint32_t t32 = static_cast<uint32_t>(t);
#if LC_TILE_Y_FASTEST
        const uint32_t rest = fast_div(t32, a.fty), b32 = fast_div(rest, a.ftx);
        ty = t32 - rest * a.fty.d;
        tx = rest - b32 * a.ftx.d;
#else
        const uint32_t rest = fast_div(t32, a.ftx), b32 = fast_div(rest, a.fty);
        tx = t32 - rest * a.ftx.d;
        ty = rest - b32 * a.fty.d;
#endif
        b = b32;
        return;
    }
#if LC_TILE_Y_FASTEST
    ty = t % a.tiles_y;
    const int64_t rest = t / a.tiles_y;
    tx = rest % a.tiles_x;
    b = rest / a.tiles_x;
#else
    tx = t % a.tiles_x;
    const int64_t rest = t / a.tiles_x;
    ty = rest % a.tiles_y;
    b = rest / a.tiles_y;
#endif
}

// Flat batch index -> batch coordinates b0 (outermost) .. b2.
__device__ __forceinline__ void batch_coords(const TileArgs &a, int64_t b, int32_t &b0, int32_t &b1, int32_t &b2) {
    b0 = b1 = b2 = 0;
    if (a.narrow) {
        uint32_t q = static_cast<uint32_t>(b);
        if (a.nb == 3) { const uint32_t n = fast_div(q, a.fbe[2]); b2 = static_cast<int32_t>(q - n * a.fbe[2].d); q = n; }
        if (a.nb >= 2) { const uint32_t n = fast_div(q, a.fbe[1]); b1 = static_cast<int32_t>(q - n * a.fbe[1].d); q = n; }
        if (a.nb >= 1) b0 = static_cast<int32_t>(q);  // the outermost batch index is below its extent
    } else {
        if (a.nb == 3) { b2 = static_cast<int32_t>(b % a.be[2]); b /= a.be[2]; }
        if (a.nb >= 2) { b1 = static_cast<int32_t>(b % a.be[1]); b /= a.be[1]; }
        if (a.nb >= 1) { b0 = static_cast<int32_t>(b % a.be[0]); }
    }
}

template <int W, bool SHORT>
__device__ __forceinline__ void tile_issue_load(const CUtensorMap *tmap, const TileArgs &a, int64_t t,
                                                uint32_t dst, uint32_t bar) {
    using C = TileCfg<W, SHORT>;
    int64_t tx, ty, b;
    tile_coords(a, t, tx, ty, b);
    int32_t b0, b1, b2;  // batch coordinates, outermost first
    batch_coords(a, b, b0, b1, b2);
    const int32_t c0 = static_cast<int32_t>(ty * C::TY * (W == 16 ? 2 : 1));
    const int32_t c1 = static_cast<int32_t>(tx * C::R);
    ptx::mbar_arrive_expect_tx(bar, C::TILE_BYTES);
    // tensor dims: (Y, X, batch innermost .. outermost)
    switch (a.nb) {
        case 0: ptx::tma_load_2d(dst, tmap, c0, c1, bar); break;
        case 1: ptx::tma_load_3d(dst, tmap, c0, c1, b0, bar); break;
        case 2: ptx::tma_load_4d(dst, tmap, c0, c1, b1, b0, bar); break;
        default: ptx::tma_load_5d(dst, tmap, c0, c1, b2, b1, b0, bar); break;
    }
}

// Micro-block mb of a tile -> (16-byte chunk c, row group mr).  With line
// stores, lane l of a warp's 32 micro-blocks takes chunk 4 g + (l & 3) and
// one of 8 consecutive row groups; the row-group bit that varies inside a
// quarter warp (8 lanes, one shared-memory wavefront of 16-byte reads) is
// the one that changes the swizzle phase (row & 7) of the rows read: bit 0
// for 4-byte words (V = 4), 1 for 8-byte, 2 for 16-byte words.
template <typename C>
__device__ __forceinline__ void micro_block(int mb, int &c, int &mr) {
    if constexpr (C::LINES) {
        constexpr int CQ = C::CPR / 4;
        const int l = mb & 31, g = mb >> 5, m3 = l >> 2;
        int lo = m3;
        if constexpr (C::V == 2) lo = ((m3 & 1) << 1) | ((m3 >> 1) & 1) | (m3 & 4);
        else if constexpr (C::V == 1) lo = ((m3 & 1) << 2) | (m3 >> 1);
        c = (g % CQ) * 4 + (l & 3);
        mr = (g / CQ) * 8 + lo;
    } else {
        c = mb % C::CPR;
        mr = mb / C::CPR;
    }
}

// Tile t = (batch, ty, tx): TMA brings source rows [tx*R, tx*R + R) x words
// [ty*TY, ty*TY + TY) (BOXB bytes per row) into a stage.  Micro-block mb =
// (row group mr, 16-byte chunk c; micro_block): V rows x 16 bytes,
// transposed in registers into V destination chunks, destination rows
// ty*TY + c*V + q, words tx*R + mr*V .. + V.  Without line stores the 8
// lanes of a 16-byte shared-memory wavefront read 8 consecutive chunks of one
// box row, i.e. all 32 banks once: conflict-free with no swizzle; with line
// stores they read 4 chunks of two rows whose swizzle phases differ.
template <int W, bool SHORT>
__global__ void __launch_bounds__(TileCfg<W, SHORT>::NT)
    k_tile_transpose(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ TileArgs a) {
    using C = TileCfg<W, SHORT>;
    constexpr int V = C::V;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    const int tid = threadIdx.x;
    const int64_t n_local = a.n_tiles > blockIdx.x ? (a.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t bar0 = ptx::smem_addr(bars);
    uint32_t tile0 = bar0 + 128;
    if constexpr (C::SWZ) tile0 = (tile0 + 1023u) & ~1023u;  // the swizzle's phase follows address bits 7-9
    const uint8_t *tiles = smem + (tile0 - bar0);
    if (tid == 0) {
        ptx::prefetch_tensormap(&tmap);
        for (int s = 0; s < C::S; ++s) ptx::mbar_init(bar0 + 8 * s, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int64_t i = 0; i < lmin(C::S, n_local); ++i)
            tile_issue_load<W, SHORT>(&tmap, a, blockIdx.x + i * gridDim.x, tile0 + i * C::TILE_BYTES, bar0 + 8 * i);

    for (int64_t i = 0; i < n_local; ++i) {
        const int s = static_cast<int>(i % C::S);
        const uint32_t parity = static_cast<uint32_t>((i / C::S) & 1);
        const int64_t t = blockIdx.x + i * gridDim.x;
#if LC_TILE_POLL_ONE
        __shared__ int stage_ok;
        if (tid == 0) stage_ok = ptx::mbar_wait_bounded(bar0 + 8 * s, parity, a.timeout_ns) ? 1 : 0;
        __syncthreads();
        const bool ok = stage_ok != 0;
#else
        const bool ok = ptx::mbar_wait_bounded(bar0 + 8 * s, parity, a.timeout_ns);
#endif
        if (ok) {
            int64_t tx, ty, b;
            tile_coords(a, t, tx, ty, b);
            uint8_t *dbase = a.dst;
            if (a.narrow) {
                uint32_t q = static_cast<uint32_t>(b);
                for (int k = a.nb - 1; k > 0; --k) {
                    const uint32_t n = fast_div(q, a.fbe[k]);
                    dbase += static_cast<int64_t>(q - n * a.fbe[k].d) * a.bd[k];
                    q = n;
                }
                if (a.nb > 0) dbase += static_cast<int64_t>(q) * a.bd[0];
            } else {
                for (int k = a.nb - 1; k >= 0; --k) {
                    dbase += (b % a.be[k]) * a.bd[k];
                    b /= a.be[k];
                }
            }
            const uint8_t *st = tiles + static_cast<size_t>(s) * C::TILE_BYTES;
            for (int mb = tid; mb < C::MB; mb += C::NT) {
                int c, mr;
                micro_block<C>(mb, c, mr);
                const int64_t x0 = tx * C::R + int64_t(mr) * V;
                if (x0 >= a.eX) continue;  // rows past the tensor (TMA filled them)
                uint32_t in[V][4], out[V][4];
                // With 8 or more rows a micro-block, every row group starts on the
                // same swizzle phase; lanes of odd row groups read their rows in the
                // order r ^ 4 so that the two row groups of a quarter warp sit on
                // different phases, and put the rows back in order in registers.
                constexpr bool FLIP = C::SWZ && C::LINES && V >= 8;
                const int fl = FLIP ? (mr & 1) * 4 : 0;
#pragma unroll
                for (int r = 0; r < V; ++r) {
                    const int row = mr * V + (r ^ fl);
                    const int pc = C::SWZ ? (c ^ (row & 7)) : c;
                    const uint4 q = *reinterpret_cast<const uint4 *>(st + row * C::BOXB + pc * 16);
                    in[r][0] = q.x; in[r][1] = q.y; in[r][2] = q.z; in[r][3] = q.w;
                }
                if constexpr (FLIP) {
                    if (fl) {
#pragma unroll
                        for (int r = 0; r < V; ++r) {
                            if (r & 4) continue;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint32_t t = in[r][k];
                                in[r][k] = in[r ^ 4][k];
                                in[r ^ 4][k] = t;
                            }
                        }
                    }
                }
                transpose_chunk<W>(in, out);
                const int64_t y0 = ty * C::TY + int64_t(c) * V;
                const int nx = static_cast<int>(lmin(V, a.eX - x0));
#pragma unroll
                for (int q = 0; q < V; ++q) {
                    if (y0 + q < a.eY) {
                        uint8_t *p = dbase + (y0 + q) * a.dY + x0 * W;
                        if (nx == V)
                            store_out<uint4>(p, make_uint4(out[q][0], out[q][1], out[q][2], out[q][3]));
                        else
                            store_partial<W>(p, out[q], nx);
                    }
                }
            }
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                report_error(LC_ERR_TIMEOUT, LC_KERNEL_TILE_TRANSPOSE);
                for (int64_t q = i; q < lmin(i + C::S, n_local); ++q)
                    ptx::mbar_wait_bounded(bar0 + 8 * (q % C::S), static_cast<uint32_t>((q / C::S) & 1),
                                           a.timeout_ns);
            }
            return;
        }
        if (tid == 0 && i + C::S < n_local)
            tile_issue_load<W, SHORT>(&tmap, a, blockIdx.x + (i + C::S) * gridDim.x, tile0 + s * C::TILE_BYTES,
                               bar0 + 8 * s);
    }
}

// ---- Tile transpose through TMA stores --------------------------------------
//
// Boxes of 128-byte source rows land in a ring under the TMA 128-byte swizzle.
// A warp takes 8 consecutive row groups x 4 chunks: lane (i, cq) reads the V
// rows of row group mr = 8 g + i at chunk c in the order r ^ f(i), so that the
// 8 lanes of a quarter warp read 8 different swizzle phases (conflict-free),
// puts them back in order with conditional register swaps, transposes V x V
// words in registers and writes its V destination chunks into an output tile
// laid out as the destination box (TY rows of R words), the quarter warp
// writing 128 contiguous bytes.  One thread then stores the output tile with
// a TMA tensor store through a destination tensor map, which clips it at the
// tensor's edges (its contiguous mode in 16-byte steps: the form takes only
// destination rows of whole 16-byte chunks), and refills the stage; O output
// tiles rotate, each reused once its store has read it.
// Sizes (bytes a side) that take TMA stores, per word width (unless the
// direct form applies): 1- and 2-byte words above LC_TS_MIN_BYTES_NARROW,
// 4-byte words at every size, 8- and 16-byte words up to
// LC_TS_MAX_BYTES_WIDE.  Measured on GB300 over square and 4:1 transposes of
// 64 MiB - 1.5 GiB a side (L2 flushed by a read between launches below 258
// MiB a side, launches back to back above), against the ring with thread
// stores: 1-byte words 91.1-96.8 % of the copy peak against 80.2-87.4 % above
// 256 MiB (84.8-86.9 % against 91.7-94.8 % at 128 MiB); 2-byte words
// 92.2-97.6 % against 81.9-91.0 % above 256 MiB, except 87.3 % against
// 89.2 % on the 16384^2 transpose; 4-byte words 88.9-96.5 % against
// 84.2-96.2 % (never more than a point behind); 8-byte words 92.3-96.4 %
// against 83.5-84.4 % up to 256 MiB, 86.2-91.3 % against 88.3-93.9 % above;
// 16-byte words 94.8-97.5 % against 78.9-88.4 % up to 256 MiB, 85.5-91.8 %
// against 88.1-95.2 % above.  2-byte words whose destination rows are a
// multiple of LC_TS_W2_PITCH_RING bytes apart keep thread stores: 87.5-87.6 %
// against 88.9-89.4 % (32 KiB rows), 91.0-91.6 % against 92.5-92.8 % (64 KiB),
// where rows 16 KiB apart measured 93.8-94.0 % against 92.6 % and rows 24-48
// KiB apart (not powers of two) 94.2-95.3 % against 70.3-86.6 %.
#ifndef LC_TS_W2_PITCH_RING
#define LC_TS_W2_PITCH_RING (32 << 10)
#endif
#ifndef LC_TS_MIN_BYTES_NARROW
#define LC_TS_MIN_BYTES_NARROW (256ll << 20)
#endif
#ifndef LC_TS_MAX_BYTES_WIDE
#define LC_TS_MAX_BYTES_WIDE (256ll << 20)
#endif
#ifndef LC_TS_ROWS_NARROW
#define LC_TS_ROWS_NARROW 256
#endif
#ifndef LC_TS_ROWS_W8
#define LC_TS_ROWS_W8 128
#endif
#ifndef LC_TS_ROWS_W16
#define LC_TS_ROWS_W16 128
#endif
// Ring stages (4: 89.6-90.0 % on the 8192^2 4-byte transpose) and output
// tiles; CTAs of 512 threads measured 91.1-91.5 %.
#ifndef LC_TS_STAGES
#define LC_TS_STAGES 3
#endif
#ifndef LC_TS_OUT
#define LC_TS_OUT 2
#endif
#ifndef LC_TS_THREADS
#define LC_TS_THREADS 256
#endif

template <int W> struct TsCfg {
    static constexpr int V = 16 / W;
    static constexpr int MULT = W == 16 ? 2 : 1;  // 16-byte words travel as two 8-byte TMA elements
    static constexpr int TY = 128 / W;            // words of Y per tile: one 128-byte box row
    static constexpr int R = W == 16 ? LC_TS_ROWS_W16 : W == 8 ? LC_TS_ROWS_W8 : LC_TS_ROWS_NARROW;
    static constexpr int S = LC_TS_STAGES, O = LC_TS_OUT;
    static constexpr int TILE_BYTES = 128 * R;    // an input stage, and an output tile (TY rows x R words)
    static constexpr int MB = 8 * R / V;          // micro-blocks: 8 chunks x R / V row groups
    static constexpr int NT = MB < LC_TS_THREADS ? MB : LC_TS_THREADS;
    static constexpr int SMEM = 2048 + (S + O) * TILE_BYTES;  // barriers, alignment slack, ring, outputs
    static_assert(R * MULT <= 256 && (R / V) % 8 == 0 && NT % 32 == 0 && MB % NT == 0, "whole warps of octets");
    static_assert(SMEM <= 227 * 1024, "ring and output tiles fit");
};

template <int W>
__device__ __forceinline__ void ts_issue_load(const CUtensorMap *tmap, const TileArgs &a, int64_t t, uint32_t dst,
                                              uint32_t bar) {
    using C = TsCfg<W>;
    int64_t tx, ty, b;
    tile_coords(a, t, tx, ty, b);
    int32_t b0, b1, b2;
    batch_coords(a, b, b0, b1, b2);
    const int32_t c0 = static_cast<int32_t>(ty * C::TY * C::MULT), c1 = static_cast<int32_t>(tx * C::R);
    ptx::mbar_arrive_expect_tx(bar, C::TILE_BYTES);
    switch (a.nb) {  // tensor dims: (Y, X, batch innermost .. outermost)
        case 0: ptx::tma_load_2d(dst, tmap, c0, c1, bar); break;
        case 1: ptx::tma_load_3d(dst, tmap, c0, c1, b0, bar); break;
        case 2: ptx::tma_load_4d(dst, tmap, c0, c1, b1, b0, bar); break;
        default: ptx::tma_load_5d(dst, tmap, c0, c1, b2, b1, b0, bar); break;
    }
}

template <int W>
__device__ __forceinline__ void ts_issue_store(const CUtensorMap *smap, const TileArgs &a, int64_t t, uint32_t src) {
    using C = TsCfg<W>;
    int64_t tx, ty, b;
    tile_coords(a, t, tx, ty, b);
    int32_t b0, b1, b2;
    batch_coords(a, b, b0, b1, b2);
    // tensor dims: (X, Y, batch innermost .. outermost)
    int32_t c[5] = {static_cast<int32_t>(tx * C::R * C::MULT), static_cast<int32_t>(ty * C::TY), 0, 0, 0};
    if (a.nb == 1) c[2] = b0;
    else if (a.nb == 2) { c[2] = b1; c[3] = b0; }
    else if (a.nb == 3) { c[2] = b2; c[3] = b1; c[4] = b0; }
    bulk::tma_store(smap, 2 + a.nb, c, src);
    bulk::commit();
}

template <int W>
__global__ void __launch_bounds__(TsCfg<W>::NT)
    k_tile_tstore(const __grid_constant__ CUtensorMap lmap, const __grid_constant__ CUtensorMap smap,
                  const __grid_constant__ TileArgs a) {
    using C = TsCfg<W>;
    constexpr int V = C::V;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int64_t n_local = a.n_tiles > blockIdx.x ? (a.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t bar0 = ptx::smem_addr(smem);
    const uint32_t ring0 = (bar0 + 128u + 1023u) & ~1023u;  // the swizzle's phase follows address bits 7-9
    const uint32_t out0 = ring0 + C::S * C::TILE_BYTES;
    const uint8_t *ring = smem + (ring0 - bar0);
    uint8_t *outp = smem + (out0 - bar0);
    if (tid == 0) {
        ptx::prefetch_tensormap(&lmap);
        ptx::prefetch_tensormap(&smap);
        for (int s = 0; s < C::S; ++s) ptx::mbar_init(bar0 + 8 * s, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int64_t i = 0; i < lmin(C::S, n_local); ++i)
            ts_issue_load<W>(&lmap, a, blockIdx.x + i * gridDim.x, ring0 + i * C::TILE_BYTES, bar0 + 8 * i);

    for (int64_t i = 0; i < n_local; ++i) {
        const int s = static_cast<int>(i % C::S), o = static_cast<int>(i % C::O);
        const int64_t t = blockIdx.x + i * gridDim.x;
        if (tid == 0 && i >= C::O) bulk::wait_read<C::O - 1>();  // output tile o: its last store has read it
        const bool ok = ptx::mbar_wait_bounded(bar0 + 8 * s, static_cast<uint32_t>((i / C::S) & 1), a.timeout_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                report_error(LC_ERR_TIMEOUT, LC_KERNEL_TILE_TRANSPOSE);
                bulk::wait_all();
                for (int64_t q = i; q < lmin(i + C::S, n_local); ++q)
                    ptx::mbar_wait_bounded(bar0 + 8 * (q % C::S), static_cast<uint32_t>((q / C::S) & 1),
                                           a.timeout_ns);
            }
            return;
        }
        const uint8_t *st = ring + s * C::TILE_BYTES;
        uint8_t *ot = outp + o * C::TILE_BYTES;
        for (int mb = tid; mb < C::MB; mb += C::NT) {
            const int l = mb & 31, g = mb >> 5, i8 = l & 7;
            const int c = (g & 1) * 4 + (l >> 3);  // 16-byte chunk of the box row
            const int mr = (g >> 1) * 8 + i8;     // row group
            const int f = V >= 8 ? i8 : (i8 * V) >> 3;
            uint32_t in[V][4], out[V][4];
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int row = mr * V + (k ^ f);
                const uint4 q = *reinterpret_cast<const uint4 *>(st + row * 128 + ((c ^ (row & 7)) << 4));
                in[k][0] = q.x; in[k][1] = q.y; in[k][2] = q.z; in[k][3] = q.w;
            }
            // in[k] holds row k ^ f: swap by each set bit of f to put row k there
#pragma unroll
            for (int bit = 1; bit < 8 && bit < V; bit <<= 1) {
                if (f & bit) {
#pragma unroll
                    for (int k = 0; k < V; ++k) {
                        if (k & bit) continue;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t tmp = in[k][e];
                            in[k][e] = in[k ^ bit][e];
                            in[k ^ bit][e] = tmp;
                        }
                    }
                }
            }
            transpose_chunk<W>(in, out);
#pragma unroll
            for (int q = 0; q < V; ++q)
                *reinterpret_cast<uint4 *>(ot + (c * V + q) * (C::R * W) + mr * 16) =
                    make_uint4(out[q][0], out[q][1], out[q][2], out[q][3]);
        }
        bulk::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            ts_issue_store<W>(&smap, a, t, out0 + o * C::TILE_BYTES);
            if (i + C::S < n_local)
                ts_issue_load<W>(&lmap, a, blockIdx.x + (i + C::S) * gridDim.x, ring0 + s * C::TILE_BYTES,
                                 bar0 + 8 * s);
        }
    }
    if (tid == 0) bulk::wait_all();
}

// ---- Direct tile transpose (no TMA, no shared memory) --------------------
//
// A warp takes a tile of RB row blocks x CL chunks: lane (rb, c) loads the V
// source rows of its block, 16 bytes each at chunk c, straight from global
// memory, transposes the V x V block in registers (transpose_chunk) and
// stores its V destination chunks.  One load instruction of the warp reads
// RB segments of CL * 16 contiguous bytes (one per source row), one store
// writes CL destination rows, RB * 16 bytes each.  Taken only when both
// extents are whole blocks (multiples of V), so that every block is either
// in the tensor or out of it.
// Largest copy (bytes a side) that takes the direct form, per word width (0:
// never).  Measured on GB300 (same sweep as the TMA-store sizes): 1-byte
// words 92.3-93.9 % of the copy peak up to 96 MiB against 80.7-88.8 % for the
// swizzled ring, 90.2-91.6 % against 91.7-94.8 % at 123-128 MiB, 69-83 %
// from 256 MiB; 2-byte words 91.4 % against 88.9 % at 64 MiB, 91.8-96.3 %
// against 93.9-97.0 % at 94-128 MiB.  4- and 8-byte words never gained
// (86.6-87.9 % against 90.8-90.9 %, 83.9-87.8 against 93.5 % at 8192^2).
#ifndef LC_DIRECT_MAX_BYTES_W1
#define LC_DIRECT_MAX_BYTES_W1 (96ll << 20)
#endif
#ifndef LC_DIRECT_MAX_BYTES_W2
#define LC_DIRECT_MAX_BYTES_W2 (64ll << 20)
#endif
// Threads per CTA: 256 for 1-byte words (83.8 % with 512), 512 for 2-byte
// words (91.1-91.6 % with 256).
#ifndef LC_DIRECT_THREADS_W1
#define LC_DIRECT_THREADS_W1 256
#endif
#ifndef LC_DIRECT_THREADS_W2
#define LC_DIRECT_THREADS_W2 512
#endif
#ifndef LC_DIRECT_THREADS_WIDE
#define LC_DIRECT_THREADS_WIDE 256
#endif
// 16-byte chunks per source row segment: 8 (128-byte loads, 64-byte store
// segments), 4 (64-byte loads, 128-byte stores) or 2.  With 8, the 8192^2
// 1-byte transpose ran at 64.6-73.3 %, the 2-byte one at 83.2-83.6 %; with
// 2, at 87.1-87.5 % and 77.8 %.
#ifndef LC_DIRECT_CL
#define LC_DIRECT_CL 4
#endif
#ifndef LC_DIRECT_CL_W1
#define LC_DIRECT_CL_W1 LC_DIRECT_CL
#endif
#ifndef LC_DIRECT_CL_W2
#define LC_DIRECT_CL_W2 LC_DIRECT_CL
#endif
#ifndef LC_DIRECT_CL_W4
#define LC_DIRECT_CL_W4 LC_DIRECT_CL
#endif
#ifndef LC_DIRECT_CL_W8
#define LC_DIRECT_CL_W8 LC_DIRECT_CL
#endif

template <int W> struct DirectCfg {
    static constexpr int V = 16 / W;
    static constexpr int CL = W == 1 ? LC_DIRECT_CL_W1 : W == 2 ? LC_DIRECT_CL_W2 : W == 4 ? LC_DIRECT_CL_W4
                                                                                        : LC_DIRECT_CL_W8;
    static constexpr int RB = 32 / CL;
    static constexpr int ROWS = RB * V;  // source rows (X) per warp tile
    static constexpr int COLS = CL * V;  // words (Y) per warp tile
    static constexpr int NT = W == 1 ? LC_DIRECT_THREADS_W1 : W == 2 ? LC_DIRECT_THREADS_W2 : LC_DIRECT_THREADS_WIDE;
    static constexpr int MINB = NT >= 512 ? 1 : 512 / NT;  // at most 128 registers a thread
    static_assert(CL == 2 || CL == 4 || CL == 8, "lanes split as 32 / CL row blocks x CL chunks");
};
// Warp tiles per round, all loads issued first (2: 76-77 % and 87.6 % for
// the 8192^2 1- and 2-byte transposes).
#ifndef LC_DIRECT_U
#define LC_DIRECT_U 1
#endif

struct DirectArgs {
    const uint8_t *src;  // address of source word offset 0
    uint8_t *dst;        // address of destination word offset 0
    int64_t eX, eY;      // words; both multiples of V
    int64_t sX, dY;      // bytes: source stride of X, destination stride of Y
    int32_t nb;          // batch modes (<= 3), outermost first
    int64_t be[3], bs[3], bd[3];  // extents; source and destination strides (bytes)
    int64_t tiles_x, tiles_y, n_tiles;  // warp tiles, fewer than 2^32 (copies of at most 256 MiB)
    int32_t narrow;      // always 1: tile and batch indices split by 32-bit invariant divisors
    FastDiv ftx, fty, fbe[3];
};

__device__ __forceinline__ uint4 direct_load(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int W>
__global__ void __launch_bounds__(DirectCfg<W>::NT, DirectCfg<W>::MINB)
    k_tile_direct(const __grid_constant__ DirectArgs a) {
    using C = DirectCfg<W>;
    constexpr int V = C::V, CL = C::CL, RB = C::RB, U = LC_DIRECT_U;
    const int lane = threadIdx.x & 31, c = lane % CL, rb = lane / CL;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (; t < a.n_tiles; t += U * warps) {
        uint32_t in[U][V][4];
        uint8_t *dp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            dp[u] = nullptr;
            const int64_t tu = t + u * warps;
            if (tu >= a.n_tiles) continue;
            int64_t tx, ty, b;
            tile_coords(a, tu, tx, ty, b);
            const int64_t x0 = tx * (RB * V) + rb * V, y0 = ty * (CL * V) + c * V;
            if (x0 >= a.eX || y0 >= a.eY) continue;  // a block past the tensor
            const uint8_t *sp = a.src + x0 * a.sX + y0 * W;
            uint8_t *d = a.dst + y0 * a.dY + x0 * W;
            uint32_t q = static_cast<uint32_t>(b);
            for (int k = a.nb - 1; k > 0; --k) {
                const uint32_t n = fast_div(q, a.fbe[k]);
                const int64_t bk = q - n * a.fbe[k].d;
                sp += bk * a.bs[k];
                d += bk * a.bd[k];
                q = n;
            }
            if (a.nb > 0) { sp += int64_t(q) * a.bs[0]; d += int64_t(q) * a.bd[0]; }  // below its extent
            dp[u] = d;
#pragma unroll
            for (int r = 0; r < V; ++r) {
                const uint4 v = direct_load(sp + r * a.sX);
                in[u][r][0] = v.x; in[u][r][1] = v.y; in[u][r][2] = v.z; in[u][r][3] = v.w;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (!dp[u]) continue;
            if constexpr (W == 1) {
                // four output rows at a time, so that each input word dies as it is used
#pragma unroll
                for (int tw = 0; tw < 4; ++tw) {
                    uint32_t o[4][4];
                    transpose_bytes_word(in[u], tw, o[0], o[1], o[2], o[3]);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        store_out<uint4>(dp[u] + (4 * tw + k) * a.dY, make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]));
                }
            } else {
                uint32_t out[V][4];
                transpose_chunk<W>(in[u], out);
#pragma unroll
                for (int q = 0; q < V; ++q)
                    store_out<uint4>(dp[u] + q * a.dY, make_uint4(out[q][0], out[q][1], out[q][2], out[q][3]));
            }
        }
    }
}

// Whether a copy of `bytes` a side with w-byte words takes the short boxes.
static bool tile_short(int w, int64_t bytes) { return w <= 4 && bytes <= LC_TILE_SHORT_MAX_BYTES; }

template <int W, bool SHORT>
static void geometry_of(int *rows, int *cols, int *stages, int *threads) {
    using C = TileCfg<W, SHORT>;
    *rows = C::R;
    *cols = C::TY;
    *stages = C::S;
    *threads = C::NT;
}

template <int W>
static void direct_geometry_of(int *rows, int *cols, int *threads) {
    *rows = DirectCfg<W>::ROWS;
    *cols = DirectCfg<W>::COLS;
    *threads = DirectCfg<W>::NT;
}

template <int W>
static void tstore_geometry_of(int *rows, int *cols, int *stages, int *threads) {
    *rows = TsCfg<W>::R;
    *cols = TsCfg<W>::TY;
    *stages = TsCfg<W>::S;
    *threads = TsCfg<W>::NT;
}

bool tile_tstore_geometry(int w, int64_t bytes, int64_t eX, int64_t dY_bytes, int *rows, int *cols, int *stages,
                          int *threads) {
    // a tensor store clips the destination's contiguous mode in 16-byte steps
    // (measured: a 71-word row of 2-byte words got its 72nd word written), so
    // the form takes only destination rows of whole 16-byte chunks
    const bool sized = w <= 2 ? bytes > LC_TS_MIN_BYTES_NARROW : w == 4 ? true : bytes <= LC_TS_MAX_BYTES_WIDE;
    if (!sized || (eX * w) % 16) return false;
    if (w == 2 && dY_bytes % LC_TS_W2_PITCH_RING == 0) return false;
    switch (w) {
        case 1: tstore_geometry_of<1>(rows, cols, stages, threads); break;
        case 2: tstore_geometry_of<2>(rows, cols, stages, threads); break;
        case 4: tstore_geometry_of<4>(rows, cols, stages, threads); break;
        case 8: tstore_geometry_of<8>(rows, cols, stages, threads); break;
        default: tstore_geometry_of<16>(rows, cols, stages, threads); break;
    }
    return true;
}

bool tile_direct_geometry(int w, int64_t bytes, int64_t eX, int64_t eY, int *rows, int *cols, int *threads) {
    const int64_t max_bytes = w == 1 ? LC_DIRECT_MAX_BYTES_W1 : w == 2 ? LC_DIRECT_MAX_BYTES_W2 : 0;
    if (bytes > max_bytes) return false;
    if (eX % (16 / w) || eY % (16 / w)) return false;
    switch (w) {
        case 1: direct_geometry_of<1>(rows, cols, threads); break;
        case 2: direct_geometry_of<2>(rows, cols, threads); break;
        case 4: direct_geometry_of<4>(rows, cols, threads); break;
        default: direct_geometry_of<8>(rows, cols, threads); break;
    }
    return true;
}

void tile_geometry(int w, int64_t bytes, int *rows, int *cols, int *stages, int *threads) {
    const bool sh = tile_short(w, bytes);
    switch (w) {
        case 1: sh ? geometry_of<1, true>(rows, cols, stages, threads) : geometry_of<1, false>(rows, cols, stages, threads); break;
        case 2: sh ? geometry_of<2, true>(rows, cols, stages, threads) : geometry_of<2, false>(rows, cols, stages, threads); break;
        case 4: sh ? geometry_of<4, true>(rows, cols, stages, threads) : geometry_of<4, false>(rows, cols, stages, threads); break;
        case 8: geometry_of<8, false>(rows, cols, stages, threads); break;
        default: geometry_of<16, false>(rows, cols, stages, threads); break;
    }
}

namespace {

template <int W, bool SHORT>
int launch_tile_t(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    using C = TileCfg<W, SHORT>;
    const TilePlan &tp = p.tile;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return LC_ERR_CUDA;
    const int rank = 2 + tp.batch.n;
    const int mult = W == 16 ? 2 : 1;  // 16-byte words travel as two 8-byte TMA elements
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], estr[5];
    dims[0] = static_cast<cuuint64_t>(tp.Y.e * mult);
    dims[1] = static_cast<cuuint64_t>(tp.X.e);
    strides[0] = static_cast<cuuint64_t>(tp.X.s * W);
    for (int i = 0; i < tp.batch.n; ++i) {  // innermost batch mode first
        const Mode &b = tp.batch.m[tp.batch.n - 1 - i];
        dims[2 + i] = static_cast<cuuint64_t>(b.e);
        strides[1 + i] = static_cast<cuuint64_t>(b.s * W);
    }
    box[0] = static_cast<cuuint32_t>(C::BOXB / (W / mult));
    box[1] = static_cast<cuuint32_t>(C::R);
    for (int i = 2; i < 5; ++i) box[i] = 1;
    for (int i = 0; i < 5; ++i) estr[i] = 1;
    CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (W == 2) dt = CU_TENSOR_MAP_DATA_TYPE_UINT16;
    else if (W == 4) dt = CU_TENSOR_MAP_DATA_TYPE_UINT32;
    else if (W >= 8) dt = CU_TENSOR_MAP_DATA_TYPE_UINT64;
    CUtensorMap tmap;
    std::memset(&tmap, 0, sizeof(tmap));
    void *base = const_cast<uint8_t *>(src + p.src_off * W);
    if (enc(&tmap, dt, static_cast<cuuint32_t>(rank), base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, C::SWZ ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return LC_ERR_UNSUPPORTED;  // the driver refused this tensor shape

    TileArgs a{};
    a.dst = dst + p.dst_off * W;
    a.eX = tp.X.e;
    a.eY = tp.Y.e;
    a.dY = tp.Y.d * W;
    a.nb = tp.batch.n;
    int64_t nbatch = 1;
    for (int i = 0; i < tp.batch.n; ++i) {
        a.be[i] = tp.batch.m[i].e;
        a.bd[i] = tp.batch.m[i].d * W;
        nbatch *= tp.batch.m[i].e;
    }
    a.tiles_x = (tp.X.e + C::R - 1) / C::R;
    a.tiles_y = (tp.Y.e + C::TY - 1) / C::TY;
    a.n_tiles = a.tiles_x * a.tiles_y * nbatch;
    // 32-bit index math for the short boxes only: measured on GB300 it moves
    // the 8192^2 2-byte transpose at 87.8 % against 83.2 % with 64-bit
    // division, but the 256-row boxes of the larger transposes at 84-86 %
    // against 91.6-93.8 % (16384^2 2-byte, 8192^2 8- and 16-byte words).
    a.narrow = SHORT && a.n_tiles < (int64_t(1) << 32);
    if (a.narrow) {
        a.ftx = make_fastdiv(static_cast<uint32_t>(a.tiles_x));
        a.fty = make_fastdiv(static_cast<uint32_t>(a.tiles_y));
        for (int i = 0; i < tp.batch.n; ++i) a.fbe[i] = make_fastdiv(static_cast<uint32_t>(tp.batch.m[i].e));
    }
    a.timeout_ns = wait_limit_ns();

    const void *fn = reinterpret_cast<const void *>(&k_tile_transpose<W, SHORT>);
    int sms, per;
    if (prepare(fn, C::NT, C::SMEM, C::SMEM, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t grid = lmin(a.n_tiles, int64_t(sms) * per);
    k_tile_transpose<W, SHORT><<<static_cast<unsigned>(grid), C::NT, C::SMEM, stream>>>(tmap, a);
    return finish_launch();
}

// The tile arguments shared by the ring forms: extents, destination stride
// of Y, batch modes, tile counts for R x TY tiles, 32-bit divisors when the
// tile count allows them.
static TileArgs ring_args(const Plan &p, uint8_t *dst, int w, int R, int TY, bool narrow_ok) {
    const TilePlan &tp = p.tile;
    TileArgs a{};
    a.dst = dst + p.dst_off * w;
    a.eX = tp.X.e;
    a.eY = tp.Y.e;
    a.dY = tp.Y.d * w;
    a.nb = tp.batch.n;
    int64_t nbatch = 1;
    for (int i = 0; i < tp.batch.n; ++i) {
        a.be[i] = tp.batch.m[i].e;
        a.bd[i] = tp.batch.m[i].d * w;
        nbatch *= tp.batch.m[i].e;
    }
    a.tiles_x = (tp.X.e + R - 1) / R;
    a.tiles_y = (tp.Y.e + TY - 1) / TY;
    a.n_tiles = a.tiles_x * a.tiles_y * nbatch;
    a.narrow = narrow_ok && a.n_tiles < (int64_t(1) << 32);
    if (a.narrow) {
        a.ftx = make_fastdiv(static_cast<uint32_t>(a.tiles_x));
        a.fty = make_fastdiv(static_cast<uint32_t>(a.tiles_y));
        for (int i = 0; i < tp.batch.n; ++i) a.fbe[i] = make_fastdiv(static_cast<uint32_t>(tp.batch.m[i].e));
    }
    a.timeout_ns = wait_limit_ns();
    return a;
}

static CUtensorMapDataType tma_type(int w) {
    return w == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : w == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
         : w == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT64;
}

template <int W>
int launch_tstore_t(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    using C = TsCfg<W>;
    const TilePlan &tp = p.tile;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return LC_ERR_CUDA;
    const int rank = 2 + tp.batch.n;
    // load map: (Y, X, batch innermost first) over the source, boxes of one
    // 128-byte row x R rows, swizzled; store map: (X, Y, batch) over the
    // destination, boxes of R words x TY rows
    cuuint64_t ld_dims[5], ld_str[4], st_dims[5], st_str[4];
    cuuint32_t ld_box[5], st_box[5], estr[5];
    ld_dims[0] = static_cast<cuuint64_t>(tp.Y.e * C::MULT);
    ld_dims[1] = static_cast<cuuint64_t>(tp.X.e);
    ld_str[0] = static_cast<cuuint64_t>(tp.X.s * W);
    st_dims[0] = static_cast<cuuint64_t>(tp.X.e * C::MULT);
    st_dims[1] = static_cast<cuuint64_t>(tp.Y.e);
    st_str[0] = static_cast<cuuint64_t>(tp.Y.d * W);
    for (int i = 0; i < tp.batch.n; ++i) {
        const Mode &b = tp.batch.m[tp.batch.n - 1 - i];
        ld_dims[2 + i] = st_dims[2 + i] = static_cast<cuuint64_t>(b.e);
        ld_str[1 + i] = static_cast<cuuint64_t>(b.s * W);
        st_str[1 + i] = static_cast<cuuint64_t>(b.d * W);
    }
    ld_box[0] = static_cast<cuuint32_t>(128 / (W / C::MULT));
    ld_box[1] = static_cast<cuuint32_t>(C::R);
    st_box[0] = static_cast<cuuint32_t>(C::R * C::MULT);
    st_box[1] = static_cast<cuuint32_t>(C::TY);
    for (int i = 2; i < 5; ++i) ld_box[i] = st_box[i] = 1;
    for (int i = 0; i < 5; ++i) estr[i] = 1;
    const CUtensorMapDataType dt = tma_type(W / C::MULT);
    CUtensorMap lmap, smap;
    std::memset(&lmap, 0, sizeof(lmap));
    std::memset(&smap, 0, sizeof(smap));
    void *sbase = const_cast<uint8_t *>(src + p.src_off * W);
    void *dbase = dst + p.dst_off * W;
    if (enc(&lmap, dt, static_cast<cuuint32_t>(rank), sbase, ld_dims, ld_str, ld_box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&smap, dt, static_cast<cuuint32_t>(rank), dbase, st_dims, st_str, st_box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return LC_ERR_UNSUPPORTED;  // the driver refused this tensor shape
    const TileArgs a = ring_args(p, dst, W, C::R, C::TY, true);
    const void *fn = reinterpret_cast<const void *>(&k_tile_tstore<W>);
    int sms, per;
    if (prepare(fn, C::NT, C::SMEM, C::SMEM, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t grid = lmin(a.n_tiles, int64_t(sms) * per);
    k_tile_tstore<W><<<static_cast<unsigned>(grid), C::NT, C::SMEM, stream>>>(lmap, smap, a);
    return finish_launch();
}

template <int W>
int launch_direct_t(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    using C = DirectCfg<W>;
    constexpr int V = C::V, CL = C::CL, RB = C::RB;
    const TilePlan &tp = p.tile;
    if (reinterpret_cast<uintptr_t>(src + p.src_off * W) % 16 || reinterpret_cast<uintptr_t>(dst + p.dst_off * W) % 16)
        return LC_ERR_UNSUPPORTED;  // the planner checked the pointers it was given
    DirectArgs a{};
    a.src = src + p.src_off * W;
    a.dst = dst + p.dst_off * W;
    a.eX = tp.X.e;
    a.eY = tp.Y.e;
    a.sX = tp.X.s * W;
    a.dY = tp.Y.d * W;
    a.nb = tp.batch.n;
    int64_t nbatch = 1;
    for (int i = 0; i < tp.batch.n; ++i) {
        a.be[i] = tp.batch.m[i].e;
        a.bs[i] = tp.batch.m[i].s * W;
        a.bd[i] = tp.batch.m[i].d * W;
        nbatch *= tp.batch.m[i].e;
    }
    a.tiles_x = (tp.X.e + RB * V - 1) / (RB * V);
    a.tiles_y = (tp.Y.e + CL * V - 1) / (CL * V);
    a.n_tiles = a.tiles_x * a.tiles_y * nbatch;
    if (a.n_tiles >= (int64_t(1) << 32)) return LC_ERR_UNSUPPORTED;  // not on copies the planner sends here
    a.narrow = 1;
    a.ftx = make_fastdiv(static_cast<uint32_t>(a.tiles_x));
    a.fty = make_fastdiv(static_cast<uint32_t>(a.tiles_y));
    for (int i = 0; i < tp.batch.n; ++i) a.fbe[i] = make_fastdiv(static_cast<uint32_t>(tp.batch.m[i].e));
    const void *fn = reinterpret_cast<const void *>(&k_tile_direct<W>);
    int sms, per;
    if (prepare(fn, C::NT, 0, 0, &sms, &per) != cudaSuccess) return LC_ERR_CUDA;
    const int64_t wpb = C::NT / 32;
    const int64_t grid = lmin((a.n_tiles + wpb - 1) / wpb, int64_t(sms) * per);
    k_tile_direct<W><<<static_cast<unsigned>(grid), C::NT, 0, stream>>>(a);
    return finish_launch();
}

}  // namespace

int launch_tile(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream) {
    if (p.tile.tstore) {
        switch (p.w) {
            case 1: return launch_tstore_t<1>(p, src, dst, stream);
            case 2: return launch_tstore_t<2>(p, src, dst, stream);
            case 4: return launch_tstore_t<4>(p, src, dst, stream);
            case 8: return launch_tstore_t<8>(p, src, dst, stream);
            case 16: return launch_tstore_t<16>(p, src, dst, stream);
        }
    }
    if (p.tile.direct) {
        switch (p.w) {
            case 1: return launch_direct_t<1>(p, src, dst, stream);
            case 2: return launch_direct_t<2>(p, src, dst, stream);
            case 4: return launch_direct_t<4>(p, src, dst, stream);
            case 8: return launch_direct_t<8>(p, src, dst, stream);
        }
    }
    const bool sh = tile_short(p.w, p.total * p.w);
    switch (p.w) {
        case 1: return sh ? launch_tile_t<1, true>(p, src, dst, stream) : launch_tile_t<1, false>(p, src, dst, stream);
        case 2: return sh ? launch_tile_t<2, true>(p, src, dst, stream) : launch_tile_t<2, false>(p, src, dst, stream);
        case 4: return sh ? launch_tile_t<4, true>(p, src, dst, stream) : launch_tile_t<4, false>(p, src, dst, stream);
        case 8: return launch_tile_t<8, false>(p, src, dst, stream);
        case 16: return launch_tile_t<16, false>(p, src, dst, stream);
    }
    return LC_ERR_UNSUPPORTED;
}

cudaError_t take_error_tile(unsigned long long *v) { return take_module_error(v); }

}  // namespace lc
