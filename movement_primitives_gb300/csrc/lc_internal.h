// Internal planner structures shared by the host planner (plan.cpp) and the
// kernel launchers (the k_*.cu translation units).  Not part of the ABI.
#pragma once

#include <cstdint>

#include "layout_copy.h"

namespace lc {

constexpr int kMaxModes = LC_MAX_RANK + 1;  // the tile mode rides along

// One mode of the aligned iteration: extent and the element stride on each
// side (the "extent / src_str / dst_str" of the permute_layout page).
struct Mode {
    int64_t e, s, d;
};

struct ModeList {
    int n = 0;
    Mode m[kMaxModes];
};

// [outer, threads, vec] vector copy over the destination-ordered modes.
struct VecPlan {
    ModeList outer;   // every mode but the contiguous run, outermost first
    int64_t run = 1;  // words in the run contiguous on both sides
    int vec = 1;      // words per vector (vec * w in {1,2,4,8,16} bytes)
};

// Warp register-staged permute of dense units of U = 32 * P words.
struct WarpPlan {
    ModeList unit;    // unit modes, logical order (the page's extent order)
    ModeList batch;   // modes enumerating the units, outermost first
    int64_t U = 0;
    int P = 0, k = 0, shift = 0, mask = 0, cr = 0, cw = 0;
    int64_t units_per_stage = 1;
    int64_t n_units = 0;
};

// TMA tile transpose: X is contiguous in dst, Y contiguous in src.
struct TilePlan {
    Mode X{}, Y{};
    ModeList batch;   // at most 3 (TMA tensors have at most 5 dims)
    int R = 0;        // source rows (X) per tile
    int TY = 0;       // words (Y) per 128-byte tile row
    int S = 0;        // pipeline stages (0: the direct form, no TMA ring)
    int threads = 0;
    int direct = 0;   // 1: whole V x V blocks, loaded straight into registers
    int tstore = 0;   // 1: the ring form whose output tiles leave by TMA tensor stores
};

// TMA tensor copy: the modes of the destination order, innermost first, as
// tensor dimensions of both tensor maps; box[k] words of dimension k per tile
// (in TMA elements: 16-byte words travel as two 8-byte elements).  Ring
// depth and tile size are compile-time knobs so that variants can be measured.
#ifndef LC_TMA_STAGES
#define LC_TMA_STAGES 6
#endif
#ifndef LC_TMA_TILE_BYTES
#define LC_TMA_TILE_BYTES 16384
#endif
struct TmaPlan {
    int rank = 0;
    int box[5] = {0, 0, 0, 0, 0};
    int64_t stage_bytes = 0;
};

// Warp-shuffle permute: blocks of V x V words (V = 16 / w) whose rows are
// 16-byte chunks of the source and whose columns are 16-byte chunks of the
// destination.  Lane a of a block's group moves the chunk at source word
// offset a * sa + k * sk and destination word offset a * da + k * dk of
// block k of its batch entry.
struct ShflPlan {
    int V = 0;
    int64_t sa = 0, sk = 0, da = 0, dk = 0;  // words
    int64_t kb = 0;                          // blocks per batch entry
    int64_t n_blocks = 0;
    ModeList batch;                          // outermost first
};

// Chunk swizzle of the shared tile of the shared-memory transpose: chunk k
// of row x is stored in chunk slot k ^ ((x >> shift) & mask).
struct SmemSwizzle {
    int shift = 0, mask = 0, cr = 0, cw = 0;
};

struct Plan {
    int kernel = LC_KERNEL_AUTO;
    int w = 0;                 // word bytes moved (after fusion)
    int fused = 1;             // inner-run words fused into one word
    int64_t src_off = 0, dst_off = 0;  // base offsets, in words of w bytes
    int64_t total = 0;         // words moved
    // byte ranges [lo, hi) each side reaches, relative to its pointer
    int64_t src_lo = 0, src_hi = 0, dst_lo = 0, dst_hi = 0;
    ModeList logical;          // logical order, jointly coalesced (original w)
    ModeList sorted;           // destination-stride order (fused w)
    VecPlan vec;
    WarpPlan warp;
    TilePlan tile;       // also the X / Y / batch split of the shared-memory transpose
    SmemSwizzle smem_swz;
    TmaPlan tma;
    ShflPlan shfl;
    // the caller's layouts and tile count (the staged class plans from them)
    lc_tile_layout src_l{}, dst_l{};
    int64_t n_tiles = 0;
};

// Pointer facts the planner needs (alignment of the two base addresses).
struct PtrInfo {
    uintptr_t src = 0, dst = 0;
    bool check = false;   // false for lc_plan: pointers assumed 256-byte aligned
    bool no_tma = false;  // a side in page-locked host memory: plain loads and stores only
};

// Threads of one staged-tile CTA when the planner launches the class.
constexpr int kStagedThreads = 256;

int make_plan(const lc_tile_layout *src, const lc_tile_layout *dst, int32_t w,
              int64_t n_tiles, int32_t kernel, const PtrInfo &ptr, Plan *out);
void fill_info(const Plan &p, lc_plan_info *info);

// A copy under a loop-layout override.  The thread digits and the slot
// digits are each sorted by their stride (ascending), so digit i of a
// thread index (or slot index) is (index / stride_i) % e_i; `weight` is the
// row-major weight of the digit's mode in the tile's flat index.
struct LoopDigit {
    int64_t e = 1, weight = 0;
};
struct LoopPlan {
    int w = 0;
    int64_t n_tiles = 0;
    int64_t N = 0;                     // words per tile
    int64_t src_off = 0, dst_off = 0;  // words
    int64_t sts = 0, dts = 0;          // tile strides, words
    ModeList logical;                  // one tile's modes, logical order
    int nt = 0, ns = 0;
    LoopDigit td[LC_MAX_RANK], sd[LC_MAX_RANK];
    int64_t T = 0, L = 0;
    int64_t inner_run = 1;  // innermost non-unit loop mode's extent when it is a slot mode of stride 1
    int vec = 1;            // words moved per vector
    // The loop's and the tile's mixed radices nest (their suffix products
    // form one divisibility chain) and a tile's byte span fits 31 bits: a
    // point's offsets are then the thread part's plus the slot part's.
    bool split = false;
};
int check_loop(const lc_loop_layout *loop, int64_t n, LoopPlan *out);
int make_loop_plan(const lc_tile_layout *src, const lc_tile_layout *dst, int32_t w, int64_t n_tiles,
                   const lc_loop_layout *loop, const PtrInfo &ptr, LoopPlan *out);

// Bank simulator ("permute_layout", section "Algorithm", step 2).
void phase_degrees(const ModeList &unit, int w, int k, int shift, int *rd, int *wd);
// Returns 0 when conflict-free (k, shift) found; 1 otherwise (best returned).
int choose_xor(const ModeList &unit, int w, int *k, int *shift, int *rd, int *wd);

// Geometry of the shared-memory transpose for w-byte words: a tile is TX
// source rows by TYW words; each row is staged as RB bytes of aligned C-byte
// chunks starting at the chunk boundary at or below the row's first word, so
// a row holds its lead-in (0 .. C - w bytes) and TYW words.
struct SmemGeo {
    int C, RB, TX, TYW;
};
// Tile rows (TX) and words (TYW) per width: compile-time knobs so that
// variants can be measured.
#ifndef LC_SMEM_TX_W1
#define LC_SMEM_TX_W1 64
#endif
#ifndef LC_SMEM_TYW_W1
#define LC_SMEM_TYW_W1 252
#endif
#ifndef LC_SMEM_TX_W2
#define LC_SMEM_TX_W2 64
#endif
#ifndef LC_SMEM_TYW_W2
#define LC_SMEM_TYW_W2 124
#endif
#ifndef LC_SMEM_TX_W4
#define LC_SMEM_TX_W4 64
#endif
constexpr SmemGeo smem_geometry(int w) {
    return w == 1   ? SmemGeo{4, 256, LC_SMEM_TX_W1, LC_SMEM_TYW_W1}
           : w == 2 ? SmemGeo{4, 256, LC_SMEM_TX_W2, LC_SMEM_TYW_W2}
           : w == 4 ? SmemGeo{4, 256, LC_SMEM_TX_W4, 64}
           : w == 8 ? SmemGeo{8, 512, 64, 64}
                    : SmemGeo{16, 512, 32, 32};
}

// TMA tile transpose geometry for w-byte words and `bytes` moved a side
// (source rows and words per tile, ring stages, threads), from the kernel's
// own compile-time table.
void tile_geometry(int w, int64_t bytes, int *rows, int *cols, int *stages, int *threads);
// The direct form of the tile transpose (no TMA, no shared memory): taken
// for the enabled word widths on copies of at most the short-box size a
// side when both extents are whole V x V blocks; false leaves the outputs
// alone.
bool tile_direct_geometry(int w, int64_t bytes, int64_t eX, int64_t eY, int *rows, int *cols, int *threads);
// The ring form with TMA tensor stores, by word width and bytes a side, for
// destination rows of whole 16-byte chunks (eX words) dY_bytes apart; false
// leaves the outputs alone.
bool tile_tstore_geometry(int w, int64_t bytes, int64_t eX, int64_t dY_bytes, int *rows, int *cols, int *stages,
                          int *threads);

// Shared tile swizzle of the shared-memory transpose for w-byte words:
// smallest (mask, shift) that keeps both copies conflict-free.
SmemSwizzle choose_smem_swizzle(int w);

// Joint coalescing and shard alignment, exposed for the swizzle queries.
int align_shards(const lc_tile_layout *src, const lc_tile_layout *dst, ModeList *out);

// Host-buffer copies (host_copy.cu, host_copy_static.cu): the byte spans the
// tiles of each side reach, relative to that side's pointer.
struct HostSpan {
    int64_t lo, hi;
};

inline int64_t cosize_of(const lc_tile_layout &l) {
    int64_t c = 1;
    for (int k = 0; k < l.rank; ++k) {
        if (l.shape[k] == 0) return 0;
        c += (l.shape[k] - 1) * l.stride[k];
    }
    return c;
}

inline int64_t words_of(const lc_tile_layout &l) {
    int64_t n = 1;
    for (int k = 0; k < l.rank; ++k) n *= l.shape[k];
    return n;
}

inline int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

// Word size, cosizes and tile strides (words) of both sides of a copy.
struct HostSides {
    const lc_tile_layout *s = nullptr, *d = nullptr;
    int64_t w = 0, scos = 0, dcos = 0, sts = 0, dts = 0;
    // the destination image covers its span exactly (tiles packed, each tile
    // dense), so nothing of the span needs to be staged in first
    bool dst_dense = false;
    HostSpan src(int64_t t0, int64_t t1) const {
        return HostSpan{(s->offset + t0 * sts) * w, (s->offset + (t1 - 1) * sts + scos) * w};
    }
    HostSpan dst(int64_t t0, int64_t t1) const {
        return HostSpan{(d->offset + t0 * dts) * w, (d->offset + (t1 - 1) * dts + dcos) * w};
    }
    // device bytes of one staging slot for `tiles` tiles: both spans, each
    // rounded up to 256 bytes
    int64_t slot_bytes(int64_t tiles) const {
        const HostSpan a = src(0, tiles), b = dst(0, tiles);
        return round256(a.hi - a.lo) + round256(b.hi - b.lo);
    }
};

inline HostSides host_sides(const lc_tile_layout &src, const lc_tile_layout &dst, int64_t w, int64_t n_tiles) {
    HostSides h;
    h.s = &src;
    h.d = &dst;
    h.w = w;
    h.scos = cosize_of(src);
    h.dcos = cosize_of(dst);
    h.sts = src.tile_stride ? src.tile_stride : h.scos;
    h.dts = dst.tile_stride ? dst.tile_stride : h.dcos;
    h.dst_dense = words_of(dst) == h.dcos && (n_tiles == 1 || h.dts == h.dcos);
    return h;
}

// Fast unsigned 32-bit division by an invariant divisor: q = n / d for every
// 32-bit n (Granlund & Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, the round-up multiplier with the extra add).
struct FastDiv {
    uint32_t d = 1, m = 1;
    int32_t s = 0;
};
FastDiv make_fastdiv(uint32_t d);

// Bank simulator on one warp-wide shared access of `width`-byte words at the
// 32 lanes' byte addresses: the most distinct 4-byte words one bank serves in
// a 128-byte wavefront.
int access_degree_vec(const int64_t *byte_addr, int width);

// int64 multiply / add that report overflow (false) instead of wrapping.
bool mul_ok_ext(int64_t a, int64_t b, int64_t *r);
bool add_ok_ext(int64_t a, int64_t b, int64_t *r);

}  // namespace lc
