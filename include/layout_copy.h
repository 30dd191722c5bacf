/*
 * layout_copy.h -- C ABI of the GB300 (sm_103a) strided tile layout copy.
 *
 * A TileLayout S[shape : stride] maps a logical index (i_0 .. i_{r-1}) to the
 * element offset  offset + sum_k i_k * stride_k  (Apache TVM docs
 * "permute_layout", section "Algorithm", step 3, `project`; "copy ->
 * gmem_smem", section "Demonstration program", `TileLayout(S[shape])`).
 * lc_layout_copy moves, for every tile t in [0, n_tiles) and every logical
 * index i, the elem_bytes-byte word at
 *     src + (src.offset + t * src.tile_stride + sum_k i_k * src.stride_k) * elem_bytes
 * to
 *     dst + (dst.offset + t * dst.tile_stride + sum_k i_k * dst.stride_k) * elem_bytes.
 * Both layouts are indexed by the same logical index: their non-unit extents
 * must be equal, in order ("copy -> gmem_smem", section "What it accepts",
 * row "dtype / shape"; "permute_layout", section "What it accepts", row
 * "operands").  Words are moved as raw bits; nothing is converted.  Bytes of
 * dst outside the destination image are never written.
 *
 * Conventions for every entry point
 *   - Strides and offsets count ELEMENTS of elem_bytes bytes, not bytes.
 *   - Layout structs are read during the call and not retained.
 *   - Device pointers are plain CUDA device addresses owned by the caller;
 *     the library never allocates, frees or retains user buffers.
 *   - `stream` is a cudaStream_t (the type below is the same pointer type);
 *     NULL is the legacy default stream.  Launches are asynchronous on it.
 *   - Every function returns an lc_status (0 = LC_OK); nothing throws or
 *     aborts across the ABI.  On an error nothing has been launched, except
 *     LC_ERR_CUDA, which reports the CUDA runtime's launch error.
 *   - One process, one GPU: the current CUDA device of the calling thread.
 */
#ifndef LAYOUT_COPY_H_
#define LAYOUT_COPY_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LC_MAX_RANK 8

/* Same pointer type as cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st *lc_stream_t;

/* A TileLayout plus this library's batching fields.
 *   rank         1..LC_MAX_RANK
 *   shape[k]     >= 0; unit modes (extent 1) are ignored when pairing modes
 *   stride[k]    elements; >= 0 on the source (0 = broadcast read),
 *                > 0 on the destination for every non-unit mode
 *   offset       >= 0, element offset of tile 0
 *   tile_stride  >= 0, elements between consecutive tiles; 0 means the
 *                layout's cosize, 1 + sum_k (shape_k - 1) * stride_k, i.e.
 *                tiles packed back to back.  The pages show a single tile
 *                or a serial `pipe` loop ("permute_layout", section
 *                "Demonstration program"); tiles are that loop, batched. */
typedef struct {
    int32_t rank;
    int64_t shape[LC_MAX_RANK];
    int64_t stride[LC_MAX_RANK];
    int64_t offset;
    int64_t tile_stride;
} lc_tile_layout;

typedef enum {
    LC_OK = 0,
    LC_ERR_NULL = 1,            /* a required pointer is NULL */
    LC_ERR_RANK = 2,            /* rank outside 1..LC_MAX_RANK */
    LC_ERR_SHAPE = 3,           /* negative extent or n_tiles, or P not whole */
    LC_ERR_EXTENT_MISMATCH = 4, /* non-unit extents differ ("extent mismatch") */
    LC_ERR_ELEM_BYTES = 5,      /* elem_bytes not in {1,2,4,8,16} */
    LC_ERR_BAD_STRIDE = 6,      /* negative stride/offset, or 0 on dst */
    LC_ERR_NOT_INJECTIVE = 7,   /* two logical indices share a dst offset */
    LC_ERR_OVERLAP = 8,         /* src and dst byte ranges overlap (other than
                                   an exact in-place unit permute) */
    LC_ERR_ALIGN = 9,           /* pointer not aligned to elem_bytes */
    LC_ERR_NO_SWIZZLE = 10,     /* no conflict-free XOR swizzle ("fail") */
    LC_ERR_CUDA = 11,           /* CUDA runtime error at launch */
    LC_ERR_TIMEOUT = 12,        /* a bounded device wait gave up */
    LC_ERR_UNSUPPORTED = 13,    /* a forced kernel class cannot take this copy */
    LC_ERR_OVERFLOW = 14,       /* an offset does not fit in 63 bits */
    LC_ERR_STAGING = 15,        /* a staging buffer is too small */
    LC_ERR_LOOP_LAYOUT = 16,    /* a loop layout is not an exact partition */
    LC_ERR_UNDECIDED = 17,      /* the destination could not be shown one-to-one:
                                   no stride split settles it and the modes left
                                   hold over 2^24 words to enumerate */
    LC_ERR_NOT_MAPPED = 18      /* lc_layout_copy_mapped: a byte range is not
                                   memory the device can address (pageable host
                                   memory, or a range leaving its mapping) */
} lc_status;

/* Kernel classes (the planner picks one; lc_layout_copy_ex can force one). */
typedef enum {
    LC_KERNEL_AUTO = 0,
    /* [outer, threads, vec] vector copy: the destination-ordered logical
     * index is split into vectors of the widest of 16/8/4/2/1 bytes that keep
     * every per-thread pointer aligned ("copy -> gmem_smem", sections
     * "Algorithm" steps 1-3; TileLang "loop_mapping.py" partition).  Takes
     * every valid copy; the fast path for copies whose innermost mode is
     * contiguous on both sides (identity copies, row gathers, axis permutes
     * that keep the last axis). */
    LC_KERNEL_VEC_COPY = 1,
    /* Warp register-staged permute: units of 32*P elements, dense on both
     * sides, are staged in a per-warp shared-memory slot with 16-byte
     * coalesced loads ("copy -> gmem_smem" [outer, threads, vec] split), each
     * unit is permuted in place through registers with the per-lane XOR
     * swizzle j = r ^ ((lane >> shift) & mask) chosen by the bank simulator
     * ("permute_layout", section "Algorithm"), and the slot leaves with
     * 16-byte stores.  Small transposed units. */
    LC_KERNEL_WARP_PERMUTE = 2,
    /* Tile transpose: TMA tensor loads of 128- or 256-byte x R-row tiles
     * into a shared-memory ring (mbarrier pipelined), 16-byte shared reads,
     * an in-register transpose of the sub-16-byte elements, 16-byte
     * coalesced global stores.  Large 2-D transposes with batch modes.  Its
     * direct form (1- and 2-byte words, both extents whole 16-byte blocks,
     * at most 96 / 64 MiB a side) loads each block's rows with 16-byte
     * global loads straight into registers instead: no TMA and no shared
     * memory.  Its TMA-store form stages each transposed tile in shared
     * memory and stores it with a TMA tensor store: destination rows of
     * whole 16-byte chunks, 4-byte words at every size, 1- and 2-byte words
     * above 256 MiB a side (2-byte words not with destination rows a
     * multiple of 32 KiB apart), 8- and 16-byte words up to 256 MiB
     * (lc_plan_info.tile_form). */
    LC_KERNEL_TILE_TRANSPOSE = 3,
    /* Shared-memory transpose for any alignment: tiles of 64 source rows
     * (32 for 16-byte words), each row staged as aligned chunks (4 bytes for
     * words of up to 4 bytes, else the word) from the chunk boundary at or
     * below its first word; copied global -> shared in source order and
     * shared -> global in destination order, one word per store ("copy ->
     * gmem_smem", its two copies around a swizzled shared layout); the chunk
     * swizzle slot = k ^ ((x >> shift) & mask) is chosen by the bank
     * simulator so that both copies are conflict-free.  Transposes whose
     * strides or bases the TMA path cannot take. */
    LC_KERNEL_SMEM_TRANSPOSE = 4,
    /* TMA tensor copy: the innermost mode is contiguous on both sides (at
     * least 64 bytes, a multiple of 16) and every other stride is a multiple
     * of 16 bytes, at most 5 modes.  Boxes of whole inner modes (about
     * 16 KiB) go global -> shared by TMA tensor loads and shared -> global by
     * TMA tensor stores through a second tensor map with the destination
     * strides; one thread per CTA drives a 6-stage ring.  Axis permutes that
     * keep the last axis, strided slices, row gathers. */
    LC_KERNEL_TMA_COPY = 5,
    /* Warp-shuffle permute: of the mode contiguous in the source and the mode
     * contiguous in the destination, one spans exactly 16 bytes (V = 16 /
     * elem_bytes words, elem_bytes <= 8) and the other a multiple of V
     * words: the scale-factor transpose of "permute_layout" ("Demonstration
     * program", a (4, 32) fp32 block written with strides (1, 4)) and its
     * mirror.  Groups of V lanes load one V x V block as V 16-byte chunks,
     * transpose it in registers by warp shuffles and store V 16-byte chunks;
     * no shared memory.  Other strides and both bases must be 16-byte
     * aligned. */
    LC_KERNEL_WARP_SHUFFLE = 6,
    /* Staged tile copy ("copy -> gmem_smem", its demonstration program): one
     * CTA of 256 threads per tile, global -> shared through the source
     * layout, a barrier, shared -> global through the destination layout,
     * the shared tile swizzled by the library's choice; tiles of at most
     * LC_STAGED_MAX_BYTES (lc_layout_copy_staged sets threads, swizzle and
     * traces). */
    LC_KERNEL_SMEM_STAGED = 7
} lc_kernel;

/* What the planner decided for one copy (filled by lc_plan). */
typedef struct {
    int32_t kernel;            /* lc_kernel */
    int32_t elem_bytes;        /* word size moved (after fusing a contiguous
                                  inner run into wider words) */
    int32_t n_modes;           /* canonical modes, outermost first */
    int64_t extent[LC_MAX_RANK + 1];
    int64_t src_stride[LC_MAX_RANK + 1];
    int64_t dst_stride[LC_MAX_RANK + 1];
    int64_t total;             /* logical words moved (all tiles) */
    /* vector copy */
    int32_t vec;               /* words per vector */
    int64_t run;               /* words in the contiguous inner run (1 if none) */
    /* warp permute (P, XOR swizzle); shared-memory transpose (swizzle) */
    int32_t unit_modes;        /* number of modes in one unit (innermost) */
    int32_t P;                 /* words per lane per unit */
    int32_t k, shift, mask;    /* XOR swizzle (mask = 2^k - 1) */
    int32_t conflicts_read, conflicts_write;
    int64_t units_per_chunk;
    /* tile transpose (also the shared-memory transpose's tile and the TMA
     * tensor copy's box) */
    int32_t tile_rows;         /* R: source rows per tile (per warp tile in the direct form) */
    int32_t tile_cols;         /* words per tile row */
    int32_t stages;            /* TMA ring stages; 0: the tile transpose's direct form
                                  (1- and 2-byte words in whole 16-byte blocks, loaded
                                  straight into registers: no TMA, no shared memory) */
    /* reserved, always 0: each launch sizes its grid from the device's SM
     * count and the kernel's occupancy, which the host-only planner does not
     * query */
    int32_t grid, block, smem_bytes;
    /* tile transpose: 0 the TMA ring with thread stores, 1 the direct form
     * (stages 0), 2 the TMA ring whose output tiles leave by TMA tensor
     * stores; 0 for the other classes */
    int32_t tile_form;
} lc_plan_info;

/* The copy.  Validates, plans (host only, microseconds), launches one
 * kernel on `stream`.  n_tiles >= 0; a copy of zero words returns LC_OK
 * without launching (and then src/dst may be NULL).
 * In place: src and dst may be the same memory when every dense unit of the
 * warp-permute class is read and written at the same bytes (same base
 * address, equal batch and tile strides) -- the aliasing case of
 * "permute_layout" (its introduction: the permute tolerates aliased buffers); each
 * warp stages whole units before writing them back.  Any other overlap of
 * the two byte ranges is refused with LC_ERR_OVERLAP.
 * Errors: LC_ERR_NULL, _RANK, _SHAPE, _EXTENT_MISMATCH, _ELEM_BYTES,
 * _BAD_STRIDE, _NOT_INJECTIVE, _OVERLAP, _ALIGN, _OVERFLOW (before any
 * launch); LC_ERR_CUDA (launch failed).  Device-side wait timeouts are
 * reported later by lc_last_device_error. */
int lc_layout_copy(const void *src, const lc_tile_layout *src_layout,
                   void *dst, const lc_tile_layout *dst_layout,
                   int32_t elem_bytes, int64_t n_tiles, lc_stream_t stream);

/* As lc_layout_copy, with the kernel class forced (LC_KERNEL_AUTO = let the
 * planner choose).  LC_ERR_UNSUPPORTED when the forced class cannot take the
 * copy.  Meant for tests and benchmarks that compare classes. */
int lc_layout_copy_ex(const void *src, const lc_tile_layout *src_layout,
                      void *dst, const lc_tile_layout *dst_layout,
                      int32_t elem_bytes, int64_t n_tiles, int32_t kernel,
                      lc_stream_t stream);

/* The copy between two HOST buffers.  The tiles are split into chunks that
 * are moved host -> device, permuted and moved device -> host through
 * `staging`, a caller-owned device buffer of at least staging_bytes bytes
 * (lc_host_staging_bytes gives the size for full pipelining, three chunk
 * slots; a smaller buffer gets smaller chunks).  Uploads, permutes and downloads run on two internal copy streams
 * and on `stream`, overlapped chunk by chunk and ordered by events; the work
 * is queued behind what `stream` already holds, and `stream` resumes after the
 * last download, so synchronising `stream` completes the copy.  Host buffers
 * should be page-locked for the transfers to overlap.  Bytes of dst_host
 * outside the destination image keep their values (when the image has holes
 * the chunk's span is uploaded first).  Layout semantics as lc_layout_copy;
 * host ranges may not overlap (LC_ERR_OVERLAP).  Errors: as lc_layout_copy,
 * plus LC_ERR_STAGING when staging_bytes cannot hold one chunk, LC_ERR_ALIGN
 * when staging is not 256-byte aligned.  The library creates its two copy streams and their
 * events once per device and allocates no memory. */
int lc_layout_copy_host(const void *src_host, const lc_tile_layout *src_layout,
                        void *dst_host, const lc_tile_layout *dst_layout,
                        int32_t elem_bytes, int64_t n_tiles, void *staging,
                        int64_t staging_bytes, lc_stream_t stream);

/* The copy between buffers in page-locked host memory, run by the copy
 * kernels themselves over the CPU-GPU link: no staging buffer and no copy
 * engine, every word crosses the link once each way, and the permute happens
 * on the way (the same operation as lc_layout_copy: Apache TVM docs "copy ->
 * gmem_smem" and "permute_layout"; the layouts, the word size and the tiles
 * have the same meaning).  src_host and dst_host are host addresses of
 * memory the device can address: page-locked and mapped (cudaHostAlloc /
 * torch pin_memory, or cudaHostRegister'd), or device memory.  Each byte
 * range the layouts reach, [first, last] on each side, is looked up with
 * cudaPointerGetAttributes: both ends must be addressable and contiguous in
 * the device's view, else LC_ERR_NOT_MAPPED (nothing is launched).  The plan
 * takes only kernel classes that move words with plain loads and stores (the
 * warp shuffle and warp permutes, the tile transpose's direct form, the
 * shared-memory transpose, the staged and vector copies): no TMA tensor map
 * is built over host memory.  When both buffers are device memory the call
 * is lc_layout_copy's.  Asynchronous on `stream`; the caller keeps
 * both buffers alive and unmodified (src) until the stream has run the copy.
 * It allocates nothing and needs no staging memory, so callers that cannot
 * allocate device memory and hold page-locked buffers can use it in place
 * of lc_layout_copy_host_static.  Errors: as lc_layout_copy, plus
 * LC_ERR_NOT_MAPPED.  Measured on GB300 (a Grace host): the 2^20-tile
 * scale-factor permute moves 336-338 GB/s of link traffic, host to host,
 * where the copy engines move 340 GB/s in both directions at once and
 * lc_layout_copy_host 320. */
int lc_layout_copy_mapped(const void *src_host, const lc_tile_layout *src_layout, void *dst_host,
                          const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles,
                          lc_stream_t stream);

/* Staging bytes lc_layout_copy_host needs for this copy (three slots of a
 * chunk of about 48 MiB of source tiles -- at least one tile, at most 1024
 * chunks -- when the tiles can be chunked, else the whole source and
 * destination spans); 0 for invalid arguments. */
int64_t lc_host_staging_bytes(const lc_tile_layout *src_layout,
                              const lc_tile_layout *dst_layout,
                              int32_t elem_bytes, int64_t n_tiles);

/* Bytes of the staging array built into the library for
 * lc_layout_copy_host_static (on every GPU that loads the library, for the
 * life of the process). */
#define LC_STATIC_STAGING_BYTES (32 * 1024 * 1024)

/* lc_layout_copy_host for callers that cannot allocate device memory.  (The
 * source pages have no counterpart: this is a deployment convenience.)  Some
 * callers cannot hand over a staging buffer: a plugin inside an application
 * whose own allocator owns all device memory and gives none out, or code
 * that must avoid cudaMalloc because it can synchronise the whole device.
 * This entry point stages through an LC_STATIC_STAGING_BYTES array that
 * lives in the library and allocates and frees nothing.  Chunks of tiles are
 * uploaded, permuted and downloaded in order on `stream` alone (no overlap
 * between transfers); synchronise `stream` to finish.  The copies are
 * asynchronous only for page-locked host buffers; with pageable buffers
 * CUDA makes them synchronous with the host, and the result is the same.
 * Set-up: the first call on a device, with that device current, looks up
 * the array's device address (loading the library's code onto the device if
 * needed) before it checks anything else, so any call completes it; that
 * first call must not itself run inside a stream capture.  The address is
 * kept for the life of the process: do not call this entry point on a
 * device after cudaDeviceReset on it.  Every call shares the array and it
 * keeps the previous call's bytes (nothing in it needs to start at zero);
 * calls that overlap on the GPU, e.g. on two streams, race on it --
 * serialise them.
 * Errors: as lc_layout_copy_host; LC_ERR_STAGING when even one tile's
 * source and destination spans (each rounded up to 256 bytes) exceed
 * LC_STATIC_STAGING_BYTES, or when the whole copy must fit at once (one
 * tile, or destination tiles that interleave) and does not.  Every check
 * that can refuse the copy runs before anything is queued; an LC_ERR_CUDA
 * from a later chunk leaves the chunks before it queued on `stream` (a
 * partial copy). */
int lc_layout_copy_host_static(const void *src_host, const lc_tile_layout *src_layout,
                               void *dst_host, const lc_tile_layout *dst_layout,
                               int32_t elem_bytes, int64_t n_tiles, lc_stream_t stream);

/* Largest window of lc_window_sum_f32. */
#define LC_WINDOW_SUM_MAX 64

/* Window sum through a cooperatively fetched shared-memory chunk (MLC course
 * "Ep7: GPU and Hardware Acceleration", section "Window Sum Example", which
 * has window 3):  b[i] = a[i] + a[i+1] + ... + a[i+window-1] for i in
 * [0, n_out), float32 additions left to right.  `a` (device) holds
 * n_out + window - 1 floats, `b` (device) n_out floats; 4-byte aligned,
 * non-overlapping.  Asynchronous on `stream`.  Errors: LC_ERR_SHAPE (n_out < 0
 * or window outside 1..LC_WINDOW_SUM_MAX), LC_ERR_NULL, LC_ERR_ALIGN,
 * LC_ERR_OVERLAP, LC_ERR_OVERFLOW, LC_ERR_CUDA. */
int lc_window_sum_f32(const float *a, float *b, int64_t n_out, int32_t window,
                      lc_stream_t stream);

/* The planner alone: validation and the plan lc_layout_copy_ex would launch
 * for (layouts, elem_bytes, n_tiles, kernel), without touching the GPU.
 * Pointer checks (NULL, alignment, overlap) are skipped.  `out` must not be
 * NULL. */
int lc_plan(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout,
            int32_t elem_bytes, int64_t n_tiles, int32_t kernel,
            lc_plan_info *out);

/* XOR swizzle of the warp permute ("permute_layout", section "Algorithm",
 * steps 1-2; section "What it accepts", row "bank-freedom").  Both layouts
 * describe ONE warp's shard: unit modes are dropped, the non-unit modes are
 * paired in order and neighbours contiguous on both sides are merged, giving
 * extent / src_str / dst_str with P = prod(extent) / 32 words per lane.  The
 * bank simulator (32 banks of 4-byte words; 128-byte wavefronts, i.e. 32
 * lanes for words up to 4 bytes, 16 lanes for 8, 8 lanes for 16; a bank's
 * degree is the number of distinct 4-byte words it serves) tries k = 0 ..
 * log2(P) (k = 0 only when P is not a power of two) and, for each k, shift =
 * 0 .. 5-k, and returns the first pair whose read phase and write phase both
 * have degree 1; mask = 2^k - 1.  Offsets of the layouts are ignored
 * (addresses are relative to a 128-byte-aligned base).
 * Outputs (all must be non-NULL): k, shift, mask, and the worst bank degree
 * of each phase at that choice.  LC_ERR_NO_SWIZZLE when no pair is
 * conflict-free (outputs then hold the pair with the lowest worst degree);
 * LC_ERR_SHAPE when prod(extent) is not a multiple of 32. */
int lc_choose_swizzle(const lc_tile_layout *src_layout,
                      const lc_tile_layout *dst_layout, int32_t elem_bytes,
                      int32_t *k, int32_t *shift, int32_t *mask,
                      int32_t *conflicts_read, int32_t *conflicts_write);

/* The bank simulator itself for one given (k, shift), same model and
 * alignment as lc_choose_swizzle: worst degree of each phase. */
int lc_swizzle_conflicts(const lc_tile_layout *src_layout,
                         const lc_tile_layout *dst_layout, int32_t elem_bytes,
                         int32_t k, int32_t shift, int32_t *conflicts_read,
                         int32_t *conflicts_write);

/* The synthesized [outer, threads, vec] partition of one global <-> shared
 * copy executed by `threads` threads ("copy -> gmem_smem", section
 * "Algorithm" steps 1-2, section "How inputs change the algorithm"): the
 * global layout drives the canonical (stride-descending) order, vector
 * widths of 16, 8, 4, 2, 1 bytes are tried widest first, and a width of vec
 * words is accepted when the innermost mode is contiguous on both sides with
 * an extent that is a multiple of vec, every other stride on both sides and
 * both offsets are multiples of vec, and threads * vec divides the element
 * count.  Outputs: vec (words) and outer = count / (threads * vec).
 * LC_ERR_SHAPE ("declines") when the element count is not a multiple of
 * `threads`. */
int lc_gmem_smem_partition(const lc_tile_layout *global_layout,
                           const lc_tile_layout *shared_layout,
                           int32_t elem_bytes, int32_t threads,
                           int32_t *vec, int64_t *outer);

/* Synchronises `stream`, then reads and clears this device's error word,
 * which kernels set when a bounded wait gives up (LC_ERR_TIMEOUT).
 * Returns LC_OK when the word was clear; LC_ERR_CUDA if the stream reported
 * an error.  `detail` (may be NULL) receives the raw word. */
int lc_last_device_error(lc_stream_t stream, uint64_t *detail);

/* Failure-path check: launches one tiny kernel that waits on a shared-memory
 * barrier nothing ever arrives at, giving up after timeout_ns nanoseconds
 * (clamped to 1 us .. 1 s), so that the bounded-wait error path can be
 * tested without hanging anything.  lc_last_device_error then reports
 * LC_ERR_TIMEOUT. */
int lc_debug_wait_timeout(int64_t timeout_ns, lc_stream_t stream);

/* ---- P4's warp permute on shared-memory buffers ------------------------
 * Apache TVM docs "permute_layout" define the permute as a warp-scope op
 * between two layout-carrying buffers in shared memory, safe when they
 * alias.  lc_warp_unit is one such op, planned on the host: the aligned
 * modes of one unit (logical order, last mode fastest; strides in words),
 * P = words per lane (the unit holds 32 * P words), and the XOR swizzle
 * j = r ^ ((lane >> shift) & mask) chosen by the bank simulator.  The
 * device side is in layout_copy_device.cuh (warp_unit_offsets,
 * warp_unit_permute). */
#define LC_WARP_UNIT_MAX_P 32

typedef struct {
    int32_t n_modes;
    int32_t extent[LC_MAX_RANK];
    int32_t src_stride[LC_MAX_RANK];
    int32_t dst_stride[LC_MAX_RANK];
    int32_t P, k, shift, mask;
    int32_t conflicts_read, conflicts_write;  /* worst bank degree per phase */
    int32_t src_cosize, dst_cosize;           /* words each buffer spans */
} lc_warp_unit;

/* Plans one warp-scope permute of a single tile (n_tiles = 1) between
 * buffers with these layouts ("permute_layout", sections "What it accepts"
 * and "Algorithm").  Host only.  Errors: as lc_layout_copy's validation;
 * LC_ERR_SHAPE when the element count is not 32 * P with 1 <= P <=
 * LC_WARP_UNIT_MAX_P, or a stride or span does not fit 31 bits;
 * LC_ERR_NO_SWIZZLE when no (k, shift) is conflict-free -- `out` then holds
 * the pair with the lowest worst degree and the op still runs correctly. */
int lc_warp_unit_plan(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout,
                      int32_t elem_bytes, lc_warp_unit *out);

/* Runs the op on n_units units, each staged in shared memory.  src holds
 * n_units source buffers back to back (unit i at i * src_cosize * elem_bytes
 * bytes), dst likewise with dst_cosize.  For each unit, a warp copies the
 * source buffer into shared buffer A and (in_place = 0, unless the
 * destination image is the whole buffer: its strides form an exact mixed
 * radix) the destination buffer into shared buffer B, permutes A -> B
 * (in_place = 0) or A -> A (in_place = 1,
 * the aliased form: the destination layout is applied inside A, which needs
 * src_cosize >= dst_cosize), and copies the destination buffer back to dst.
 * Bytes of the destination buffer outside its image keep their values
 * (in_place = 0) or hold A's (in_place = 1).  A warp stages up to 8 units
 * at a time (2 KiB of each buffer kind), copying them in 16-byte chunks when
 * both buffer sizes are multiples of 16 bytes.  Each buffer must fit
 * LC_WARP_UNIT_MAX_BYTES.  Asynchronous on `stream`.  Errors: LC_ERR_NULL,
 * LC_ERR_SHAPE (buffers too large, bad counts), LC_ERR_ALIGN (pointers not
 * 16-byte aligned), LC_ERR_OVERLAP (src and dst ranges overlap),
 * LC_ERR_CUDA. */
#define LC_WARP_UNIT_MAX_BYTES 8192
int lc_warp_unit_run(const void *src, void *dst, const lc_warp_unit *unit, int32_t elem_bytes,
                     int64_t n_units, int32_t in_place, lc_stream_t stream);

/* ---------------------------------------------------------------------------
 * The global <-> shared copy of Apache TVM docs "copy -> gmem_smem" as a
 * device primitive for kernels that stage through shared memory.
 *
 * A shared buffer may be swizzled: the byte at shared offset o (as its
 * layout places it) is stored at
 *     o ^ (((o >> row_log2) & ((1 << bits) - 1)) << chunk_log2),
 * i.e. the `bits`-bit field above row_log2 is XORed into the index of the
 * 2^chunk_log2-byte chunk; bytes inside a chunk keep their order.  The page
 * names a swizzle without giving its formula; this XOR form is the library's
 * reading (the per-row XOR of "permute_layout" applied to chunks).  bits = 0
 * is no swizzle; otherwise row_log2 >= chunk_log2 + bits (so that the map is
 * one-to-one) and the chunk holds at least one element.
 * ------------------------------------------------------------------------- */
typedef struct {
    int32_t bits;
    int32_t chunk_log2;
    int32_t row_log2;
} lc_smem_swizzle;

/* One copy between a global and a shared buffer by `threads` threads, in the
 * [outer, threads, vec] split ("copy -> gmem_smem", section "Algorithm"
 * steps 1-3): the modes in the global side's canonical order (stride
 * descending, neighbours contiguous on both sides merged), vectors of `vec`
 * elements, round f of thread tid moving elements
 * [(f * threads + tid) * vec, + vec) of that order.  When threads * vec does
 * not divide the element count, the last round is partial and the threads
 * past the end do nothing (`guarded`; TileLang "loop_mapping.py": such
 * threads get no work behind a guard).  Filled by lc_gmem_smem_plan; read
 * by lc_device::gmem_smem_copy in layout_copy_device.cuh. */
typedef struct {
    int32_t n_modes;
    int64_t extent[LC_MAX_RANK];
    int64_t g_stride[LC_MAX_RANK];   /* elements */
    int64_t s_stride[LC_MAX_RANK];   /* elements */
    int64_t g_offset, s_offset;      /* elements */
    int32_t elem_bytes, vec, threads;
    int64_t outer;                   /* rounds: ceil(total / (threads * vec)) */
    int64_t total;                   /* elements (< 2^31) */
    int32_t guarded;
    lc_smem_swizzle swizzle;
    /* vector-start indices are split into mode digits by multiplying:
     * digit i of n is n - q * extent[i], q = (umulhi(n, div_m[i]) + n) >> div_s[i] */
    uint32_t div_m[LC_MAX_RANK];
    int32_t div_s[LC_MAX_RANK];
} lc_gmem_smem;

/* Plans one global <-> shared copy: the two layouts index the same logical
 * elements (equal non-unit extents, as for lc_layout_copy; tile_stride is
 * ignored), `threads` in 1..1024, `swizzle` the shared buffer's swizzle
 * (NULL = none).  The vector is the widest of 16, 8, 4, 2, 1 bytes with the
 * innermost mode contiguous on both sides and a multiple of it, every other
 * stride and both offsets multiples of it, and -- with a swizzle -- at most
 * one chunk ("copy -> gmem_smem", section "How inputs change the algorithm",
 * last paragraph).  Host only.  Errors: LC_ERR_NULL, LC_ERR_RANK,
 * LC_ERR_EXTENT_MISMATCH, LC_ERR_ELEM_BYTES, LC_ERR_BAD_STRIDE (a negative
 * stride or offset, or a swizzle that is not one-to-one or splits an
 * element), LC_ERR_SHAPE (threads outside 1..1024, 2^31 elements or more). */
int lc_gmem_smem_plan(const lc_tile_layout *global_layout, const lc_tile_layout *shared_layout,
                      int32_t elem_bytes, int32_t threads, const lc_smem_swizzle *swizzle,
                      lc_gmem_smem *out);

/* Largest shared tile of lc_layout_copy_staged, in bytes. */
#define LC_STAGED_MAX_BYTES (96 * 1024)

/* "copy -> gmem_smem"'s demonstration program as a copy: each tile is
 * staged through shared memory by one CTA of `threads` threads (a multiple
 * of 32, at most 1024), copy 1 global -> shared through the source layout
 * (the source drives the canonical order), a CTA barrier, copy 2 shared ->
 * global through the destination layout (the destination drives), both by
 * lc_device::gmem_smem_copy.  The shared tile holds the tile's logical box
 * row-major, under `swizzle` (NULL: the library picks, with its bank
 * simulator, the swizzle that makes both copies' shared accesses least
 * conflicted).  Tiles are spread over a grid of resident CTAs.
 *   trace_in, trace_out  NULL, or n_tiles * N int64 words of device memory
 *          (N = the tile's element count) receiving, at tile * N + the
 *          element's row-major index in the tile, f * threads + tid of the
 *          round and thread that moved it in copy 1 / copy 2.
 * Results equal lc_layout_copy's.  Asynchronous on `stream`.  Errors: as
 * lc_layout_copy (source and destination may not overlap), plus
 * LC_ERR_SHAPE when a tile's box exceeds LC_STAGED_MAX_BYTES (after
 * rounding up to the swizzle's span, 2^(chunk_log2 + bits) bytes) or
 * `threads` is invalid, and lc_gmem_smem_plan's errors for the swizzle. */
int lc_layout_copy_staged(const void *src, const lc_tile_layout *src_layout, void *dst,
                          const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles,
                          int32_t threads, const lc_smem_swizzle *swizzle, int64_t *trace_in,
                          int64_t *trace_out, lc_stream_t stream);

/* ---------------------------------------------------------------------------
 * Loop-layout override of the default partition (TileLang tutorial
 * "loop_mapping.py", module docstring).  The default plan flattens the nest
 * row-major, groups vector_size consecutive points, rotates the groups over
 * num_thread threads and turns the rest into a per-thread serial loop; a
 * ``loop_layout=`` annotation replaces that plan.  The page says no more, so
 * this library reads an override as follows.
 *
 * The nest is one tile's logical box (the non-unit extents both layouts
 * share, in logical order).  A point's row-major flat index is read as
 * mixed-radix digits over the loop layout's extents (mode 0 slowest) and
 *     thread = sum_k digit_k * thread_stride[k],
 *     slot   = sum_k digit_k * slot_stride[k].
 * The override must be an exact partition: the extents multiply to the
 * tile's element count N, each non-unit mode has exactly one of its two
 * strides non-zero, and the thread modes and the slot modes, each sorted by
 * stride, form mixed radices (the smallest stride 1, each next stride the
 * previous stride times its extent).  Then the points fill
 * [0, T) x [0, L) with T * L = N, T the product of the thread extents and L
 * of the slot extents, one point per (thread, slot).  The default plan is
 * the override (N / (T V): slot stride V), (T: thread stride 1),
 * (V: slot stride 1) -- lc_loop_layout_default.
 * ------------------------------------------------------------------------- */
#define LC_LOOP_MAX_THREADS 1024

typedef struct {
    int32_t rank;                       /* 1..LC_MAX_RANK */
    int64_t shape[LC_MAX_RANK];         /* >= 0 */
    int64_t thread_stride[LC_MAX_RANK]; /* >= 0 */
    int64_t slot_stride[LC_MAX_RANK];   /* >= 0 */
} lc_loop_layout;

/* The default plan for n_elems points, num_thread threads and vectors of
 * vector_size points, written as an override into `out` (three modes; unit
 * modes kept).  Host only.  Errors: LC_ERR_NULL; LC_ERR_SHAPE when a count
 * is below 1 (n_elems below 0) or num_thread * vector_size does not divide
 * n_elems (the page's guarded case, which no exact partition expresses). */
int lc_loop_layout_default(int64_t n_elems, int32_t num_thread, int32_t vector_size,
                           lc_loop_layout *out);

/* Checks that `loop` is an exact partition of n_elems points and reports
 * its threads T and slots per thread L.  Host only.  Errors: LC_ERR_NULL,
 * LC_ERR_RANK, LC_ERR_SHAPE (negative extent or n_elems, or the extents'
 * product is not n_elems), LC_ERR_BAD_STRIDE (a negative stride, or a
 * non-unit mode with both or neither stride non-zero), LC_ERR_LOOP_LAYOUT
 * (the thread or slot modes leave gaps or collide, or T exceeds
 * LC_LOOP_MAX_THREADS). */
int lc_loop_layout_info(const lc_loop_layout *loop, int64_t n_elems, int32_t *num_threads,
                        int64_t *slots_per_thread);

/* What lc_layout_copy_loop would do for these layouts, with both base
 * pointers assumed 16-byte aligned (host only, like lc_plan):
 *   num_threads, slots_per_thread  T and L of the override
 *   points_per_tile                N = T * L
 *   vec                            words moved per vector (1 = single words)
 *   split                          1 when the loop's and the tile's radices
 *                                  nest and a tile spans under 2^31 bytes:
 *                                  offsets are a per-thread part plus a
 *                                  per-slot part from a shared table
 * Errors: as lc_layout_copy_loop's validation. */
typedef struct {
    int32_t num_threads;
    int64_t slots_per_thread;
    int64_t points_per_tile;
    int32_t vec;
    int32_t split;
} lc_loop_plan_info;

int lc_loop_plan(const lc_tile_layout *src_layout, const lc_tile_layout *dst_layout, int32_t elem_bytes,
                 int64_t n_tiles, const lc_loop_layout *loop, lc_loop_plan_info *out);

/* lc_layout_copy with the partition given by `loop` instead of the
 * library's planner: each tile is one CTA of T threads (tiles spread over
 * the grid), and thread t moves its slots 0 .. L-1 in order, the point of
 * slot s being the one the override maps to (t, s).  Where the innermost
 * loop mode is a slot mode of slot stride 1, runs of consecutive slots that
 * are contiguous on both sides move as one vector of the widest of 16, 8,
 * 4, 2 bytes that keeps every pointer aligned ("loop_mapping.py": points
 * that share a lane vectorize; "copy -> gmem_smem" for the width rule).
 * The copied words equal lc_layout_copy's; only who moves them differs.
 *   trace  NULL, or n_tiles * N int64 words of device memory that receive
 *          trace[tile * N + flat] = t * L + s for every point moved (flat =
 *          the point's row-major index in the tile), to observe the
 *          partition.
 * Asynchronous on `stream`.  Errors: as lc_layout_copy (source and
 * destination may not overlap at all), plus lc_loop_layout_info's errors
 * for the tile's element count. */
int lc_layout_copy_loop(const void *src, const lc_tile_layout *src_layout,
                        void *dst, const lc_tile_layout *dst_layout,
                        int32_t elem_bytes, int64_t n_tiles, const lc_loop_layout *loop,
                        int64_t *trace, lc_stream_t stream);

/* Row-major strides of `shape` (the layout S[shape] with no strides given,
 * "copy -> gmem_smem", section "Demonstration program",
 * `TileLayout(S[shape])`): stride[rank-1] = 1, stride[k] = stride[k+1] *
 * max(shape[k+1], 1).  Host only.  Errors: LC_ERR_NULL, LC_ERR_RANK,
 * LC_ERR_SHAPE (negative extent), LC_ERR_OVERFLOW. */
int lc_row_major_strides(int32_t rank, const int64_t *shape, int64_t *stride);

/* Elements a buffer must hold for n_tiles tiles of `layout`: offset +
 * (n_tiles - 1) * tile_stride + cosize (tile_stride 0 = the cosize), or the
 * offset alone when no word is addressed (n_tiles = 0 or a zero extent).
 * Host only.  Returns -1 for an invalid layout or count, or on overflow. */
int64_t lc_layout_footprint(const lc_tile_layout *layout, int64_t n_tiles);

/* Human-readable name of a status / kernel class (static strings). */
const char *lc_status_string(int32_t status);
const char *lc_kernel_name(int32_t kernel);

#ifdef __cplusplus
}
#endif

#endif /* LAYOUT_COPY_H_ */
