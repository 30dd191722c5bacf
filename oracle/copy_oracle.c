/*
 * Plain CPU definition of the strided tile layout copy.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is part of the oracle: only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it.  The
 * product library never links, loads or calls it, and it shares no code,
 * header or table with the CUDA path.
 *
 * What it computes (Apache TVM docs "copy -> gmem_smem", section "Algorithm",
 * and "permute_layout", section "Algorithm"): a layout maps a logical index
 * (i_0 .. i_{r-1}) to the element offset  base + sum_k i_k * stride_k  (the
 * "project" of the permute page, the "layout.apply" of the copy page).  The
 * copy moves, for every tile t and every logical index i, the w-byte word at
 * the source offset to the destination offset, both layouts being indexed by
 * the SAME logical index (both pages require equal extents).  Tile t adds
 * t * tile_stride on each side.
 *
 * The caller (oracle/definition.py) has already paired the non-unit modes of
 * the two layouts, so this loop sees one extent list and two stride lists.
 * The logical index is walked row-major, last index fastest, exactly like the
 * row-major flatten of the TileLang "loop_mapping.py" tutorial.  Words are
 * moved as raw bytes: no arithmetic touches the payload.
 */
#include <stdint.h>
#include <string.h>

#define ORACLE_MAX_RANK 16

int oracle_copy(const unsigned char *src, unsigned char *dst, int32_t w,
                int32_t rank, const int64_t *extent,
                const int64_t *src_stride, const int64_t *dst_stride,
                int64_t src_base, int64_t dst_base,
                int64_t src_tile_stride, int64_t dst_tile_stride,
                int64_t tile_begin, int64_t tile_end)
{
    int64_t idx[ORACLE_MAX_RANK];
    if (rank < 0 || rank > ORACLE_MAX_RANK || w <= 0)
        return -1;
    for (int k = 0; k < rank; ++k)
        if (extent[k] <= 0)
            return 0; /* empty logical box: nothing to move */

    for (int64_t t = tile_begin; t < tile_end; ++t) {
        for (int k = 0; k < rank; ++k)
            idx[k] = 0;
        for (;;) {
            int64_t so = src_base + t * src_tile_stride;
            int64_t d_o = dst_base + t * dst_tile_stride;
            for (int k = 0; k < rank; ++k) {
                so += idx[k] * src_stride[k];
                d_o += idx[k] * dst_stride[k];
            }
            memcpy(dst + d_o * (int64_t)w, src + so * (int64_t)w, (size_t)w);

            /* advance the logical index, last mode fastest */
            int k = rank - 1;
            while (k >= 0) {
                if (++idx[k] < extent[k])
                    break;
                idx[k] = 0;
                --k;
            }
            if (k < 0)
                break;
        }
    }
    return 0;
}
