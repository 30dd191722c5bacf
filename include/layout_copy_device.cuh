/* Device side of the warp-scope permute between layout-carrying buffers
 * (Apache TVM docs "permute_layout", section "Algorithm", step 3: two
 * register-staged phases under the per-lane XOR swizzle).
 *
 * Usage inside a kernel, all 32 lanes of a warp together:
 *
 *     int32_t soff[PMAX], doff[PMAX];
 *     lc_device::warp_unit_offsets<W, PMAX>(unit, lane, soff, doff);  // once
 *     lc_device::warp_unit_permute<W, PMAX>(dst, src, unit.P, soff, doff);
 *
 * `unit` comes from lc_warp_unit_plan on the host (pass it by value or in
 * constant memory).  src and dst are byte addresses of the two buffers,
 * normally in shared memory, each aligned to the word size W; they may be
 * the same buffer or overlap in any way: every lane reads all of its P words
 * into registers, the warp synchronises, and only then does any lane write.
 * PMAX is a compile-time bound >= unit.P (at most LC_WARP_UNIT_MAX_P).
 * With the simulator's (k, shift), neither phase has shared-memory bank
 * conflicts (unit.conflicts_read / conflicts_write report the degrees). */
#ifndef LAYOUT_COPY_DEVICE_CUH_
#define LAYOUT_COPY_DEVICE_CUH_

#include <cuda_runtime.h>

#include <cstdint>

#include "layout_copy.h"

namespace lc_device {

template <int W> struct unit_word;
template <> struct unit_word<1> { using type = uint8_t; };
template <> struct unit_word<2> { using type = uint16_t; };
template <> struct unit_word<4> { using type = uint32_t; };
template <> struct unit_word<8> { using type = uint2; };
template <> struct unit_word<16> { using type = uint4; };

/* Element offsets of flat index `flat` of a unit (last mode fastest). */
__device__ __forceinline__ void unit_point(const lc_warp_unit &u, int32_t flat, int32_t &so, int32_t &dof) {
    so = 0;
    dof = 0;
    for (int i = u.n_modes - 1; i >= 0; --i) {
        const int32_t c = flat % u.extent[i];
        flat /= u.extent[i];
        so += c * u.src_stride[i];
        dof += c * u.dst_stride[i];
    }
}

/* Byte offsets, inside the two buffers, of the P words lane `lane` moves:
 * step r takes iteration j = r ^ ((lane >> shift) & mask), the logical index
 * unflatten(lane + 32 j) over the unit's extents (last mode fastest), and its
 * offset on each side.  When 32 lies on the divisibility chain of the unit's
 * suffix products (every suffix product divides 32 or is a multiple of it),
 * the lane digits and the j digits of lane + 32 j are disjoint, so its
 * offsets are those of lane plus those of 32 j: each lane unflattens its own
 * index and 32 * lane, and the j parts travel by warp shuffles.  Otherwise
 * each step unflattens its index.  Call with all 32 lanes of the warp. */
template <int W, int PMAX>
__device__ __forceinline__ void warp_unit_offsets(const lc_warp_unit &u, int lane, int32_t (&soff)[PMAX],
                                                  int32_t (&doff)[PMAX]) {
    bool nests = true;
    int32_t suffix = 1;
    for (int i = u.n_modes - 1; i >= 0; --i) {
        suffix *= u.extent[i];
        nests = nests && (suffix % 32 == 0 || 32 % suffix == 0);
    }
    const int sw = (lane >> u.shift) & u.mask;
    if (nests) {
        int32_t ls, ld, js, jd;
        unit_point(u, lane, ls, ld);
        unit_point(u, lane < u.P ? 32 * lane : 0, js, jd);
#pragma unroll
        for (int r = 0; r < PMAX; ++r) {
            const int j = (r ^ sw) & 31;
            soff[r] = (ls + __shfl_sync(0xffffffffu, js, j)) * W;
            doff[r] = (ld + __shfl_sync(0xffffffffu, jd, j)) * W;
        }
        return;
    }
#pragma unroll(PMAX <= 8 ? PMAX : 1)
    for (int r = 0; r < PMAX; ++r) {
        int32_t so, dof;
        unit_point(u, lane + 32 * (r ^ sw), so, dof);
        soff[r] = so * W;
        doff[r] = dof * W;
    }
}

/* The two phases for one unit: read src, synchronise the warp, write dst,
 * synchronise again (so the warp may reuse either buffer at once). */
template <int W, int PMAX>
__device__ __forceinline__ void warp_unit_permute(void *dst, const void *src, int P, const int32_t (&soff)[PMAX],
                                                  const int32_t (&doff)[PMAX]) {
    using T = typename unit_word<W>::type;
    const uint8_t *s = static_cast<const uint8_t *>(src);
    uint8_t *d = static_cast<uint8_t *>(dst);
    T regs[PMAX];
#pragma unroll
    for (int r = 0; r < PMAX; ++r)
        if (r < P) regs[r] = *reinterpret_cast<const T *>(s + soff[r]);
    __syncwarp();
#pragma unroll
    for (int r = 0; r < PMAX; ++r)
        if (r < P) *reinterpret_cast<T *>(d + doff[r]) = regs[r];
    __syncwarp();
}

}  // namespace lc_device

#endif /* LAYOUT_COPY_DEVICE_CUH_ */
