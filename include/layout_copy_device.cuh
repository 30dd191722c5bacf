/* Device side of the warp-scope permute between layout-carrying buffers
 * (Apache TVM docs "permute_layout", section "Algorithm", step 3: two
 * register-staged phases under the per-lane XOR swizzle), and of the
 * global <-> shared copy of "copy -> gmem_smem" (gmem_smem_copy, below).
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

/* ---- "copy -> gmem_smem": the global <-> shared copy -------------------
 *
 * Usage inside a kernel, all `plan.threads` threads of the copy together
 * (tid in [0, plan.threads)):
 *
 *     lc_device::gmem_smem_copy<W>(plan, global_base, shared_base, tid, true);   // global -> shared
 *     __syncthreads();
 *     lc_device::gmem_smem_copy<W>(plan2, global2, shared_base, tid, false);     // shared -> global
 *
 * `plan` comes from lc_gmem_smem_plan on the host (pass it by value or in
 * constant memory); W = plan.elem_bytes.  Element offsets are relative to
 * the two base pointers; global_base must be aligned to the vector
 * (plan.vec * W bytes) after adding plan.g_offset elements, shared_base to
 * 16 bytes.  Each thread runs its rounds f = 0 .. plan.outer - 1, stopping
 * at the first vector past the element count (the guard), and moves its
 * vector with one plan.vec * W-byte access on each side; the shared address
 * goes through plan.swizzle.  `trace` (NULL, or one int64 per shared element
 * offset) receives f * threads + tid for every element moved. */

/* Stored position of shared byte offset o under the swizzle. */
__device__ __forceinline__ uint32_t smem_swizzle(const lc_smem_swizzle &z, uint32_t o) {
    return o ^ (((o >> z.row_log2) & ((1u << z.bits) - 1u)) << z.chunk_log2);
}

template <int B> struct vec_word;
template <> struct vec_word<1> { using type = uint8_t; };
template <> struct vec_word<2> { using type = uint16_t; };
template <> struct vec_word<4> { using type = uint32_t; };
template <> struct vec_word<8> { using type = uint2; };
template <> struct vec_word<16> { using type = uint4; };

template <int B>
__device__ __forceinline__ void move_bytes(void *to, const void *from) {
    using T = typename vec_word<B>::type;
    *reinterpret_cast<T *>(to) = *reinterpret_cast<const T *>(from);
}

template <int W>
__device__ __forceinline__ void gmem_smem_copy(const lc_gmem_smem &p, void *global, void *shared, int tid,
                                               bool global_to_shared, int64_t *trace = nullptr) {
    uint8_t *const gb = static_cast<uint8_t *>(global);
    uint8_t *const sb = static_cast<uint8_t *>(shared);
    const int vb = p.vec * W;
    for (int64_t f = 0; f < p.outer; ++f) {
        const int64_t first = (f * p.threads + tid) * p.vec;
        if (first >= p.total) break;  // the guard: nothing past the element count
        uint32_t rest = static_cast<uint32_t>(first);
        int64_t g = p.g_offset, s = p.s_offset;
        for (int i = p.n_modes - 1; i >= 0; --i) {
            const uint32_t q = static_cast<uint32_t>(
                (static_cast<uint64_t>(__umulhi(rest, p.div_m[i])) + rest) >> p.div_s[i]);
            const uint32_t c = rest - q * static_cast<uint32_t>(p.extent[i]);
            g += static_cast<int64_t>(c) * p.g_stride[i];
            s += static_cast<int64_t>(c) * p.s_stride[i];
            rest = q;
        }
        uint8_t *gp = gb + g * W;
        uint8_t *sp = sb + smem_swizzle(p.swizzle, static_cast<uint32_t>(s * W));
        uint8_t *to = global_to_shared ? sp : gp;
        const uint8_t *from = global_to_shared ? gp : sp;
        switch (vb) {
            case 16: move_bytes<16>(to, from); break;
            case 8: move_bytes<8>(to, from); break;
            case 4: move_bytes<4>(to, from); break;
            case 2: move_bytes<2>(to, from); break;
            default: move_bytes<1>(to, from); break;
        }
        if (trace)
            for (int v = 0; v < p.vec; ++v) trace[s + v] = f * p.threads + tid;
    }
}

}  // namespace lc_device

#endif /* LAYOUT_COPY_DEVICE_CUH_ */
