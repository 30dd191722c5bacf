// TMA tensor stores from shared memory and their bulk-group completion,
// written from the public PTX ISA (cp.async.bulk.tensor, shared::cta ->
// global, bulk_group completion; cp.async.bulk.wait_group; fence.proxy.async).
#pragma once

#include <cstdint>

namespace lc {
namespace bulk {

// One tensor store of the box at shared address `src` to coordinates c[0 ..
// rank) of the tensor map, in the issuing thread's current bulk group.
__device__ __forceinline__ void tma_store(const void *tmap, int rank, const int32_t (&c)[5], uint32_t src) {
    switch (rank) {
        case 2:
            asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
                         "r"(src), "r"(c[0]), "r"(c[1])
                         : "memory");
            break;
        case 3:
            asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                             tmap),
                         "r"(src), "r"(c[0]), "r"(c[1]), "r"(c[2])
                         : "memory");
            break;
        case 4:
            asm volatile(
                "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(tmap),
                "r"(src), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3])
                : "memory");
            break;
        default:
            asm volatile(
                "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
                    tmap),
                "r"(src), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4])
                : "memory");
            break;
    }
}

__device__ __forceinline__ void commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the newest N bulk groups have finished reading shared memory.
template <int N>
__device__ __forceinline__ void wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// All bulk groups have completed.
__device__ __forceinline__ void wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Shared memory written by threads is read by the async proxy (TMA) next.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace bulk
}  // namespace lc
