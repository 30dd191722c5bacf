// Host-side launch interface between the ABI (api.cu) and the kernel
// translation units.  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "lc_internal.h"

namespace lc {

// Limit of every bounded device wait (LC_WAIT_TIMEOUT_NS overrides 2 s).
uint64_t wait_limit_ns();

// Opts `fn` into `attr_smem` bytes of dynamic shared memory on the current
// device (once) and reports the SM count and resident blocks per SM.
cudaError_t prepare(const void *fn, int threads, int smem, int attr_smem, int *sms, int *per_sm);

inline int finish_launch() { return cudaGetLastError() == cudaSuccess ? LC_OK : LC_ERR_CUDA; }

int launch_vec(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream);
int launch_warp(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream);
int launch_shuffle(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream);
int launch_staged(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream);
int launch_staged_layouts(const void *src, const lc_tile_layout *src_layout, void *dst,
                          const lc_tile_layout *dst_layout, int32_t elem_bytes, int64_t n_tiles, int32_t threads,
                          const lc_smem_swizzle *swizzle, int64_t *trace_in, int64_t *trace_out,
                          cudaStream_t stream);
int launch_tile(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream);
int launch_smem(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream);
int launch_tma_copy(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream);
int launch_loop(const LoopPlan &lp, const uint8_t *src, uint8_t *dst, int64_t *trace, cudaStream_t stream);

// Launches the plan's kernel class.  With `fallback`, a TMA plan whose tensor
// map the driver refuses runs on the non-TMA class of the same copy instead
// (tile transpose -> shared-memory transpose, tensor copy -> vector copy).
int launch_plan(const Plan &p, const uint8_t *src, uint8_t *dst, cudaStream_t stream, bool fallback);

// Error words of the modules whose kernels wait on barriers (each
// translation unit holds its own), read and cleared by lc_last_device_error.
cudaError_t take_error_tile(unsigned long long *v);
cudaError_t take_error_tma_copy(unsigned long long *v);
cudaError_t take_error_warp1(unsigned long long *v);
cudaError_t take_error_warp2(unsigned long long *v);
cudaError_t take_error_warp4(unsigned long long *v);
cudaError_t take_error_warp8(unsigned long long *v);
cudaError_t take_error_warp16(unsigned long long *v);

}  // namespace lc
