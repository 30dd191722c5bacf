// Warp permute kernels for 2-byte words (see k_warp.cuh).
#include "k_warp.cuh"

namespace lc {

int launch_warp_width2(int P, const WarpArgs &a, cudaStream_t s) { return launch_warp_w<2>(P, a, s); }
int launch_unit_width2(const UnitArgs &a, cudaStream_t s) { return launch_unit_w<2>(a, s); }
cudaError_t take_error_warp2(unsigned long long *v) { return take_module_error(v); }

}  // namespace lc
