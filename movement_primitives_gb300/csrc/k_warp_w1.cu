// Warp permute kernels for 1-byte words (see k_warp.cuh).
#include "k_warp.cuh"

namespace lc {

int launch_warp_width1(int P, const WarpArgs &a, cudaStream_t s) { return launch_warp_w<1>(P, a, s); }
int launch_unit_width1(const UnitArgs &a, cudaStream_t s) { return launch_unit_w<1>(a, s); }
cudaError_t take_error_warp1(unsigned long long *v) { return take_module_error(v); }

}  // namespace lc
