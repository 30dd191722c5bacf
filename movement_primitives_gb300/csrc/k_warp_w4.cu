// Warp permute kernels for 4-byte words (see k_warp.cuh).
#include "k_warp.cuh"

namespace lc {

int launch_warp_width4(int P, const WarpArgs &a, cudaStream_t s) { return launch_warp_w<4>(P, a, s); }
int launch_unit_width4(const UnitArgs &a, cudaStream_t s) { return launch_unit_w<4>(a, s); }
cudaError_t take_error_warp4(unsigned long long *v) { return take_module_error(v); }

}  // namespace lc
