// gemm_pair256.cu -- instantiations of the CTA-pair kernel with 256 x 256
// tiles (gemm_kernel_pair.cuh) for the plain GEMM, the plain GEMM with an
// addend, and both grouped layouts.
#include "gemm_pair_launch.cuh"

namespace fp8g {

static_assert(PairCfg<256>::kPanelCols == PairCfg<128>::kPanelCols, "one D view serves both pair tile widths");

cudaError_t launch_pair_256(int kind, const LaunchArgs &a) { return pair_launch_kind<256>(kind, a); }

int max_active_pairs_256(int dev) { return pair_max_active<256>(dev); }

}  // namespace fp8g
