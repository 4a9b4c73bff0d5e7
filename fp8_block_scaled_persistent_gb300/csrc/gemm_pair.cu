// gemm_pair.cu -- instantiations of the CTA-pair kernel with 256 x 128 tiles
// (gemm_kernel_pair.cuh) for the plain GEMM, the plain GEMM with an addend,
// and both grouped layouts, and the dispatch over both pair tile widths.
#include "gemm_pair_launch.cuh"

namespace fp8g {

cudaError_t launch_pair_256(int kind, const LaunchArgs &a);   // gemm_pair256.cu
int max_active_pairs_256(int dev);

int pair_panel_cols() { return PairCfg<128>::kPanelCols; }

int max_active_pairs(int dev, int block_n)
{
    return block_n == 256 ? max_active_pairs_256(dev) : pair_max_active<128>(dev);
}

cudaError_t launch_pair(int kind, int block_n, const LaunchArgs &a)
{
    if (block_n == 256)
        return launch_pair_256(kind, a);
    if (block_n == 128)
        return pair_launch_kind<128>(kind, a);
    return cudaErrorInvalidValue;
}

}  // namespace fp8g
