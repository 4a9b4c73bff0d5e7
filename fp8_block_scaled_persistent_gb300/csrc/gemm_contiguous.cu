// gemm_contiguous.cu -- instantiations of the grouped kernel with the
// contiguous layout (GemmType::GroupedContiguous).
#include "launch_impl.cuh"

namespace fp8g {

cudaError_t launch_contiguous(int block_n, const LaunchArgs &a)
{
    if (block_n == 256)
        return launch_one<256, kKindContiguous, false>(a);
    return launch_one<128, kKindContiguous, false>(a);
}

}  // namespace fp8g
