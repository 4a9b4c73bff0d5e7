// gemm_masked.cu -- instantiations of the grouped kernel with the masked
// layout (GemmType::GroupedMasked).
#include "launch_impl.cuh"

namespace fp8g {

cudaError_t launch_masked(int block_n, const LaunchArgs &a)
{
    if (block_n == 256)
        return launch_one<256, kKindMasked, false>(a);
    return launch_one<128, kKindMasked, false>(a);
}

}  // namespace fp8g
