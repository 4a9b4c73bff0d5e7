// gemm_nt_acc.cu -- instantiations of the plain GEMM with an fp32 addend
// (kKindNTAcc, D = bf16(C + A B^T scaled)): 128- and 256-column tiles, and
// the split-K schedule (128-column tiles).
#include "launch_impl.cuh"

namespace fp8g {

cudaError_t launch_nt_acc(int block_n, bool split, const LaunchArgs &a)
{
    if (split)
        return block_n == 256 ? launch_one<256, kKindNTAcc, true>(a) : launch_one<128, kKindNTAcc, true>(a);
    if (block_n == 256)
        return launch_one<256, kKindNTAcc, false>(a);
    return launch_one<128, kKindNTAcc, false>(a);
}

}  // namespace fp8g
