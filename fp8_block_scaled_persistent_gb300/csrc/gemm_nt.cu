// gemm_nt.cu -- instantiations of the plain (GemmType::Normal) kernel:
// 128- and 256-column tiles, and the split-K schedule (128-column tiles).
#include "launch_impl.cuh"

namespace fp8g {

int smem_bytes_for(int block_n)
{
    return block_n == 256 ? Cfg<256>::kSmemBytes : Cfg<128>::kSmemBytes;
}

int panel_cols_for(int block_n)
{
    return block_n == 256 ? Cfg<256>::kPanelCols : Cfg<128>::kPanelCols;
}

cudaError_t launch_nt(int block_n, bool split, const LaunchArgs &a)
{
    if (split)
        return block_n == 256 ? launch_one<256, kKindNT, true>(a) : launch_one<128, kKindNT, true>(a);
    if (block_n == 256)
        return launch_one<256, kKindNT, false>(a);
    return launch_one<128, kKindNT, false>(a);
}

}  // namespace fp8g
