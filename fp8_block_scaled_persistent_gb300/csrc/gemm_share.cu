// gemm_share.cu -- instantiations of the one-CTA kernel launched in clusters
// of two CTAs that share each A tile over DSMEM (fp8_gemm_kernel with SHARE):
// 256-column tiles, unsplit, for the plain GEMM and both grouped layouts.
#include "launch_impl.cuh"

namespace fp8g {

cudaError_t launch_share(int kind, const LaunchArgs &a)
{
    switch (kind) {
    case kKindNT: return launch_one<256, kKindNT, false, true>(a);
    case kKindContiguous: return launch_one<256, kKindContiguous, false, true>(a);
    case kKindMasked: return launch_one<256, kKindMasked, false, true>(a);
    default: return cudaErrorInvalidValue;
    }
}

int max_active_share_pairs(int dev) { return share_max_active<256>(dev); }

}  // namespace fp8g
