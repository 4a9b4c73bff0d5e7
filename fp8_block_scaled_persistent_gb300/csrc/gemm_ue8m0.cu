// gemm_ue8m0.cu -- launch of the power-of-two-scale kernel
// (gemm_kernel_ue8m0.cuh): one CTA per SM, 512 threads, programmatic stream
// serialisation.
#include <atomic>

#include "gemm_kernel_ue8m0.cuh"

#ifndef FP8G_PDL
#define FP8G_PDL 1
#endif
#include "launch.h"

namespace fp8g {

int ue8m0_block_n() { return Ue8m0Cfg::kBN; }

int ue8m0_panel_cols() { return Ue8m0Cfg::kPanelCols; }

cudaError_t launch_ue8m0(const LaunchArgs &a)
{
    static std::atomic<unsigned long long> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(fp8_gemm_ue8m0_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Ue8m0Cfg::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid, 1, 1);
    cfg.blockDim = dim3(Ue8m0Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Ue8m0Cfg::kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = FP8G_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fp8_gemm_ue8m0_kernel, a.tmap_a, a.tmap_b, a.tmap_d, a.p);
}

}  // namespace fp8g
