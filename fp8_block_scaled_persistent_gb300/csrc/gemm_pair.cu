// gemm_pair.cu -- instantiations and launch of the CTA-pair kernel
// (gemm_kernel_pair.cuh): clusters of two CTAs, one 256 x 128 tile per pair,
// for the plain GEMM, the plain GEMM with an addend, and both grouped layouts.
#include <atomic>
#include <mutex>

#include "gemm_kernel_pair.cuh"

#ifndef FP8G_PDL
#define FP8G_PDL 1
#endif
#include "launch.h"

namespace fp8g {

namespace {

constexpr int kPairBN = 128;

template <int KIND>
cudaError_t set_smem_attr(int dev)
{
    static std::atomic<unsigned long long> done{0};
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit)
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_pair_kernel<kPairBN, KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg<kPairBN>::kSmemBytes);
    if (e == cudaSuccess)
        done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <int KIND>
cudaError_t launch_pair_one(const LaunchArgs &a)
{
    auto kern = fp8_gemm_pair_kernel<kPairBN, KIND>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if ((e = set_smem_attr<KIND>(dev)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<kPairBN>::kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic stream serialisation, as for the one-CTA kernel
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = FP8G_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a.tmap_a, a.tmap_b, a.tmap_d, a.tmap_sfa, a.tmap_sfb, a.p);
}

}  // namespace

int pair_panel_cols() { return PairCfg<kPairBN>::kPanelCols; }

int pair_block_n() { return kPairBN; }

// Clusters of two this kernel can keep resident at once on device `dev`
// (one CTA per SM; a pair needs two SMs of the same cluster-capable group).
int max_active_pairs(int dev)
{
    static std::mutex mu;
    static int cache[64] = {};
    if (dev < 0 || dev >= 64)
        return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] > 0)
        return cache[dev];
    if (set_smem_attr<kKindNT>(dev) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    cfg.gridDim = dim3(2 * sms, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<kPairBN>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_pair_kernel<kPairBN, kKindNT>, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    cache[dev] = n;
    return n;
}

cudaError_t launch_pair(int kind, const LaunchArgs &a)
{
    switch (kind) {
    case kKindNT: return launch_pair_one<kKindNT>(a);
    case kKindNTAcc: return launch_pair_one<kKindNTAcc>(a);
    case kKindContiguous: return launch_pair_one<kKindContiguous>(a);
    case kKindMasked: return launch_pair_one<kKindMasked>(a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fp8g
