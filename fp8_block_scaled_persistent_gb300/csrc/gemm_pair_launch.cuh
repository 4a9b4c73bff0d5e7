// gemm_pair_launch.cuh -- launch of one CTA-pair kernel instantiation:
// clusters of two CTAs, one CTA per SM, the configuration's dynamic shared
// memory, programmatic stream serialisation.
#pragma once

#include <atomic>
#include <mutex>

#include "gemm_kernel_pair.cuh"

#ifndef FP8G_PDL
#define FP8G_PDL 1
#endif
#include "launch.h"

namespace fp8g {

template <int BN, int KIND>
cudaError_t pair_set_smem_attr(int dev)
{
    static std::atomic<unsigned long long> done{0};
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit)
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_pair_kernel<BN, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg<BN>::kSmemBytes);
    if (e == cudaSuccess)
        done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <int BN, int KIND>
cudaError_t pair_launch_one(const LaunchArgs &a)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if ((e = pair_set_smem_attr<BN, KIND>(dev)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<BN>::kSmemBytes;
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
    return cudaLaunchKernelEx(&cfg, fp8_gemm_pair_kernel<BN, KIND>, a.tmap_a, a.tmap_b, a.tmap_d, a.tmap_sfa,
                              a.tmap_sfb, a.tmap_c, a.p);
}

template <int BN>
cudaError_t pair_launch_kind(int kind, const LaunchArgs &a)
{
    switch (kind) {
    case kKindNT: return pair_launch_one<BN, kKindNT>(a);
    case kKindNTAcc: return pair_launch_one<BN, kKindNTAcc>(a);
    case kKindContiguous: return pair_launch_one<BN, kKindContiguous>(a);
    case kKindMasked: return pair_launch_one<BN, kKindMasked>(a);
    default: return cudaErrorInvalidValue;
    }
}

// Clusters of two that can be resident at once (cached per device).
template <int BN>
int pair_max_active(int dev)
{
    static std::mutex mu;
    static int cache[64] = {};
    if (dev < 0 || dev >= 64)
        return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] > 0)
        return cache[dev];
    if (pair_set_smem_attr<BN, kKindNT>(dev) != cudaSuccess)
        return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sms, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<BN>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_pair_kernel<BN, kKindNT>, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    cache[dev] = n;
    return n;
}

}  // namespace fp8g
