// launch_impl.cuh -- one launch of a kernel instantiation (persistent grid,
// kNumThreads threads, the configuration's dynamic shared memory).
#pragma once

#include <atomic>

#include "gemm_kernel.cuh"

#ifndef FP8G_PDL
#define FP8G_PDL 1
#endif
#include "launch.h"

namespace fp8g {

template <int BN, int KIND, bool SPLIT, bool SHARE = false>
cudaError_t launch_one(const LaunchArgs &a)
{
    auto kern = fp8_gemm_kernel<BN, KIND, SPLIT, SHARE>;
    constexpr int smem = Cfg<BN>::kSmemBytes;
    // The opt-in shared-memory size is a per-device function attribute.
    static std::atomic<unsigned long long> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    // programmatic stream serialisation: the kernel may be scheduled while the
    // previous kernel on the stream finishes; it waits (griddepcontrol.wait)
    // before it reads or writes global memory
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = FP8G_PDL;
    // A sharing: clusters of two CTAs (a.grid is even)
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = SHARE ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, a.tmap_a, a.tmap_b, a.tmap_d, a.tmap_sfa, a.tmap_sfb, a.tmap_a2, a.tmap_b2,
                              a.tmap_c, a.p);
}

// Clusters of two of the A-sharing instantiation that can be resident at once
// on device `dev` (cached; 0 on failure).
template <int BN>
int share_max_active(int dev)
{
    static std::atomic<int> cache[64];
    if (dev < 0 || dev >= 64)
        return 0;
    const int c = cache[dev].load();
    if (c > 0)
        return c;
    auto kern = fp8_gemm_kernel<BN, kKindNT, false, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN>::kSmemBytes) != cudaSuccess)
        return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sms, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<BN>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    cache[dev].store(n);
    return n;
}

}  // namespace fp8g
