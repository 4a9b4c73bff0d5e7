// gemm_ue8m0_pair.cu -- launch of the power-of-two-scale kernel on CTA pairs
// (gemm_kernel_ue8m0_pair.cuh): clusters of two CTAs, one CTA per SM, 512
// threads, programmatic stream serialisation.
#include <atomic>
#include <mutex>

#include "gemm_kernel_ue8m0_pair.cuh"

#ifndef FP8G_PDL
#define FP8G_PDL 1
#endif
#include "launch.h"

namespace fp8g {

namespace {

cudaError_t ue8m0_pair_set_smem_attr(int dev)
{
    static std::atomic<unsigned long long> done{0};
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit)
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_ue8m0_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Ue8m0PairCfg::kSmemBytes);
    if (e == cudaSuccess)
        done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

}  // namespace

int ue8m0_pair_block_n() { return Ue8m0PairCfg::kBN; }

cudaError_t launch_ue8m0_pair(const LaunchArgs &a)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if ((e = ue8m0_pair_set_smem_attr(dev)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid, 1, 1);
    cfg.blockDim = dim3(Ue8m0PairCfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Ue8m0PairCfg::kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = FP8G_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fp8_gemm_ue8m0_pair_kernel, a.tmap_a, a.tmap_b, a.tmap_d, a.p);
}

int ue8m0_pair_max_active(int dev)
{
    static std::mutex mu;
    static int cache[64] = {};
    if (dev < 0 || dev >= 64)
        return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] > 0)
        return cache[dev];
    if (ue8m0_pair_set_smem_attr(dev) != cudaSuccess)
        return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sms, 1, 1);
    cfg.blockDim = dim3(Ue8m0PairCfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Ue8m0PairCfg::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_ue8m0_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    cache[dev] = n;
    return n;
}

}  // namespace fp8g
