// gemm_narrow.cu -- launch of the narrow-slice kernel (gemm_kernel_narrow.cuh)
// for the plain GEMM with M <= 128: work units of one slice of
// narrow_block_n() columns and one of narrow_ksplit() K parts (a CTA takes
// units c, c + grid, ...), 192 threads, programmatic stream serialisation.
#include <atomic>

#include "gemm_kernel_narrow.cuh"

#ifndef FP8G_PDL
#define FP8G_PDL 1
#endif
// slice width, K blocks per copy and K parts, per A box height (64 rows:
// M <= 64).  Two K parts halve each CTA's share of A (with 128 rows A's
// copies otherwise rival B's) and let 150 CTAs rather than 112 stream B;
// measured on 64 x 7168 x 16384, 64-column slices over the whole K range
// took 26.9 us, 96-column slices in two K parts 25.6 us.
#ifndef FP8G_NARROW64_BN
#define FP8G_NARROW64_BN 96
#endif
#ifndef FP8G_NARROW64_KD
#define FP8G_NARROW64_KD 2
#endif
#ifndef FP8G_NARROW64_KSPLIT
#define FP8G_NARROW64_KSPLIT 2
#endif
#ifndef FP8G_NARROW128_BN
#define FP8G_NARROW128_BN 96
#endif
#ifndef FP8G_NARROW128_KD
#define FP8G_NARROW128_KD 2
#endif
#ifndef FP8G_NARROW128_KSPLIT
#define FP8G_NARROW128_KSPLIT 2
#endif
#include "launch.h"

namespace fp8g {

namespace {

// as many stages as 192 KB of operands hold
constexpr int stages_for(int bn, int a_rows, int kd) { return (192 * 1024) / (kd * (a_rows + bn) * kBK); }

template <int BN, int A_ROWS, int KD, int KSPLIT>
cudaError_t launch_narrow_one(const LaunchArgs &a)
{
    constexpr int S = stages_for(BN, A_ROWS, KD);
    using C = NarrowCfg<BN, A_ROWS, KD, S, KSPLIT>;
    auto kern = fp8_gemm_narrow_kernel<BN, A_ROWS, KD, S, KSPLIT>;
    static std::atomic<unsigned long long> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = FP8G_PDL;
    // two K parts: the two CTAs of a slice are a cluster (a.grid is even)
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = KSPLIT == 2 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, a.tmap_a, a.tmap_b, a.tmap_sfa, a.tmap_sfb, a.p);
}

// Clusters of two of an instantiation that can be resident at once on device
// `dev` (cached; 0 on failure).
template <int BN, int A_ROWS, int KD>
int max_clusters_one(int dev)
{
    constexpr int S = stages_for(BN, A_ROWS, KD);
    using C = NarrowCfg<BN, A_ROWS, KD, S, 2>;
    static std::atomic<int> cache[64];
    if (dev < 0 || dev >= 64)
        return 0;
    const int c = cache[dev].load();
    if (c > 0)
        return c;
    auto kern = fp8_gemm_narrow_kernel<BN, A_ROWS, KD, S, 2>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
        return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sms, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
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

}  // namespace

int narrow_block_n(int a_box_rows) { return a_box_rows == 64 ? FP8G_NARROW64_BN : FP8G_NARROW128_BN; }

int narrow_kd(int a_box_rows) { return a_box_rows == 64 ? FP8G_NARROW64_KD : FP8G_NARROW128_KD; }

int narrow_scale_chunk() { return kNarrowChunk; }

int narrow_ksplit(int a_box_rows) { return a_box_rows == 64 ? FP8G_NARROW64_KSPLIT : FP8G_NARROW128_KSPLIT; }

int narrow_max_clusters(int dev, int a_box_rows)
{
    if (a_box_rows == 64) {
        if constexpr (FP8G_NARROW64_KSPLIT == 2)
            return max_clusters_one<FP8G_NARROW64_BN, 64, FP8G_NARROW64_KD>(dev);
        return 0;
    }
    if constexpr (FP8G_NARROW128_KSPLIT == 2)
        return max_clusters_one<FP8G_NARROW128_BN, 128, FP8G_NARROW128_KD>(dev);
    return 0;
}

cudaError_t launch_narrow(const LaunchArgs &a)
{
    if (a.p.a_box_rows == 64)
        return launch_narrow_one<FP8G_NARROW64_BN, 64, FP8G_NARROW64_KD, FP8G_NARROW64_KSPLIT>(a);
    if (a.p.a_box_rows == 128)
        return launch_narrow_one<FP8G_NARROW128_BN, 128, FP8G_NARROW128_KD, FP8G_NARROW128_KSPLIT>(a);
    return cudaErrorInvalidValue;
}

}  // namespace fp8g
