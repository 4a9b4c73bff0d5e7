// gemm_ue8m0_common.cuh -- what the one-CTA and the CTA-pair power-of-two-
// scale kernels share: the one-CTA configuration (the pair kernel reuses its
// scale-slot layout) and the bf16 panel store from packed pairs.
#pragma once

#include "gemm_kernel.cuh"

namespace fp8g {

#ifndef FP8G_UE8M0_STAGES
#define FP8G_UE8M0_STAGES 4
#endif

struct Ue8m0Cfg {
    static constexpr int kBN = 256;
    static constexpr int kThreads = 512;            // 16 warps
    static constexpr int kStages = FP8G_UE8M0_STAGES;
    static constexpr int kABytes = kBM * kBK;       // 16 KB
    static constexpr int kBBytes = kBN * kBK;       // 32 KB
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kChunk = 8;                // K blocks per scale chunk
    static constexpr int kChunks = 2;               // scale chunks in tensor memory
    static constexpr int kSlotCols = 12;            // per K block: A 4 columns, B 2 x 4 columns
    static constexpr int kScaleCol0 = kBN;          // scale ring after the accumulator
    static constexpr int kPanelCols = 64;
    static constexpr int kPanelBytes = 32 * kPanelCols * 2;
    static constexpr int kColsPerWarp = kBN / 2;    // two drain warps per TMEM lane quarter
    static constexpr int kPanelsPerWarp = kColsPerWarp / kPanelCols;
    // staging panels per warp: with 4 operand stages one (the warp's two
    // panels pass through it one after the other), else two
    static constexpr int kStagingPanels = kStages >= 4 ? 1 : 2;
    static constexpr int kStagingBytes = kNumEpiWarps * kStagingPanels * kPanelBytes;
    static constexpr int kBarriers = 2 * kStages + 2 + 2 * kChunks + 1;
    static constexpr int kSmemBytes =
        kStages * kStageBytes + kStagingBytes + kBarriers * 8 + 16 + 1024 /* alignment slack */;
    static constexpr int kStagingWarp0 = 12;
    static_assert(kScaleCol0 + kChunks * kChunk * kSlotCols <= kTmemCols, "tensor memory");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0 && kStagingBytes % 1024 == 0, "alignment");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// Writes PC columns (one staging panel) of this warp's 32 rows to D from
// packed bf16 pairs (see store_panel).
template <int PC>
__device__ __forceinline__ void store_panel_packed(const uint32_t *w, uint8_t *panel, const CUtensorMap *tmap_d,
                                                   const Params &p, int x, int y_row0, int rows_ok, int lane)
{
    constexpr int NC = PC / 8;          // 16-byte chunks per row
    if (rows_ok == 32) {
        const uint32_t base = smem_u32(panel) + lane * (PC * 2);
        const int sw = ((lane * PC * 2) >> 7) & (NC - 1);
#pragma unroll
        for (int c = 0; c < NC; ++c)
            st_shared_v4(base + ((c ^ sw) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmap_d, panel, x, y_row0);
            bulk_commit_group();
        }
    } else if (lane < rows_ok) {
        uint4 *dst = reinterpret_cast<uint4 *>(p.d + (size_t)(y_row0 + lane) * p.N + x);
#pragma unroll
        for (int c = 0; c < NC; ++c)
            if (x + 8 * c < p.N)
                dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

}  // namespace fp8g
