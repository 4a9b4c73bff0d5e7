// gemm_kernel_ue8m0.cuh -- the FP8 (E4M3) GEMM with power-of-two (UE8M0)
// block scales, on the tensor cores' block-scaled MMA.
//
// What is computed: the method's GEMM (DeepGEMM fp8_gemm.cuh: one A scale per
// row per 128-wide K block, one B scale per 128 x 128 block) with every scale
// a power of two, stored as a UE8M0 byte e (value 2^(e - 127)):
//
//   D[m][n] = bf16( sum_k 2^(ea[k][m] - 127) * 2^(eb[n/128][k] - 127) *
//                   sum_{t < 128} A[m][128k+t] * B[n][128k+t] )
//
// How (the "TCGen05 Copy Instruction" tutorial's closing section on
// block-scaled MMA, where the scales are held in tensor memory next to the
// accumulator; design ours): tcgen05.mma.kind::mxf8f6f4.block_scale applies
// each row's and column's scale inside the MMA, so the fp32 accumulator in
// tensor memory takes the whole K sum and no per-K-block promotion pass is
// needed.  A power-of-two scale times an E4M3 product is exact, so the only
// roundings are the MMA's fp32 accumulation and the final bf16.
//
// One CTA per SM, 512 threads, tiles of 128 x 256:
//   warp 0      TMA producer: A 128 x 128 and B 256 x 128 e4m3 tiles,
//               128-byte swizzled, into a 4-stage ring.
//   warp 1      MMA issuer: per K block 4 x (128 x 256 x 32) block-scaled
//               MMAs accumulating into tensor-memory columns 0 .. 255; one
//               commit per K block frees the operand stage; one commit at
//               the end of a tile hands the accumulator to the epilogue.
//   warps 4-11  epilogue: at the end of a tile, each reads its 32 rows x
//               128 columns of the accumulator (two tcgen05.ld), releases it
//               for the next tile, converts to bf16 (round to nearest even)
//               and TMA-stores through a swizzled staging panel, one 64-column
//               panel after the other (predicated row stores where the tile
//               straddles M).
//   warps 12-15 scale staging: the scale bytes of each K block go into a
//               ring of tensor-memory slots, written by tcgen05.st (each
//               warp its 32 lanes), eight K blocks per chunk, two chunks.
//   warps 2-3   idle.
//
// The scale slot of a K block is 12 columns: 4 for A, 4 + 4 for B's two
// 128-column blocks.  Every column of a slot holds, in each lane, the scale
// byte repeated in all four byte positions, so that whichever byte (the
// instruction's scale-factor id) and whichever of a row's four columns the
// MMA reads, it reads that row's or that column block's scale: A's lane m
// holds row m's byte in all four A columns; B's two blocks fill their four
// columns uniformly.
//
// Every wait is bounded; on expiry the CTA records an error, drains, frees its
// tensor memory and returns.
#pragma once

#include "gemm_ue8m0_common.cuh"

namespace fp8g {

__global__ void __launch_bounds__(Ue8m0Cfg::kThreads, 1)
    fp8_gemm_ue8m0_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ Params p)
{
#if defined(__CUDA_ARCH__)
    using C = Ue8m0Cfg;
    constexpr int S = C::kStages;
    constexpr int BN = C::kBN;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + S * C::kABytes;
    uint8_t *sm_stage_d = sm_b + S * C::kBBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm_stage_d + C::kStagingBytes);
    uint64_t *full = bar;                    // S: A/B tiles landed (TMA transactions)
    uint64_t *empty = full + S;              // S: the stage's MMAs finished
    uint64_t *acc_full = empty + S;          // the tile's accumulator is complete
    uint64_t *acc_empty = acc_full + 1;      // the epilogue has read it (8 warps)
    uint64_t *sc_full = acc_empty + 1;       // kChunks: a scale chunk is in tensor memory (4 warps)
    uint64_t *sc_empty = sc_full + C::kChunks;   // kChunks: the MMAs reading it finished
    uint64_t *drain = sc_empty + C::kChunks;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kNumEpiWarps);
        for (int i = 0; i < C::kChunks; ++i) {
            mbar_init(&sc_full[i], 4);
            mbar_init(&sc_empty[i], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_shared();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        prefetch_tensormap(&tmap_d);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    const WaitCtl ctl{abort_flag, p.error_word, p.timeout_ns};

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        Scheduler<BN, kKindNT, false> sched(p, false);
        Work w;
        Ring ring;
        uint32_t issued = 0, issued_parity = 0;
        bool ok = true;
        while (ok && sched.next(w)) {
            if (!bounds_ok(w.a_row0 >= 0 && w.a_row0 < p.a_rows_total && w.n_blk >= 0 && w.n_blk * BN < p.N,
                           ctl)) {
                ok = false;
                break;
            }
            const int b_row0 = w.n_blk * BN;
            for (int k = 0; k < p.kb; ++k) {
                if (!mbar_wait(&empty[ring.i], ring.ph ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[ring.i], C::kStageBytes);
                tma_load_2d(sm_a + ring.i * C::kABytes, &tmap_a, &full[ring.i], k * kBK, w.a_row0);
                tma_load_2d(sm_b + ring.i * C::kBBytes, &tmap_b, &full[ring.i], k * kBK, b_row0);
                issued |= 1u << ring.i;
                issued_parity = (issued_parity & ~(1u << ring.i)) | (ring.ph << ring.i);
                ring.template next<S>();
            }
        }
        for (int i = 0; i < S; ++i)
            if (issued & (1u << i))
                mbar_wait_drain(&full[i], (issued_parity >> i) & 1u, p.timeout_ns);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        Scheduler<BN, kKindNT, false> sched(p, false);
        Work w;
        Ring ring, sring;
        uint32_t acc_ph = 0;
        constexpr uint32_t idesc = idesc_mx_e4m3(kBM, BN);
        bool ok = true;
        while (ok && sched.next(w)) {
            // the previous tile's accumulator has been read
            if (!mbar_wait(acc_empty, acc_ph ^ 1u, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            // chunk by chunk of K blocks: the scale chunk's wait stays out
            // of the per-K-block loop, whose shape costs the issuing thread
            // ~200 cycles per K block otherwise (measured)
            for (int k0 = 0; k0 < p.kb; k0 += C::kChunk) {
                if (!mbar_wait(&sc_full[sring.i], sring.ph, ctl)) {
                    ok = false;
                    break;
                }
                const int n = min(C::kChunk, p.kb - k0);
                const uint32_t slot = tmem_base + C::kScaleCol0 + sring.i * C::kChunk * C::kSlotCols;
                // one K block: its operands, four MMAs, the commit that frees
                // the stage; a whole chunk runs fully unrolled (no loop
                // branch per K block on the issuing thread)
                auto kblock = [&](int kc) -> bool {
                    const int k = k0 + kc;
                    if (!mbar_wait(&full[ring.i], ring.ph, ctl)) {
                        return false;
                    }
                    tc_fence_after_sync();
                    const uint64_t a0 = sdesc_kmajor_sw128(smem_u32(sm_a + ring.i * C::kABytes));
                    const uint64_t b0 = sdesc_kmajor_sw128(smem_u32(sm_b + ring.i * C::kBBytes));
                    const uint32_t sfa = slot + kc * C::kSlotCols;
                    const uint32_t sfb = sfa + 4;
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)
                        mma_mxf8f6f4(tmem_base, a0 + 2 * kk, b0 + 2 * kk, idesc, sfa, sfb,
                                     (k | kk) != 0 ? 1u : 0u);
                    mma_commit(&empty[ring.i]);
                    ring.template next<S>();
                    return true;
                };
                if (n == C::kChunk) {
#pragma unroll
                    for (int kc = 0; kc < C::kChunk; ++kc)
                        if (!kblock(kc)) {
                            ok = false;
                            break;
                        }
                } else {
                    for (int kc = 0; kc < n; ++kc)
                        if (!kblock(kc)) {
                            ok = false;
                            break;
                        }
                }
                if (!ok)
                    break;
                mma_commit(&sc_empty[sring.i]);   // the chunk's scale slots may be rewritten
                sring.template next<C::kChunks>();
            }
            if (!ok)
                break;
            mma_commit(acc_full);
            acc_ph ^= 1u;
        }
        mma_commit(drain);
        mbar_wait_drain(drain, 0, p.timeout_ns);
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kNumEpiWarps) {
        // ------------------------------------------------ epilogue warps
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3;
        const int h = ew >> 2;
        uint8_t *panels = sm_stage_d + ew * C::kStagingPanels * C::kPanelBytes;
        Scheduler<BN, kKindNT, false> sched(p, false);
        Work w;
        uint32_t acc_ph = 0;
        while (sched.next(w)) {
            if (!warp_wait(acc_full, acc_ph, ctl))
                break;
            __syncwarp();
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + h * C::kColsPerWarp;
            uint32_t pk0[32], pk1[32];
            {
                uint32_t v[64];
                tmem_ld_32x32b_x64(taddr, v);
                tmem_wait_ld(v);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk0[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                tmem_ld_32x32b_x64(taddr + 64, v);
                tmem_wait_ld(v);
                // the accumulator may be overwritten by the next tile
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acc_empty);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk1[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            }
            acc_ph ^= 1u;
            int rows_ok = min(max(w.valid_rows - 32 * q, 0), 32);
            const int y_row0 = w.a_row0 + 32 * q;
            const int x = w.n_blk * BN + h * C::kColsPerWarp;
            if (rows_ok > 0 && !bounds_ok(y_row0 >= 0 && y_row0 + rows_ok <= p.d_rows_total, ctl))
                rows_ok = 0;
            // the previous tile's stores have read this warp's panels
            if (lane == 0)
                bulk_wait_group_read<0>();
            __syncwarp();
            if (rows_ok > 0) {
                if (x < p.N)
                    store_panel_packed<C::kPanelCols>(pk0, panels, &tmap_d, p, x, y_row0, rows_ok, lane);
                if (x + C::kPanelCols < p.N) {
                    uint8_t *second = panels + (C::kStagingPanels - 1) * C::kPanelBytes;
                    if (C::kStagingPanels == 1) {
                        // one panel buffer: the first panel's store has read it
                        if (lane == 0)
                            bulk_wait_group_read<0>();
                        __syncwarp();
                    }
                    store_panel_packed<C::kPanelCols>(pk1, second, &tmap_d, p, x + C::kPanelCols, y_row0, rows_ok,
                                                      lane);
                }
            }
        }
        if (lane == 0)
            bulk_wait_group<0>();
        __syncwarp();
    } else if (warp >= C::kStagingWarp0) {
        // ------------------------------------------------ scale staging warps
        const int q = warp & 3;               // the TMEM lane quarter this warp writes
        Scheduler<BN, kKindNT, false> sched(p, false);
        Work w;
        Ring sring;
        bool ok = true;
        while (ok && sched.next(w)) {
            const int row = w.a_row0 + 32 * q + lane;
            const bool row_ok = row < p.rows;
            const int nblk0 = 2 * w.n_blk;
            const bool nb1_ok = nblk0 + 1 < p.nb;
            if (!bounds_ok(nblk0 >= 0 && nblk0 < p.nb && w.a_row0 >= 0, ctl)) {
                ok = false;
                break;
            }
            for (int k0 = 0; k0 < p.kb; k0 += C::kChunk) {
                const int n = min(C::kChunk, p.kb - k0);
                if (!warp_wait(&sc_empty[sring.i], sring.ph ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                tc_fence_after_sync();
                uint32_t ea[C::kChunk], eb0[C::kChunk], eb1[C::kChunk];
#pragma unroll
                for (int j = 0; j < C::kChunk; ++j) {
                    ea[j] = eb0[j] = eb1[j] = 127u;
                    if (j < n) {
                        if (row_ok)
                            ea[j] = __ldg(p.sfa_e + (size_t)(k0 + j) * p.sfa_ld + row);
                        eb0[j] = __ldg(p.sfb_e + (size_t)nblk0 * p.kb + k0 + j);
                        if (nb1_ok)
                            eb1[j] = __ldg(p.sfb_e + (size_t)(nblk0 + 1) * p.kb + k0 + j);
                    }
                }
                const uint32_t slot0 = tmem_base + ((uint32_t)(32 * q) << 16) + C::kScaleCol0 +
                                       sring.i * C::kChunk * C::kSlotCols;
#pragma unroll
                for (int j = 0; j < C::kChunk; ++j) {
                    if (j < n) {
                        const uint32_t a = ea[j] * 0x01010101u, b0 = eb0[j] * 0x01010101u,
                                       b1 = eb1[j] * 0x01010101u;
                        const uint32_t col = slot0 + j * C::kSlotCols;
                        tmem_st_32x32b_x4(col, a, a, a, a);
                        tmem_st_32x32b_x8(col + 4, b0, b0, b0, b0, b1, b1, b1, b1);
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sc_full[sring.i]);
                sring.template next<C::kChunks>();
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
#endif
}

}  // namespace fp8g
