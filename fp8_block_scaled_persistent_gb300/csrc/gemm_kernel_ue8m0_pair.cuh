// gemm_kernel_ue8m0_pair.cuh -- the power-of-two-scale GEMM
// (gemm_kernel_ue8m0.cuh) on CTA pairs: one 256 x 256 output tile per
// cluster of two CTAs on neighbouring SMs, through the block-scaled
// tcgen05.mma.cta_group::2.
//
// What is computed is that of the one-CTA UE8M0 kernel: every scale a power
// of two, applied inside the block-scaled MMA, one fp32 accumulator per tile
// in tensor memory, bf16 out.
//
// Why pairs: the one-CTA kernel's SM loads 48 KB of operands per K block of a
// 128 x 256 tile through its TMA unit, and its four-stage ring turns over
// slower than the tensor pipe consumes it.  Here each CTA loads its own 128
// rows of A and its half (128 rows) of B -- 32 KB per SM per K block for the
// same 128 x 256 share of the output -- into a six-stage ring, and the
// leader's single MMA of M = 256 covers both SMs.
//
//   warp 0      TMA producer (both CTAs): A 128 x 128 and B 128 x 128 e4m3
//               tiles, counted on the leader's full barrier
//               (cp.async.bulk.tensor .cta_group::2 with a remote
//               arrive.expect_tx from the peer).
//   warp 1      MMA issuer (leader only): per K block 4 x (256 x 256 x 32)
//               block-scaled MMAs into columns 0 .. 255 of both CTAs' tensor
//               memory; one commit per K block, multicast to both CTAs'
//               empty barriers; one at the end of a tile to both acc_full.
//   warps 4-11  epilogue (both CTAs): drain the CTA's 128 x 256 accumulator,
//               release it on the leader's acc_empty (remote arrive), bf16
//               conversion and TMA stores, as in the one-CTA kernel.
//   warps 12-15 scale staging (both CTAs): each CTA's tensor memory gets
//               the A scales of its own 128 rows and the B scales of both
//               128-column blocks of the tile, in the one-CTA kernel's slot
//               layout; the leader's sc_full counts both CTAs' warps (remote
//               arrives), the MMA's chunk commit frees both CTAs' slots.
//
// Every wait is bounded; an expiry raises both CTAs' abort flags, both drain
// and meet at the final cluster barrier, then wait a short grace period for
// copies in flight before they free tensor memory.
#pragma once

#include "gemm_kernel_pair.cuh"
#include "gemm_ue8m0_common.cuh"

namespace fp8g {

#ifndef FP8G_UE8M0_PAIR_STAGES
#define FP8G_UE8M0_PAIR_STAGES 6
#endif

struct Ue8m0PairCfg {
    static constexpr int kBN = 256;                 // pair tile 256 x 256
    static constexpr int kBHalfRows = kBN / 2;      // B rows each CTA loads
    static constexpr int kThreads = 512;
    static constexpr int kStages = FP8G_UE8M0_PAIR_STAGES;
    static constexpr int kABytes = kBM * kBK;       // 16 KB
    static constexpr int kBBytes = kBHalfRows * kBK;    // 16 KB
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kChunk = Ue8m0Cfg::kChunk;
    static constexpr int kChunks = Ue8m0Cfg::kChunks;
    static constexpr int kSlotCols = Ue8m0Cfg::kSlotCols;
    static constexpr int kScaleCol0 = kBN;
    static constexpr int kPanelCols = 64;
    static constexpr int kPanelBytes = 32 * kPanelCols * 2;
    static constexpr int kColsPerWarp = kBN / 2;
    static constexpr int kStagingPanels = 1;
    static constexpr int kStagingBytes = kNumEpiWarps * kStagingPanels * kPanelBytes;
    static constexpr int kBarriers = 2 * kStages + 2 + 2 * kChunks + 1;
    static constexpr int kSmemBytes =
        kStages * kStageBytes + kStagingBytes + kBarriers * 8 + 16 + 1024 /* alignment slack */;
    static constexpr int kStagingWarp0 = 12;
    static_assert(kScaleCol0 + kChunks * kChunk * kSlotCols <= kTmemCols, "tensor memory");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0 && kStagingBytes % 1024 == 0, "alignment");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

__global__ void __launch_bounds__(Ue8m0PairCfg::kThreads, 1)
    fp8_gemm_ue8m0_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                               const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ Params p)
{
#if defined(__CUDA_ARCH__)
    using C = Ue8m0PairCfg;
    constexpr int S = C::kStages;
    constexpr int BN = C::kBN;

    // the same layout in both CTAs (the leader's descriptors and scale
    // addresses name the peer's tiles and columns by the same offsets)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + S * C::kABytes;
    uint8_t *sm_stage_d = sm_b + S * C::kBBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm_stage_d + C::kStagingBytes);
    uint64_t *full = bar;                    // S: leader: both CTAs' A/B tiles landed
    uint64_t *empty = full + S;              // S: the stage's MMAs finished (multicast commit)
    uint64_t *acc_full = empty + S;          // the tile's accumulator is complete (multicast commit)
    uint64_t *acc_empty = acc_full + 1;      // leader: both epilogues have read it (16 warps)
    uint64_t *sc_full = acc_empty + 1;       // kChunks: leader: both CTAs' scale chunk is in tensor memory
    uint64_t *sc_empty = sc_full + C::kChunks;   // kChunks: the MMAs reading it finished (multicast)
    uint64_t *drain = sc_empty + C::kChunks;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 2);             // one arrive.expect_tx per producer
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * kNumEpiWarps);
        for (int i = 0; i < C::kChunks; ++i) {
            mbar_init(&sc_full[i], 2 * 4);      // four staging warps per CTA
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
    __syncthreads();
    // both CTAs' barriers exist before any remote arrival or copy reaches them
    cluster_sync();
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_alloc_permit_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int *>(abort_flag)), (uint32_t)rank ^ 1u);
    const WaitCtl ctl{abort_flag, p.error_word, p.timeout_ns, peer_abort};

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        PairScheduler<kKindNT> sched(p, false);
        PairWork w;
        Ring ring;
        const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
        uint32_t issued = 0, issued_parity = 0;
        bool ok = true;
        while (ok && sched.next(w)) {
            if (!bounds_ok(w.n_blk >= 0 && w.n_blk * BN < p.N && w.a_row0 >= 0 &&
                               (w.valid_rows == 0 || (w.a_row0 < p.a_rows_total && w.valid_rows <= kBM)),
                           ctl)) {
                ok = false;
                break;
            }
            const int b_row0 = w.n_blk * BN + rank * C::kBHalfRows;
            for (int k = 0; k < p.kb; ++k) {
                if (!mbar_wait(&empty[ring.i], ring.ph ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = leader_full + 8u * ring.i;
                mbar_arrive_expect_tx_cluster(fb, C::kStageBytes);
                tma_load_2d_pair(sm_a + ring.i * C::kABytes, &tmap_a, fb, k * kBK, w.a_row0);
                tma_load_2d_pair(sm_b + ring.i * C::kBBytes, &tmap_b, fb, k * kBK, b_row0);
                issued |= 1u << ring.i;
                issued_parity = (issued_parity & ~(1u << ring.i)) | (ring.ph << ring.i);
                ring.template next<S>();
            }
        }
        // both CTAs' copies count on the leader's barriers: the leader waits
        // for every fill it started (the peer started the same ones unless
        // the pair aborted)
        if (rank == 0)
            for (int i = 0; i < S; ++i)
                if (issued & (1u << i))
                    mbar_wait_drain(&full[i], (issued_parity >> i) & 1u, p.timeout_ns);
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------ MMA issuer (leader)
        PairScheduler<kKindNT> sched(p, false);
        PairWork w;
        Ring ring, sring;
        uint32_t acc_ph = 0;
        constexpr uint32_t idesc = idesc_mx_e4m3(2 * kBM, BN);
        bool ok = true;
        while (ok && sched.next(w)) {
            // both CTAs' epilogues have read the previous tile's accumulator
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
                // branch per K block on the issuing thread: 42.2 -> 41.6 us at
                // 4096 x 7168 x 2048)
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
                        mma_mxf8f6f4_pair(tmem_base, a0 + 2 * kk, b0 + 2 * kk, idesc, sfa, sfb,
                                          (k | kk) != 0 ? 1u : 0u);
                    mma_commit_pair(&empty[ring.i], 0x3);
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
                mma_commit_pair(&sc_empty[sring.i], 0x3);   // the chunk's scale slots may be rewritten
                sring.template next<C::kChunks>();
            }
            if (!ok)
                break;
            mma_commit_pair(acc_full, 0x3);
            acc_ph ^= 1u;
        }
        // all MMAs issued above complete before either CTA frees its tensor memory
        mma_commit_pair(drain, 0x1);
        mbar_wait_drain(drain, 0, p.timeout_ns);
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kNumEpiWarps) {
        // ------------------------------------------------ epilogue warps (both CTAs)
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3;
        const int h = ew >> 2;
        uint8_t *panels = sm_stage_d + ew * C::kStagingPanels * C::kPanelBytes;
        const uint32_t leader_acc_empty = mapa_shared(smem_u32(acc_empty), 0);
        PairScheduler<kKindNT> sched(p, false);
        PairWork w;
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
                // the accumulator may be overwritten by the pair's next tile
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(leader_acc_empty);
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
            // the previous tile's stores have read this warp's panel
            if (lane == 0)
                bulk_wait_group_read<0>();
            __syncwarp();
            if (rows_ok > 0) {
                if (x < p.N)
                    store_panel_packed<C::kPanelCols>(pk0, panels, &tmap_d, p, x, y_row0, rows_ok, lane);
                if (x + C::kPanelCols < p.N) {
                    // one panel buffer: the first panel's store has read it
                    if (lane == 0)
                        bulk_wait_group_read<0>();
                    __syncwarp();
                    store_panel_packed<C::kPanelCols>(pk1, panels, &tmap_d, p, x + C::kPanelCols, y_row0, rows_ok,
                                                      lane);
                }
            }
        }
        if (lane == 0)
            bulk_wait_group<0>();
        __syncwarp();
    } else if (warp >= C::kStagingWarp0) {
        // ------------------------------------------------ scale staging warps (both CTAs)
        const int q = warp & 3;               // the TMEM lane quarter this warp writes
        const uint32_t leader_sc_full = mapa_shared(smem_u32(sc_full), 0);
        PairScheduler<kKindNT> sched(p, false);
        PairWork w;
        Ring sring;
        bool ok = true;
        while (ok && sched.next(w)) {
            // this CTA's rows' A scales; the B scales of both 128-column
            // blocks of the pair tile
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
                    mbar_arrive_cluster(leader_sc_full + 8u * sring.i);
                sring.template next<C::kChunks>();
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // no remote arrival, copy signal or MMA write reaches either CTA after this
    cluster_sync();
    if (__syncthreads_or(*abort_flag)) {
        // an aborted pair may have stopped with operand copies in flight that
        // no barrier it still waits on counts: give them time to land
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull)
            __nanosleep(1000);
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
#endif
}

}  // namespace fp8g
