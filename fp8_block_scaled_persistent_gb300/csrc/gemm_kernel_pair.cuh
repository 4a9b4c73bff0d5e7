// gemm_kernel_pair.cuh -- the CTA-pair variant of the FP8 block-scaled GEMM:
// one 256 x BN output tile (BN = 128 or 256) per cluster of two CTAs on
// neighbouring SMs.
//
// What is computed is the same as in gemm_kernel.cuh (DeepGEMM fp8_gemm.cuh,
// fp8_gemm_kernel: each 128-wide K block's partial promoted with
// scale_a * scale_b into an fp32 accumulator, bf16 out).  What differs is how
// the pair shares work (the DeepGEMM page reaches the same sharing with TMA
// multicast over a cluster, tma_copy<kNumTMAMulticast>; here nothing is
// multicast):
//
//   * rank 0 of the cluster (the leader) issues tcgen05.mma.cta_group::2 with
//     M = 256, N = BN: each CTA holds its own 128 rows of A and its own BN/2
//     rows (half) of B in its shared memory, and each CTA's tensor memory
//     receives its 128 rows x BN columns of the partial.  At BN = 256 each
//     SM loads 32 KB per K block for a 128 x 256 share of the output, where a
//     128 x 256 tile on one SM loads 48 KB;
//   * at BN = 128 the 512 tensor-memory columns hold four partial buffers per
//     CTA (three K blocks of slack for the "MMA completes -> epilogue reads
//     -> buffer freed" round trip), at BN = 256 two;
//   * both producers load into their own CTA but signal the leader's
//     full barrier (cp.async.bulk.tensor .cta_group::2, each producer adding
//     its own bytes with a remote arrive.expect_tx); the leader's one commit
//     per K block is multicast to the stage's empty barrier in both CTAs,
//     which frees the stage for both producers and tells both epilogues that
//     the partial is ready; the epilogue warps of both CTAs release a tensor
//     memory buffer on the leader's barrier (remote arrive).
//
// Roles per CTA are those of the one-CTA kernel (warp 0 producer, warp 1 MMA
// issuer -- idle in the second CTA --, warps 4-11 epilogue; with the fp32
// addend at BN = 256, warp 2 copies each tile's C of the CTA's own 128 rows
// into the staging area in two halves and stores the bf16 tile, as the
// one-CTA kernel's addend/store warp does).  Scales are per CTA: each loads
// the A scales of its own rows and the B scales of the tile's 128 columns
// into its own scale ring.
//
// Every wait is bounded.  A wait that runs out raises the abort flag of both
// CTAs; both then drain and meet at the final cluster barrier, after which
// an aborted pair waits a short grace period for copies still in flight
// before it frees tensor memory and exits.
#pragma once

#include "gemm_kernel.cuh"

namespace fp8g {

// Pair tiles are 256 x BN: each CTA holds 128 rows of A and BN/2 rows of B
// per K block, and receives a 128 x BN partial in its tensor memory.
//   BN = 128: four partial buffers per CTA (the round trip has three K
//             blocks of slack) and 24 KB of operands per SM per K block, but
//             only 256 tensor cycles per K block for the one issuing thread;
//   BN = 256: two partial buffers, 512 tensor cycles per K block, and 32 KB
//             of operands per SM per K block where a 128 x 256 tile on one SM
//             loads 48 KB.
template <int BN>
struct PairCfg {
    static_assert(BN == 128 || BN == 256, "pair tiles are 256 x 128 or 256 x 256");
    static constexpr int kPairRows = 2 * kBM;          // output rows per pair tile
    static constexpr int kBHalfRows = BN / 2;          // B rows each CTA loads
    static constexpr int kStages = BN == 128 ? 7 : 4;  // A/B operand ring
    static constexpr int kAccBufs = kTmemCols / BN;    // partial buffers per CTA
    static constexpr int kScaleSlots = 4;
    static constexpr int kABytes = kBM * kBK;          // 16 KB
    static constexpr int kBBytes = kBHalfRows * kBK;   // 8 or 16 KB
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSfbRows = BN / 128;
    static constexpr int kSlotSfaBytes = kScaleChunk * kBM * 4;
    static constexpr int kSlotSfbStride = 128;
    static constexpr int kSlotBytes = kSlotSfaBytes + kSlotSfbStride * kSfbRows;
    static constexpr int kSlotTxBytes = kSlotSfaBytes + (kScaleChunk + 4) * 4 * kSfbRows;
    static constexpr int kColsPerThread = BN / 2;      // two warps per TMEM lane quarter
    static constexpr int kPanelCols = 64;              // 128-byte rows, 128-byte swizzle
    static constexpr int kPanelBytes = 32 * kPanelCols * 2;
    static constexpr int kPanelsPerWarp = kColsPerThread / kPanelCols;
    static constexpr int kStagingBytes = kNumEpiWarps * kPanelsPerWarp * kPanelBytes;
    static constexpr int kBarriers = 2 * kStages + kAccBufs + 2 * kScaleSlots + 4;
    static constexpr int kSmemBytes = kStages * kStageBytes + kStagingBytes + kScaleSlots * kSlotBytes +
                                      kBarriers * 8 + 16 + 1024 /* alignment slack */;
    // registers per thread after reallocation: the epilogue holds BN/2
    // accumulator columns; the launch allocation is 384 x 168 = 64512
    static constexpr int kRegsCtl = BN == 128 ? 72 : 40;
    static constexpr int kRegsEpi = BN == 128 ? 208 : 232;
    static_assert(128 * kRegsCtl + 256 * kRegsEpi <= kNumThreads * kLaunchRegs,
                  "register reallocation exceeds the launch allocation");
    static_assert(kSlotTxBytes <= kSlotBytes, "scale slot");
    static_assert(kSlotBytes % 128 == 0 && kSlotSfaBytes % 128 == 0 && kStagingBytes % 1024 == 0 &&
                      kABytes % 1024 == 0 && kBBytes % 1024 == 0 && kPanelBytes % 1024 == 0,
                  "TMA destinations and sources must stay 128-byte (swizzled: 1024-byte) aligned");
    static_assert(kStages >= kAccBufs, "the epilogue's wait on a stage's MMA completion must not alias");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// The same K-block promotion as promote_block, releasing the buffer on the
// leader's barrier (a shared::cluster address) once its last load landed.
template <int COLS, int LD>
__device__ __forceinline__ void promote_block_pair(float (&acc)[COLS], uint32_t taddr, const float *pa,
                                                   const float *pb, uint32_t tempty_cluster_addr, int lane)
{
    constexpr int NCH = COLS / LD;
    static_assert(COLS % LD == 0, "column split");
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        uint32_t v[LD];
        tmem_ld(taddr + c * LD, v);
        if (c == 0)
            s = *pa * *pb;
        tmem_wait_ld(v);
        if (c + 1 == NCH) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(tempty_cluster_addr);
        }
        fma_cols<LD>(acc + c * LD, v, s);
    }
}

// Work unit of one CTA of a pair: its 128 rows of a 256-row pair tile.
struct PairWork {
    int g, m_blk, n_blk, tile;
    int a_row0;      // this CTA's first row in A's (and D's) 2-D view
    int sfa_x;       // this CTA's first row in SFA's M-major view (within the group when masked)
    int valid_rows;  // rows of this CTA's half that belong in D (0 .. 128)
};

// The tile sequence of one pair.  Both CTAs, and every role in each, run
// their own copy and see the same sequence of tiles.
//   plain      pair tile t = (256-row block, 128-column block), banded
//              rasterisation as in the one-CTA scheduler;
//   contiguous pair tiles come in two passes.  Pass 0 multiplies both
//              128-row blocks of a pair tile by the B of the first block's
//              group, and stores the second block's rows only if it has the
//              same group.  Pass 1 exists only for pair tiles whose two
//              blocks belong to different groups: it multiplies them by the
//              second block's B and stores the second block's rows.  (Both
//              CTAs of an MMA pair must read the same B.)  A block whose
//              index is -1 is skipped; any other index outside [0, G) is
//              skipped and reported;
//   masked     per group, ceil(count / 256) row blocks x the column blocks.
template <int KIND>
struct PairScheduler {
    const Params &p;
    int next_tile;
    int walk_g = 0, walk_base = 0, walk_tiles = -1, walk_count = 0;
    bool report;

    __device__ PairScheduler(const Params &pp, bool report_bad_groups) : p(pp), report(report_bad_groups)
    {
        next_tile = (int)blockIdx.x / 2;
    }

    // (read from special registers when needed rather than held)
    __device__ __forceinline__ int npairs() const { return (int)gridDim.x / 2; }
    __device__ __forceinline__ int rank() const { return (int)cluster_ctarank(); }

    __device__ __forceinline__ bool group_ok(int g) const { return g >= 0 && g < p.G; }

    __device__ bool next(PairWork &w)
    {
        if constexpr (KIND == kKindNT || KIND == kKindNTAcc) {
            if (next_tile >= p.num_tiles)
                return false;
            const int t = next_tile;
            next_tile += npairs();
            raster(t, p.num_m_blocks, p.num_n_blocks, p.group_m, w.m_blk, w.n_blk);
            w.g = 0;
            w.tile = t;
            w.a_row0 = w.m_blk * (2 * kBM) + kBM * rank();
            w.sfa_x = w.a_row0;
            w.valid_rows = min(max(p.rows - w.a_row0, 0), kBM);
            return true;
        } else if constexpr (KIND == kKindContiguous) {
            const int T = p.num_tiles / 2;     // pair tiles of one pass
            while (next_tile < p.num_tiles) {
                const int t = next_tile;
                next_tile += npairs();
                const bool pass1 = t >= T;
                raster(pass1 ? t - T : t, p.num_m_blocks, p.num_n_blocks, p.group_m, w.m_blk, w.n_blk);
                const int r0 = w.m_blk * (2 * kBM);
                const int g0 = __ldg(p.layout + r0);
                const int g1 = r0 + kBM < p.rows ? __ldg(p.layout + r0 + kBM) : -1;
                const bool ok0 = group_ok(g0), ok1 = group_ok(g1);
                if (!pass1 && report && ((!ok0 && g0 != -1) || (!ok1 && g1 != -1 && r0 + kBM < p.rows)))
                    atomicOr(p.error_word, kErrBadGroupBit);
                bool live0, live1;
                if (!pass1) {
                    if (ok0) {
                        w.g = g0;
                        live0 = true;
                        live1 = ok1 && g1 == g0;
                    } else if (ok1) {
                        w.g = g1;
                        live0 = false;
                        live1 = true;
                    } else {
                        continue;
                    }
                } else {
                    if (!(ok0 && ok1 && g1 != g0))
                        continue;
                    w.g = g1;
                    live0 = false;
                    live1 = true;
                }
                w.tile = t;
                w.a_row0 = r0 + kBM * rank();
                w.sfa_x = w.a_row0;
                w.valid_rows = (rank() ? live1 : live0) ? kBM : 0;
                return true;
            }
            return false;
        } else {  // masked
            const int t = next_tile;
            for (;;) {
                if (walk_g >= p.G)
                    return false;
                if (walk_tiles < 0) {
                    walk_count = min(max(__ldg(p.layout + walk_g), 0), p.rows);
                    walk_tiles = ((walk_count + 2 * kBM - 1) / (2 * kBM)) * p.num_n_blocks;
                }
                if (t < walk_base + walk_tiles)
                    break;
                walk_base += walk_tiles;
                walk_tiles = -1;
                ++walk_g;
            }
            next_tile += npairs();
            const int mb = (walk_count + 2 * kBM - 1) / (2 * kBM);
            raster(t - walk_base, mb, p.num_n_blocks, mb, w.m_blk, w.n_blk);
            w.g = walk_g;
            w.tile = t;
            const int row_in_group = w.m_blk * (2 * kBM) + kBM * rank();
            w.a_row0 = walk_g * p.rows + row_in_group;
            w.sfa_x = row_in_group;
            w.valid_rows = min(max(walk_count - row_in_group, 0), kBM);
            return true;
        }
    }
};

template <int BN, int KIND>
__global__ void __launch_bounds__(kNumThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ CUtensorMap tmap_sfa,
                         const __grid_constant__ CUtensorMap tmap_sfb, const __grid_constant__ CUtensorMap tmap_c,
                         const __grid_constant__ Params p)
{
#if defined(__CUDA_ARCH__)
    using C = PairCfg<BN>;
    constexpr int S = C::kStages;
    constexpr int NACC = C::kAccBufs;
    constexpr int SR = C::kScaleSlots;
    constexpr int COLS = C::kColsPerThread;
    // the addend at 256-column tiles: warp 2 copies C into the staging area
    // and stores the tile, as in the one-CTA kernel (each CTA of the pair
    // handles the C of its own 128 rows)
    constexpr bool kHelperC = KIND == kKindNTAcc && BN == 256;
    static_assert(!kHelperC || (COLS == 2 * kAddendHalfCols &&
                                C::kPanelsPerWarp * C::kPanelBytes >= 32 * kAddendHalfCols * 4),
                  "addend halves");

    // shared memory, the same layout in both CTAs (the leader's descriptors
    // name the peer's operand tiles by the same offsets):
    // [A stages][B stages][D staging][scale slots][barriers][tmem addr, abort]
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + S * C::kABytes;
    uint8_t *sm_stage_d = sm_b + S * C::kBBytes;
    uint8_t *sm_scales = sm_stage_d + C::kStagingBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm_scales + SR * C::kSlotBytes);
    uint64_t *full = bar;              // S:  leader: both CTAs' A/B tiles landed
    uint64_t *empty = full + S;        // S:  the stage's MMAs finished (multicast commit)
    uint64_t *tempty = empty + S;      // NACC: leader: both epilogues finished reading a TMEM buffer
    uint64_t *sfull = tempty + NACC;   // SR: scale slot landed (local)
    uint64_t *sempty = sfull + SR;     // SR: epilogue finished reading a scale slot (local)
    uint64_t *drain = sempty + SR;
    uint64_t *c_full = drain + 1;      // a half tile of C landed in the staging area (local)
    uint64_t *c_free = c_full + 1;     // every epilogue warp has added the first half
    uint64_t *d_ready = c_free + 1;    // every epilogue warp has left its bf16 rows in the staging area
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(d_ready + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 2);            // one arrive.expect_tx per producer
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NACC; ++i)
            mbar_init(&tempty[i], 2 * kNumEpiWarps);
        for (int i = 0; i < SR; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], kNumEpiWarps);
        }
        mbar_init(drain, 1);
        mbar_init(c_full, 1);
        mbar_init(c_free, kNumEpiWarps);
        mbar_init(d_ready, kNumEpiWarps);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_shared();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        prefetch_tensormap(&tmap_d);
        prefetch_tensormap(&tmap_sfa);
        prefetch_tensormap(&tmap_sfb);
        if (kHelperC)
            prefetch_tensormap(&tmap_c);
    }
    __syncthreads();
    // both CTAs' barriers are initialised before any remote arrival or copy
    // signal can reach them, and both are present for the allocation
    cluster_sync();
    if (warp == 1) {
        // one warp of each CTA allocates, together, the same columns in both
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

    if (warp < kEpiWarp0) {
        regs_dealloc<C::kRegsCtl>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            PairScheduler<KIND> sched(p, false);
            PairWork w;
            Ring ring, sring;
            const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
            uint32_t issued = 0, issued_parity = 0, sissued = 0, sissued_parity = 0;
            bool ok = true;
            while (ok && sched.next(w)) {
                if (!bounds_ok(w.g >= 0 && w.g < p.G && w.n_blk >= 0 && w.n_blk * BN < p.N && w.a_row0 >= 0 &&
                                   (w.valid_rows == 0 || (w.a_row0 < p.a_rows_total && w.valid_rows <= kBM)),
                               ctl)) {
                    ok = false;
                    break;
                }
                const int b_row0 = w.g * p.N + w.n_blk * BN + rank * C::kBHalfRows;
                const int sfa_y0 = (KIND == kKindMasked) ? w.g * p.kb : 0;
                const int sfb_x0 = (w.g * p.nb + (w.n_blk * BN) / 128) * p.kb;
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
                    if (k % kScaleChunk == 0) {
                        // the scales of this CTA's rows for the chunk of K blocks starting here
                        if (!mbar_wait(&sempty[sring.i], sring.ph ^ 1u, ctl)) {
                            ok = false;
                            break;
                        }
                        uint8_t *slot = sm_scales + sring.i * C::kSlotBytes;
                        mbar_arrive_expect_tx(&sfull[sring.i], C::kSlotTxBytes);
                        tma_load_2d(slot, &tmap_sfa, &sfull[sring.i], w.sfa_x, sfa_y0 + k);
#pragma unroll
                        for (int j = 0; j < C::kSfbRows; ++j)
                            tma_load_1d(slot + C::kSlotSfaBytes + C::kSlotSfbStride * j, &tmap_sfb,
                                        &sfull[sring.i], (sfb_x0 + j * p.kb + k) & ~3);
                        sissued |= 1u << sring.i;
                        sissued_parity = (sissued_parity & ~(1u << sring.i)) | (sring.ph << sring.i);
                        sring.template next<SR>();
                    }
                    ring.template next<S>();
                }
            }
            // the operand copies of both CTAs count on the leader's barriers:
            // the leader waits for every fill it started (the peer started the
            // same ones unless the pair aborted); scale copies are local
            if (rank == 0)
                for (int i = 0; i < S; ++i)
                    if (issued & (1u << i))
                        mbar_wait_drain(&full[i], (issued_parity >> i) & 1u, p.timeout_ns);
            for (int i = 0; i < SR; ++i)
                if (sissued & (1u << i))
                    mbar_wait_drain(&sfull[i], (sissued_parity >> i) & 1u, p.timeout_ns);
        } else if (kHelperC && warp == 2 && lane == 0) {
            // ------------------------------------------------ addend/store (accumulate)
            // Per tile, in this CTA's staging area: once the previous tile's
            // stores have read it, C's first half (64 of each epilogue warp's
            // 128 columns, one 3-D box of 4 x 32 rows x 16 fp32 columns per
            // warp); when every warp has added it, the second half; when
            // every warp has left its bf16 rows there, the tile's stores.
            // Rows past M and columns past N arrive as zeros.
            PairScheduler<KIND> sched(p, false);
            PairWork w;
            uint32_t ph = 0, c_issued = 0;
            bool pending = false, ok = true;
            while (ok && sched.next(w)) {
                if (pending)
                    bulk_wait_group_read<0>();
                const int chunk0 = (w.n_blk * BN) / 16;     // the tile's first 16-column slab of C
                for (int rd = 0; rd < 2 && ok; ++rd) {
                    if (rd == 1 && !mbar_wait(c_free, ph, ctl)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(c_full, kNumEpiWarps * C::kPanelsPerWarp * C::kPanelBytes);
#pragma unroll 1
                    for (int e = 0; e < kNumEpiWarps; ++e)
                        tma_load_3d(sm_stage_d + e * C::kPanelsPerWarp * C::kPanelBytes, &tmap_c, c_full, 0,
                                    w.a_row0 + 32 * (e & 3), chunk0 + (e >> 2) * (COLS / 16) + rd * 4);
                    ++c_issued;
                }
                if (!ok || !mbar_wait(d_ready, ph, ctl)) {
                    ok = false;
                    break;
                }
                ph ^= 1u;
#pragma unroll 1
                for (int e = 0; e < kNumEpiWarps; ++e) {
                    // the epilogue's rule: full 32-row slabs go by TMA, others
                    // were written by their warp directly
                    if (w.valid_rows - 32 * (e & 3) < 32)
                        continue;
                    for (int pi = 0; pi < C::kPanelsPerWarp; ++pi) {
                        const int x = w.n_blk * BN + (e >> 2) * COLS + pi * C::kPanelCols;
                        if (x < p.N)
                            tma_store_2d(&tmap_d,
                                         sm_stage_d + e * C::kPanelsPerWarp * C::kPanelBytes + pi * C::kPanelBytes,
                                         x, w.a_row0 + 32 * (e & 3));
                    }
                }
                bulk_commit_group();
                pending = true;
            }
            // every store is done and the last addend copy has landed before
            // the CTA exits
            bulk_wait_group<0>();
            if (c_issued)
                mbar_wait_drain(c_full, (c_issued - 1) & 1u, p.timeout_ns);
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer (leader)
            PairScheduler<KIND> sched(p, false);
            PairWork w;
            Ring ring, acc;
            constexpr uint32_t idesc = idesc_e4m3_f32(2 * kBM, BN);
            bool ok = true;
            while (ok && sched.next(w)) {
                for (int k = 0; k < p.kb; ++k) {
                    if (!mbar_wait(&tempty[acc.i], acc.ph ^ 1u, ctl) || !mbar_wait(&full[ring.i], ring.ph, ctl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + acc.i * BN;
                    const uint64_t a0 = sdesc_kmajor_sw128(smem_u32(sm_a + ring.i * C::kABytes));
                    const uint64_t b0 = sdesc_kmajor_sw128(smem_u32(sm_b + ring.i * C::kBBytes));
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)  // +32 bytes along K = +2 in the address field
                        mma_f8f6f4_pair(d_tmem, a0 + 2 * kk, b0 + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                    // one commit per K block, to the stage's empty barrier of
                    // both CTAs: frees the stage for both producers and tells
                    // both epilogues that TMEM buffer acc.i is complete
                    mma_commit_pair(&empty[ring.i], 0x3);
                    ring.template next<S>();
                    acc.template next<NACC>();
                }
            }
            // all MMAs issued above complete before either CTA frees its tensor memory
            mma_commit_pair(drain, 0x1);
            mbar_wait_drain(drain, 0, p.timeout_ns);
        }
    } else {
        regs_alloc<C::kRegsEpi>();
        // ------------------------------------------------ epilogue warps (both CTAs)
        const int ew = warp - kEpiWarp0;     // 0..7
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int h = ew >> 2;               // column half of the tile
        const int row_in_tile = 32 * q + lane;
        const int sfb_row = (BN == 256) ? h : 0;   // the warp's 128-column block of the tile
        uint8_t *panels = sm_stage_d + ew * C::kPanelsPerWarp * C::kPanelBytes;
        const uint32_t leader_tempty = mapa_shared(smem_u32(tempty), 0);

        if (KIND == kKindMasked && blockIdx.x == 0 && ew == 0) {
            for (int g = lane; g < p.G; g += 32) {
                const int c = __ldg(p.layout + g);
                if (c < 0 || c > p.rows)
                    atomicOr(p.error_word, kErrBadGroupBit);
            }
        }

        PairScheduler<KIND> sched(p, rank == 0 && ew == 0 && lane == 0);
        PairWork w;
        Ring ring, acc_ring, sring;
        bool ok = true;
        uint32_t cph = 0;       // phase of c_full this warp waits for next (addend/store warp)
        // with the addend/store warp, half 0 of C is added halfway through
        // the tile's K blocks, which releases the staging area for half 1;
        // below 8 K blocks both halves are added after the loop.  Measured on
        // 4096 x 7168 x 2048 (16 K blocks), adding half 0 after K block 4,
        // 6, 8, 10, 11 or 12: 66.0, 62.7, 62.1, 62.1, 62.8, 65.0 us
        const bool c_early = p.kb >= 8;
        const int k_c0 = p.kb / 2;
        // wait for half rd of C, add it and, for the first half, hand the
        // staging area back
        auto take_c = [&](float (&a)[COLS], int rd) -> bool {
            if (!warp_wait(c_full, cph, ctl))
                return false;
            cph ^= 1u;
            __syncwarp();
            add_c_box<COLS>(a, panels, lane, rd);
            __syncwarp();           // every lane's reads before the area is reused
            if (rd == 0 && lane == 0)
                mbar_arrive(c_free);
            return true;
        };
        (void)take_c;
        (void)c_early;
        (void)k_c0;
        while (ok && sched.next(w)) {
            float acc[COLS];
            if (KIND == kKindNTAcc && !bounds_ok(w.a_row0 + w.valid_rows <= p.rows || w.valid_rows == 0, ctl)) {
                ok = false;
                break;
            }
            if constexpr (KIND == kKindNTAcc && !kHelperC) {
                // the addend starts the accumulator (the only CTA of the tile)
                Work w1;
                w1.a_row0 = w.a_row0;
                w1.n_blk = w.n_blk;
                w1.kb1 = p.kb;
                w1.valid_rows = w.valid_rows;
                init_from_c<BN, COLS>(acc, p, w1, q, h, lane);
            } else {
#pragma unroll
                for (int i = 0; i < COLS; ++i)
                    acc[i] = 0.f;
            }

            for (int k = 0; k < p.kb; ++k) {
                const int kc = k % kScaleChunk;
                if (!warp_all((kc != 0 || mbar_wait(&sfull[sring.i], sring.ph, ctl)) &&
                              mbar_wait(&empty[ring.i], ring.ph, ctl))) {
                    ok = false;
                    break;
                }
                __syncwarp();
                tc_fence_after_sync();
                const uint8_t *slot = sm_scales + sring.i * C::kSlotBytes;
                const float *pa = reinterpret_cast<const float *>(slot) + kc * kBM + row_in_tile;
                const int sfb_idx0 = (w.g * p.nb + (w.n_blk * BN) / 128 + sfb_row) * p.kb + (k - kc);
                const float *pb = reinterpret_cast<const float *>(slot + C::kSlotSfaBytes +
                                                                  C::kSlotSfbStride * sfb_row) + (sfb_idx0 & 3) + kc;

                // promote, and hand the buffer back to the leader's MMA issuer
                const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + acc_ring.i * BN + h * COLS;
                promote_block_pair<COLS, 64>(acc, taddr, pa, pb, leader_tempty + 8u * acc_ring.i, lane);
                acc_ring.template next<NACC>();
                ring.template next<S>();
                if (kc == kScaleChunk - 1 || k + 1 == p.kb) {
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&sempty[sring.i]);
                    sring.template next<SR>();
                }
                if constexpr (kHelperC) {
                    if (c_early && k == k_c0 && !take_c(acc, 0)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok)
                break;

            // ---- bf16 store of this warp's 32 rows x COLS columns
            int rows_ok = min(max(w.valid_rows - 32 * q, 0), 32);
            const int y_row0 = w.a_row0 + 32 * q;
            if (rows_ok > 0 && !bounds_ok(y_row0 >= 0 && y_row0 + rows_ok <= p.d_rows_total, ctl))
                rows_ok = 0;
            const int x = w.n_blk * BN + h * COLS;
            if constexpr (kHelperC) {
                // the addend/store warp waited for the previous tile's stores
                // before copying C here; the second half (and, for short K,
                // the first) goes in now
                if ((!c_early && !take_c(acc, 0)) || !take_c(acc, 1)) {
                    ok = false;
                    break;
                }
            } else {
                // the previous tile's store has had a whole tile to read this
                // warp's panel; make sure it has
                if (lane == 0)
                    bulk_wait_group_read<0>();
                __syncwarp();
            }
            constexpr int PC = C::kPanelCols;
#pragma unroll
            for (int pi = 0; pi < COLS / PC; ++pi)
                if (x + pi * PC < p.N && rows_ok > 0)
                    store_panel<PC, false, !kHelperC>(acc + pi * PC, panels + pi * C::kPanelBytes, &tmap_d, p,
                                                      x + pi * PC, y_row0, rows_ok, lane);
            if constexpr (kHelperC) {
                // the full 32-row slabs are in the staging area: the
                // addend/store warp stores them
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(d_ready);
            }
        }
        if constexpr (KIND == kKindNTAcc)
            cp_async_wait_all();
        if (lane == 0)
            bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    // no remote arrival, copy signal or MMA write reaches either CTA after this
    cluster_sync();
    if (__syncthreads_or(*abort_flag)) {
        // an aborted pair may have stopped with operand copies in flight that
        // no barrier it still waits on counts: give them time to land before
        // the shared memory is released
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
