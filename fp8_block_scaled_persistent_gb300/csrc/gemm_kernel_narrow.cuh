// gemm_kernel_narrow.cuh -- the plain FP8 (E4M3) GEMM for at most 128 rows of
// A: one CTA per narrow column slice of the output (48 or 64 columns), the
// whole K range each, no split and so no partial sums to publish or reduce.
//
// What is computed: the method's GEMM (DeepGEMM fp8_gemm.cuh, fp8_gemm_kernel:
// each 128-wide K block's partial product is formed on its own in fp32 and
// promoted into an fp32 accumulator with scale_a(row, k) * scale_b(n/128, k),
// rounded to bf16 at the end), in the same K order as the one-CTA kernel.
//
// Why a kernel of its own: with M <= 128 the work is one stream of B from
// HBM.  Split over K (the one-CTA kernel's stream-K schedule), every CTA whose
// K range ends inside a tile publishes an fp32 partial and another reduces it,
// and those partials' trips through the memory system set the tail of the
// launch.  Here each CTA streams B[BN slice rows][K] once (BN = 48 or 64) and
// stores its outputs itself.  A 48-column slice may straddle one boundary of
// the 128-column scale blocks: its scale slots then hold both blocks' B
// scales and each 16-column chunk of the slice takes its block's.  The narrow
// tile makes each K block small (6 or 8 KB of B), so the per-K-block costs
// are batched: every copy brings KD consecutive K blocks (one 3-D box of A,
// one of B), and the MMA issuer, the epilogue and the buffer releases work a
// whole copy (a "group" of KD K blocks) at a time.
//
// 192 threads (six warps):
//   warp 0      TMA producer: per group one box of A (KD x A_ROWS rows x
//               128 B) and one of B (KD x BN rows x 128 B), 128-byte swizzled,
//               into an S-stage ring; the scales of kScaleChunk K blocks at a
//               time (128 A scales per K block, the slice's B scales) into a
//               scale ring.
//   warp 1      MMA issuer (and tensor-memory owner): per group, 4 x
//               tcgen05.mma kind::f8f6f4 (128 x BN x 32) per K block, each K
//               block into its own 64-column buffer of the group, then one
//               commit, which frees the stage and tells the epilogue the group
//               is complete.  512 columns hold 512 / (64 KD) groups.
//   warps 2-5   epilogue, one per tensor-memory lane quarter (warp & 3): per
//               K block a tcgen05.ld of its 32 rows x BN columns and
//               acc += (sa*sb) * P in fp32 registers; the group is released
//               once its last load has landed.  At the end of a slice, bf16
//               (round to nearest even) row stores; rows past M and columns
//               past N are not written.
// With A_ROWS = 64 (M <= 64) only the first 64 rows of A are loaded: the MMA
// still forms 128 rows, whose upper half reads the stage's next bytes (in
// bounds: B follows A in every stage) and is never read back.
//
// Every wait is bounded; on expiry the CTA records an error, drains its copies
// in flight, frees its tensor memory and returns.
#pragma once

#include "gemm_kernel.cuh"

namespace fp8g {

template <int BN, int A_ROWS, int KD, int S>
struct NarrowCfg {
    static_assert(BN == 48 || BN == 64, "slice width");
    static_assert(A_ROWS == 64 || A_ROWS == 128, "A box rows");
    static_assert(KD == 2 || KD == 4, "K blocks per copy (a divisor of kScaleChunk)");
    static constexpr int kBN = BN;                          // output columns (B rows) per CTA
    static constexpr int kBufCols = 64;                     // tensor-memory columns per K block
    // 128-column scale blocks a slice can touch
    static constexpr int kSfbRows = (128 % BN == 0) ? 1 : 2;
    static constexpr int kThreads = 192;
    static constexpr int kEpi0 = 2;                         // warps 2..5: the epilogue
    static constexpr int kABlockBytes = A_ROWS * kBK;       // one K block of A
    static constexpr int kBBlockBytes = kBN * kBK;          // one K block of B
    static constexpr int kABytes = KD * kABlockBytes;
    static constexpr int kBBytes = KD * kBBlockBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;   // A then B
    static constexpr int kGroups = kTmemCols / (KD * kBufCols);    // tensor-memory groups
    static constexpr int kScaleSlots = 4;
    static constexpr int kSlotSfaBytes = kScaleChunk * kBM * 4;
    static constexpr int kSlotBytes = kSlotSfaBytes + 128 * kSfbRows;
    static constexpr int kSlotTxBytes = kSlotSfaBytes + (kScaleChunk + 4) * 4 * kSfbRows;
    static constexpr int kBarriers = 2 * S + kGroups + 2 * kScaleSlots + 1;
    static constexpr int kSmemBytes = S * kStageBytes + kScaleSlots * kSlotBytes + kBarriers * 8 + 16 +
                                      1024 /* alignment slack */;
    static_assert(kABlockBytes % 1024 == 0 && kBBlockBytes % 1024 == 0 && kStageBytes % 1024 == 0 &&
                      kSlotBytes % 128 == 0,
                  "every K block's tiles start on a 1024-byte boundary (128-byte swizzle)");
    // the MMA reads 128 rows of A from each K block's tile: with a 64-row box
    // the last K block's upper half lies in the same stage's B tiles
    static_assert(A_ROWS == 128 || kBM * kBK <= kABlockBytes + kBBytes, "MMA reads stay inside the stage");
    // the epilogue's wait on a stage's MMA completion must not alias: the
    // stage's next use needs the group this warp releases first
    static_assert(S >= kGroups, "stages >= tensor-memory groups");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// This thread's row of one K block's partial: BN columns from taddr on.
template <int BN>
__device__ __forceinline__ void narrow_ld(uint32_t taddr, uint32_t (&v)[BN])
{
    if constexpr (BN == 64) {
        tmem_ld_32x32b_x64(taddr, v);
        tmem_wait_ld(v);
    } else {
        uint32_t v0[32], v1[16];
        tmem_ld_32x32b_x32(taddr, v0);
        tmem_ld_32x32b_x16(taddr + 32, v1);
        tmem_wait_ld(v0);
        tmem_wait_ld(v1);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = v0[i];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[32 + i] = v1[i];
    }
}

template <int BN, int A_ROWS, int KD, int S>
__global__ void __launch_bounds__(NarrowCfg<BN, A_ROWS, KD, S>::kThreads, 1)
    fp8_gemm_narrow_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                           const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                           const __grid_constant__ Params p)
{
#if defined(__CUDA_ARCH__)
    using C = NarrowCfg<BN, A_ROWS, KD, S>;
    constexpr int BC = C::kBufCols;
    constexpr int NG = C::kGroups;
    constexpr int SR = C::kScaleSlots;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sm_stage = smem;                                   // S x [A | B]
    uint8_t *sm_scales = sm_stage + S * C::kStageBytes;         // SR scale slots
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm_scales + SR * C::kSlotBytes);
    uint64_t *full = bar;                  // S: a group's A/B tiles landed (TMA transactions)
    uint64_t *empty = full + S;            // S: the group's MMAs finished (stage free, partials ready)
    uint64_t *tempty = empty + S;          // NG: the epilogue read the group's buffers (4 warps)
    uint64_t *sfull = tempty + NG;         // SR: a scale chunk landed
    uint64_t *sempty = sfull + SR;         // SR: the epilogue is done with it (4 warps)
    uint64_t *drain = sempty + SR;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NG; ++i)
            mbar_init(&tempty[i], 4);
        for (int i = 0; i < SR; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        fence_proxy_async_shared();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        prefetch_tensormap(&tmap_sfa);
        prefetch_tensormap(&tmap_sfb);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // a programmatic dependent of the previous kernel on the stream: nothing
    // in global memory is touched before that grid has completed
    grid_dependency_wait();
    grid_launch_dependents();

    const WaitCtl ctl{abort_flag, p.error_word, p.timeout_ns};
    const int slices = p.num_n_blocks;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        Ring ring, sring;
        uint32_t issued = 0, issued_parity = 0, sissued = 0, sissued_parity = 0;
        bool ok = bounds_ok(p.a_box_rows == A_ROWS && p.rows <= A_ROWS, ctl);
        for (int s = blockIdx.x; ok && s < slices; s += gridDim.x) {
            const int b_row0 = s * BN;
            if (!bounds_ok(b_row0 < p.N, ctl)) {
                ok = false;
                break;
            }
            const int sfb0 = (b_row0 / 128) * p.kb;     // the slice's column block in the flat SFB
            for (int k0 = 0; k0 < p.kb; k0 += KD) {
                if (!mbar_wait(&empty[ring.i], ring.ph ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                // K blocks past the end arrive as zeros and are never used;
                // the transaction count is always the whole boxes'
                uint8_t *st = sm_stage + ring.i * C::kStageBytes;
                mbar_arrive_expect_tx(&full[ring.i], C::kStageBytes);
                tma_load_3d(st, &tmap_a, &full[ring.i], 0, 0, k0);
                tma_load_3d(st + C::kABytes, &tmap_b, &full[ring.i], 0, b_row0, k0);
                issued |= 1u << ring.i;
                issued_parity = (issued_parity & ~(1u << ring.i)) | (ring.ph << ring.i);
                ring.template next<S>();
                if (k0 % kScaleChunk == 0) {
                    if (!mbar_wait(&sempty[sring.i], sring.ph ^ 1u, ctl)) {
                        ok = false;
                        break;
                    }
                    uint8_t *slot = sm_scales + sring.i * C::kSlotBytes;
                    mbar_arrive_expect_tx(&sfull[sring.i], C::kSlotTxBytes);
                    tma_load_2d(slot, &tmap_sfa, &sfull[sring.i], 0, k0);
                    // the slice's column block and, for a slice that may
                    // straddle, the next one (past the last block: zeros)
#pragma unroll
                    for (int j = 0; j < C::kSfbRows; ++j)
                        tma_load_1d(slot + C::kSlotSfaBytes + 128 * j, &tmap_sfb, &sfull[sring.i],
                                    (sfb0 + j * p.kb + k0) & ~3);
                    sissued |= 1u << sring.i;
                    sissued_parity = (sissued_parity & ~(1u << sring.i)) | (sring.ph << sring.i);
                    sring.template next<SR>();
                }
            }
        }
        // every copy this thread started has landed before the CTA exits
        for (int i = 0; i < S; ++i)
            if (issued & (1u << i))
                mbar_wait_drain(&full[i], (issued_parity >> i) & 1u, p.timeout_ns);
        for (int i = 0; i < SR; ++i)
            if (sissued & (1u << i))
                mbar_wait_drain(&sfull[i], (sissued_parity >> i) & 1u, p.timeout_ns);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        Ring ring, acc;
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
        bool ok = true;
        for (int s = blockIdx.x; ok && s < slices; s += gridDim.x) {
            for (int k0 = 0; k0 < p.kb; k0 += KD) {
                const int nk = min(KD, p.kb - k0);
                if (!mbar_wait(&tempty[acc.i], acc.ph ^ 1u, ctl) || !mbar_wait(&full[ring.i], ring.ph, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t st = smem_u32(sm_stage + ring.i * C::kStageBytes);
                const uint32_t d0 = tmem_base + acc.i * (KD * BC);
                // K block j of the group: its own buffer; the first MMA overwrites
                auto kblock = [&](int j) {
                    const uint64_t a0 = sdesc_kmajor_sw128(st + j * C::kABlockBytes);
                    const uint64_t b0 = sdesc_kmajor_sw128(st + C::kABytes + j * C::kBBlockBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)  // +32 bytes along K = +2 in the address field
                        mma_f8f6f4(d0 + j * BC, a0 + 2 * kk, b0 + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                };
                if (nk == KD) {
#pragma unroll
                    for (int j = 0; j < KD; ++j)
                        kblock(j);
                } else {
                    for (int j = 0; j < nk; ++j)
                        kblock(j);
                }
                mma_commit(&empty[ring.i]);
                ring.template next<S>();
                acc.template next<NG>();
            }
        }
        // all MMAs issued above complete before tensor memory is freed
        mma_commit(drain);
        mbar_wait_drain(drain, 0, p.timeout_ns);
    } else if (warp >= C::kEpi0 && warp < C::kEpi0 + 4) {
        // ------------------------------------------------ epilogue warps
        const int q = warp & 3;                  // the TMEM lane quarter this warp may access
        const int row = 32 * q + lane;           // row of A / D
        const bool quarter_live = p.rows > 32 * q;
        Ring ring, acc, sring;
        bool ok = true;
        for (int s = blockIdx.x; ok && s < slices; s += gridDim.x) {
            const int col0 = s * BN;
            const int sfb0 = (col0 / 128) * p.kb;
            // columns of the slice before the next 128-column block starts
            const int jb = 128 * (col0 / 128 + 1) - col0;
            float accum[BN];
#pragma unroll
            for (int i = 0; i < BN; ++i)
                accum[i] = 0.f;
            for (int k0 = 0; k0 < p.kb; k0 += KD) {
                const int nk = min(KD, p.kb - k0);
                const int kc0 = k0 % kScaleChunk;        // the group's place in its scale chunk
                int got = 1;
                if (lane == 0)
                    got = ((kc0 != 0 || mbar_wait(&sfull[sring.i], sring.ph, ctl)) &&
                           mbar_wait(&empty[ring.i], ring.ph, ctl))
                              ? 1
                              : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                __syncwarp();           // orders lane 0's barrier waits before every lane's reads
                tc_fence_after_sync();
                if (quarter_live) {
                    const uint8_t *slot = sm_scales + sring.i * C::kSlotBytes;
                    const float *pa = reinterpret_cast<const float *>(slot) + kc0 * kBM + row;
                    // the B scales of the chunk's column block(s), from the
                    // aligned groups of 4 the producer copied (the next
                    // block's group starts at the same offset: kb is the
                    // block stride and the chunk start is shared)
                    const float *pb = reinterpret_cast<const float *>(slot + C::kSlotSfaBytes) +
                                      ((sfb0 + k0 - kc0) & 3) + kc0;
                    const float *pb1 = reinterpret_cast<const float *>(slot + C::kSlotSfaBytes + 128) +
                                       ((sfb0 + p.kb + k0 - kc0) & 3) + kc0;
                    const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + acc.i * (KD * BC);
#pragma unroll
                    for (int j = 0; j < KD; ++j) {
                        if (j < nk) {
                            const float sa = pa[j * kBM];
                            const float s0 = sa * pb[j];
                            const float s1 = (C::kSfbRows > 1 && jb < BN) ? sa * pb1[j] : s0;
                            uint32_t v[BN];
                            narrow_ld<BN>(taddr + j * BC, v);
                            if (j + 1 == nk)
                                release_tmem(&tempty[acc.i], lane);
#pragma unroll
                            for (int c = 0; c < BN / 16; ++c)
                                fma_cols<16>(accum + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(v + 16 * c),
                                             16 * c < jb ? s0 : s1);
                        }
                    }
                } else {
                    release_tmem(&tempty[acc.i], lane);   // rows past M: nothing to read
                }
                ring.template next<S>();
                acc.template next<NG>();
                if (kc0 + KD == kScaleChunk || k0 + KD >= p.kb) {
                    // the chunk's last group: its scale slot may be refilled
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&sempty[sring.i]);
                    sring.template next<SR>();
                }
            }
            if (!ok)
                break;
            // ---- bf16 row stores (16 bytes at a time; N is a multiple of 16)
            if (row < p.rows && bounds_ok(row < p.d_rows_total, ctl)) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.d + (size_t)row * p.N + col0);
#pragma unroll
                for (int c = 0; c < BN / 8; ++c) {
                    if (col0 + 8 * c < p.N)
                        dst[c] = make_uint4(pack_bf16x2(accum[8 * c], accum[8 * c + 1]),
                                            pack_bf16x2(accum[8 * c + 2], accum[8 * c + 3]),
                                            pack_bf16x2(accum[8 * c + 4], accum[8 * c + 5]),
                                            pack_bf16x2(accum[8 * c + 6], accum[8 * c + 7]));
                }
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
