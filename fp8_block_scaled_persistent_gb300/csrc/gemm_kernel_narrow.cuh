// gemm_kernel_narrow.cuh -- the plain FP8 (E4M3) GEMM for at most 128 rows of
// A: one CTA per narrow column slice of the output (48, 64 or 96 columns),
// over the whole K range or over one of two K parts.
//
// What is computed: the method's GEMM (DeepGEMM fp8_gemm.cuh, fp8_gemm_kernel:
// each 128-wide K block's partial product is formed on its own in fp32 and
// promoted into an fp32 accumulator with scale_a(row, k) * scale_b(n/128, k),
// rounded to bf16 at the end).
//
// Why a kernel of its own: with M <= 128 the work is one stream of B from
// HBM.  Split over K the one-CTA kernel's way (stream-K), every CTA whose K
// range ends inside a tile publishes an fp32 partial and another reduces it,
// and those partials' trips through the memory system set the tail of the
// launch.  Here the work units are (slice, K part) pairs, KSPLIT parts per
// slice, and every CTA's range lies inside one slice:
//   KSPLIT = 1  each CTA streams B[BN slice rows][K] once and stores its
//               outputs itself (nothing published);
//   KSPLIT = 2  the two CTAs of a slice, a cluster of two, stream one K half
//               each (half of A per CTA: with 128 rows of A, A's copies rival
//               B's), then trade halves of the slice over distributed shared
//               memory: each stores the fp32 partial of the columns the other
//               finalises straight into the other's shared memory, waits for
//               the other's, adds it (P0 + P1: fp32 addition commutes, so both
//               orders give the same bits) and stores its half.  Every CTA
//               sends before it waits, so the waits end; nothing goes through
//               global memory, so no workspace.
// The library's build (gemm_narrow.cu) runs two K parts of 96-column slices
// for both A box heights; one part (and 48- or 64-column slices) measured
// slower and stays a build option.
// A slice whose width does not divide 128 may straddle one boundary of the
// 128-column scale blocks: its scale slots then hold both blocks' B scales
// and each 16-column chunk of the slice takes its block's.  The narrow tile
// makes each K block small (6 to 12 KB of B), so the per-K-block costs are
// batched: every copy brings KD consecutive K blocks (one 3-D box of A, one
// of B), and the MMA issuer, the epilogue and the buffer releases work a
// whole copy (a "group" of KD K blocks) at a time.
//
// 192 threads (six warps):
//   warp 0      TMA producer: per group one box of A (KD x A_ROWS rows x
//               128 B) and one of B (KD x BN rows x 128 B), 128-byte swizzled,
//               into an S-stage ring; the scales of kNarrowChunk K blocks at a
//               time (128 A scales per K block, the slice's B scales) into a
//               scale ring.
//   warp 1      MMA issuer (and tensor-memory owner): per group, 4 x
//               tcgen05.mma kind::f8f6f4 (128 x BN x 32) per K block, each K
//               block into its own buffer of the group, then one commit,
//               which frees the stage and tells the epilogue the group is
//               complete.
//   warps 2-5   epilogue, one per tensor-memory lane quarter (warp & 3): per
//               K block tcgen05.ld of its 32 rows x BN columns and
//               acc += (sa*sb) * P in fp32 registers; the group is released
//               once its last load has landed.  Every lane waits and every
//               lane arrives (warp_wait in ptx.cuh).  At the end of a unit, the
//               trade of halves (KSPLIT = 2) and bf16 (round to nearest even)
//               row stores; rows past M and columns past N are not written.
// With A_ROWS = 64 (M <= 64) only the first 64 rows of A are loaded: the MMA
// still forms 128 rows, whose upper half reads the stage's next bytes (in
// bounds: B follows A in every stage) and is never read back.
//
// Every wait is bounded; on expiry the CTA records an error, drains its copies
// in flight, frees its tensor memory and returns.
#pragma once

#include "gemm_kernel.cuh"

// K blocks per scale copy (a multiple of the K blocks per operand copy)
#ifndef FP8G_NARROW_CHUNK
#define FP8G_NARROW_CHUNK 8
#endif

namespace fp8g {

constexpr int kNarrowChunk = FP8G_NARROW_CHUNK;

template <int BN, int A_ROWS, int KD, int S, int KSPLIT>
struct NarrowCfg {
    static_assert(BN == 48 || BN == 64 || BN == 96, "slice width");
    static_assert(KSPLIT == 1 || (KSPLIT == 2 && BN % 32 == 0), "K parts (a traded half is whole float4s)");
    static_assert(A_ROWS == 64 || A_ROWS == 128, "A box rows");
    static_assert((KD == 2 || KD == 4) && kNarrowChunk % KD == 0, "K blocks per copy (a divisor of the chunk)");
    static constexpr int kBN = BN;                          // output columns (B rows) per CTA
    static constexpr int kBufCols = BN <= 64 ? 64 : 128;    // tensor-memory columns per K block
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
    static constexpr int kScaleSlots = 32 / kNarrowChunk;      // 32 K blocks of scales in flight
    static constexpr int kSlotSfaBytes = kNarrowChunk * kBM * 4;
    static constexpr int kSlotBytes = kSlotSfaBytes + 128 * kSfbRows;
    static constexpr int kSlotTxBytes = kSlotSfaBytes + (kNarrowChunk + 4) * 4 * kSfbRows;
    static_assert((kNarrowChunk + 4) * 4 <= 128, "a B scale row of a slot");
    // KSPLIT = 2: the partner's traded half, [BN/8 float4 columns][128 rows]
    static constexpr int kXBytes = KSPLIT == 2 ? (BN / 2) * kBM * 4 : 0;
    static constexpr int kBarriers = 2 * S + kGroups + 2 * kScaleSlots + 1 + 2;
    static constexpr int kSmemBytes = S * kStageBytes + kScaleSlots * kSlotBytes + kXBytes + kBarriers * 8 + 16 +
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
    static_assert(kGroups >= 2, "the MMA fills one group while the epilogue reads another");
    // the two column pieces of one K block's partial (tcgen05.ld of 16, 32 or
    // 64 columns each)
    static constexpr int kPiece0 = BN >= 64 ? 64 : 32;
    static constexpr int kPiece1 = BN - kPiece0;
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// acc[c] += (c < jb ? s0 : s1) * v[c - C0] for the 16-column chunks of one
// piece of a K block's partial (columns C0 .. C0 + NV of the slice).
template <int C0, int NV, int BN>
__device__ __forceinline__ void promote_piece(float (&acc)[BN], const uint32_t (&v)[NV], int jb, float s0, float s1)
{
#pragma unroll
    for (int c = 0; c < NV / 16; ++c)
        fma_cols<16>(acc + C0 + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(v + 16 * c),
                     C0 + 16 * c < jb ? s0 : s1);
}

// The trade of halves (KSPLIT = 2) over distributed shared memory.  This
// warp's rows of columns GIVE0 .. GIVE0 + BN/2 go into the partner CTA's
// buffer (`peer_xbuf`, a shared::cluster address; [BN/8 float4 columns][128
// rows]) and its arrival on the partner's `peer_xfull` releases them; once
// this CTA's `xfull` completes (the partner's four warps), the partner's
// partial of KEEP0 .. KEEP0 + BN/2 is read from `xbuf` and added.  Before a
// later round writes the partner's buffer again, `xempty` (the partner's
// warps have read it) is awaited; after reading, this warp arrives on the
// partner's `peer_xempty` only if another round follows, so no arrival can
// reach a CTA that has exited.  Returns false if a wait ran out.
template <int GIVE0, int KEEP0, int BN>
__device__ __forceinline__ bool trade_halves(float (&acc)[BN], uint32_t peer_xbuf, const float4 *xbuf,
                                             uint64_t *xfull, uint64_t *xempty, uint32_t peer_xfull,
                                             uint32_t peer_xempty, uint32_t round, bool more, bool live, int row,
                                             int lane, const WaitCtl &ctl)
{
    constexpr int C4 = BN / 8;
    if (round > 0 && !warp_wait(xempty, (round - 1) & 1u, ctl))
        return false;
    __syncwarp();
    if (live) {
#pragma unroll
        for (int c = 0; c < C4; ++c)
            st_shared_cluster_f4(peer_xbuf + (uint32_t)(c * kBM + row) * 16u,
                                 make_float4(acc[GIVE0 + 4 * c], acc[GIVE0 + 4 * c + 1], acc[GIVE0 + 4 * c + 2],
                                             acc[GIVE0 + 4 * c + 3]));
    }
    fence_acq_rel_cluster();
    __syncwarp();
    if (lane == 0)
        mbar_arrive_release_cluster(peer_xfull);
    if (!warp_wait(xfull, round & 1u, ctl))
        return false;
    __syncwarp();
    fence_acq_rel_cluster();
    if (live) {
#pragma unroll
        for (int c = 0; c < C4; ++c) {
            const float4 v = xbuf[c * kBM + row];
            acc[KEEP0 + 4 * c] += v.x;
            acc[KEEP0 + 4 * c + 1] += v.y;
            acc[KEEP0 + 4 * c + 2] += v.z;
            acc[KEEP0 + 4 * c + 3] += v.w;
        }
    }
    if (more) {
        __syncwarp();
        if (lane == 0)
            mbar_arrive_release_cluster(peer_xempty);
    }
    return true;
}

// bf16 (round to nearest even) stores of NC columns of this thread's row,
// acc[C0 ..] to D columns x0 .., 16 bytes at a time (N is a multiple of 16).
template <int C0, int NC, int BN>
__device__ __forceinline__ void store_row(const float (&acc)[BN], __nv_bfloat16 *drow, int x0, int N)
{
    uint4 *dst = reinterpret_cast<uint4 *>(drow + x0);
#pragma unroll
    for (int c = 0; c < NC / 8; ++c) {
        if (x0 + 8 * c < N)
            dst[c] = make_uint4(pack_bf16x2(acc[C0 + 8 * c], acc[C0 + 8 * c + 1]),
                                pack_bf16x2(acc[C0 + 8 * c + 2], acc[C0 + 8 * c + 3]),
                                pack_bf16x2(acc[C0 + 8 * c + 4], acc[C0 + 8 * c + 5]),
                                pack_bf16x2(acc[C0 + 8 * c + 6], acc[C0 + 8 * c + 7]));
    }
}

template <int BN, int A_ROWS, int KD, int S, int KSPLIT>
__global__ void __launch_bounds__(NarrowCfg<BN, A_ROWS, KD, S, KSPLIT>::kThreads, 1)
    fp8_gemm_narrow_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                           const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                           const __grid_constant__ Params p)
{
#if defined(__CUDA_ARCH__)
    using C = NarrowCfg<BN, A_ROWS, KD, S, KSPLIT>;
    constexpr int BC = C::kBufCols;
    constexpr int NG = C::kGroups;
    constexpr int SR = C::kScaleSlots;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sm_stage = smem;                                   // S x [A | B]
    uint8_t *sm_scales = sm_stage + S * C::kStageBytes;         // SR scale slots
    uint8_t *sm_xbuf = sm_scales + SR * C::kSlotBytes;          // KSPLIT = 2: the partner's traded half
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm_xbuf + C::kXBytes);
    uint64_t *full = bar;                  // S: a group's A/B tiles landed (TMA transactions)
    uint64_t *empty = full + S;            // S: the group's MMAs finished (stage free, partials ready)
    uint64_t *tempty = empty + S;          // NG: the epilogue read the group's buffers (4 warps x 32 lanes)
    uint64_t *sfull = tempty + NG;         // SR: a scale chunk landed
    uint64_t *sempty = sfull + SR;         // SR: the epilogue is done with it (4 warps x 32 lanes)
    uint64_t *drain = sempty + SR;
    uint64_t *xfull = drain + 1;           // KSPLIT = 2: the partner's half landed here (its 4 warps)
    uint64_t *xempty = xfull + 1;          // KSPLIT = 2: the partner read this CTA's half (its 4 warps)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(xempty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NG; ++i)
            mbar_init(&tempty[i], 4 * 32);      // every lane of the 4 epilogue warps
        for (int i = 0; i < SR; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], 4 * 32);      // every lane of the 4 epilogue warps
        }
        mbar_init(drain, 1);
        mbar_init(xfull, 4);
        mbar_init(xempty, 4);
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
    if constexpr (KSPLIT == 2)
        cluster_sync();     // the partner's barriers exist before anything reaches them
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    // work units: (slice, K part), unit u = KSPLIT * slice + part; a part is
    // a whole number of scale chunks of K blocks (the last may be short or,
    // for a very short K, empty)
    const int units = p.num_n_blocks * KSPLIT;
    const int kb_part = KSPLIT == 1 ? p.kb : ((p.kb + 1) / 2 + kNarrowChunk - 1) / kNarrowChunk * kNarrowChunk;
    auto kb_begin = [&](int u) { return (u % KSPLIT) * kb_part; };
    auto kb_end = [&](int u) { return min(p.kb, (u % KSPLIT + 1) * kb_part); };
    // a programmatic dependent of the previous kernel on the stream: nothing
    // in global memory is read or written before that grid has completed.
    // The next kernel is let in only once this CTA's last copy is issued
    // (below): triggered at the start, its CTAs took the SMs this grid leaves
    // idle for the whole launch (64 x 7168 x 16384: 27.1 -> 26.9 us, 128 x
    // 7168 x 16384: 28.8 -> 28.4 us).
    grid_dependency_wait();

    const WaitCtl ctl{abort_flag, p.error_word, p.timeout_ns};

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        Ring ring, sring;
        uint32_t issued = 0, issued_parity = 0, sissued = 0, sissued_parity = 0;
        bool ok = bounds_ok(p.a_box_rows == A_ROWS && p.rows <= A_ROWS, ctl);
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int b_row0 = (u / KSPLIT) * BN;
            if (!bounds_ok(b_row0 < p.N, ctl)) {
                ok = false;
                break;
            }
            const int sfb0 = (b_row0 / 128) * p.kb;     // the slice's column block in the flat SFB
            for (int k0 = kb_begin(u); k0 < kb_end(u); k0 += KD) {
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
                if (k0 % kNarrowChunk == 0) {
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
        grid_launch_dependents();
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
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int k_end = kb_end(u);
            for (int k0 = kb_begin(u); k0 < k_end; k0 += KD) {
                const int nk = min(KD, k_end - k0);
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
        uint32_t round = 0;     // units this CTA has traded so far
        (void)round;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const int col0 = (u / KSPLIT) * BN;
            const int k_end = kb_end(u);
            const int sfb0 = (col0 / 128) * p.kb;
            // columns of the slice before the next 128-column block starts
            const int jb = 128 * (col0 / 128 + 1) - col0;
            float accum[BN];
#pragma unroll
            for (int i = 0; i < BN; ++i)
                accum[i] = 0.f;
            for (int k0 = kb_begin(u); k0 < k_end; k0 += KD) {
                const int nk = min(KD, k_end - k0);
                const int kc0 = k0 % kNarrowChunk;       // the group's place in its scale chunk
                if (!warp_all((kc0 != 0 || mbar_wait(&sfull[sring.i], sring.ph, ctl)) &&
                              mbar_wait(&empty[ring.i], ring.ph, ctl))) {
                    ok = false;
                    break;
                }
                __syncwarp();
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
                            // both pieces' loads in flight at once; the
                            // buffers go back once both have landed
                            uint32_t v0[C::kPiece0];
                            tmem_ld(taddr + j * BC, v0);
                            if constexpr (C::kPiece1 > 0) {
                                uint32_t v1[C::kPiece1];
                                tmem_ld(taddr + j * BC + C::kPiece0, v1);
                                tmem_wait_ld(v0);
                                tmem_wait_ld(v1);
                                if (j + 1 == nk)
                                    release_tmem(&tempty[acc.i], lane);
                                promote_piece<0>(accum, v0, jb, s0, s1);
                                promote_piece<C::kPiece0>(accum, v1, jb, s0, s1);
                            } else {
                                tmem_wait_ld(v0);
                                if (j + 1 == nk)
                                    release_tmem(&tempty[acc.i], lane);
                                promote_piece<0>(accum, v0, jb, s0, s1);
                            }
                        }
                    }
                } else {
                    release_tmem(&tempty[acc.i], lane);   // rows past M: nothing to read
                }
                ring.template next<S>();
                acc.template next<NG>();
                if (kc0 + KD == kNarrowChunk || k0 + KD >= k_end) {
                    // the chunk's last group: its scale slot may be refilled
                    // (every lane arrives)
                    mbar_arrive(&sempty[sring.i]);
                    sring.template next<SR>();
                }
            }
            if (!ok)
                break;
            const bool live = row < p.rows && bounds_ok(row < p.d_rows_total, ctl);
            __nv_bfloat16 *drow = p.d + (size_t)row * p.N;
            if constexpr (KSPLIT == 1) {
                if (live)
                    store_row<0, BN>(accum, drow, col0, p.N);
            } else {
                // the trade of halves with the slice's other K part (unit u ^ 1,
                // the other CTA of this cluster: the grid is even, so both
                // take their units in the same rounds)
                constexpr int H = BN / 2;
                const uint32_t peer = cluster_ctarank() ^ 1u;
                const uint32_t peer_xbuf = mapa_shared(smem_u32(sm_xbuf), peer);
                const uint32_t peer_xfull = mapa_shared(smem_u32(xfull), peer);
                const uint32_t peer_xempty = mapa_shared(smem_u32(xempty), peer);
                const float4 *xb = reinterpret_cast<const float4 *>(sm_xbuf);
                const bool more = u + (int)gridDim.x < units;
                const bool first = (u & 1) == 0;   // K part 0 keeps the slice's first half
                ok = first ? trade_halves<H, 0>(accum, peer_xbuf, xb, xfull, xempty, peer_xfull, peer_xempty,
                                                round, more, live, row, lane, ctl)
                           : trade_halves<0, H>(accum, peer_xbuf, xb, xfull, xempty, peer_xfull, peer_xempty,
                                                round, more, live, row, lane, ctl);
                ++round;
                if (!ok)
                    break;
                if (live) {
                    if (first)
                        store_row<0, H>(accum, drow, col0, p.N);
                    else
                        store_row<H, H>(accum, drow, col0 + H, p.N);
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // neither CTA of a trading pair leaves while the other may still store
    // into its shared memory or arrive on its barriers (after a wait that ran
    // out, too: every wait is bounded, so both get here)
    if constexpr (KSPLIT == 2)
        cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
#endif
}

}  // namespace fp8g
