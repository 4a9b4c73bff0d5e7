// gemm_kernel.cuh -- persistent, warp-specialised FP8 (E4M3) GEMM with
// fine-grained scaling for sm_103a.
//
// What is computed (DeepGEMM fp8_gemm.cuh, fp8_gemm_kernel): every 128-wide K
// block's partial product A_blk * B_blk^T is formed on its own in fp32 and
// promoted into an fp32 accumulator with scale_a(row, k) * scale_b(n/128, k);
// the accumulator is rounded to bf16 at the end.
//
// How, on Blackwell (design ours; the DeepGEMM page's Hopper kernel and the
// "TCGen05 Copy Instruction" tutorial's warp-specialised matmul are prior art):
//   warp 0      TMA producer: 128x128 A and BNx128 B e4m3 tiles, 128-byte
//               swizzled, into an S-stage shared-memory ring (full/empty
//               mbarriers, transaction-count completion).
//   warp 1      MMA issuer: one thread issues 4 x tcgen05.mma kind::f8f6f4
//               (128 x BN x 32) per K block into a FRESH tensor-memory buffer
//               (the first MMA overwrites), then commits the stage back to the
//               producer and the buffer to the epilogue.  512 TMEM columns
//               hold 512/BN such buffers, so the MMA of block k+1 runs while
//               block k is being promoted.
//   warps 2..9  epilogue: tcgen05.ld of the K block's partial, promotion
//               acc += (sa*sb) * P in fp32 registers (one row per thread,
//               BN/2 columns per warp), and at the end of a tile bf16
//               conversion into a 64-byte-swizzled staging panel and a TMA
//               store (or predicated stores where masked rows straddle).
//   scheduler   persistent: CTA c takes tiles c, c+P, ... in a banded
//               rasterisation (m fastest inside a band of m-blocks); grouped
//               layouts map tiles to groups.  A split-K ("stream-K") variant
//               gives each CTA an equal share of the (tile, K-block) units and
//               lets the last contributor of each tile reduce the fp32
//               partials in a fixed order (deterministic, no spin-wait).
//
// Every wait is bounded (see ptx.cuh); on expiry a CTA records an error,
// drains its copies in flight, frees its tensor memory and returns.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gemm_params.h"
#include "ptx.cuh"

namespace fp8g {

constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kNumThreads = 320;      // 10 warps
constexpr int kEpiWarp0 = 2;
constexpr int kNumEpiWarps = 8;
constexpr int kTmemCols = 512;
constexpr int kPanelCols = 32;        // bf16 columns per staging panel (64 B rows)
constexpr int kPanelBytes = 32 * kPanelCols * 2;

enum Kind : int { kKindNT = 0, kKindContiguous = 1, kKindMasked = 2 };

template <int BN>
struct Cfg {
    static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
    static constexpr int kStages = (BN == 256) ? 4 : 6;
    static constexpr int kAccBufs = kTmemCols / BN;
    static constexpr int kABytes = kBM * kBK;           // e4m3
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kColsPerThread = BN / 2;
    static constexpr int kStagingBytes = kNumEpiWarps * 2 * kPanelBytes;
    static constexpr int kBarrierBytes = (2 * kStages + 2 * kAccBufs + 1) * 8;
    static constexpr int kSmemBytes =
        kStages * kStageBytes + kStagingBytes + kBarrierBytes + 64 + 1024 /* alignment slack */;
};

struct Work {
    int g, m_blk, n_blk, kb0, kb1, tile;
    int a_row0;        // first row of the tile in A's (and D's) 2-D view
    int valid_rows;    // rows of the tile that belong in D
};

struct Ring {
    uint32_t i = 0, ph = 0;
    template <int N>
    __device__ __forceinline__ void next()
    {
        if (++i == N) {
            i = 0;
            ph ^= 1u;
        }
    }
};

__device__ __forceinline__ void raster(int t, int mb, int nbk, int group_m, int &m, int &n)
{
    const int per_band = group_m * nbk;
    const int band = t / per_band;
    const int first_m = band * group_m;
    const int hgt = min(group_m, mb - first_m);
    const int r = t - band * per_band;
    m = first_m + r % hgt;
    n = r / hgt;
}

// The tile sequence of one CTA.  Every role of the CTA runs its own copy and
// sees the same sequence.
template <int BN, int KIND, bool SPLIT>
struct Scheduler {
    const Params &p;
    int next_tile;
    long long u, u_end;
    int walk_g = 0, walk_base = 0, walk_tiles = -1, walk_count = 0;
    bool report;

    __device__ Scheduler(const Params &pp, bool report_bad_groups) : p(pp), report(report_bad_groups)
    {
        next_tile = blockIdx.x;
        if constexpr (SPLIT) {
            u = unit_begin(blockIdx.x);
            u_end = unit_begin(blockIdx.x + 1);
        }
    }

    __device__ __forceinline__ long long unit_begin(int c) const
    {
        return (long long)c * p.units / (long long)gridDim.x;
    }

    __device__ __forceinline__ int clamp_count(int g) const
    {
        const int c = __ldg(p.layout + g);
        return min(max(c, 0), p.rows);
    }

    __device__ bool next(Work &w)
    {
        if constexpr (SPLIT) {
            if (u >= u_end)
                return false;
            const int t = (int)(u / p.kb);
            const int k0 = (int)(u - (long long)t * p.kb);
            const long long left = u_end - u;
            const int k1 = (int)min((long long)p.kb, (long long)k0 + left);
            u += k1 - k0;
            raster(t, p.num_m_blocks, p.num_n_blocks, p.group_m, w.m_blk, w.n_blk);
            w.g = 0;
            w.tile = t;
            w.kb0 = k0;
            w.kb1 = k1;
            w.a_row0 = w.m_blk * kBM;
            w.valid_rows = min(kBM, p.rows - w.a_row0);
            return true;
        } else if constexpr (KIND == kKindNT) {
            if (next_tile >= p.num_tiles)
                return false;
            const int t = next_tile;
            next_tile += gridDim.x;
            raster(t, p.num_m_blocks, p.num_n_blocks, p.group_m, w.m_blk, w.n_blk);
            w.g = 0;
            w.tile = t;
            w.kb0 = 0;
            w.kb1 = p.kb;
            w.a_row0 = w.m_blk * kBM;
            w.valid_rows = min(kBM, p.rows - w.a_row0);
            return true;
        } else if constexpr (KIND == kKindContiguous) {
            while (next_tile < p.num_tiles) {
                const int t = next_tile;
                next_tile += gridDim.x;
                raster(t, p.num_m_blocks, p.num_n_blocks, p.group_m, w.m_blk, w.n_blk);
                const int g = __ldg(p.layout + (size_t)w.m_blk * kBM);
                if (g < 0 || g >= p.G) {
                    if (g != -1 && report)
                        atomicOr(p.error_word, kErrBadGroupBit);
                    continue;
                }
                w.g = g;
                w.tile = t;
                w.kb0 = 0;
                w.kb1 = p.kb;
                w.a_row0 = w.m_blk * kBM;
                w.valid_rows = kBM;
                return true;
            }
            return false;
        } else {  // masked
            const int t = next_tile;
            for (;;) {
                if (walk_g >= p.G)
                    return false;
                if (walk_tiles < 0) {
                    walk_count = clamp_count(walk_g);
                    walk_tiles = ((walk_count + kBM - 1) / kBM) * p.num_n_blocks;
                }
                if (t < walk_base + walk_tiles)
                    break;
                walk_base += walk_tiles;
                walk_tiles = -1;
                ++walk_g;
            }
            next_tile += gridDim.x;
            const int mb = (walk_count + kBM - 1) / kBM;
            raster(t - walk_base, mb, p.num_n_blocks, p.group_m, w.m_blk, w.n_blk);
            w.g = walk_g;
            w.tile = t;
            w.kb0 = 0;
            w.kb1 = p.kb;
            w.a_row0 = walk_g * p.rows + w.m_blk * kBM;
            w.valid_rows = min(kBM, walk_count - w.m_blk * kBM);
            return true;
        }
    }
};

// Owner CTA of split unit v when U units are shared by P CTAs in equal
// contiguous ranges [floor(c*U/P), floor((c+1)*U/P)).
__device__ __forceinline__ int unit_owner(long long v, long long U, int P)
{
    return (int)(((v + 1) * (long long)P - 1) / U);
}

// ----------------------------------------------------------------------------
// Epilogue helpers

// Writes 32 columns (one staging panel) of this warp's 32 rows to D.
// acc32 holds this thread's row, columns x .. x+31 of the output.
__device__ __forceinline__ void store_panel(const float *acc32, uint8_t *panel, const CUtensorMap *tmap_d,
                                            const Params &p, int x, int y_row0, int rows_ok, int lane,
                                            bool tma_ok)
{
    // 16-byte chunk c of row `lane` sits at chunk position c ^ ((lane >> 1) & 3)
    // of its 64-byte row (the 64-byte swizzle the D tensor map uses).
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(acc32[2 * i], acc32[2 * i + 1]);
    if (tma_ok && rows_ok == 32) {
        if (lane == 0)
            bulk_wait_group_read<1>();
        __syncwarp();
        const uint32_t base = smem_u32(panel) + lane * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            st_shared_v4(base + ((c ^ ((lane >> 1) & 3)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                         w[4 * c + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmap_d, panel, x, y_row0);
            bulk_commit_group();
        }
    } else if (lane < rows_ok) {
        // predicated row stores: only rows that belong in D are written
        uint4 *dst = reinterpret_cast<uint4 *>(p.d + (size_t)(y_row0 + lane) * p.N + x);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (x + 8 * c < p.N)
                dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

// ----------------------------------------------------------------------------
// The kernel

template <int BN, int KIND, bool SPLIT>
__global__ void __launch_bounds__(kNumThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const Params p)
{
#if defined(__CUDA_ARCH__)
    using C = Cfg<BN>;
    constexpr int S = C::kStages;
    constexpr int NACC = C::kAccBufs;
    constexpr int COLS = C::kColsPerThread;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + S * C::kABytes;
    uint8_t *sm_stage_d = sm_b + S * C::kBBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm_stage_d + C::kStagingBytes);
    uint64_t *full = bar;
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + NACC;
    uint64_t *drain = tempty + NACC;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kNumEpiWarps);
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

    const WaitCtl ctl{abort_flag, p.error_word, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            Scheduler<BN, KIND, SPLIT> sched(p, false);
            Work w;
            Ring ring;
            uint32_t issued = 0, issued_parity = 0;
            bool ok = true;
            while (ok && sched.next(w)) {
                const int b_row0 = w.g * p.N + w.n_blk * BN;
                for (int k = w.kb0; k < w.kb1; ++k) {
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
            // every fill this thread started has landed before the CTA exits
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s))
                    mbar_wait_drain(&full[s], (issued_parity >> s) & 1u, p.timeout_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            Scheduler<BN, KIND, SPLIT> sched(p, false);
            Work w;
            Ring ring, acc;
            constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
            bool ok = true;
            while (ok && sched.next(w)) {
                for (int k = w.kb0; k < w.kb1; ++k) {
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
                        mma_f8f6f4(d_tmem, a0 + 2 * kk, b0 + 2 * kk, idesc, kk > 0 ? 1u : 0u);
                    mma_commit(&empty[ring.i]);
                    mma_commit(&tfull[acc.i]);
                    ring.template next<S>();
                    acc.template next<NACC>();
                }
            }
            // all MMAs issued above complete before tensor memory is freed
            mma_commit(drain);
            mbar_wait_drain(drain, 0, p.timeout_ns);
        }
    } else {
        // ------------------------------------------------ epilogue warps
        const int ew = warp - kEpiWarp0;     // 0..7
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int h = ew >> 2;               // column half of the tile
        const int row_in_tile = 32 * q + lane;
        uint8_t *panels = sm_stage_d + ew * 2 * kPanelBytes;
        uint32_t panel_ctr = 0;

        if (KIND == kKindMasked && blockIdx.x == 0 && ew == 0) {
            for (int g = lane; g < p.G; g += 32) {
                const int c = __ldg(p.layout + g);
                if (c < 0 || c > p.rows)
                    atomicOr(p.error_word, kErrBadGroupBit);
            }
        }

        Scheduler<BN, KIND, SPLIT> sched(p, ew == 0 && lane == 0);
        Work w;
        Ring acc_ring;
        bool ok = true;
        while (ok && sched.next(w)) {
            float acc[COLS];
#pragma unroll
            for (int i = 0; i < COLS; ++i)
                acc[i] = 0.f;

            // scale sources for this thread's row and this warp's 128-column block
            const int m_local = w.m_blk * kBM + row_in_tile;              // row inside the group
            const bool row_ok = m_local < p.rows;
            const float *sfa_row =
                p.sfa + (KIND == kKindMasked ? (size_t)w.g * p.kb * p.sfa_ld : 0) + m_local;
            const int nbc = (w.n_blk * BN + h * COLS) / 128;
            const bool col_ok = nbc < p.nb;
            const float *sfb_row = p.sfb + ((size_t)w.g * p.nb + nbc) * p.kb;

            float sa_cur = row_ok ? ld_nc_f32(sfa_row + (size_t)w.kb0 * p.sfa_ld) : 0.f;
            int chunk = w.kb0 & ~31;
            float sb_cur = (col_ok && chunk + lane < p.kb) ? ld_nc_f32(sfb_row + chunk + lane) : 0.f;
            float sb_nxt = 0.f;

            for (int k = w.kb0; k < w.kb1; ++k) {
                // prefetch the next K block's A scale and, at a 32-block
                // boundary, the next chunk of B scales
                const float sa_nxt =
                    (row_ok && k + 1 < w.kb1) ? ld_nc_f32(sfa_row + (size_t)(k + 1) * p.sfa_ld) : 0.f;
                if ((k & 31) == 0 && k != w.kb0)
                    sb_cur = sb_nxt;
                if ((k & 31) == 0 || k == w.kb0) {
                    const int nc = (k & ~31) + 32;
                    sb_nxt = (col_ok && nc + lane < p.kb && nc < w.kb1) ? ld_nc_f32(sfb_row + nc + lane) : 0.f;
                }
                const float sb = __shfl_sync(0xffffffffu, sb_cur, k & 31);
                const float s = sa_cur * sb;
                sa_cur = sa_nxt;

                int got = 1;
                if (lane == 0)
                    got = mbar_wait(&tfull[acc_ring.i], acc_ring.ph, ctl) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();

                const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + acc_ring.i * BN + h * COLS;
                uint32_t v0[16], v1[16];
                tmem_ld_32x32b_x16(taddr, v0);
                tmem_wait_ld(v0);
#pragma unroll
                for (int c = 0; c < COLS / 16; ++c) {
                    uint32_t(&cur)[16] = (c & 1) ? v1 : v0;
                    uint32_t(&nxt)[16] = (c & 1) ? v0 : v1;
                    if (c + 1 < COLS / 16)
                        tmem_ld_32x32b_x16(taddr + 16 * (c + 1), nxt);
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        float2 a2 = make_float2(acc[16 * c + i], acc[16 * c + i + 1]);
                        const float2 p2 = make_float2(__uint_as_float(cur[i]), __uint_as_float(cur[i + 1]));
                        a2 = __ffma2_rn(make_float2(s, s), p2, a2);
                        acc[16 * c + i] = a2.x;
                        acc[16 * c + i + 1] = a2.y;
                    }
                    if (c + 1 < COLS / 16) {
                        tmem_wait_ld(nxt);
                        if (c + 2 == COLS / 16) {
                            // every column of this buffer is in registers now
                            tc_fence_before_sync();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(&tempty[acc_ring.i]);
                        }
                    }
                }
                acc_ring.template next<NACC>();
            }
            if (!ok)
                break;

            if constexpr (SPLIT) {
                if (!(w.kb0 == 0 && w.kb1 == p.kb)) {
                    // split tile: publish this CTA's partial for this warp's
                    // 32 x COLS region, take a ticket; the last contributor
                    // sums all partials in CTA order and stores the tile.
                    const int t = w.tile;
                    const int P = gridDim.x;
                    const int c_lo = unit_owner((long long)t * p.kb, p.units, P);
                    const int c_hi = unit_owner((long long)(t + 1) * p.kb - 1, p.units, P);
                    auto slot_of = [&](int c) {
                        const long long first_tile = ((long long)c * p.units / P) / p.kb;
                        return 2 * c + ((long long)t == first_tile ? 0 : 1);
                    };
                    constexpr int F4 = COLS / 4;
                    auto region = [&](int c) {
                        return reinterpret_cast<float4 *>(p.partials) +
                               ((size_t)slot_of(c) * kNumEpiWarps + ew) * F4 * 32;
                    };
                    float4 *mine = region(blockIdx.x);
#pragma unroll
                    for (int j = 0; j < F4; ++j)
                        st_cg_f4(mine + j * 32 + lane,
                                 make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
                    __threadfence();
                    __syncwarp();
                    int ticket = 0;
                    int *ctr = p.counters + (size_t)t * kNumEpiWarps + ew;
                    if (lane == 0) {
                        __threadfence();
                        ticket = atomicAdd(ctr, 1);
                    }
                    ticket = __shfl_sync(0xffffffffu, ticket, 0);
                    if (ticket != c_hi - c_lo)
                        continue;       // not the last contributor
                    __threadfence();
                    // every partial, this CTA's included, is summed back from
                    // L2 in CTA order, so the result does not depend on which
                    // contributor arrived last
#pragma unroll
                    for (int i = 0; i < COLS; ++i)
                        acc[i] = 0.f;
                    for (int c = c_lo; c <= c_hi; ++c) {
                        const float4 *src = region(c);
#pragma unroll
                        for (int j = 0; j < F4; ++j) {
                            const float4 v = ld_cg_f4(src + j * 32 + lane);
                            acc[4 * j] += v.x;
                            acc[4 * j + 1] += v.y;
                            acc[4 * j + 2] += v.z;
                            acc[4 * j + 3] += v.w;
                        }
                    }
                    if (lane == 0)
                        *ctr = 0;       // leave the workspace zeroed for the next call
                }
            }

            // ---- bf16 store of this warp's 32 rows x COLS columns
            const int rows_ok = min(max(w.valid_rows - 32 * q, 0), 32);
            const int y_row0 = w.a_row0 + 32 * q;
#pragma unroll
            for (int pi = 0; pi < COLS / kPanelCols; ++pi) {
                const int x = w.n_blk * BN + h * COLS + pi * kPanelCols;
                if (x >= p.N || rows_ok == 0)
                    continue;
                uint8_t *panel = panels + (panel_ctr & 1u) * kPanelBytes;
                // TMA stores may be used unless masked rows straddle this slab
                store_panel(acc + pi * kPanelCols, panel, &tmap_d, p, x, y_row0, rows_ok, lane, true);
                if (rows_ok == 32)
                    ++panel_ctr;
            }
        }
        if (lane == 0)
            bulk_wait_group<0>();
        __syncwarp();
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
