// gemm_kernel.cuh -- persistent, warp-specialised FP8 (E4M3) GEMM with
// fine-grained scaling for sm_103a.
//
// What is computed (DeepGEMM fp8_gemm.cuh, fp8_gemm_kernel): every 128-wide K
// block's partial product A_blk * B_blk^T is formed on its own in fp32 and
// promoted into an fp32 accumulator with scale_a(row, k) * scale_b(n/128, k);
// the accumulator is rounded to bf16 at the end.
//
// How, on Blackwell (design ours; the DeepGEMM page's Hopper kernel and the
// "TCGen05 Copy Instruction" tutorial's warp-specialised matmul are prior art).
// Three warpgroups of four warps:
//   warp 0      TMA producer: 128x128 A and BNx128 B e4m3 tiles, 128-byte
//               swizzled, into an S-stage shared-memory ring (with an even S,
//               two K blocks per copy: one 3-D box fills two stages), and the
//               scales of kScaleChunk K blocks at a time (128 A scales per K
//               block, the B scales of the tile's 128-column blocks) into a
//               scale ring.  mbarrier transaction counts signal completion.
//   warp 1      MMA issuer: one thread issues 4 x tcgen05.mma kind::f8f6f4
//               (128 x BN x 32) per K block into a FRESH tensor-memory buffer
//               (the first MMA overwrites) and commits once per K block.  That
//               one commit both frees the operand stage and tells the
//               epilogue the buffer is complete: each commit drains the tensor
//               pipe, so there is only one.  512 TMEM columns hold 512/BN
//               buffers, so the MMA of block k+1 runs while k is promoted.
//   warp 2      with an fp32 addend and whole-tile staging (accumulate,
//               256-column tiles, unsplit): the addend/store warp.  One thread
//               TMA-loads each tile's C into the staging area, half a tile at a
//               time, and TMA-stores the bf16 tile the epilogue leaves there,
//               so the epilogue warps neither copy C nor wait for stores.
//               Otherwise (and warp 3 always) idle: it only gives its
//               registers away.
//   warps 4-11  epilogue: tcgen05.ld of the K block's partial, promotion
//               acc += (sa*sb) * P in fp32 registers (one row per thread,
//               BN/2 columns per warp), and at the end of a tile bf16
//               conversion into swizzled staging panels and TMA stores (or
//               predicated stores where masked rows straddle).  Every lane
//               waits on the MMA completion itself and every lane arrives on
//               the buffer's release (see warp_wait in ptx.cuh).
// Registers: the control warpgroup drops to kRegsCtl with setmaxnreg and the
// epilogue warpgroups rise to kRegsEpi (the accumulator is BN/2 registers).
//   scheduler   persistent: CTA c takes tiles c, c+P, ... in a banded
//               rasterisation (m fastest inside a band of m-blocks); grouped
//               layouts map tiles to groups.  A split-K ("stream-K") variant
//               gives each CTA an equal share of the (tile, K-block) units and
//               lets the highest contributor of each tile reduce the fp32
//               partials in a fixed order (deterministic).
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

#ifndef FP8G_STAGES_256
#define FP8G_STAGES_256 3
#endif
#ifndef FP8G_FULL_TILE_STAGING
#define FP8G_FULL_TILE_STAGING 1
#endif
#ifndef FP8G_PANEL_COLS_FULL
#define FP8G_PANEL_COLS_FULL 64
#endif

namespace fp8g {

constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kNumThreads = 384;      // 3 warpgroups of 4 warps
constexpr int kEpiWarp0 = 4;          // warpgroups 1 and 2 are the epilogue
constexpr int kNumEpiWarps = 8;
constexpr int kTmemCols = 512;
// Registers per thread after reallocation: warpgroup 0 (producer, MMA, two
// idle warps) gives registers to the epilogue warpgroups.  The launch
// allocation is 384 x 168 = 64512; 128 x 40 + 256 x 232 = 64512.
constexpr int kRegsCtl = 40;
constexpr int kRegsEpi = 232;
constexpr int kLaunchRegs = 168;
static_assert(128 * kRegsCtl + 256 * kRegsEpi <= kNumThreads * kLaunchRegs,
              "register reallocation exceeds the launch allocation");

template <int BN>
struct Cfg {
    static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
    // With whole-tile staging the epilogue drops a whole bf16 tile into
    // shared memory and moves on; TMA stores drain it during the next tile.
    static constexpr bool kFullTileStaging = BN == 256 && FP8G_FULL_TILE_STAGING != 0;
    static constexpr int kStages = (BN == 256) ? FP8G_STAGES_256 : 6;   // A/B operand ring
    static constexpr int kAccBufs = kTmemCols / BN;                     // TMEM partial buffers
    static constexpr int kScaleSlots = 4;                               // scale chunk ring
    static constexpr int kABytes = kBM * kBK;                           // e4m3
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSfbRows = BN / 128;                           // 128-column blocks per tile
    // scale slot (one chunk of kScaleChunk K blocks): the A scales as
    // [kScaleChunk][128 rows], then per column block the kScaleChunk + 4 B
    // scales from the 16-byte aligned group that holds the chunk's first one.
    // Every TMA destination in shared memory starts on a 128-byte boundary.
    static constexpr int kSlotSfaBytes = kScaleChunk * kBM * 4;
    static constexpr int kSlotSfbStride = 128;
    static constexpr int kSlotBytes = kSlotSfaBytes + kSlotSfbStride * kSfbRows;
    static constexpr int kSlotTxBytes = kSlotSfaBytes + (kScaleChunk + 4) * 4 * kSfbRows;
    static_assert((kScaleChunk + 4) * 4 <= kSlotSfbStride && (kScaleChunk + 4) % 4 == 0, "B scale box");
    static constexpr int kColsPerThread = BN / 2;
    // Pair loads: one 3-D copy per operand fills two consecutive stages with
    // two consecutive K blocks of the same tile (fewer, larger copies for the
    // SM's TMA unit).  Pairs start at even stages only, hence an even stage
    // count.
    static constexpr bool kPairLoads = kStages % 2 == 0;
    // output panels: 32 rows x kPanelCols bf16, TMA-stored with the swizzle
    // of their row width
    static constexpr int kPanelCols = kFullTileStaging ? FP8G_PANEL_COLS_FULL : 16;
    static constexpr int kPanelBytes = 32 * kPanelCols * 2;
    static constexpr int kPanelsPerWarp = kFullTileStaging ? (BN / 2) / kPanelCols : 2;
    static constexpr int kStagingBytes = kNumEpiWarps * kPanelsPerWarp * kPanelBytes;
    static constexpr int kBarriers = 2 * kStages + kAccBufs + 2 * kScaleSlots + 1 + 3;
    static constexpr int kSmemBytes = kStages * kStageBytes + kStagingBytes + kScaleSlots * kSlotBytes +
                                      kBarriers * 8 + 16 + 1024 /* alignment slack */;
    static_assert(kSlotTxBytes <= kSlotBytes, "scale slot");
    static_assert(kSlotBytes % 128 == 0 && kSlotSfaBytes % 128 == 0 && kStagingBytes % 1024 == 0 &&
                      kABytes % 1024 == 0 && kBBytes % 1024 == 0 && kPanelBytes % 1024 == 0,
                  "TMA destinations and sources must stay 128-byte (swizzled: 1024-byte) aligned");
    static_assert(kPanelCols == 16 || kPanelCols == 32 || kPanelCols == 64, "panel width");
    static_assert(kStages >= kAccBufs, "the epilogue's wait on a stage's MMA completion must not alias");
    static_assert(kSmemBytes <= 232448, "shared memory");
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
//
// SHARE (clusters of two CTAs sharing the A tile over DSMEM): the tile index
// runs over (m-block, pair of n-blocks) and the two CTAs of a cluster take
// the same one, rank r computing n-block 2j + r; a rank whose n-block lies
// past N computes on whatever B its view holds and stores nothing.
template <int BN, int KIND, bool SPLIT, bool SHARE = false>
struct Scheduler {
    const Params &p;
    int next_tile;
    int u, u_end;
    int walk_g = 0, walk_base = 0, walk_tiles = -1, walk_count = 0;
    bool report;

    __device__ Scheduler(const Params &pp, bool report_bad_groups) : p(pp), report(report_bad_groups)
    {
        next_tile = SHARE ? (int)blockIdx.x / 2 : (int)blockIdx.x;
        if constexpr (SPLIT) {
            u = unit_begin(blockIdx.x);
            u_end = unit_begin(blockIdx.x + 1);
        }
    }

    __device__ __forceinline__ int stride() const { return SHARE ? (int)gridDim.x / 2 : (int)gridDim.x; }
    __device__ __forceinline__ int n_cols() const { return SHARE ? (p.num_n_blocks + 1) / 2 : p.num_n_blocks; }
    // the CTA's n-block of raster column c, and whether it lies inside N
    __device__ __forceinline__ int n_of(int c) const { return SHARE ? 2 * c + (int)cluster_ctarank() : c; }

    // the host keeps units * CTAs below 2^31
    __device__ __forceinline__ int unit_begin(int c) const
    {
        return (int)((unsigned)c * (unsigned)p.units / gridDim.x);
    }

    __device__ __forceinline__ int clamp_count(int g) const
    {
        const int c = __ldg(p.layout + g);
        return min(max(c, 0), p.rows);
    }

    __device__ bool next(Work &w)
    {
        if constexpr (SPLIT) {
            // the CTA's units [u, u_end) are taken tile by tile from the END
            // of the range: a tile's highest contributor then works on its
            // share of the tile last, like every other contributor, and can
            // be the one that reduces the tile
            if (u >= u_end)
                return false;
            const int t = (u_end - 1) / p.kb;
            const int k1 = u_end - t * p.kb;
            const int k0 = max(0, u - t * p.kb);
            u_end = t * p.kb + k0;
            raster(t, p.num_m_blocks, p.num_n_blocks, p.group_m, w.m_blk, w.n_blk);
            w.g = 0;
            w.tile = t;
            w.kb0 = k0;
            w.kb1 = k1;
            w.a_row0 = w.m_blk * kBM;
            w.valid_rows = min(kBM, p.rows - w.a_row0);
            return true;
        } else if constexpr (KIND == kKindNT || KIND == kKindNTAcc) {
            if (next_tile >= p.num_tiles)
                return false;
            const int t = next_tile;
            next_tile += stride();
            raster(t, p.num_m_blocks, n_cols(), p.group_m, w.m_blk, w.n_blk);
            w.n_blk = n_of(w.n_blk);
            w.g = 0;
            w.tile = t;
            w.kb0 = 0;
            w.kb1 = p.kb;
            w.a_row0 = w.m_blk * kBM;
            w.valid_rows = w.n_blk < p.num_n_blocks ? min(kBM, p.rows - w.a_row0) : 0;
            return true;
        } else if constexpr (KIND == kKindContiguous) {
            while (next_tile < p.num_tiles) {
                const int t = next_tile;
                next_tile += stride();
                raster(t, p.num_m_blocks, n_cols(), p.group_m, w.m_blk, w.n_blk);
                w.n_blk = n_of(w.n_blk);
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
                w.valid_rows = w.n_blk < p.num_n_blocks ? kBM : 0;
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
                    walk_tiles = ((walk_count + kBM - 1) / kBM) * n_cols();
                }
                if (t < walk_base + walk_tiles)
                    break;
                walk_base += walk_tiles;
                walk_tiles = -1;
                ++walk_g;
            }
            next_tile += stride();
            const int mb = (walk_count + kBM - 1) / kBM;
            raster(t - walk_base, mb, n_cols(), p.group_m, w.m_blk, w.n_blk);
            w.n_blk = n_of(w.n_blk);
            w.g = walk_g;
            w.tile = t;
            w.kb0 = 0;
            w.kb1 = p.kb;
            w.a_row0 = walk_g * p.rows + w.m_blk * kBM;
            w.valid_rows = w.n_blk < p.num_n_blocks ? min(kBM, walk_count - w.m_blk * kBM) : 0;
            return true;
        }
    }
};

// Owner CTA of split unit v when U units are shared by P CTAs in equal
// contiguous ranges [floor(c*U/P), floor((c+1)*U/P)).
__device__ __forceinline__ int unit_owner(int v, int U, int P)
{
    return (int)(((unsigned)(v + 1) * (unsigned)P - 1u) / (unsigned)U);
}

// ----------------------------------------------------------------------------
// Epilogue helpers

// Writes PC columns (one staging panel) of this warp's 32 rows to D.
// accp holds this thread's row, columns x .. x+PC-1 of the output.
template <int PC, bool kWaitBuffer, bool kIssue = true>
__device__ __forceinline__ void store_panel(const float *accp, uint8_t *panel, const CUtensorMap *tmap_d,
                                            const Params &p, int x, int y_row0, int rows_ok, int lane)
{
    constexpr int NW = PC / 2;          // bf16x2 words per row
    constexpr int NC = PC / 8;          // 16-byte chunks per row
    uint32_t w[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i)
        w[i] = pack_bf16x2(accp[2 * i], accp[2 * i + 1]);
    if (rows_ok == 32) {
        // all 32 rows belong in D: stage the panel and let TMA store it.
        // TMA's swizzle XORs the 16-byte chunk index with address bits 7..9:
        // chunk c of row r sits at c ^ ((r * row_bytes) >> 7 & (NC - 1)).
        if (kWaitBuffer) {
            // two alternating panel buffers: the one before last must be read
            if (lane == 0)
                bulk_wait_group_read<1>();
            __syncwarp();
        }
        const uint32_t base = smem_u32(panel) + lane * (PC * 2);
        const int sw = ((lane * PC * 2) >> 7) & (NC - 1);
#pragma unroll
        for (int c = 0; c < NC; ++c)
            st_shared_v4(base + ((c ^ sw) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (kIssue && lane == 0) {      // (otherwise the addend/store warp issues it)
            tma_store_2d(tmap_d, panel, x, y_row0);
            bulk_commit_group();
        }
    } else if (lane < rows_ok) {
        // predicated row stores: only rows that belong in D are written
        uint4 *dst = reinterpret_cast<uint4 *>(p.d + (size_t)(y_row0 + lane) * p.N + x);
#pragma unroll
        for (int c = 0; c < NC; ++c)
            if (x + 8 * c < p.N)
                dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

// ----------------------------------------------------------------------------
// Epilogue: per-K-block promotion

template <int N>
__device__ __forceinline__ void fma_cols(float *acc, const uint32_t (&v)[N], float s)
{
    const float2 s2 = make_float2(s, s);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        float2 a2 = make_float2(acc[i], acc[i + 1]);
        a2 = __ffma2_rn(s2, make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), a2);
        acc[i] = a2.x;
        acc[i + 1] = a2.y;
    }
}

__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld_32x32b_x16(taddr, r); }
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld_32x32b_x32(taddr, r); }
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[64]) { tmem_ld_32x32b_x64(taddr, r); }

// Hands a tensor-memory buffer back: every lane arrives (the barrier counts
// 32 per warp), as every lane waited (all-lane releases measured 1-2.5%
// faster than __syncwarp and one lane's arrival on the fp32-scale shapes).
__device__ __forceinline__ void release_tmem(uint64_t *bar, int lane)
{
    (void)lane;
    tc_fence_before_sync();
    mbar_arrive(bar);
}

// acc[0 .. COLS) += s * (this thread's row of the K block's partial in TMEM,
// columns taddr.col .. +COLS), LD columns per tcgen05.ld, with s = *pa * *pb
// (the K block's A and B scales in shared memory), read while the first TMEM
// load is in flight.  The buffer is handed back to the MMA issuer as soon as
// its last load landed.
template <int COLS, int LD>
__device__ __forceinline__ void promote_block(float (&acc)[COLS], uint32_t taddr, const float *pa, const float *pb,
                                              uint64_t *tempty_bar, int lane)
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
        if (c + 1 == NCH)
            release_tmem(tempty_bar, lane);
        fma_cols<LD>(acc + c * LD, v, s);
    }
}

// The accumulator's start with an addend (TCGen05 Copy Instruction, the
// matmul-accumulate example: C is placed in the accumulator before the first
// product is added).  Only the CTA that stores the tile -- the only one, or a
// split tile's highest contributor, which holds the last K block -- starts
// from C; every other contributor starts from zero, so C enters each sum once.
// The loads are issued before the first MMA completion is awaited.
template <int BN, int COLS>
__device__ __forceinline__ void init_from_c(float (&acc)[COLS], const Params &p, const Work &w, int q, int h,
                                            int lane)
{
    const int r = 32 * q + lane;          // row within the tile
    const int col0 = w.n_blk * BN + h * COLS;
    const bool live = w.kb1 == p.kb && r < w.valid_rows;
    // rows are 16-byte aligned (N % 16 == 0, C 16-byte aligned) and col0 is a
    // multiple of 64, so every float4 below is aligned
    const float4 *src = reinterpret_cast<const float4 *>(p.c + (size_t)(w.a_row0 + (live ? r : 0)) * p.N + col0);
#pragma unroll
    for (int j = 0; j < COLS / 4; ++j) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live && col0 + 4 * j < p.N)
            v = __ldg(src + j);
        acc[4 * j] = v.x;
        acc[4 * j + 1] = v.y;
        acc[4 * j + 2] = v.z;
        acc[4 * j + 3] = v.w;
    }
}

// With whole-tile staging the addend goes through shared memory instead:
// each warp's 32 rows x COLS columns of C pass through its staging area --
// idle between the previous tile's stores and this tile's -- one half (64
// columns) at a time, copied by coalesced cp.async (each instruction covers
// two rows of 256 bytes) and read back one row per thread.  Half 0 is copied
// three K blocks into the tile; three K blocks before its end half 0 is added
// and half 1 copied; half 1 is added after the last K block (shorter ranges
// do both halves after the loop).  The 16-byte chunk c of row r sits at
// c ^ (r & 15), so the copies and the row-wise reads both spread over every
// bank.  (Prefetching C into L2 at the start of the tile, an evict-first L2
// policy on the copies, other copy positions and doing both halves after the
// loop were each measured slower or no faster.)
constexpr int kAddendHalfCols = 64;     // one half: 32 rows x 256 bytes

template <int BN, int COLS>
__device__ __forceinline__ void copy_c_half(uint8_t *stage, const Params &p, const Work &w, int q, int h, int lane,
                                             int rows_ok, int rd)
{
    const uint32_t s0 = smem_u32(stage);
    const int c16 = lane & 15;          // the 16-byte chunk this lane copies
    const int x = w.n_blk * BN + h * COLS + rd * kAddendHalfCols + 4 * c16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = 2 * i + (lane >> 4);
        const bool live = r < rows_ok && x < p.N;
        const float *src = live ? p.c + (size_t)(w.a_row0 + 32 * q + r) * p.N + x : p.c;
        cp_async_16(s0 + r * 256 + ((c16 ^ (r & 15)) << 4), src, live ? 16u : 0u);
    }
    cp_async_commit();
}

template <int COLS>
__device__ __forceinline__ void add_c_half(float (&acc)[COLS], const uint8_t *stage, int lane, int rd)
{
    cp_async_wait_all();
    __syncwarp();
    // eight loads in flight before the first of their adds
    const uint32_t row = smem_u32(stage) + lane * 256;
#pragma unroll
    for (int c0 = 0; c0 < 16; c0 += 8) {
        float4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            v[c] = ld_shared_f4_nc(row + (((c0 + c) ^ (lane & 15)) << 4));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float *a = acc + rd * kAddendHalfCols + 4 * (c0 + c);
            a[0] += v[c].x;
            a[1] += v[c].y;
            a[2] += v[c].z;
            a[3] += v[c].w;
        }
    }
    __syncwarp();                       // read by every lane before the next half lands
}

// The same addition from the addend/store warp's TMA copy of a half: four
// slabs of 32 rows x 16 fp32 columns (64 bytes a row), 64-byte swizzled
// (16-byte chunk c of row r at c ^ ((r >> 1) & 3)), so each group of eight
// lanes reads all 32 banks.  The warp's bf16 rows later overwrite this area,
// and lane r's row lands on other lanes' C: the closing __syncwarp in the
// caller orders every lane's reads first.
template <int COLS>
__device__ __forceinline__ void add_c_box(float (&acc)[COLS], const uint8_t *stage, int lane, int rd)
{
    const uint32_t row = smem_u32(stage) + lane * 64;
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int b0 = 0; b0 < 4; b0 += 2) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = ld_shared_f4_nc(row + (b0 + (i >> 2)) * 2048 + (((i & 3) ^ sw) << 4));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float *a = acc + rd * kAddendHalfCols + 16 * (b0 + (i >> 2)) + 4 * (i & 3);
            a[0] += v[i].x;
            a[1] += v[i].y;
            a[2] += v[i].z;
            a[3] += v[i].w;
        }
    }
}

// ----------------------------------------------------------------------------
// The kernel

// SHARE: launched in clusters of two CTAs that compute neighbouring n-blocks
// of the same m-block (so the same A tiles; the TVM TIRx "copy_async ->
// dsmem" page's two-CTA shared-to-shared bulk copy, used as the one-GPU
// alternative to the multicast of the DeepGEMM page's tma_copy).  Rank 0
// loads each A tile from global memory; its warp 2 forwards it into rank 1's
// shared memory with one cp.async.bulk.shared::cluster, counted on rank 1's
// full barrier.  Each CTA loads its own B.  Both MMA issuers commit to the
// stage's empty barrier of both CTAs (count 2), so a stage is refilled only
// once both CTAs' MMAs -- and hence the forward, which rank 1's MMA waited
// for -- are done with it.
template <int BN, int KIND, bool SPLIT, bool SHARE = false>
__global__ void __launch_bounds__(kNumThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ CUtensorMap tmap_sfa,
                    const __grid_constant__ CUtensorMap tmap_sfb, const __grid_constant__ CUtensorMap tmap_a2,
                    const __grid_constant__ CUtensorMap tmap_b2, const __grid_constant__ CUtensorMap tmap_c,
                    const __grid_constant__ Params p)
{
#if defined(__CUDA_ARCH__)
    using C = Cfg<BN>;
    static_assert(!SHARE || (!SPLIT && !C::kPairLoads), "A sharing: unsplit schedules, one K block per copy");
    // the addend/store warp (warp 2): accumulate, whole-tile staging, unsplit
    constexpr bool kHelperC = KIND == kKindNTAcc && C::kFullTileStaging && !SPLIT;
    static_assert(!(kHelperC && SHARE), "warp 2 has one role");
    constexpr int S = C::kStages;
    constexpr int NACC = C::kAccBufs;
    constexpr int SR = C::kScaleSlots;
    constexpr int COLS = C::kColsPerThread;

    // shared memory: [A stages][B stages][D staging][scale slots][barriers][tmem addr, abort]
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + S * C::kABytes;
    uint8_t *sm_stage_d = sm_b + S * C::kBBytes;
    uint8_t *sm_scales = sm_stage_d + C::kStagingBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm_scales + SR * C::kSlotBytes);
    uint64_t *full = bar;              // S:  A/B tiles landed (TMA transactions)
    uint64_t *empty = full + S;        // S:  MMAs of the stage finished (one commit per K block)
    uint64_t *tempty = empty + S;      // NACC: epilogue finished reading a TMEM buffer
    uint64_t *sfull = tempty + NACC;   // SR: scale slot landed (TMA transactions)
    uint64_t *sempty = sfull + SR;     // SR: epilogue finished reading a scale slot
    uint64_t *drain = sempty + SR;
    uint64_t *c_full = drain + 1;      // a half tile of C landed in the staging area (TMA transactions)
    uint64_t *c_free = c_full + 1;     // every epilogue warp has added the first half
    uint64_t *d_ready = c_free + 1;    // every epilogue warp has left its bf16 rows in the staging area
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(d_ready + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t rank = SHARE ? cluster_ctarank() : 0u;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], SHARE ? 2 : 1);   // both CTAs' MMA commits when sharing
        }
        for (int i = 0; i < NACC; ++i)
            mbar_init(&tempty[i], kNumEpiWarps * 32);   // every lane of every epilogue warp
        for (int i = 0; i < SR; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], kNumEpiWarps * 32);   // every lane of every epilogue warp
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
        if (C::kPairLoads && p.kb >= 2) {
            prefetch_tensormap(&tmap_a2);
            prefetch_tensormap(&tmap_b2);
        }
        if (kHelperC)
            prefetch_tensormap(&tmap_c);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    if constexpr (SHARE)
        cluster_sync();     // the peer's barriers exist before anything reaches them
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Launched as a programmatic dependent of the previous kernel on the
    // stream, the set-up above (barriers, tensor memory, descriptor prefetch)
    // may overlap that kernel's tail; nothing in global memory is touched
    // before the previous grid has completed and its writes are visible.  The
    // next kernel may then be scheduled as SMs free up.
    grid_dependency_wait();

    const WaitCtl ctl{abort_flag, p.error_word, p.timeout_ns,
                      SHARE ? mapa_shared(smem_u32(const_cast<int *>(abort_flag)), rank ^ 1u) : 0u};

    // Each role sits inside the branch that sets its register budget, so the
    // epilogue is only reachable with the larger one.
    if (warp < kEpiWarp0) {
        regs_dealloc<kRegsCtl>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer
            Scheduler<BN, KIND, SPLIT, SHARE> sched(p, false);
            Work w;
            Ring ring, sring;
            uint32_t issued = 0, issued_parity = 0, sissued = 0, sissued_parity = 0;
            bool second = false;    // this K block's operands came with the previous block's
            bool ok = true;
            while (ok && sched.next(w)) {
                // the work unit lies inside the problem (the bounds-checking build)
                if (!bounds_ok(w.g >= 0 && w.g < p.G && w.kb0 >= 0 && w.kb0 < w.kb1 && w.kb1 <= p.kb &&
                                   w.a_row0 >= 0 && w.a_row0 < p.a_rows_total && w.n_blk >= 0 &&
                                   (w.valid_rows == 0 || (w.n_blk * BN < p.N && w.valid_rows <= kBM)),
                               ctl)) {
                    ok = false;
                    break;
                }
                const int b_row0 = w.g * p.N + w.n_blk * BN;
                const int sfa_y0 = (KIND == kKindMasked) ? w.g * p.kb : 0;
                const int sfb_x0 = (w.g * p.nb + (w.n_blk * BN) / 128) * p.kb;
                for (int k = w.kb0; k < w.kb1; ++k) {
                    if (!second) {
                        // a pair starts on an even stage and needs the next K
                        // block in the same work unit
                        const bool pair = C::kPairLoads && (ring.i & 1u) == 0 && k + 1 < w.kb1;
                        if (!mbar_wait(&empty[ring.i], ring.ph ^ 1u, ctl) ||
                            (pair && !mbar_wait(&empty[ring.i + 1], ring.ph ^ 1u, ctl))) {
                            ok = false;
                            break;
                        }
                        const uint32_t a_bytes = (uint32_t)p.a_box_rows * kBK;
                        if (pair) {
                            // both tiles signal the first stage's barrier; the
                            // second stage's barrier completes its phase with a
                            // plain arrival, so that every barrier keeps one
                            // phase per use of its stage (the MMA warp does not
                            // wait on it: it waited on the first one)
                            mbar_arrive_expect_tx(&full[ring.i], 2 * (a_bytes + C::kBBytes));
                            if (p.a_box_rows == kBM) {
                                tma_load_3d(sm_a + ring.i * C::kABytes, &tmap_a2, &full[ring.i], 0, w.a_row0, k);
                            } else {
                                // a short A box: one 2-D copy per stage (a 3-D box would pack
                                // the two K blocks' rows together)
                                tma_load_2d(sm_a + ring.i * C::kABytes, &tmap_a, &full[ring.i], k * kBK, w.a_row0);
                                tma_load_2d(sm_a + (ring.i + 1) * C::kABytes, &tmap_a, &full[ring.i], (k + 1) * kBK,
                                            w.a_row0);
                            }
                            tma_load_3d(sm_b + ring.i * C::kBBytes, &tmap_b2, &full[ring.i], 0, b_row0, k);
                            mbar_arrive(&full[ring.i + 1]);
                            issued |= 2u << ring.i;
                            issued_parity = (issued_parity & ~(2u << ring.i)) | (ring.ph << (ring.i + 1));
                        } else {
                            // when sharing, rank 1's A arrives from rank 0 (same byte count)
                            mbar_arrive_expect_tx(&full[ring.i], a_bytes + C::kBBytes);
                            if (!SHARE || rank == 0)
                                tma_load_2d(sm_a + ring.i * C::kABytes, &tmap_a, &full[ring.i], k * kBK, w.a_row0);
                            tma_load_2d(sm_b + ring.i * C::kBBytes, &tmap_b, &full[ring.i], k * kBK, b_row0);
                        }
                        issued |= 1u << ring.i;
                        issued_parity = (issued_parity & ~(1u << ring.i)) | (ring.ph << ring.i);
                        second = pair;
                    } else {
                        second = false;
                    }
                    if ((k - w.kb0) % kScaleChunk == 0) {
                        // the scales of the chunk of K blocks starting here
                        if (!mbar_wait(&sempty[sring.i], sring.ph ^ 1u, ctl)) {
                            ok = false;
                            break;
                        }
                        uint8_t *slot = sm_scales + sring.i * C::kSlotBytes;
                        mbar_arrive_expect_tx(&sfull[sring.i], C::kSlotTxBytes);
                        tma_load_2d(slot, &tmap_sfa, &sfull[sring.i], w.m_blk * kBM, sfa_y0 + k);
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
            // the next kernel on the stream is let in once this CTA's last
            // copy is issued (at the start, its CTAs took the SMs this grid
            // leaves idle; masked 16 x 256 x 7168 x 2048: 56.8 -> 55.8 us)
            grid_launch_dependents();
            // every fill this thread started has landed before the CTA exits
            for (int i = 0; i < S; ++i)
                if (issued & (1u << i))
                    mbar_wait_drain(&full[i], (issued_parity >> i) & 1u, p.timeout_ns);
            for (int i = 0; i < SR; ++i)
                if (sissued & (1u << i))
                    mbar_wait_drain(&sfull[i], (sissued_parity >> i) & 1u, p.timeout_ns);
        } else if (SHARE && warp == 2 && lane == 0 && rank == 0) {
            // ------------------------------------------------ A forwarder (rank 0 of a sharing pair)
            // once a stage's tiles have landed here, copy its A tile into the
            // same stage of rank 1; the stage cannot be refilled before rank 1's
            // MMA (which waits for this copy) is done with it
            Scheduler<BN, KIND, SPLIT, SHARE> sched(p, false);
            Work w;
            Ring ring;
            const uint32_t peer_a = mapa_shared(smem_u32(sm_a), 1);
            const uint32_t peer_full = mapa_shared(smem_u32(full), 1);
            bool ok = true;
            while (ok && sched.next(w)) {
                for (int k = w.kb0; k < w.kb1; ++k) {
                    if (!mbar_wait(&full[ring.i], ring.ph, ctl)) {
                        ok = false;
                        break;
                    }
                    bulk_copy_to_cluster(peer_a + ring.i * C::kABytes, sm_a + ring.i * C::kABytes, C::kABytes,
                                         peer_full + 8u * ring.i);
                    ring.template next<S>();
                }
            }
        } else if (kHelperC && warp == 2 && lane == 0) {
            // ------------------------------------------------ addend/store (accumulate)
            // Per tile: once the previous tile's stores have read the staging
            // area, C's first half (64 of each warp's 128 columns) goes into
            // it, one 3-D box of 4 x 32 rows x 16 fp32 columns per epilogue
            // warp; when every warp has added it, the second half; when every
            // warp has left its bf16 rows there, the tile's stores.  Rows past
            // M and columns past N arrive as zeros.
            Scheduler<BN, KIND, SPLIT, SHARE> sched(p, false);
            Work w;
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
                    // the epilogue's rule: full 32-row slabs go by TMA, others were
                    // written by their warp directly
                    if (w.valid_rows - 32 * (e & 3) < 32)
                        continue;
                    for (int pi = 0; pi < COLS / C::kPanelCols; ++pi) {
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
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------ MMA issuer
            Scheduler<BN, KIND, SPLIT, SHARE> sched(p, false);
            Work w;
            Ring ring, acc;
            constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
            bool second = false;    // this K block's operands came with the previous block's
            bool ok = true;
            while (ok && sched.next(w)) {
                for (int k = w.kb0; k < w.kb1; ++k) {
                    // the producer's pairing rule
                    const bool pair = !second && C::kPairLoads && (ring.i & 1u) == 0 && k + 1 < w.kb1;
                    if (!mbar_wait(&tempty[acc.i], acc.ph ^ 1u, ctl) ||
                        (!second && !mbar_wait(&full[ring.i], ring.ph, ctl))) {
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
                    // One commit per K block (each commit drains the tensor
                    // pipe): it frees the operand stage for the producer and
                    // tells the epilogue that TMEM buffer acc.i is complete
                    // (when sharing, in both CTAs of the pair).
                    if constexpr (SHARE)
                        mma_commit_multicast(&empty[ring.i], 0x3);
                    else
                        mma_commit(&empty[ring.i]);
                    second = pair;
                    ring.template next<S>();
                    acc.template next<NACC>();
                }
            }
            // all MMAs issued above complete before tensor memory is freed
            mma_commit(drain);
            mbar_wait_drain(drain, 0, p.timeout_ns);
        }
    } else {
        regs_alloc<kRegsEpi>();
        // ------------------------------------------------ epilogue warps
        const int ew = warp - kEpiWarp0;     // 0..7
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int h = ew >> 2;               // column half of the tile
        const int row_in_tile = 32 * q + lane;
        const int sfb_row = (BN == 256) ? h : 0;
        uint8_t *panels = sm_stage_d + ew * C::kPanelsPerWarp * C::kPanelBytes;
        uint32_t panel_ctr = 0;
        (void)panel_ctr;

        if (KIND == kKindMasked && blockIdx.x == 0 && ew == 0) {
            for (int g = lane; g < p.G; g += 32) {
                const int c = __ldg(p.layout + g);
                if (c < 0 || c > p.rows)
                    atomicOr(p.error_word, kErrBadGroupBit);
            }
        }

        Scheduler<BN, KIND, SPLIT, SHARE> sched(p, ew == 0 && lane == 0 && rank == 0);
        Work w;
        Ring ring, acc_ring, sring;
        bool ok = true;
        uint32_t cph = 0;       // phase of c_full this warp waits for next (addend/store warp)
        while (ok && sched.next(w)) {
            float acc[COLS];
            // staged addend (kKindNTAcc, whole-tile staging): the rows this
            // warp adds C to (none unless this CTA stores the tile), and the
            // K blocks after which half 0 is copied and then added (with
            // half 1 copied); short ranges do both halves after the loop
            constexpr bool kStagedC = KIND == kKindNTAcc && C::kFullTileStaging && !kHelperC;
            static_assert(!kStagedC || (COLS == 2 * kAddendHalfCols &&
                                        C::kPanelsPerWarp * C::kPanelBytes >= 32 * kAddendHalfCols * 4),
                          "addend halves");
            const int c_rows = (kStagedC && w.kb1 == p.kb) ? min(max(w.valid_rows - 32 * q, 0), 32) : 0;
            const bool c_early = w.kb1 - w.kb0 >= 8;
            const int k_copy0 = w.kb0 + 3, k_add0 = w.kb1 - 3;
            // with the addend/store warp, half 0 is added six K blocks into
            // the tile (halfway, for shorter ranges): its copy has landed by
            // then, and the copy of half 1 that this releases has the rest of
            // the tile to land (adding it three blocks before the end, like
            // the cp.async path, left the epilogue waiting for half 1: 4096 x
            // 7168 x 2048 took 81.9 us, against 70.6 us this way)
            const int k_c0 = w.kb0 + min(6, (w.kb1 - w.kb0) / 2);
            // with the addend/store warp: wait for half rd of C, add it and,
            // for the first half, hand the staging area back
            auto take_c = [&](int rd) -> bool {
                if (!warp_wait(c_full, cph, ctl))
                    return false;
                cph ^= 1u;
                __syncwarp();
                add_c_box<COLS>(acc, panels, lane, rd);
                __syncwarp();           // every lane's reads before the area is reused
                if (rd == 0 && lane == 0)
                    mbar_arrive(c_free);
                return true;
            };
            (void)take_c;
            if (KIND == kKindNTAcc &&
                !bounds_ok(w.a_row0 + w.valid_rows <= p.rows && w.n_blk * BN < p.N, ctl)) {
                ok = false;
                break;
            }
            if constexpr (KIND == kKindNTAcc && !C::kFullTileStaging) {
                init_from_c<BN, COLS>(acc, p, w, q, h, lane);
            } else {
#pragma unroll
                for (int i = 0; i < COLS; ++i)
                    acc[i] = 0.f;
            }

            for (int k = w.kb0; k < w.kb1; ++k) {
                // the K block's scales (landed long ago: the producer runs
                // up to S + NACC blocks ahead), then its MMA completion.  The
                // stage barrier cannot have moved on: MMA k+S needs the TMEM
                // buffer this warp frees after block k+S-NACC >= k.
                const int kc = (k - w.kb0) % kScaleChunk;     // position in the scale chunk
                const int k0 = k - kc;
                if (!warp_all((kc != 0 || mbar_wait(&sfull[sring.i], sring.ph, ctl)) &&
                              mbar_wait(&empty[ring.i], ring.ph, ctl))) {
                    ok = false;
                    break;
                }
                __syncwarp();
                tc_fence_after_sync();
                // the scales are read inside promote_block, after the first
                // TMEM load is issued; the B part starts at the aligned group
                // of 4 that holds the chunk's first B scale, and the flat SFB
                // index picks the element
                const uint8_t *slot = sm_scales + sring.i * C::kSlotBytes;
                const float *pa = reinterpret_cast<const float *>(slot) + kc * kBM + row_in_tile;
                const int sfb_idx0 = (w.g * p.nb + (w.n_blk * BN) / 128 + sfb_row) * p.kb + k0;
                const float *pb = reinterpret_cast<const float *>(slot + C::kSlotSfaBytes +
                                                                  C::kSlotSfbStride * sfb_row) + (sfb_idx0 & 3) + kc;

                const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + acc_ring.i * BN + h * COLS;
                if (w.valid_rows > 32 * q)
                    promote_block<COLS, 64>(acc, taddr, pa, pb, &tempty[acc_ring.i], lane);
                else
                    release_tmem(&tempty[acc_ring.i], lane);   // rows past M: nothing to read
                acc_ring.template next<NACC>();
                ring.template next<S>();
                if (kc == kScaleChunk - 1 || k + 1 == w.kb1) {
                    // last K block of the chunk: the slot may be refilled
                    // (released after the TMEM buffer, off its critical path;
                    // every lane arrives)
                    mbar_arrive(&sempty[sring.i]);
                    sring.template next<SR>();
                }
                if constexpr (kHelperC) {
                    if (c_early && k == k_c0 && !take_c(0)) {
                        ok = false;
                        break;
                    }
                }
                if constexpr (kStagedC) {
                    if (c_rows > 0 && c_early && k == k_copy0) {
                        // the previous tile's stores have read the staging area
                        if (lane == 0)
                            bulk_wait_group_read<0>();
                        __syncwarp();
                        copy_c_half<BN, COLS>(panels, p, w, q, h, lane, c_rows, 0);
                    }
                    if (c_rows > 0 && c_early && k == k_add0) {
                        add_c_half<COLS>(acc, panels, lane, 0);
                        copy_c_half<BN, COLS>(panels, p, w, q, h, lane, c_rows, 1);
                    }
                }
            }
            if (!ok)
                break;

            bool has_out = true;
            if constexpr (SPLIT) {
                // a warp whose 32 rows all lie past M (M <= 96) neither
                // publishes nor reduces: every contributor of the tile sees the
                // same rows, so the region's counter is simply never used
                const bool warp_rows = w.valid_rows > 32 * q;
                if (!warp_rows)
                    has_out = false;
                if (warp_rows && !(w.kb0 == 0 && w.kb1 == p.kb)) {
                    // split tile: contributors c_lo .. c_hi (CTA order) each
                    // hold the partial of their K range.  All but c_hi publish
                    // theirs for this warp's 32 x COLS region and bump the
                    // region's counter; c_hi (which works on its share last)
                    // waits for the counter, sums the published partials in CTA
                    // order, adds its own and stores the tile.
                    const int t = w.tile;
                    const int P = gridDim.x;
                    const int c_lo = unit_owner(t * p.kb, p.units, P);
                    const int c_hi = unit_owner((t + 1) * p.kb - 1, p.units, P);
                    auto slot_of = [&](int c) {
                        const int first_tile = (int)((unsigned)c * (unsigned)p.units / (unsigned)P) / p.kb;
                        return 2 * c + (t == first_tile ? 0 : 1);
                    };
                    constexpr int F4 = COLS / 4;
                    auto region = [&](int c) {
                        return reinterpret_cast<float4 *>(p.partials) +
                               ((size_t)slot_of(c) * kNumEpiWarps + ew) * F4 * 32;
                    };
                    int *ctr = p.counters + (size_t)t * kNumEpiWarps + ew;
                    if (!bounds_ok(t >= 0 && t < p.num_tiles && c_lo >= 0 && c_lo <= (int)blockIdx.x &&
                                       (int)blockIdx.x <= c_hi && c_hi < P && slot_of((int)blockIdx.x) < 2 * P,
                                   ctl)) {
                        ok = false;
                        break;
                    }
                    if ((int)blockIdx.x != c_hi) {
                        float4 *mine = region(blockIdx.x);
#pragma unroll
                        for (int j = 0; j < F4; ++j)
                            st_cg_f4(mine + j * 32 + lane,
                                     make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
                        __threadfence();
                        __syncwarp();
                        if (lane == 0)
                            red_release_add(ctr, 1);
                        has_out = false;
                    } else {
                        int got = 1;
                        if (lane == 0)
                            got = wait_counter(ctr, c_hi - c_lo, ctl) ? 1 : 0;
                        got = __shfl_sync(0xffffffffu, got, 0);
                        if (!got) {
                            ok = false;
                            break;
                        }
                        __threadfence();
                        // this CTA's partial, then the published ones in CTA
                        // order: one fixed sequence of additions per tile,
                        // however the contributors' timing falls
                        for (int c = c_lo; c < c_hi; ++c) {
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
                            *ctr = 0;   // leave the workspace zeroed for the next call
                    }
                }
            }

            // ---- bf16 store of this warp's 32 rows x COLS columns
            int rows_ok = has_out ? min(max(w.valid_rows - 32 * q, 0), 32) : 0;
            const int y_row0 = w.a_row0 + 32 * q;
            if (rows_ok > 0 && !bounds_ok(y_row0 >= 0 && y_row0 + rows_ok <= p.d_rows_total, ctl))
                rows_ok = 0;
            if constexpr (kHelperC) {
                // the addend/store warp has waited for the previous tile's
                // stores; each lane overwrites only its own row of C below
                if ((!c_early && !take_c(0)) || !take_c(1)) {
                    ok = false;
                    break;
                }
            } else if constexpr (C::kFullTileStaging) {
                // the previous tile's stores have had a whole tile to read
                // this warp's staging area; make sure they are done
                if (lane == 0)
                    bulk_wait_group_read<0>();
                __syncwarp();
                if constexpr (kStagedC) {
                    if (c_rows > 0) {
                        if (!c_early) {
                            copy_c_half<BN, COLS>(panels, p, w, q, h, lane, c_rows, 0);
                            add_c_half<COLS>(acc, panels, lane, 0);
                            copy_c_half<BN, COLS>(panels, p, w, q, h, lane, c_rows, 1);
                        }
                        add_c_half<COLS>(acc, panels, lane, 1);
                    }
                }
            }
            constexpr int PC = C::kPanelCols;
#pragma unroll
            for (int pi = 0; pi < COLS / PC; ++pi) {
                const int x = w.n_blk * BN + h * COLS + pi * PC;
                if (x >= p.N || rows_ok == 0)
                    continue;
                // TMA store unless the slab's rows straddle the end of D's rows
                if constexpr (C::kFullTileStaging) {
                    store_panel<PC, false, !kHelperC>(acc + pi * PC, panels + pi * C::kPanelBytes, &tmap_d, p, x,
                                                      y_row0, rows_ok, lane);
                } else {
                    uint8_t *buf = panels + (panel_ctr & 1u) * C::kPanelBytes;
                    store_panel<PC, true>(acc + pi * PC, buf, &tmap_d, p, x, y_row0, rows_ok, lane);
                    if (rows_ok == 32)
                        ++panel_ctr;
                }
            }
            if constexpr (kHelperC) {
                // the full 32-row slabs are in the staging area: the
                // addend/store warp stores them
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(d_ready);
            }
        }
        if constexpr (KIND == kKindNTAcc)
            cp_async_wait_all();        // no addend copy lands after an abort either
        if (lane == 0)
            bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (SHARE) {
        // no commit, forwarded tile or abort store reaches either CTA after this
        cluster_sync();
        if (__syncthreads_or(*abort_flag)) {
            // an aborted pair may have stopped with a forwarded tile in flight
            // that no barrier it still waits on counts: give it time to land
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 200000ull)
                __nanosleep(1000);
        }
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
#endif
}

}  // namespace fp8g
