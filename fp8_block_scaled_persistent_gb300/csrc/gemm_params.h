// gemm_params.h -- the kernel's by-value argument block (host and device).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace fp8g {

// The operation a kernel instantiation computes.  kKindNTAcc: the plain GEMM
// with an fp32 addend, D = bf16(C + A B^T scaled).
enum Kind : int { kKindNT = 0, kKindContiguous = 1, kKindMasked = 2, kKindNTAcc = 3 };

// Bits of the sticky device-side error word.
enum : int { kErrTimeoutBit = 1, kErrBadGroupBit = 2, kErrBoundsBit = 4 };

// K blocks whose scales one scale copy brings in: the A scales of 128 rows x
// kScaleChunk K blocks (one 2-D box) and, per 128-column block, the B scales
// of those K blocks (one 1-D box of kScaleChunk + 4 values from the 16-byte
// aligned start).  Chunks start at each work unit's first K block.
constexpr int kScaleChunk = 8;

struct Params {
    int rows;          // NT: M, contiguous: M_total, masked: M_max
    int N, K, G;
    int kb, nb;        // K/128, ceil(N/128)
    int sfa_ld;        // round_up(rows, 4)
    const float *sfa;
    const float *sfb;
    const uint8_t *sfa_e;  // power-of-two scales: UE8M0 bytes, layouts of sfa and sfb
    const uint8_t *sfb_e;
    const int *layout; // contiguous: m_indices; masked: masked_m
    __nv_bfloat16 *d;
    const float *c;    // NT with an addend: fp32 [rows][N], read-only, not overlapping d
    int num_m_blocks;  // ceil(rows/128) (masked: per group, at most)
    int num_n_blocks;  // ceil(N/BN)
    int group_m;       // rasterisation band height, in m-blocks
    int num_tiles;     // NT and contiguous
    int units;         // split: num_tiles * kb (the host keeps units * CTAs < 2^31)
    float *partials;   // split: 2 * gridDim.x slots of 128 x BN fp32
    int *counters;     // split: num_tiles * 8 counters of published partials
    int *error_word;
    unsigned long long timeout_ns;
    // extents of the 2-D views (rows), for the bounds-checking build
    int a_rows_total;  // A: rows (masked: G * M_max)
    int b_rows_total;  // B: G * N
    int d_rows_total;  // D: rows (masked: G * M_max)
    // rows of A each copy brings (128, or 64 for the plain GEMM with M <= 64:
    // the MMA's rows 64..127 then read whatever the stage holds, and no warp
    // stores, publishes or reduces them)
    int a_box_rows;
};

}  // namespace fp8g
