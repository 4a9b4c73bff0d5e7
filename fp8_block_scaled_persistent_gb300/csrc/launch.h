// launch.h -- host-side launch interface between the C ABI (api.cu) and the
// kernel instantiations (gemm_nt.cu, gemm_nt_acc.cu, gemm_contiguous.cu,
// gemm_masked.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_params.h"

namespace fp8g {

struct LaunchArgs {
    CUtensorMap tmap_a, tmap_b, tmap_d, tmap_sfa, tmap_sfb;
    // A and B viewed as [K/128][rows][128 B] with boxes two K blocks deep
    // (zeroed, and never used, when K/128 < 2)
    CUtensorMap tmap_a2, tmap_b2;
    // the fp32 addend C [rows][N] viewed as [N/16][rows][16] with boxes of
    // 4 x 32 rows x 16 columns, for the accumulate kernel whose addend/store
    // warp copies it (zeroed, and never used, otherwise)
    CUtensorMap tmap_c{};
    Params p;
    int grid;
    cudaStream_t stream;
};

// Dynamic shared memory a launch with tiles of `block_n` columns needs.
int smem_bytes_for(int block_n);

// Width, in bf16 columns, of the output panels the kernel TMA-stores for
// tiles of `block_n` columns (the D tensor map's box is 32 rows x this).
int panel_cols_for(int block_n);

cudaError_t launch_nt(int block_n, bool split, const LaunchArgs &a);
cudaError_t launch_nt_acc(int block_n, bool split, const LaunchArgs &a);   // a.p.c set
cudaError_t launch_contiguous(int block_n, const LaunchArgs &a);
cudaError_t launch_masked(int block_n, const LaunchArgs &a);

// The CTA-pair kernel (gemm_pair.cu, gemm_pair256.cu): clusters of two CTAs,
// one tile of 256 rows x block_n (128 or 256) columns per pair.  `kind` is a
// Kind; a.grid is twice the number of pairs; the tensor maps are those of
// make_pair_maps in api.cu (B boxes of block_n/2 rows, D panels of
// pair_panel_cols() columns).
cudaError_t launch_pair(int kind, int block_n, const LaunchArgs &a);
int pair_panel_cols();
// Clusters of two that can be resident at once on device `dev` (0 on failure).
int max_active_pairs(int dev, int block_n);

// The one-CTA kernel in clusters of two sharing each A tile over DSMEM
// (gemm_share.cu): 256-column tiles, unsplit; `kind` is kKindNT,
// kKindContiguous or kKindMasked; the tensor maps are make_maps' for
// block_n 256; a.p.num_tiles counts (m-block, pair of n-blocks) tiles and
// a.grid is twice the number of clusters.
cudaError_t launch_share(int kind, const LaunchArgs &a);
int max_active_share_pairs(int dev);

// The power-of-two-scale kernel (gemm_ue8m0.cu): tiles of 128 x
// ue8m0_block_n(), a.p.sfa_e / a.p.sfb_e set; tensor maps tmap_a (boxes of
// 128 rows), tmap_b (boxes of ue8m0_block_n() rows), tmap_d (panels of
// ue8m0_panel_cols() columns).
cudaError_t launch_ue8m0(const LaunchArgs &a);
int ue8m0_block_n();
int ue8m0_panel_cols();
// The same on CTA pairs (256 x 256 tiles): tmap_a boxes of 128 rows, tmap_b
// boxes of ue8m0_pair_block_n() / 2 rows, tmap_d panels of
// ue8m0_panel_cols() columns; a.grid = 2 x clusters.
cudaError_t launch_ue8m0_pair(const LaunchArgs &a);
int ue8m0_pair_block_n();
// Clusters of two of the pair kernel that can be resident at once (0 on failure).
int ue8m0_pair_max_active(int dev);

// The narrow-slice kernel for the plain GEMM with M <= 128 (gemm_narrow.cu):
// work units of one slice of narrow_block_n(a_box_rows) columns and one of
// narrow_ksplit(a_box_rows) K parts.  a.p.a_box_rows (64 when M <= 64, else
// 128) picks the instantiation; a.p.num_n_blocks counts slices; tmap_a and
// tmap_b view A and B as [K/128][rows][128 B] with boxes of a_box_rows (A) or
// the slice width (B) rows x narrow_kd(a_box_rows) K blocks; tmap_sfa and
// tmap_sfb are make_maps'.  With two K parts the two CTAs of a slice are a
// cluster of two that trade halves over distributed shared memory: a.grid is
// even and at most 2 x narrow_max_clusters().
cudaError_t launch_narrow(const LaunchArgs &a);
int narrow_block_n(int a_box_rows);
int narrow_kd(int a_box_rows);
int narrow_ksplit(int a_box_rows);
// K blocks per scale copy: tmap_sfa boxes of 128 x this, tmap_sfb of this + 4.
int narrow_scale_chunk();
// Clusters of two of the two-K-part instantiation for `a_box_rows` that can
// be resident at once on device `dev` (0 on failure or with one K part).
int narrow_max_clusters(int dev, int a_box_rows);

}  // namespace fp8g
