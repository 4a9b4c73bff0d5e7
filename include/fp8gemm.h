/*
 * fp8gemm.h -- C ABI of the GB300 (sm_103a) FP8 block-scaled GEMM library.
 *
 * Operation (every GEMM entry point; fp8_gemm_nt_accumulate adds C first):
 *
 *   D[m][n] = bf16( sum_{k < K/128} SFA[k][m] * SFB[n/128][k] *
 *                   sum_{t < 128} A[m][128k+t] * B[n][128k+t] )
 *
 * A and B hold OCP E4M3FN bytes.  A carries one fp32 scale per row per
 * 128-wide K block, B one fp32 scale per 128x128 block.  Each 128-K partial
 * product is accumulated in fp32 and promoted into an fp32 accumulator with
 * its two scales; D is rounded to bf16 (round to nearest even).
 * Source: DeepGEMM fp8_gemm.cuh -- fp8_gemm_kernel (per-128-channel scaling
 * checks, the math warp-groups' promotion of each K block with
 * scale_a * scale_b, the bf16 epilogue) and the Gemm class's TMA descriptor
 * factories, which fix the layouts below.
 *
 * Layouts (row-major, C order; every pointer is a DEVICE pointer):
 *   A    e4m3 [M][K]                 masked: [G][M_max][K]
 *   SFA  fp32 [K/128][sfa_ld(M)]     masked: [G][K/128][sfa_ld(M_max)]
 *        (M-major: SFA[k][m] scales A[m][128k .. 128k+127]; the leading
 *        dimension is M rounded up to a multiple of 4, as the Gemm class's
 *        make_2d_tma_scales_a_desc pads it; pad entries are never read)
 *   B    e4m3 [G][N][K]              (G = 1 for fp8_gemm_nt; "NT": K is the
 *        contiguous dimension of both operands)
 *   SFB  fp32 [G][ceil(N/128)][K/128]
 *   D    bf16 [M][N]                 masked: [G][M_max][N]
 *
 * Requirements (checked on the host before anything is launched):
 *   K % 128 == 0 and K > 0 (the kernel's BLOCK_K == 128 scaling contract);
 *   N % 16 == 0 (16-byte rows of D for the tensor-memory-access store);
 *   A, B, D, SFA and SFB 16-byte aligned;
 *   contiguous: M_total % 128 == 0 (every 128-row block belongs to one group).
 *
 * Ownership and synchronisation: the caller owns every buffer.  Calls are
 * asynchronous on `stream` and allocate nothing.  The host never reads the
 * device-side group layout (m_indices, masked_m), so no call synchronises.
 * Calls on different streams may run concurrently if their workspaces differ.
 *
 * Errors: every entry point returns an fp8g_status.  Argument errors are
 * returned synchronously and nothing is launched.  Errors found on the
 * device (a bounded wait that ran out, a group index out of range) are
 * recorded in a per-device sticky flag that fp8_gemm_get_device_error
 * reads and clears.  Nothing aborts, prints or throws.
 */
#ifndef FP8GEMM_H
#define FP8GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *fp8g_stream_t;

enum fp8g_status {
    FP8G_OK = 0,
    FP8G_ERR_INVALID_ARG = 1,  /* null pointer, negative size, G <= 0        */
    FP8G_ERR_UNSUPPORTED = 2,  /* K % 128, N % 16, M_total % 128, size limits */
    FP8G_ERR_MISALIGNED = 3,   /* pointer alignment (see Requirements)        */
    FP8G_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed           */
    FP8G_ERR_TIMEOUT = 5,      /* device: a bounded pipeline wait ran out     */
    FP8G_ERR_BAD_GROUP = 6,    /* device: group index / count out of range    */
    FP8G_ERR_WORKSPACE = 7,    /* workspace smaller than a forced split needs */
    FP8G_ERR_SCRATCH_LIMIT = 8, /* fp8_gemm_nt_noalloc: static scratch too small */
    FP8G_ERR_BOUNDS = 9        /* device: a bounds check of the checking build failed */
};

enum fp8g_kind {
    FP8G_KIND_NT = 0,
    FP8G_KIND_GROUPED_CONTIGUOUS = 1,
    FP8G_KIND_GROUPED_MASKED = 2
};

/*
 * Plain GEMM: D[M][N] = A[M][K] * B[N][K]^T with the scales above.
 * Source: DeepGEMM fp8_gemm.cuh, fp8_gemm_kernel with GemmType::Normal.
 * M == 0 or N == 0 is a no-op.  `workspace` (device memory, may be NULL) lets
 * problems with fewer output tiles than SMs split K across SMs; its size
 * comes from fp8_gemm_workspace_size.  It must be zero-filled before its
 * first use; every successful call leaves it zero-filled again (after a
 * device error, zero it again before reuse).  With no or too small a
 * workspace the call runs unsplit and still returns FP8G_OK.
 */
int fp8_gemm_nt(const void *A, const float *SFA, const void *B, const float *SFB,
                void *D, int M, int N, int K,
                void *workspace, size_t workspace_bytes, fp8g_stream_t stream);

/*
 * Plain GEMM with an fp32 addend:
 *   D[m][n] = bf16( C[m][n] + sum_k SFA[k][m] * SFB[n/128][k] * S_k(m, n) )
 * with S_k the 128-wide K block's product of A and B as above.  C is DEVICE
 * fp32 [M][N] (row-major, leading dimension N), 16-byte aligned, read only,
 * and must not overlap D; D keeps fp8_gemm_nt's bf16 layout.  Only the
 * thread block that stores a tile adds C into its fp32 accumulator, so C is
 * added exactly once (also when K is split across blocks); the result is
 * rounded to bf16 once.
 * Source: TCGen05 Copy Instruction (Triton Gluon tutorial), the matmul-
 * accumulate example (C is placed in the accumulator, then the product of A
 * and B is accumulated on top of it).
 * Everything else -- requirements, workspace (size from fp8_gemm_workspace_size
 * with kind FP8G_KIND_NT), schedules, errors -- is fp8_gemm_nt's.  C == NULL or
 * C overlapping D returns FP8G_ERR_INVALID_ARG, a C not 16-byte aligned
 * FP8G_ERR_MISALIGNED; M == 0 or N == 0 is a no-op.
 */
int fp8_gemm_nt_accumulate(const void *A, const float *SFA, const void *B, const float *SFB,
                           const float *C, void *D, int M, int N, int K,
                           void *workspace, size_t workspace_bytes, fp8g_stream_t stream);

/*
 * Plain GEMM with power-of-two (UE8M0) scales:
 *   D[m][n] = bf16( sum_k 2^(SFA_e[k][m] - 127) * 2^(SFB_e[n/128][k] - 127) *
 *                   sum_{t < 128} A[m][128k+t] * B[n][128k+t] )
 * The method's granularity is kept (one scale per row of A per 128-wide K
 * block, one per 128 x 128 block of B); each scale is a UE8M0 byte e of the
 * OCP MX formats, value 2^(e - 127) (0xFF is not a valid scale).  The tensor
 * cores' block-scaled MMA applies the scales, so the fp32 sum over all of K
 * stays in tensor memory: the product of two power-of-two scales and an
 * E4M3 product is exact, and the only roundings are the fp32 accumulation
 * and the final bf16.
 * Layouts (device pointers): A e4m3 [M][K], B e4m3 [N][K], D bf16 [M][N] as
 * for fp8_gemm_nt; SFA_e uint8 [K/128][fp8_gemm_sfa_ld(M)] (M-major, pad
 * entries never read), SFB_e uint8 [ceil(N/128)][K/128].  SFA_e and SFB_e
 * need no alignment; A, B and D 16 bytes.  K % 128 == 0, N % 16 == 0.
 * No workspace; M == 0 or N == 0 is a no-op.  Errors as for fp8_gemm_nt.
 * Source: TCGen05 Copy Instruction (Triton Gluon tutorial), the closing
 * section on block-scaled MMA (scales held in tensor memory beside the
 * accumulator), applied to the scaling of DeepGEMM fp8_gemm.cuh.
 */
int fp8_gemm_nt_ue8m0(const void *A, const void *SFA_e, const void *B, const void *SFB_e,
                      void *D, int M, int N, int K, fp8g_stream_t stream);

/*
 * Grouped GEMM, contiguous layout (MoE experts): rows of A are concatenated
 * over groups; m_indices[r] (device int32 [M_total]) names the group of row
 * r, and row r is multiplied by B[m_indices[r]].  Every 128-row block must
 * hold one group: the kernel reads m_indices at the first row of each block.
 * A block whose index is -1 is skipped and its D rows are left untouched;
 * any other index outside [0, G) is skipped too and raises FP8G_ERR_BAD_GROUP
 * in the device flag.
 * Source: DeepGEMM fp8_gemm.cuh, GemmType::GroupedContiguous (B descriptor
 * spans N * kNumGroups rows; the scheduler maps a block to its group).
 */
int fp8_gemm_grouped_contiguous(const void *A, const float *SFA, const void *B,
                                const float *SFB, void *D, const int *m_indices,
                                int M_total, int N, int K, int G,
                                void *workspace, size_t workspace_bytes,
                                fp8g_stream_t stream);

/*
 * Grouped GEMM, masked layout (MoE decode): group g computes rows
 * 0 .. masked_m[g]-1 of its [M_max][K] slice of A against B[g]; D rows at or
 * beyond masked_m[g] are left untouched.  masked_m is device int32 [G]; a
 * count above M_max is clamped to M_max and a negative one treated as 0, both
 * raising FP8G_ERR_BAD_GROUP in the device flag.
 * Source: DeepGEMM fp8_gemm.cuh, GemmType::GroupedMasked (A, D and scales_a
 * descriptors span kNumGroups slices of shape_m rows).
 */
int fp8_gemm_grouped_masked(const void *A, const float *SFA, const void *B,
                            const float *SFB, void *D, const int *masked_m,
                            int G, int M_max, int N, int K,
                            void *workspace, size_t workspace_bytes,
                            fp8g_stream_t stream);

/*
 * Bytes of workspace the given problem can use (0 if it never splits K).
 * kind is an fp8g_kind (FP8G_KIND_NT also for fp8_gemm_nt_accumulate); for NT
 * pass G = 1; M is M, M_total or M_max.
 * Pure host function: needs no GPU.  Assumes the current device's SM count
 * if a device is present, else 152.
 */
size_t fp8_gemm_workspace_size(int kind, int M, int N, int K, int G);

/*
 * Synchronises `stream`, then returns and clears the current device's sticky
 * device-side error (FP8G_OK if none; FP8G_ERR_BOUNDS wins over
 * FP8G_ERR_TIMEOUT, which wins over FP8G_ERR_BAD_GROUP).  FP8G_ERR_CUDA if the
 * synchronisation itself failed.  FP8G_ERR_BOUNDS comes only from the
 * bounds-checking build of this library (libfp8gemm_debug.so, compiled with
 * FP8G_DEBUG_BOUNDS=1): its kernels check that every tile, group, K-block,
 * split-slot and counter index and every store lies inside the problem, and
 * skip the access (and stop the block) instead of faulting when one does not.
 */
int fp8_gemm_get_device_error(fp8g_stream_t stream);

/* Static, human-readable text for a status code (never NULL). */
const char *fp8_gemm_status_string(int status);

/* Leading dimension of SFA for M rows: M rounded up to a multiple of 4. */
int fp8_gemm_sfa_ld(int M);

/*
 * Tuning and test control (process-wide; 0 restores the automatic choice):
 *   block_n     : 128 or 256 columns per output tile;
 *   split_ctas  : > 0 forces the split-K schedule over that many CTAs (with
 *                 128-column tiles unless block_n says 256; needs a workspace
 *                 of fp8_gemm_workspace_size_for bytes), < 0 forbids splitting.
 *                 A forced count above the device's SM count makes the GEMM
 *                 calls return FP8G_ERR_UNSUPPORTED: all CTAs of a split
 *                 schedule must be resident at once (one per SM), because a
 *                 tile's reducing CTA waits for the others' partials.
 * Returns FP8G_ERR_INVALID_ARG for values outside those sets.  The
 * environment variable FP8G_FORCE_CONFIG="block_n[,split_ctas]", read when
 * the library loads, sets the same values (a malformed value is ignored);
 * this call replaces them.
 */
int fp8_gemm_set_override(int block_n, int split_ctas);

/*
 * CTA-pair kernel choice (process-wide):
 *   mode  1 : run every unsplit plain, addend, contiguous and masked call on
 *             CTA pairs -- clusters of two CTAs on neighbouring SMs that
 *             share one 256 x 256 output tile (256 x 128 under a block_n
 *             override of 128) through tcgen05.mma.cta_group::2 (each CTA
 *             loads its own 128 rows of A and half of the tile's B; nothing
 *             is multicast); and every fp8_gemm_nt_ue8m0 call on CTA pairs
 *             sharing 256 x 256 tiles through the block-scaled
 *             tcgen05.mma.cta_group::2 (each CTA holds the scales of its own
 *             rows and of all 256 columns in its tensor memory);
 *   mode  2 : run every unsplit plain, contiguous and masked call (not the
 *             addend variant) with 128 x 256 tiles in clusters of two CTAs
 *             that compute neighbouring n-blocks of one m-block: the first
 *             CTA loads each A tile and copies it into the second one's
 *             shared memory (cp.async.bulk.shared::cluster), so the pair
 *             reads A from global memory once.  A block_n override other than
 *             256 turns it off.  Source: TVM TIRx, the "copy_async -> dsmem"
 *             two-CTA shared-to-shared bulk copy;
 *   mode  0 : the automatic choice (the default): CTA pairs with 256 x 256
 *             tiles for an unsplit plain call, with or without the addend
 *             (fp8_gemm_nt, fp8_gemm_nt_noalloc, fp8_gemm_nt_accumulate),
 *             when no block_n override is set, the
 *             problem has at least one pair tile per pair the GPU holds at
 *             once, and the pair tiles cover at most an eighth more of D
 *             than the one-CTA tiles would (M = 384 stays on one CTA), and
 *             for fp8_gemm_nt_ue8m0 with M > 128; one CTA per tile for
 *             everything else;
 *   mode -1 : never use CTA pairs.
 * Results are the same to within fp32 rounding order (bit-identical on
 * exactly representable inputs).  Returns FP8G_ERR_INVALID_ARG for other
 * values.  The environment variable FP8G_PAIR_MODE ("-1", "0", "1" or "2"), read
 * when the library loads, sets the same value; this call replaces it.
 * Source of the sharing: DeepGEMM fp8_gemm.cuh, tma_copy<kNumTMAMulticast>
 * and the cluster launch of Gemm::run (the pages share one m-block's A across
 * the CTAs of a cluster; here the pair shares its B and each CTA's partial
 * stays in its own tensor memory).
 */
int fp8_gemm_set_pair_mode(int mode);

/*
 * Narrow-slice kernel choice for fp8_gemm_nt and fp8_gemm_nt_noalloc
 * (process-wide).  With M <= 128 the GEMM is one stream of B.  The
 * narrow-slice kernel gives each CTA one 96-column slice of the output and
 * one of two K parts (each CTA reads half of A; one CTA per SM, work units
 * taken in turn beyond that).  The two CTAs of a slice, a cluster of two,
 * trade halves of their fp32 partials over distributed shared memory; each
 * adds the other's (P0 + P1, the same bits in either order) and stores its
 * half.  It needs no workspace (a workspace passed in is left untouched).
 * Each copy brings several consecutive K blocks of A and B; the promotion
 * with the scales is the same as everywhere else (DeepGEMM fp8_gemm.cuh,
 * fp8_gemm_kernel: per 128-wide K block, scale_a * scale_b).
 *   mode  1 : every fp8_gemm_nt / fp8_gemm_nt_noalloc call with M <= 128
 *             and K >= 512;
 *   mode  0 : the automatic choice (the default): as mode 1, with at least
 *             8 K blocks per K part and between half the SM count and the SM
 *             count of work units;
 *   mode -1 : never.
 * A block_n or split override (fp8_gemm_set_override) rules it out.  Results
 * equal the other schedules' to within fp32 rounding order (bit-identical on
 * exactly representable inputs).  Returns FP8G_ERR_INVALID_ARG for other
 * values.  The environment variable FP8G_NARROW_MODE ("-1", "0" or "1"), read
 * when the library loads, sets the same value; this call replaces it.
 * fp8_gemm_workspace_size(FP8G_KIND_NT, ...) still reports the split-K
 * schedule's workspace (fp8_gemm_nt_accumulate, which never runs narrow,
 * uses the same size).
 */
int fp8_gemm_set_narrow_mode(int mode);

/* Workspace bytes for an explicit split over `split_ctas` CTAs with tiles of
 * `block_n` columns (the size fp8_gemm_workspace_size reports for the
 * automatic choice). */
size_t fp8_gemm_workspace_size_for(int M, int N, int K, int block_n, int split_ctas);

/*
 * Upper bound, in nanoseconds, on every pipeline wait inside the kernels
 * (default 2e9).  A wait that runs out records FP8G_ERR_TIMEOUT, drains the
 * block's copies in flight, frees its tensor memory and returns.  Must be >= 1e6.
 */
int fp8_gemm_set_wait_timeout_ns(uint64_t ns);

/*
 * fp8_gemm_nt_noalloc: fp8_gemm_nt for callers that cannot allocate device
 * memory -- for example code that runs inside an allocator or memory-pool
 * callback, plug-ins whose host framework owns every device allocation, or
 * real-time loops that forbid allocation once they have started -- and so
 * cannot provide the workspace the split-K schedule needs.  The paper has
 * no counterpart to this entry point.
 *
 * Same operation, layouts and requirements as fp8_gemm_nt; the caller still
 * passes A, SFA, B, SFB and D.  The split-K scratch (counters and fp32
 * partials) is a static device array of 24 MiB (25,165,824 bytes) inside
 * this library; every GPU that loads the library holds it until the process
 * exits.  Nothing is allocated per call: no cudaMalloc, no cudaFree.
 *   - Schedule: fp8_gemm_nt's, given all the workspace it asks for, whenever
 *     that fits the array -- always the case for the automatic tile width on
 *     a GPU with up to 190 SMs.  When it does not fit (a forced 256-column
 *     tile width through fp8_gemm_set_override, or a GPU with more SMs) the
 *     call quietly takes the best automatic schedule that fits the array,
 *     down to the unsplit one, and still returns FP8G_OK.
 *   - Only a forced split count (fp8_gemm_set_override's split_ctas > 0)
 *     whose scratch exceeds the array returns FP8G_ERR_SCRATCH_LIMIT, and
 *     then nothing is launched.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Every call shares the one array and clears its counters (an async
 *     memset on `stream`) before launching; calls that overlap on the GPU
 *     (different streams, or several host threads) race on it and must be
 *     serialised by the caller.
 */
int fp8_gemm_nt_noalloc(const void *A, const float *SFA, const void *B, const float *SFB,
                        void *D, int M, int N, int K, fp8g_stream_t stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int fp8_gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8GEMM_H */
