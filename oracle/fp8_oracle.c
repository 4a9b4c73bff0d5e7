/*
 * fp8_oracle.c -- CPU oracle for the FP8 (E4M3) GEMM with fine-grained scaling.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or constant with the CUDA library and it
 * never calls it.
 *
 * What it computes (plain definition, written out with no blocking, fusion or
 * reordering beyond what the definition states):
 *
 *   dec(q)      OCP E4M3FN decode of one byte (exact in fp64)
 *   S_k(m,n)  = sum_{t=0}^{127} dec(A[m][128k+t]) * dec(B[n][128k+t])
 *   acc(m,n)  = sum_{k=0}^{K/128-1} (SFA[k][m] * SFB[n/128][k]) * S_k(m,n)
 *   D(m,n)    = bf16_rne(acc(m,n))        (one rounding, fp64 -> bf16)
 *
 * and, with an fp32 addend C[M][N] (oracle_gemm_nt_acc_rows),
 *
 *   D(m,n)    = bf16_rne(C(m,n) + acc(m,n))
 *
 * and, with power-of-two scales stored as UE8M0 exponent bytes
 * (oracle_gemm_nt_ue8m0_rows; same granularity and layouts, one byte each),
 *
 *   acc(m,n)  = sum_k 2^(ea[k][m] - 127) * 2^(eb[n/128][k] - 127) * S_k(m,n)
 *
 * Sources (page title, section):
 *   - DeepGEMM fp8_gemm.cuh, fp8_gemm_kernel, the math warp-groups: each
 *     128-wide K block is accumulated on its own (the MMA overwrites a fresh
 *     accumulator per K block) and then promoted into the final accumulator
 *     with scale_a(row, k) * scale_b(k) (the "promote with scales" step).
 *   - same kernel, the B-scale load: B scales are indexed by the column's
 *     128-column block and the K block, i.e. SFB laid out [ceil(N/128)][K/128].
 *   - same file, Gemm::make_2d_tma_scales_a_desc: A scales are stored
 *     M-major, [K/128][round_up(M, 4)], one fp32 per row per K block.
 *   - same kernel, the epilogue: the fp32 result is converted to bf16 with
 *     round-to-nearest-even.
 *   - TCGen05 Copy Instruction (Gluon tutorial), the matmul-accumulate
 *     example: the fp32 addend C is placed in the accumulator first and the
 *     product of A and B is accumulated on top of it, so D = A B^T + C.
 *   - TCGen05 Copy Instruction (Gluon tutorial), the closing section on
 *     block-scaled MMA: its scales are supplied through tensor memory; the
 *     hardware form of such scales is the 8-bit exponent-only UE8M0 format
 *     of the OCP microscaling (MX) specification: value 2^(e - 127), and
 *     e = 255 is NaN.
 *   - the grouped layouts (contiguous: one group index per row; masked: a
 *     per-group valid-row count, rows beyond it untouched) follow the same
 *     file's GemmType::GroupedContiguous / GroupedMasked descriptor shapes.
 *
 * Precision: the pages fix fp32 accumulation on the GPU; the oracle uses fp64
 * throughout.  Every E4M3 product has at most 8 significant bits and a 128
 * term sum of them spans fewer than 53 bits, so S_k is exact; only the scale
 * multiply and the sum over K blocks round (at ~1e-16 relative).  The result
 * is therefore the exact real value rounded once to bf16, up to a sub-ulp
 * double-rounding chance.
 *
 * Pins (tests/test_oracle_pins.py): exhaustive decode against a library cast
 * and the format's named special values, bf16 rounding against a library cast
 * and hand-made tie patterns, brute force against an independent dequantise-
 * then-matmul formulation, exact small-integer closed forms, the scale-
 * doubling invariant and the grouped-to-dense reductions.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* OCP 8-bit floating point, E4M3 "FN" variant: 1 sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits, no infinities, NaN = S.1111.111.                */
double oracle_e4m3_to_f64(uint8_t q)
{
    int s = (q >> 7) & 1;
    int e = (q >> 3) & 0xF;
    int m = q & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);           /* subnormal: 0.m * 2^-6 */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);   /* normal: 1.m * 2^(e-7) */
    return s ? -v : v;
}

/* bf16 = the upper 16 bits of an IEEE binary32: 8 exponent bits (bias 127),
 * 7 stored mantissa bits.  Round x (fp64) once to the nearest bf16 value,
 * ties to the value with an even last mantissa bit; overflow goes to +-Inf;
 * NaN goes to the canonical quiet NaN 0x7FC0.                               */
uint16_t oracle_f64_to_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs(x);
    uint16_t sign = (uint16_t)(neg << 15);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;

    /* a = f * 2^E with f in [0.5, 1): the leading bit has weight 2^(E-1).   */
    int E;
    (void)frexp(a, &E);
    int lead = E - 1;
    /* Quantum (weight of the last kept bit): 2^(lead-7) for normals, and
     * the fixed subnormal quantum 2^-133 below the smallest normal 2^-126. */
    int qexp = (lead >= -126) ? (lead - 7) : (-133);
    double n = ldexp(a, -qexp);                  /* exact: power-of-2 scale */
    double fl = floor(n);
    double frac = n - fl;                        /* exact: n < 2^9 */
    double r;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;   /* tie: to even */
    double v = ldexp(r, qexp);
    if (v >= ldexp(1.0, 128))
        return sign | 0x7F80;                    /* rounded past the max */

    /* v is a bf16 value, hence exactly representable in binary32. */
    float f = (float)v;
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return sign | (uint16_t)((bits >> 16) & 0x7FFF);
}

double oracle_bf16_to_f64(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* The decode of every code, filled once from oracle_e4m3_to_f64 when the
 * library loads, so the inner loop below does not call ldexp per term.    */
static double e4m3_value[256];

__attribute__((constructor)) static void oracle_fill_decode_table(void)
{
    for (int q = 0; q < 256; ++q)
        e4m3_value[q] = oracle_e4m3_to_f64((uint8_t)q);
}

/* ------------------------------------------------------------------------ */
/* One output element before rounding.
 *   a_row : K bytes of A's row m
 *   b_row : K bytes of B's row n
 *   sfa   : pointer to SFA[0][m]; the scale of K block k is sfa[k * sfa_ld]
 *   sfb   : pointer to SFB[n/128][0]; the scale of K block k is sfb[k]      */
double oracle_element_f64(const uint8_t *a_row, const uint8_t *b_row,
                          const float *sfa, long sfa_ld, const float *sfb, int K)
{
    int kb = K / 128;
    double acc = 0.0;
    for (int k = 0; k < kb; ++k) {
        double s_k = 0.0;
        for (int t = 0; t < 128; ++t)
            s_k += e4m3_value[a_row[128 * k + t]] *
                   e4m3_value[b_row[128 * k + t]];
        double scale = (double)sfa[(long)k * sfa_ld] * (double)sfb[k];
        acc += scale * s_k;
    }
    return acc;
}

/* Round-up of M to a multiple of 4: the leading dimension of SFA
 * (Gemm::make_2d_tma_scales_a_desc pads M to 16 bytes of fp32).            */
static long sfa_ld_of(int M) { return ((long)M + 3) / 4 * 4; }

/* ------------------------------------------------------------------------ */
/* Plain GEMM, D[M][N] = A[M][K] * B[N][K]^T with the scales above.
 * acc (optional, may be NULL) receives the unrounded fp64 values.           */
void oracle_gemm_nt(const uint8_t *A, const float *SFA, const uint8_t *B,
                    const float *SFB, int M, int N, int K,
                    uint16_t *D, double *acc)
{
    long ld = sfa_ld_of(M);
    int kb = K / 128;
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            double v = oracle_element_f64(A + (long)m * K, B + (long)n * K,
                                          SFA + m, ld,
                                          SFB + (long)(n / 128) * kb, K);
            if (acc)
                acc[(long)m * N + n] = v;
            D[(long)m * N + n] = oracle_f64_to_bf16_rne(v);
        }
    }
}

/* The same definition, evaluated only for the listed rows (for sampled
 * checks of large problems).  Row i of the output is rows[i] of D.          */
void oracle_gemm_nt_rows(const uint8_t *A, const float *SFA, const uint8_t *B,
                         const float *SFB, int M, int N, int K,
                         const int *rows, int nrows, uint16_t *D_rows,
                         double *acc_rows)
{
    long ld = sfa_ld_of(M);
    int kb = K / 128;
    for (int i = 0; i < nrows; ++i) {
        int m = rows[i];
        for (int n = 0; n < N; ++n) {
            double v = oracle_element_f64(A + (long)m * K, B + (long)n * K,
                                          SFA + m, ld,
                                          SFB + (long)(n / 128) * kb, K);
            if (acc_rows)
                acc_rows[(long)i * N + n] = v;
            D_rows[(long)i * N + n] = oracle_f64_to_bf16_rne(v);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Grouped, contiguous layout: rows of A are concatenated over groups and
 * group_of_row[r] names the B matrix (B is [G][N][K], SFB [G][nb][kb]) that
 * row r multiplies.  A row whose group index is outside [0, G) produces no
 * output: its D row is left as it was.  SFA is [kb][round_up(M_total, 4)].
 * Only the listed rows are evaluated (pass all rows for a full product).    */
void oracle_gemm_grouped_contiguous_rows(const uint8_t *A, const float *SFA,
                                         const uint8_t *B, const float *SFB,
                                         const int *group_of_row, int M_total,
                                         int N, int K, int G,
                                         const int *rows, int nrows,
                                         uint16_t *D_rows)
{
    long ld = sfa_ld_of(M_total);
    int kb = K / 128;
    int nb = (N + 127) / 128;
    for (int i = 0; i < nrows; ++i) {
        int m = rows[i];
        int g = group_of_row[m];
        if (g < 0 || g >= G)
            continue;
        const uint8_t *Bg = B + (long)g * N * K;
        const float *SFBg = SFB + (long)g * nb * kb;
        for (int n = 0; n < N; ++n) {
            double v = oracle_element_f64(A + (long)m * K, Bg + (long)n * K,
                                          SFA + m, ld,
                                          SFBg + (long)(n / 128) * kb, K);
            D_rows[(long)i * N + n] = oracle_f64_to_bf16_rne(v);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Grouped, masked layout: A is [G][M_max][K], SFA [G][kb][round_up(M_max,4)],
 * B [G][N][K], SFB [G][nb][kb], D [G][M_max][N].  Group g has valid rows
 * 0 .. masked_m[g]-1; rows at or beyond the count are left as they were.
 * Only group g_sel's listed rows are evaluated.                            */
void oracle_gemm_grouped_masked_rows(const uint8_t *A, const float *SFA,
                                     const uint8_t *B, const float *SFB,
                                     const int *masked_m, int G, int M_max,
                                     int N, int K, int g_sel,
                                     const int *rows, int nrows,
                                     uint16_t *D_rows)
{
    long ld = sfa_ld_of(M_max);
    int kb = K / 128;
    int nb = (N + 127) / 128;
    if (g_sel < 0 || g_sel >= G)
        return;
    int count = masked_m[g_sel];
    const uint8_t *Ag = A + (long)g_sel * M_max * K;
    const float *SFAg = SFA + (long)g_sel * kb * ld;
    const uint8_t *Bg = B + (long)g_sel * N * K;
    const float *SFBg = SFB + (long)g_sel * nb * kb;
    for (int i = 0; i < nrows; ++i) {
        int m = rows[i];
        if (m < 0 || m >= count || m >= M_max)
            continue;
        for (int n = 0; n < N; ++n) {
            double v = oracle_element_f64(Ag + (long)m * K, Bg + (long)n * K,
                                          SFAg + m, ld,
                                          SFBg + (long)(n / 128) * kb, K);
            D_rows[(long)i * N + n] = oracle_f64_to_bf16_rne(v);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Plain GEMM with an fp32 addend: D[M][N] = bf16(C[M][N] + A[M][K] * B[N][K]^T
 * with the scales above).  C is row-major with leading dimension N.  The
 * addend joins the fp64 sum of the scaled K blocks and the total is rounded
 * to bf16 once.  Only the listed rows are evaluated; acc_rows (optional)
 * receives the unrounded values.                                            */
void oracle_gemm_nt_acc_rows(const uint8_t *A, const float *SFA, const uint8_t *B,
                             const float *SFB, const float *C, int M, int N, int K,
                             const int *rows, int nrows, uint16_t *D_rows,
                             double *acc_rows)
{
    long ld = sfa_ld_of(M);
    int kb = K / 128;
    for (int i = 0; i < nrows; ++i) {
        int m = rows[i];
        for (int n = 0; n < N; ++n) {
            double v = (double)C[(long)m * N + n] +
                       oracle_element_f64(A + (long)m * K, B + (long)n * K,
                                          SFA + m, ld,
                                          SFB + (long)(n / 128) * kb, K);
            if (acc_rows)
                acc_rows[(long)i * N + n] = v;
            D_rows[(long)i * N + n] = oracle_f64_to_bf16_rne(v);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* UE8M0 scale byte: an unsigned biased exponent, value 2^(e - 127); 0xFF is
 * NaN.  Every other value is exact in fp64 (and in fp32: 2^-127 is a
 * binary32 subnormal).                                                      */
double oracle_ue8m0_to_f64(uint8_t e)
{
    if (e == 0xFF)
        return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* Plain GEMM with UE8M0 scales: SFA_e [K/128][round_up(M, 4)] and SFB_e
 * [ceil(N/128)][K/128] hold exponent bytes instead of fp32 values; the
 * definition is otherwise the plain one.  Only the listed rows are
 * evaluated; acc_rows (optional) receives the unrounded values.             */
void oracle_gemm_nt_ue8m0_rows(const uint8_t *A, const uint8_t *SFA_e, const uint8_t *B,
                               const uint8_t *SFB_e, int M, int N, int K,
                               const int *rows, int nrows, uint16_t *D_rows,
                               double *acc_rows)
{
    long ld = sfa_ld_of(M);
    int kb = K / 128;
    for (int i = 0; i < nrows; ++i) {
        int m = rows[i];
        for (int n = 0; n < N; ++n) {
            const uint8_t *a_row = A + (long)m * K;
            const uint8_t *b_row = B + (long)n * K;
            double acc = 0.0;
            for (int k = 0; k < kb; ++k) {
                double s_k = 0.0;
                for (int t = 0; t < 128; ++t)
                    s_k += e4m3_value[a_row[128 * k + t]] *
                           e4m3_value[b_row[128 * k + t]];
                double scale = oracle_ue8m0_to_f64(SFA_e[(long)k * ld + m]) *
                               oracle_ue8m0_to_f64(SFB_e[(long)(n / 128) * kb + k]);
                acc += scale * s_k;
            }
            if (acc_rows)
                acc_rows[(long)i * N + n] = acc;
            D_rows[(long)i * N + n] = oracle_f64_to_bf16_rne(acc);
        }
    }
}
