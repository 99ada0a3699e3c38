/*
 * fgf8_oracle.c -- plain, slow CPU oracle for the fine-grained FP8 GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is compared
 * against.  It shares no code, header, table or helper with the CUDA library
 * (fine_grained_fp8_persistent_gb300/csrc) and neither side includes the other.
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may load it.
 *
 * Every function states the passage of the pages it follows.  Page names:
 *   [DG]   "DeepGEMM dissected: a 300-line FP8 GEMM kernel" (pinghaoyang.com.cn)
 *   [TC5]  "GPU GEMM part 4: tcgen05 & Blackwell" (pinghaoyang.com.cn)
 *   [TIRx] "TIRx and high-performance GEMM (part 2)" (Tencent Cloud developer)
 *
 * Arithmetic: floating point is carried in double (fp64) wherever the pages do
 * not fix a precision.  The quantizer is the exception: it decides integer codes,
 * so its divide and its amax are done in FP32, the precision the kernel uses
 * (scale s = amax/448 and q = x/s are FP32 quantities in [DG] "how outliers wreck
 * per-tensor quantization").
 *
 * Parallelism: the loops over output rows carry an OpenMP pragma when the file is
 * built with -fopenmp.  Each output element is still computed by exactly the
 * same sequential loop, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define FGO_SCALE_F32 0
#define FGO_SCALE_UE8M0 1

/* ------------------------------------------------------------------------- */
/* E4M3 ("fn" variant: no infinities, one NaN pattern per sign)               */
/* [DG] section "The lure of FP8": 4 exponent bits, 3 mantissa bits, largest  */
/* value 448; [DG] "fine-grained quantization": smallest subnormal ~2^-9.     */
/* Bias 7.  Normals (1 + m/8) * 2^(e-7) for e in 1..15 (e=15, m=7 is NaN);    */
/* subnormals m * 2^-9.                                                        */
/* ------------------------------------------------------------------------- */

double fgo_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Code of a non-negative value r that lies exactly on the E4M3 grid, r <= 448. */
static uint8_t e4m3_code_of_grid_value(double r)
{
    int ex;
    double f;
    if (r == 0.0)
        return 0;
    if (r < ldexp(1.0, -6))                 /* subnormal: r = m * 2^-9 */
        return (uint8_t)(r / ldexp(1.0, -9));
    f = frexp(r, &ex);                      /* r = f * 2^ex, f in [0.5, 1) */
    /* r = (1 + m/8) * 2^(ex-1) -> biased exponent ex-1+7, m = (2f - 1) * 8 */
    return (uint8_t)(((ex - 1 + 7) << 3) | (int)((2.0 * f - 1.0) * 8.0));
}

/*
 * Round a real value to E4M3: round to nearest, ties to even, saturating any
 * finite magnitude above the largest value (448) to +-448, keeping the sign of
 * zero.  Works on the exact double value: the grid spacing near |v| is a power
 * of two, so |v| / spacing is exact and nearbyint() (current mode: nearest-even)
 * performs the only rounding.
 */
uint8_t fgo_e4m3_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a, spacing, r;
    int ex;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    a = fabs(v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        spacing = ldexp(1.0, -9);           /* subnormal spacing */
    } else {
        frexp(a, &ex);                      /* a in [2^(ex-1), 2^ex) */
        spacing = ldexp(1.0, ex - 1 - 3);   /* 3 mantissa bits */
    }
    r = nearbyint(a / spacing) * spacing;   /* <= 448 because a < 448 */
    return (uint8_t)(sign | e4m3_code_of_grid_value(r));
}

void fgo_e4m3_encode_array(const double *x, uint8_t *q, long n)
{
    long i;
    for (i = 0; i < n; ++i)
        q[i] = fgo_e4m3_encode(x[i]);
}

void fgo_e4m3_decode_array(const uint8_t *q, double *out, long n)
{
    long i;
    for (i = 0; i < n; ++i)
        out[i] = fgo_e4m3_decode(q[i]);
}

/* ------------------------------------------------------------------------- */
/* Scales                                                                      */
/* ------------------------------------------------------------------------- */

/* Rows padded to a multiple of 4 so every scale column starts on 16 bytes:   */
/* [DG] "why only the NT layout": activation scales are given TMA-aligned and */
/* transposed, shape (K/128, M) column-major.                                  */
long fgo_align4(long x) { return (x + 3) / 4 * 4; }

/*
 * FP32 scale of one group: s = amax / 448 in FP32 ([DG] worked example
 * s = 40/448).  A group whose amax is 0 takes s = 1 (the pages are silent; any
 * positive s quantizes an all-zero group to zeros).
 */
static float f32_scale_of(float amax)
{
    volatile float num = amax;
    if (amax == 0.0f)
        return 1.0f;
    return num / 448.0f;
}

/*
 * Power-of-two scale exponent of one group: the smallest e with
 * 2^e >= amax/448 (FP32 quotient), i.e. ceil(log2(amax/448)), clamped to the
 * UE8M0 range [-127, 127].  [DG] "fine-grained quantization": Blackwell MXFP8
 * wants power-of-two (UE8M0) scales; rounding the exponent up is the reading
 * under which no element saturates.  amax = 0 gives e = 0.
 */
static int ue8m0_exponent_of(float amax)
{
    volatile float num = amax;
    float t;
    double f;
    int ex, e;
    if (amax == 0.0f)
        return 0;
    t = num / 448.0f;
    f = frexp((double)t, &ex);              /* t = f * 2^ex, f in [0.5, 1) */
    e = (f == 0.5) ? ex - 1 : ex;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Quantize one value given the group's scale, in the precision the method    */
/* fixes: FP32 division x / s for FP32 scales, exact x * 2^-e for UE8M0.       */
static uint8_t quantize_value(float x, int fmt, float s, int e)
{
    if (fmt == FGO_SCALE_F32) {
        volatile float xv = x;
        volatile float sv = s;
        float qv = xv / sv;
        return fgo_e4m3_encode((double)qv);
    }
    return fgo_e4m3_encode(ldexp((double)x, -e));
}

/* Byte address of the UE8M0 exponent of (row r, K-block kb) in a packed table */
/* int32[ceil(nkb/4)][ld]: word (kb/4, r), byte kb%4 (little endian).           */
static size_t ue8m0_byte_index(long r, long kb, long ld)
{
    return ((size_t)(kb / 4) * (size_t)ld + (size_t)r) * 4u + (size_t)(kb % 4);
}

/*
 * 1x128 activation quantization ([DG] "fine-grained quantization": activations
 * grouped per token per 128 channels; scales computed online from the group's
 * max |x|).
 *   X   : M x K values (bf16 values widened to float), row-major.
 *   Xq  : M x K E4M3 codes, row-major.
 *   SFA : FP32   -> float[K/128][align4(M)]         (column m, row kb)
 *         UE8M0  -> uint8 view of int32[ceil(K/512)][align4(M)]; byte kb%4 of
 *                   word (kb/4, m) is e+127; unused bytes are 0.
 * K must be a multiple of 128.
 */
void fgo_quantize_1x128(const float *X, long M, long K, int fmt, uint8_t *Xq, void *SFA)
{
    long nkb = K / 128, ld = fgo_align4(M), m;
    if (fmt == FGO_SCALE_UE8M0)
        memset(SFA, 0, (size_t)((nkb + 3) / 4) * (size_t)ld * 4u);
    else
        memset(SFA, 0, (size_t)nkb * (size_t)ld * sizeof(float));
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (m = 0; m < M; ++m) {
        long kb, k;
        for (kb = 0; kb < nkb; ++kb) {
            const float *x = X + m * K + kb * 128;
            float amax = 0.0f, s = 1.0f;
            int e = 0;
            for (k = 0; k < 128; ++k)
                amax = fmaxf(amax, fabsf(x[k]));
            if (fmt == FGO_SCALE_F32) {
                s = f32_scale_of(amax);
                ((float *)SFA)[kb * ld + m] = s;
            } else {
                e = ue8m0_exponent_of(amax);
                ((uint8_t *)SFA)[ue8m0_byte_index(m, kb, ld)] = (uint8_t)(e + 127);
            }
            for (k = 0; k < 128; ++k)
                Xq[m * K + kb * 128 + k] = quantize_value(x[k], fmt, s, e);
        }
    }
}

/*
 * 128x128 weight-block quantization ([DG] "fine-grained quantization": weights
 * grouped per 128 input channels x 128 output channels, one scale per block).
 *   W   : G x N x K values, row-major per group.
 *   Wq  : G x N x K codes.
 *   SFB : FP32   -> float[G][ceil(N/128)][K/128]     (row-major, [DG] SMEM layout
 *                   section: one FP32 per 128x128 block along K)
 *         UE8M0  -> int32[G][ceil(K/512)][align4(N)]; the block exponent is
 *                   written for every row n of the block (the MMA consumes one
 *                   scale per B row: [TC5] block-scaling formula, SFB(N, SFK)).
 * A partial last block along N takes its amax over its valid rows only.
 */
void fgo_quantize_128x128(const float *W, long G, long N, long K, int fmt, uint8_t *Wq, void *SFB)
{
    long nkb = K / 128, nnb = (N + 127) / 128, ldn = fgo_align4(N), g;
    size_t sfb_per_group = (fmt == FGO_SCALE_UE8M0) ? (size_t)((nkb + 3) / 4) * (size_t)ldn * 4u
                                                    : (size_t)nnb * (size_t)nkb * sizeof(float);
    memset(SFB, 0, sfb_per_group * (size_t)G);
    for (g = 0; g < G; ++g) {
        const float *Wg = W + (size_t)g * (size_t)N * (size_t)K;
        uint8_t *Wqg = Wq + (size_t)g * (size_t)N * (size_t)K;
        uint8_t *sfg = (uint8_t *)SFB + (size_t)g * sfb_per_group;
        long nb;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (nb = 0; nb < nnb; ++nb) {
            long kb, n, k, n_end = (nb + 1) * 128 < N ? (nb + 1) * 128 : N;
            for (kb = 0; kb < nkb; ++kb) {
                float amax = 0.0f, s = 1.0f;
                int e = 0;
                for (n = nb * 128; n < n_end; ++n)
                    for (k = kb * 128; k < kb * 128 + 128; ++k)
                        amax = fmaxf(amax, fabsf(Wg[n * K + k]));
                if (fmt == FGO_SCALE_F32) {
                    s = f32_scale_of(amax);
                    ((float *)sfg)[nb * nkb + kb] = s;
                } else {
                    e = ue8m0_exponent_of(amax);
                    for (n = nb * 128; n < n_end; ++n)
                        sfg[ue8m0_byte_index(n, kb, ldn)] = (uint8_t)(e + 127);
                }
                for (n = nb * 128; n < n_end; ++n)
                    for (k = kb * 128; k < kb * 128 + 128; ++k)
                        Wqg[n * K + k] = quantize_value(Wg[n * K + k], fmt, s, e);
            }
        }
    }
}

/* Scale of A row m (within its table, leading dimension ld_a) for K-block kb. */
static double sfa_value(const void *SFA, int fmt, long m, long kb, long ld_a)
{
    if (fmt == FGO_SCALE_F32)
        return (double)((const float *)SFA)[kb * ld_a + m];
    return ldexp(1.0, (int)((const uint8_t *)SFA)[ue8m0_byte_index(m, kb, ld_a)] - 127);
}

/* Scale of B row n (one expert's table) for K-block kb. */
static double sfb_value(const void *SFB, int fmt, long n, long kb, long nkb, long ld_n)
{
    if (fmt == FGO_SCALE_F32)
        return (double)((const float *)SFB)[(n / 128) * nkb + kb];
    return ldexp(1.0, (int)((const uint8_t *)SFB)[ue8m0_byte_index(n, kb, ld_n)] - 127);
}

static size_t sfb_group_bytes(int fmt, long N, long K)
{
    long nkb = K / 128;
    if (fmt == FGO_SCALE_F32)
        return (size_t)((N + 127) / 128) * (size_t)nkb * sizeof(float);
    return (size_t)((nkb + 3) / 4) * (size_t)fgo_align4(N) * 4u;
}

static size_t sfa_table_bytes(int fmt, long rows, long K)
{
    long nkb = K / 128;
    if (fmt == FGO_SCALE_F32)
        return (size_t)nkb * (size_t)fgo_align4(rows) * sizeof(float);
    return (size_t)((nkb + 3) / 4) * (size_t)fgo_align4(rows) * 4u;
}

/*
 * One output element of the block-scaled NT GEMM:
 *   D[m,n] = sum_kb  sA[m,kb] * sB[n,kb] * sum_{k in kb} dec(Aq[m,k]) * dec(Bq[n,k])
 * This is the block-scaling formula of [TC5] "block scaling" with scale-vector
 * length 128 along K, which is the per-128-K promotion of [DG] main loop
 * (final += scale_a * scale_b * partial).  Everything is in double; the inner
 * 128-term sum of E4M3 products is exact in double.
 */
static double dot_fp8(const uint8_t *a, const uint8_t *b, long K,
                      const void *SFA, long ld_a, long m,
                      const void *SFB, long n, long N, int fmt)
{
    long nkb = K / 128, kb, k;
    long ld_n = fgo_align4(N);
    double acc = 0.0;
    (void)N;
    for (kb = 0; kb < nkb; ++kb) {
        double partial = 0.0;
        for (k = kb * 128; k < kb * 128 + 128; ++k)
            partial += fgo_e4m3_decode(a[k]) * fgo_e4m3_decode(b[k]);
        acc += sfa_value(SFA, fmt, m, kb, ld_a) * sfb_value(SFB, fmt, n, kb, nkb, ld_n) * partial;
    }
    return acc;
}

/* Dense FP8 NT GEMM, D is M x N row-major double. */
void fgo_gemm_fp8(const uint8_t *Aq, const void *SFA, const uint8_t *Bq, const void *SFB,
                  long M, long N, long K, int fmt, double *D)
{
    long m;
    long ld_a = fgo_align4(M);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (m = 0; m < M; ++m) {
        long n;
        for (n = 0; n < N; ++n)
            D[m * N + n] = dot_fp8(Aq + m * K, Bq + n * K, K, SFA, ld_a, m, SFB, n, N, fmt);
    }
}

/* Selected entries (rows[i], cols[i]) of the dense FP8 GEMM. */
void fgo_gemm_fp8_entries(const uint8_t *Aq, const void *SFA, const uint8_t *Bq, const void *SFB,
                          long M, long N, long K, int fmt,
                          const long *rows, const long *cols, long count, double *out)
{
    long i;
    long ld_a = fgo_align4(M);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (i = 0; i < count; ++i)
        out[i] = dot_fp8(Aq + rows[i] * K, Bq + cols[i] * K, K, SFA, ld_a, rows[i], SFB, cols[i], N, fmt);
}

/*
 * Grouped GEMM, contiguous layout ([DG] "two grouped layouts": tokens of one
 * expert concatenated along M; N and K shared by all experts).
 *   Aq : M x K (all segments), SFA over the M rows.
 *   Bq : G x N x K, SFB per expert (layout as fgo_quantize_128x128).
 *   m_indices[m] : expert of row m, or -1 for a padding row.
 * Rows with m_indices = -1 are left untouched in D (valid[m*N+n] = 0).
 */
void fgo_grouped_contiguous(const uint8_t *Aq, const void *SFA, const uint8_t *Bq, const void *SFB,
                            const int32_t *m_indices, long M, long N, long K, long G, int fmt,
                            double *D, uint8_t *valid)
{
    long m;
    long ld_a = fgo_align4(M);
    size_t sfb_bytes = sfb_group_bytes(fmt, N, K);
    (void)G;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (m = 0; m < M; ++m) {
        long n, g = m_indices[m];
        for (n = 0; n < N; ++n) {
            if (g < 0) {
                valid[m * N + n] = 0;
                continue;
            }
            valid[m * N + n] = 1;
            D[m * N + n] = dot_fp8(Aq + m * K, Bq + ((size_t)g * N + n) * K, K, SFA, ld_a, m,
                                   (const uint8_t *)SFB + (size_t)g * sfb_bytes, n, N, fmt);
        }
    }
}

/*
 * Grouped GEMM, masked layout ([DG] "two grouped layouts": each expert owns a
 * fixed slot of Mmax rows; a mask says how many are valid; only valid rows are
 * computed).
 *   Aq : G x Mmax x K, SFA : per expert a table over Mmax rows.
 *   Bq : G x N x K, SFB per expert.
 *   masked_m[g] : valid rows of expert g (0..Mmax).
 * D is G x Mmax x N; rows >= masked_m[g] are marked invalid.
 */
void fgo_grouped_masked(const uint8_t *Aq, const void *SFA, const uint8_t *Bq, const void *SFB,
                        const int32_t *masked_m, long G, long Mmax, long N, long K, int fmt,
                        double *D, uint8_t *valid)
{
    long g;
    size_t sfa_bytes = sfa_table_bytes(fmt, Mmax, K);
    size_t sfb_bytes = sfb_group_bytes(fmt, N, K);
    long ld_a = fgo_align4(Mmax);
    for (g = 0; g < G; ++g) {
        long m;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (m = 0; m < Mmax; ++m) {
            long n;
            size_t row = (size_t)g * Mmax + m;
            for (n = 0; n < N; ++n) {
                if (m >= masked_m[g]) {
                    valid[row * N + n] = 0;
                    continue;
                }
                valid[row * N + n] = 1;
                D[row * N + n] = dot_fp8(Aq + row * K, Bq + ((size_t)g * N + n) * K, K,
                                         (const uint8_t *)SFA + (size_t)g * sfa_bytes, ld_a, m,
                                         (const uint8_t *)SFB + (size_t)g * sfb_bytes, n, N, fmt);
            }
        }
    }
}

/*
 * Dense 16-bit NT GEMM in double: D[m,n] = sum_k A[m,k] * B[n,k].  The
 * operands are fp16 or bf16 values widened to float (exact).  [TIRx] Step 7
 * computes this product with FP32 accumulation; the oracle uses the exact sum.
 */
void fgo_gemm_f16(const float *A, const float *B, long M, long N, long K, double *D)
{
    long m;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (m = 0; m < M; ++m) {
        long n, k;
        for (n = 0; n < N; ++n) {
            double acc = 0.0;
            for (k = 0; k < K; ++k)
                acc += (double)A[m * K + k] * (double)B[n * K + k];
            D[m * N + n] = acc;
        }
    }
}

/* Selected entries of the 16-bit GEMM. */
void fgo_gemm_f16_entries(const float *A, const float *B, long M, long N, long K,
                          const long *rows, const long *cols, long count, double *out)
{
    long i;
    (void)M; (void)N;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (i = 0; i < count; ++i) {
        long k;
        double acc = 0.0;
        for (k = 0; k < K; ++k)
            acc += (double)A[rows[i] * K + k] * (double)B[cols[i] * K + k];
        out[i] = acc;
    }
}

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int fgo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void fgo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ========================================================================= */
/* 4-bit block-scaled formats: MXFP4 and NVFP4                               */
/* [TC5] section 6.1 (the block-scaled GEMM: every SV consecutive K elements */
/* of a row share one low-precision scale), 6.3 (MXFP4: E2M1 elements, E8M0  */
/* scale per 32; NVFP4: E2M1 elements, E4M3 scale per 16) and 7.1 (two 4-bit */
/* elements per byte, packed along K).                                        */
/* ========================================================================= */

#define FGO_FP4_MX 0   /* E2M1 + E8M0 scale per 32 elements along K */
#define FGO_FP4_NV 1   /* E2M1 + E4M3 scale per 16 elements along K */

/*
 * E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no infinity or NaN
 * ([TC5] section 3.5 lists e2m1 among the 4-bit element types).  Exponent
 * field 0: subnormal m * 2^-1; otherwise (1 + m/2) * 2^(e-1).  Largest 6.
 */
double fgo_e2m1_decode(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return sign ? -v : v;
}

/* Code (0..7) of a non-negative value that lies on the E2M1 grid. */
static uint8_t e2m1_code_of_grid_value(double r)
{
    int ex;
    double f;
    if (r < 1.0)
        return (uint8_t)(r * 2.0);                  /* 0 -> 0, 0.5 -> 1 */
    f = frexp(r, &ex);                              /* r = f * 2^ex, f in [0.5, 1) */
    /* r = (1 + m/2) * 2^(ex-1): exponent field ex - 1 + 1, m = (2f - 1) * 2 */
    return (uint8_t)((ex << 1) | (int)((2.0 * f - 1.0) * 2.0));
}

/*
 * Round a real value to E2M1: nearest, ties to even, finite magnitudes above 6
 * saturate to +-6, the sign of zero is kept (the same rounding reading as the
 * E4M3 encoder above).  The grid spacing near |v| is a power of two (0.5 below
 * 2, then 1, then 2), so |v| / spacing is exact and nearbyint() does the only
 * rounding.  Returns a 4-bit code.
 */
uint8_t fgo_e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v), spacing;
    if (isnan(v))
        return (uint8_t)(sign | 0x7);   /* no NaN in E2M1: the method never feeds one */
    if (a >= 6.0)
        return (uint8_t)(sign | 0x7);
    spacing = (a < 2.0) ? 0.5 : (a < 4.0) ? 1.0 : 2.0;
    return (uint8_t)(sign | e2m1_code_of_grid_value(nearbyint(a / spacing) * spacing));
}

void fgo_e2m1_encode_array(const double *x, uint8_t *q, long n)
{
    long i;
    for (i = 0; i < n; ++i)
        q[i] = fgo_e2m1_encode(x[i]);
}

void fgo_e2m1_decode_array(const uint8_t *q, double *out, long n)
{
    long i;
    for (i = 0; i < n; ++i)
        out[i] = fgo_e2m1_decode(q[i]);
}

/* Elements per scale along K. */
static long fp4_vec(int fmt) { return fmt == FGO_FP4_MX ? 32 : 16; }

/*
 * Scale byte of one group from its max |x| (FP32, the precision the kernel
 * decides codes in).
 *   MXFP4: the power of two 2^e with e = ceil(log2(amax / 6)) (FP32 quotient),
 *          clamped to [-127, 127], stored as the E8M0 byte e + 127 -- the same
 *          reading as the FP8 path's UE8M0 scales (rounding up: nothing
 *          saturates); amax = 0 gives byte 127 (scale 1).
 *   NVFP4: the E4M3 code of amax / 6 (FP32 quotient; nearest even, saturating
 *          at 448); amax = 0 gives the code of 1.0.
 */
static uint8_t fp4_scale_byte(float amax, int fmt)
{
    volatile float num = amax;
    float t;
    if (amax == 0.0f)
        return (uint8_t)(fmt == FGO_FP4_MX ? 127 : fgo_e4m3_encode(1.0));
    t = num / 6.0f;
    if (fmt == FGO_FP4_MX) {
        int ex, e;
        double f = frexp((double)t, &ex);
        e = (f == 0.5) ? ex - 1 : ex;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
        return (uint8_t)(e + 127);
    }
    return fgo_e4m3_encode((double)t);
}

/* Value of a scale byte. */
double fgo_fp4_scale_value(uint8_t b, int fmt)
{
    return fmt == FGO_FP4_MX ? ldexp(1.0, (int)b - 127) : fgo_e4m3_decode(b);
}

/*
 * 1 x SV block quantization of the rows of X (activations or weights alike:
 * the scale groups run along K for both operands, [TC5] section 6.1).
 *   X  : R x K values (bf16 values widened to float), row-major.
 *   Xq : R x K/2 bytes, row-major; byte j of a row holds element 2j in its low
 *        nibble and element 2j+1 in its high nibble ([TC5] section 7.1: two
 *        4-bit elements per byte along K).
 *   SF : uint8 view of int32[ceil(K/SV/4)][align4(R)]; byte j of word (w, r) is
 *        the scale of group 4w+j of row r; unused bytes and rows are 0.
 * The element code is E2M1(x * 2^-e) (exact scaling) for MXFP4 and
 * E2M1(x / s) with an FP32 division by the decoded E4M3 scale for NVFP4; a
 * group whose E4M3 scale is 0 (amax / 6 below the smallest subnormal) has
 * zero codes.  K must be a multiple of 64.
 */
void fgo_quantize_fp4(const float *X, long R, long K, int fmt, uint8_t *Xq, void *SF)
{
    long sv = fp4_vec(fmt), ng = K / sv, nw = (ng + 3) / 4, ld = fgo_align4(R), r;
    uint8_t *sf = (uint8_t *)SF;
    memset(SF, 0, (size_t)nw * (size_t)ld * 4u);
    memset(Xq, 0, (size_t)R * (size_t)(K / 2));
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (r = 0; r < R; ++r) {
        long g, k;
        for (g = 0; g < ng; ++g) {
            const float *x = X + r * K + g * sv;
            float amax = 0.0f;
            uint8_t b;
            double s;
            for (k = 0; k < sv; ++k) {
                float a = fabsf(x[k]);
                if (a > amax) amax = a;
            }
            b = fp4_scale_byte(amax, fmt);
            s = fgo_fp4_scale_value(b, fmt);
            sf[((size_t)(g / 4) * (size_t)ld + (size_t)r) * 4u + (size_t)(g % 4)] = b;
            for (k = 0; k < sv; ++k) {
                uint8_t c;
                if (fmt == FGO_FP4_MX) {
                    c = fgo_e2m1_encode(ldexp((double)x[k], 127 - (int)b));
                } else if (s == 0.0) {
                    c = 0;
                } else {
                    volatile float xv = x[k];
                    volatile float sv32 = (float)s;
                    float qv = xv / sv32;
                    c = fgo_e2m1_encode((double)qv);
                }
                {
                    long col = g * sv + k;
                    uint8_t *byte = Xq + r * (K / 2) + col / 2;
                    *byte = (uint8_t)(*byte | (col % 2 ? (uint8_t)(c << 4) : c));
                }
            }
        }
    }
}

/*
 * The block-scaled 4-bit NT GEMM, term by term as [TC5] section 6.1 writes it:
 *   D[i][j] = sum_k (A[i][k] * SFA[i][k/SV]) * (B[j][k] * SFB[j][k/SV])
 * in double.  Aq (M x K/2) and Bq (N x K/2) are packed as fgo_quantize_fp4
 * writes them, SFA / SFB in its scale layout.  D is M x N row-major.
 */
void fgo_gemm_fp4(const uint8_t *Aq, const void *SFA, const uint8_t *Bq, const void *SFB,
                  long M, long N, long K, int fmt, double *D)
{
    long sv = fp4_vec(fmt), lda = fgo_align4(M), ldb = fgo_align4(N), i;
    const uint8_t *sa = (const uint8_t *)SFA, *sb = (const uint8_t *)SFB;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (i = 0; i < M; ++i) {
        long j, k;
        for (j = 0; j < N; ++j) {
            double acc = 0.0;
            for (k = 0; k < K; ++k) {
                long g = k / sv;
                uint8_t ca = (uint8_t)((Aq[i * (K / 2) + k / 2] >> (4 * (k % 2))) & 0xF);
                uint8_t cb = (uint8_t)((Bq[j * (K / 2) + k / 2] >> (4 * (k % 2))) & 0xF);
                double a = fgo_e2m1_decode(ca) *
                           fgo_fp4_scale_value(sa[((size_t)(g / 4) * (size_t)lda + (size_t)i) * 4u + (size_t)(g % 4)], fmt);
                double b = fgo_e2m1_decode(cb) *
                           fgo_fp4_scale_value(sb[((size_t)(g / 4) * (size_t)ldb + (size_t)j) * 4u + (size_t)(g % 4)], fmt);
                acc += a * b;
            }
            D[i * N + j] = acc;
        }
    }
}
