/*
 * oracle.c -- plain, slow, fp64 CPU reference for the W4A16 skinny GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA library under bf16_activation_quantized_gb300/csrc.
 *
 * What it computes (definitions, not an algorithm):
 *
 *   Y[m][n] = sum_k X[m][k] * Wd[n][k]                       (fp64 throughout)
 *   Wd[n][k] = scale[n][k / G] * (nib(n, k) - 8)
 *
 * Sources (page title, then the passage):
 *  - "[ROCm][Kernel] W4A16 skinny GEMM: hand-asm kernel for gfx1151", opening
 *    paragraph: the op is an int4-weight / bf16-activation skinny GEMM with
 *    N x K weights; "Benchmark results (per-GEMM)": group-wise symmetric
 *    quantisation; section 1 "Magic-constant bf16 dequant": each weight is
 *    scale * (n - 8) for a 4-bit code n.
 *  - "Add Triton BF16xINT4 rowwise GEMM for ROCm gfx942/gfx950", section
 *    "Implementation", paragraph "Fused A-operand dot": the low nibble of a
 *    byte pairs with the even K column and the high nibble with the odd one.
 *    Paragraph "Native fused grouped kernel": group g's rows start at
 *    M_starts[g] = cumsum(M_sizes)[g] - M_sizes[g].
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *  - W orientation: row n of the packed weight is output feature n, Y = X W^T.
 *  - A negative M_sizes entry counts as 0; rows past M_total are dropped; rows
 *    of Y that no group covers are left untouched.
 *  - bf16 -> fp64 is exact; fp64 -> bf16 is round-to-nearest-even, used only
 *    for the bf16 weight probe, whose fp64 product is exact before rounding.
 *
 * Parallelism: OpenMP over output elements only; each element's k loop runs
 * serially in ascending k, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE binary32: widen and reinterpret. */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16 (ties to even), directly from fp64
 * (no detour through binary32, so there is a single rounding).  bf16 has 8
 * significant bits and binary32's exponent range: normal values with
 * exponent e have a quantum of 2^(e-7), subnormals a quantum of 2^-133. */
uint16_t oracle_f64_to_bf16(double v)
{
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);           /* a = f * 2^e, f in [0.5, 1): leading bit 2^(e-1) */
    int lead = e - 1;
    if (lead < -126) lead = -126;             /* subnormal range */
    double quantum = ldexp(1.0, lead - 7);
    double q = a / quantum;                   /* exact: a power-of-two division */
    double r = nearbyint(q);                  /* default mode: ties to even */
    double rounded = r * quantum;
    if (rounded >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)rounded;                 /* exact: rounded is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* The 4-bit code of weight (n, k) in the canonical packing: row n holds K/2
 * bytes; byte j carries k = 2j in bits 0-3 and k = 2j+1 in bits 4-7. */
int oracle_nibble(const uint8_t *w_canon, long K, long n, long k)
{
    uint8_t byte = w_canon[n * (K / 2) + k / 2];
    return (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

/* One dequantised weight, exactly, in fp64. */
double oracle_weight(const uint8_t *w_canon, const uint16_t *scales, long K, long G,
                     long n, long k)
{
    double s = oracle_bf16_to_f64(scales[n * (K / G) + k / G]);
    return s * (double)(oracle_nibble(w_canon, K, n, k) - 8);
}

/* Dense dequantised weight matrix Wd[N][K] in fp64. */
void oracle_dequant_f64(const uint8_t *w_canon, const uint16_t *scales, long N, long K,
                        long G, double *out)
{
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            out[n * K + k] = oracle_weight(w_canon, scales, K, G, n, k);
}

/* The same weights as binary32.  The product of an 8-bit bf16 significand and
 * a 4-bit integer fits binary32's 24 bits, so this conversion is exact. */
void oracle_dequant_f32(const uint8_t *w_canon, const uint16_t *scales, long N, long K,
                        long G, float *out)
{
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            out[n * K + k] = (float)oracle_weight(w_canon, scales, K, G, n, k);
}

/* The weights rounded once to bf16 (nearest, ties to even): the operand a
 * bf16 tensor-core product consumes when the scale is folded in first. */
void oracle_dequant_bf16(const uint8_t *w_canon, const uint16_t *scales, long N, long K,
                         long G, uint16_t *out)
{
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            out[n * K + k] = oracle_f64_to_bf16(oracle_weight(w_canon, scales, K, G, n, k));
}

static void set_threads(int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

/* Y[m][n] for m in [0, M), n in [0, N), straight from the definition.
 * x: bf16 bits [M][K]; y: fp64 [M][N]. */
void oracle_gemm_f64(const uint16_t *x, const uint8_t *w_canon, const uint16_t *scales,
                     long M, long N, long K, long G, double *y, int threads)
{
    set_threads(threads);
    #pragma omp parallel for collapse(2) schedule(static)
    for (long m = 0; m < M; ++m) {
        for (long n = 0; n < N; ++n) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(x[m * K + k]) *
                       oracle_weight(w_canon, scales, K, G, n, k);
            y[m * N + n] = acc;
        }
    }
}

/* Only the output columns [n_lo, n_hi): a bounded sample of a large product,
 * used to time the reference on a slice of a workload.  y is [M][N]. */
void oracle_gemm_cols_f64(const uint16_t *x, const uint8_t *w_canon, const uint16_t *scales,
                          long M, long N, long K, long G, long n_lo, long n_hi, double *y,
                          int threads)
{
    set_threads(threads);
    #pragma omp parallel for collapse(2) schedule(static)
    for (long m = 0; m < M; ++m) {
        for (long n = n_lo; n < n_hi; ++n) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(x[m * K + k]) *
                       oracle_weight(w_canon, scales, K, G, n, k);
            y[m * N + n] = acc;
        }
    }
}

/* ---- Asymmetric variant (zero points) -------------------------------------
 * The pages state only the symmetric form, scale * (n - 8).  The variant with
 * a zero point per scale group is a reading (listed in the design notes): the
 * usual int4 convention of a 4-bit integer zero z per (row, group),
 *
 *   Wd[n][k] = scale[n][k / G] * (nib(n, k) - z[n][k / G]),
 *
 * z held in the low four bits of one byte per group (zeros: uint8 [N][K/G]).
 * With every z = 8 it is the symmetric form. */
double oracle_weight_zp(const uint8_t *w_canon, const uint16_t *scales, const uint8_t *zeros,
                        long K, long G, long n, long k)
{
    long gi = n * (K / G) + k / G;
    double s = oracle_bf16_to_f64(scales[gi]);
    return s * (double)(oracle_nibble(w_canon, K, n, k) - (int)(zeros[gi] & 0x0F));
}

void oracle_dequant_zp_f32(const uint8_t *w_canon, const uint16_t *scales, const uint8_t *zeros,
                           long N, long K, long G, float *out)
{
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            out[n * K + k] = (float)oracle_weight_zp(w_canon, scales, zeros, K, G, n, k);
}

void oracle_dequant_zp_bf16(const uint8_t *w_canon, const uint16_t *scales, const uint8_t *zeros,
                            long N, long K, long G, uint16_t *out)
{
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            out[n * K + k] = oracle_f64_to_bf16(oracle_weight_zp(w_canon, scales, zeros, K, G, n, k));
}

void oracle_gemm_zp_f64(const uint16_t *x, const uint8_t *w_canon, const uint16_t *scales,
                        const uint8_t *zeros, long M, long N, long K, long G, double *y,
                        int threads)
{
    set_threads(threads);
    #pragma omp parallel for collapse(2) schedule(static)
    for (long m = 0; m < M; ++m) {
        for (long n = 0; n < N; ++n) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(x[m * K + k]) *
                       oracle_weight_zp(w_canon, scales, zeros, K, G, n, k);
            y[m * N + n] = acc;
        }
    }
}

/* Row starts of each group: the exclusive prefix sum of the (clamped) sizes. */
void oracle_group_starts(const int32_t *m_sizes, long num_groups, int64_t *starts)
{
    int64_t run = 0;
    for (long g = 0; g < num_groups; ++g) {
        starts[g] = run;
        run += m_sizes[g] > 0 ? m_sizes[g] : 0;
    }
}

/* Grouped product: group g owns X/Y rows [start_g, start_g + M_sizes[g]) and
 * uses weight block g (w_canon + g*N*K/2) and scale block g
 * (scales + g*N*(K/G)).  Rows at or past M_total are not computed. */
void oracle_gemm_grouped_f64(const uint16_t *x, const uint8_t *w_canon,
                             const uint16_t *scales, const int32_t *m_sizes,
                             long num_groups, long M_total, long N, long K, long G,
                             double *y, int threads)
{
    set_threads(threads);
    int64_t start = 0;
    for (long g = 0; g < num_groups; ++g) {
        long rows = m_sizes[g] > 0 ? m_sizes[g] : 0;
        long lo = start, hi = start + rows;
        if (hi > M_total) hi = M_total;
        const uint8_t *wg = w_canon + (size_t)g * (size_t)N * (size_t)(K / 2);
        const uint16_t *sg = scales + (size_t)g * (size_t)N * (size_t)(K / G);
        #pragma omp parallel for collapse(2) schedule(static)
        for (long m = lo; m < hi; ++m) {
            for (long n = 0; n < N; ++n) {
                double acc = 0.0;
                for (long k = 0; k < K; ++k)
                    acc += oracle_bf16_to_f64(x[m * K + k]) *
                           oracle_weight(wg, sg, K, G, n, k);
                y[m * N + n] = acc;
            }
        }
        start += rows;
    }
}

/* Element-wise sum of split-K slices in ascending slice order: the
 * reference for a partial-sum reduction, ws is [splits][count]. */
void oracle_sum_slices_f64(const float *ws, long splits, long count, double *out)
{
    for (long i = 0; i < count; ++i) {
        double acc = 0.0;
        for (long s = 0; s < splits; ++s) acc += (double)ws[s * count + i];
        out[i] = acc;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
