/*
 * fp8_oracle.c -- plain CPU restatement of the FP8 linear-layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load it; the product path never calls it.  It
 * shares no source, header, table or helper with the CUDA library.
 *
 * What it computes, and where that comes from:
 *
 *  - FP8 formats e4m3fn (max 448), e5m2 (max 57344), e4m3fnuz (max 240) and
 *    e5m2fnuz (max 57344); the two fnuz formats have one NaN code (0x80), no
 *    infinities and no negative zero, and an exponent bias one above their fn
 *    counterparts.  The maxima and the fnuz conventions are stated on "FP8
 *    Training on MI300X" (section "Discovered AMD FP8 dtype difference", which
 *    also names float8_e5m2fnuz as AMD's backward format) and on "FP8 Training
 *    on AMD GPUs with TorchTitan and TorchAO" (the question "Why does FP8
 *    training on AMD GPUs give silently wrong results ...").  The bit layouts
 *    (sign, exponent, mantissa, bias) are the public OCP 8-bit float
 *    definitions.
 *  - The scaling recipe knobs (format, recipe, margin, amax history length,
 *    amax compute algorithm) are the ones listed on "FP8 training for Flux
 *    models" (section Configuration > Key FP8 Parameters).  The scale formula
 *    is scale = fp8_max / amax / 2^margin; the quantised value is
 *    sat_rne_fp8(fp32(x) * scale) and the dequantisation multiplier is
 *    scale_inv = 1 / scale.
 *  - Forward tensors in E4M3 and gradients in E5M2 ("hybrid") follow "FP8
 *    Training on MI300X" (section "Patched nanochat/fp8.py").
 *  - Rowwise scales and colwise scales with a transposed layout follow "How
 *    PyTorch FP8 Optimizations on AMD GPUs ..." (section What Happened) and
 *    the TorchTitan/TorchAO post (the colwise-scales kernel).
 *  - The grouped GEMM over expert groups follows the same two pages (grouped
 *    GEMM for Mixture-of-Experts).
 *
 * Readings where the pages are silent (each is repeated in the design notes):
 *  - NaN input encodes to the format's NaN code; |x| above the format maximum
 *    (or +-Inf) saturates to +-max; ties round to the even code.
 *  - Current scaling: amax == 0 or non-finite gives scale 1; a scale that
 *    overflows fp32 becomes FLT_MAX.
 *  - Delayed update: a non-finite or zero window amax keeps the previous
 *    scale; a non-finite one also bumps a per-tensor counter.  The history
 *    row is shifted one slot towards the end (oldest dropped) and slot 0,
 *    which collects the current step's amax, is zeroed.
 *  - Grouped colwise layout: group e's columns start at the padded offset
 *    sum_{e'<e} roundup(m_e', 32); padding bytes are zero.
 *
 * Arithmetic: scalar C, fp32 where the method is fp32 (the x*scale product,
 * the scale divide), exact double for the FP8 rounding decision and for the
 * dequantised GEMM.  Compile with -ffp-contract=off (no fused multiply-add).
 * OpenMP only distributes independent outer iterations; every result is
 * independent of the thread count.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads for the parallel outer loops (the timed baseline also runs on one
 * core); no effect on any result: every loop iteration is independent. */
void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

#define ORC_E4M3FN 0
#define ORC_E5M2 1
#define ORC_E4M3FNUZ 2
#define ORC_E5M2FNUZ 3
#define ORC_NUM_FMT 4

#define ORC_DELAYED 0
#define ORC_TENSORWISE 1
#define ORC_ROWWISE 2

#define ORC_MOST_RECENT 0
#define ORC_MAX 1

#define ORC_LAYOUT_ROW 1
#define ORC_LAYOUT_COLT 2

/* ------------------------------------------------------------------------ */
/* FP8 codec                                                                 */
/* ------------------------------------------------------------------------ */

static int fmt_is_fnuz(int fmt) { return fmt == ORC_E4M3FNUZ || fmt == ORC_E5M2FNUZ; }
static int fmt_exp_bits(int fmt) { return (fmt == ORC_E5M2 || fmt == ORC_E5M2FNUZ) ? 5 : 4; }
static int fmt_man_bits(int fmt) { return (fmt == ORC_E5M2 || fmt == ORC_E5M2FNUZ) ? 2 : 3; }
static int fmt_bias(int fmt)
{
    if (fmt == ORC_E5M2) return 15;
    if (fmt == ORC_E5M2FNUZ) return 16;
    if (fmt == ORC_E4M3FNUZ) return 8;
    return 7;
}

/* Largest finite positive code of each format. */
int orc_fp8_max_code(int fmt)
{
    if (fmt == ORC_E5M2) return 0x7B;     /* 0 11110 11 = 1.75 * 2^15 */
    if (fmt == ORC_E4M3FNUZ) return 0x7F; /* 0 1111 111 = 1.875 * 2^7 (bias 8) */
    if (fmt == ORC_E5M2FNUZ) return 0x7F; /* 0 11111 11 = 1.75 * 2^15 (bias 16) */
    return 0x7E;                          /* 0 1111 110 = 1.75 * 2^8 */
}

int orc_fp8_nan_code(int fmt)
{
    if (fmt == ORC_E5M2) return 0x7E;
    if (fmt_is_fnuz(fmt)) return 0x80;
    return 0x7F;
}

/* Exact value of an 8-bit code, from the sign / exponent / mantissa fields. */
double orc_fp8_decode(int code, int fmt)
{
    int eb = fmt_exp_bits(fmt), mb = fmt_man_bits(fmt), bias = fmt_bias(fmt);
    int sign = (code >> 7) & 1;
    int e = (code >> mb) & ((1 << eb) - 1);
    int m = code & ((1 << mb) - 1);
    double mag;

    if (fmt_is_fnuz(fmt)) {
        if (code == 0x80) return NAN; /* the only NaN; there is no -0 */
    } else if (fmt == ORC_E4M3FN) {
        if (e == 15 && m == 7) return NAN; /* 0x7F / 0xFF */
    } else {                               /* e5m2: IEEE-style top exponent */
        if (e == 31) {
            if (m != 0) return NAN;
            return sign ? -INFINITY : INFINITY;
        }
    }
    if (e == 0) /* subnormal: m * 2^(1 - bias - mb) */
        mag = ldexp((double)m, 1 - bias - mb);
    else /* normal: (2^mb + m) * 2^(e - bias - mb) */
        mag = ldexp((double)((1 << mb) + m), e - bias - mb);
    return sign ? -mag : mag;
}

/* Magnitudes of codes 0 .. max_code, strictly increasing with the code. */
static double g_mag[ORC_NUM_FMT][128];
static int g_mag_ready = 0;

static void init_tables(void)
{
    if (g_mag_ready) return;
    for (int f = 0; f < ORC_NUM_FMT; f++)
        for (int c = 0; c <= orc_fp8_max_code(f); c++) g_mag[f][c] = orc_fp8_decode(c, f);
    g_mag_ready = 1;
}

/*
 * Round v to the nearest FP8 value, ties to the even code (= even mantissa),
 * saturating to +-max (a saturating cast: anything above max, or +-Inf, maps
 * to +-max).  v is an fp32 value carried exactly in a double, so every
 * comparison below is exact.
 */
int orc_fp8_encode(double v, int fmt)
{
    int top = orc_fp8_max_code(fmt);
    int neg, lo, hi, mag;
    double a;

    init_tables();
    if (isnan(v)) return orc_fp8_nan_code(fmt);
    neg = signbit(v) ? 1 : 0;
    a = fabs(v);
    if (a >= g_mag[fmt][top]) {
        mag = top;
    } else {
        /* bracket a: g_mag[lo] <= a < g_mag[hi], hi = lo + 1 */
        lo = 0;
        hi = top;
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (g_mag[fmt][mid] <= a)
                lo = mid;
            else
                hi = mid;
        }
        {
            double dlo = a - g_mag[fmt][lo], dhi = g_mag[fmt][hi] - a;
            if (dlo < dhi)
                mag = lo;
            else if (dhi < dlo)
                mag = hi;
            else
                mag = (lo % 2 == 0) ? lo : hi;
        }
    }
    if (fmt_is_fnuz(fmt) && mag == 0) return 0x00; /* unsigned zero */
    return (neg << 7) | mag;
}

double orc_fp8_max_value(int fmt) { return orc_fp8_decode(orc_fp8_max_code(fmt), fmt); }

/* ------------------------------------------------------------------------ */
/* Scales                                                                    */
/* ------------------------------------------------------------------------ */

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* scale = fp8_max / amax, then * 2^-margin; overflow becomes FLT_MAX. */
static float scale_formula(float amax, int fmt, int margin)
{
    float fmax = (float)orc_fp8_max_value(fmt);
    float s = fmax / amax;
    s = s * ldexpf(1.0f, -margin);
    if (isinf(s)) s = FLT_MAX;
    return s;
}

/* Current scaling (tensorwise / rowwise / colwise). */
void orc_current_scale(float amax, int fmt, int margin, float *scale, float *scale_inv)
{
    float s;
    if (!(amax > 0.0f) || !isfinite(amax))
        s = 1.0f;
    else
        s = scale_formula(amax, fmt, margin);
    *scale = s;
    *scale_inv = 1.0f / s;
}

/* max with NaN propagation */
static float amax_acc(float acc, float v)
{
    float a = fabsf(v);
    if (isnan(acc) || isnan(a)) return NAN;
    return a > acc ? a : acc;
}

/* ------------------------------------------------------------------------ */
/* Quantize                                                                  */
/* ------------------------------------------------------------------------ */

float orc_amax_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x);

static int64_t roundup32(int64_t m) { return (m + 31) / 32 * 32; }

/* Padded column offsets of the grouped colwise layout; returns the total. */
int64_t orc_padded_offsets(const int32_t *off, int G, int64_t *poff)
{
    int64_t acc = 0;
    for (int e = 0; e < G; e++) {
        poff[e] = acc;
        acc += roundup32((int64_t)off[e + 1] - off[e]);
    }
    poff[G] = acc;
    return acc;
}

/*
 * Full quantize of a bf16 matrix x[rows][cols] (row stride ld_x elements).
 *
 * kind DELAYED   : cast with the stored scale scale_in[0]; both layouts share
 *                  it; scale_inv = 1/scale_in[0]; amax_io[0] = max(amax_io[0],
 *                  amax(x)) (the history slot of the current step).
 * kind TENSORWISE: scale from the whole tensor's amax (current scaling);
 *                  amax_io[0] (optional) receives that amax.
 * kind ROWWISE   : q_row uses one scale per row, q_colT one per column (per
 *                  group and column when offsets != NULL); amax_io[0]
 *                  (optional) receives the whole-tensor amax.
 *
 * q_row  : [rows][cols] bytes, scale_inv_row: [1] or [rows].
 * q_colT : [cols][ldT] bytes, ldT = rows (ungrouped) or the padded total
 *          (grouped); scale_inv_col: [1], [cols] or [G][cols].
 * offsets: NULL for an ungrouped tensor, else int32 [G+1] with offsets[0] = 0
 *          and offsets[G] = rows (the row range of each group).
 */
int orc_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt, int kind,
                 int margin, int layouts, const float *scale_in, float *amax_io, uint8_t *q_row,
                 float *scale_inv_row, uint8_t *q_colT, float *scale_inv_col,
                 const int32_t *offsets, int G)
{
    int ngroups = offsets ? G : 1;
    int64_t *poff = (int64_t *)malloc(sizeof(int64_t) * (ngroups + 1));
    int64_t ldT;
    float tensor_amax = 0.0f;

    init_tables();
    if (offsets) {
        ldT = orc_padded_offsets(offsets, G, poff);
    } else {
        poff[0] = 0;
        poff[1] = rows;
        ldT = rows;
    }

    /* whole-tensor amax */
    tensor_amax = orc_amax_bf16(x, rows, cols, ld_x);

    if (kind == ORC_DELAYED || kind == ORC_TENSORWISE) {
        float s, sinv;
        if (kind == ORC_DELAYED) {
            s = scale_in[0];
            sinv = 1.0f / s;
            if (amax_io) {
                float prev = amax_io[0];
                amax_io[0] = (isnan(prev) || isnan(tensor_amax)) ? NAN
                             : (tensor_amax > prev ? tensor_amax : prev);
            }
        } else {
            orc_current_scale(tensor_amax, fmt, margin, &s, &sinv);
            if (amax_io) amax_io[0] = tensor_amax;
        }
        if (layouts & ORC_LAYOUT_ROW) {
#pragma omp parallel for schedule(static)
            for (int64_t r = 0; r < rows; r++)
                for (int64_t c = 0; c < cols; c++) {
                    float p = bf16_to_float(x[r * ld_x + c]) * s;
                    q_row[r * cols + c] = (uint8_t)orc_fp8_encode((double)p, fmt);
                }
            scale_inv_row[0] = sinv;
        }
        if (layouts & ORC_LAYOUT_COLT) {
            memset(q_colT, 0, (size_t)(cols * ldT));
#pragma omp parallel for schedule(static)
            for (int64_t c = 0; c < cols; c++)
                for (int e = 0; e < ngroups; e++) {
                    int64_t r0 = offsets ? offsets[e] : 0, r1 = offsets ? offsets[e + 1] : rows;
                    for (int64_t r = r0; r < r1; r++) {
                        float p = bf16_to_float(x[r * ld_x + c]) * s;
                        q_colT[c * ldT + poff[e] + (r - r0)] = (uint8_t)orc_fp8_encode((double)p, fmt);
                    }
                }
            scale_inv_col[0] = sinv;
        }
    } else { /* ROWWISE (current scaling per row, per column / group column) */
        if (amax_io) amax_io[0] = tensor_amax;
        if (layouts & ORC_LAYOUT_ROW) {
#pragma omp parallel for schedule(static)
            for (int64_t r = 0; r < rows; r++) {
                float am = 0.0f, s, sinv;
                for (int64_t c = 0; c < cols; c++) am = amax_acc(am, bf16_to_float(x[r * ld_x + c]));
                orc_current_scale(am, fmt, margin, &s, &sinv);
                for (int64_t c = 0; c < cols; c++) {
                    float p = bf16_to_float(x[r * ld_x + c]) * s;
                    q_row[r * cols + c] = (uint8_t)orc_fp8_encode((double)p, fmt);
                }
                scale_inv_row[r] = sinv;
            }
        }
        if (layouts & ORC_LAYOUT_COLT) {
            memset(q_colT, 0, (size_t)(cols * ldT));
#pragma omp parallel for schedule(static)
            for (int64_t c = 0; c < cols; c++)
                for (int e = 0; e < ngroups; e++) {
                    int64_t r0 = offsets ? offsets[e] : 0, r1 = offsets ? offsets[e + 1] : rows;
                    float am = 0.0f, s, sinv;
                    for (int64_t r = r0; r < r1; r++) am = amax_acc(am, bf16_to_float(x[r * ld_x + c]));
                    orc_current_scale(am, fmt, margin, &s, &sinv);
                    for (int64_t r = r0; r < r1; r++) {
                        float p = bf16_to_float(x[r * ld_x + c]) * s;
                        q_colT[c * ldT + poff[e] + (r - r0)] = (uint8_t)orc_fp8_encode((double)p, fmt);
                    }
                    scale_inv_col[(int64_t)e * cols + c] = sinv;
                }
        }
    }
    free(poff);
    return 0;
}

/* Whole-tensor amax of a bf16 matrix (NaN propagates): per-row maxima in
 * parallel, then their maximum (max is independent of the order). */
float orc_amax_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x)
{
    float acc = 0.0f;
    float *rowmax = (float *)malloc(sizeof(float) * (rows > 0 ? rows : 1));
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        float m = 0.0f;
        for (int64_t c = 0; c < cols; c++) m = amax_acc(m, bf16_to_float(x[r * ld_x + c]));
        rowmax[r] = m;
    }
    for (int64_t r = 0; r < rows; r++) acc = (isnan(acc) || isnan(rowmax[r])) ? NAN : (rowmax[r] > acc ? rowmax[r] : acc);
    free(rowmax);
    return acc;
}

/*
 * Encode selected elements only: out[i] = encode(fp32(x[i]) * scale[i]).
 * Lets tests check sampled bytes of full-size tensors one element at a time.
 */
void orc_cast_points(const uint16_t *xv, const float *scale, int64_t n, int fmt, uint8_t *out)
{
    init_tables();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        float p = bf16_to_float(xv[i]) * scale[i];
        out[i] = (uint8_t)orc_fp8_encode((double)p, fmt);
    }
}

/* ------------------------------------------------------------------------ */
/* Amax history and the delayed scale update                                 */
/* ------------------------------------------------------------------------ */

void orc_update_amax_history(float *hist, float *scale, float *scale_inv, const uint8_t *fmt, int n,
                             int L, int algo, int margin, int32_t *nonfinite_count)
{
    init_tables();
    for (int i = 0; i < n; i++) {
        float *H = hist + (int64_t)i * L;
        float a = H[0];
        if (algo == ORC_MAX)
            for (int j = 1; j < L; j++) {
                if (isnan(a) || isnan(H[j]))
                    a = NAN;
                else if (H[j] > a)
                    a = H[j];
            }
        if (isfinite(a) && a > 0.0f) {
            float s = scale_formula(a, fmt[i], margin);
            scale[i] = s;
            scale_inv[i] = 1.0f / s;
        } else if (!isfinite(a) && nonfinite_count) {
            nonfinite_count[i] += 1;
        }
        for (int j = L - 1; j >= 1; j--) H[j] = H[j - 1];
        H[0] = 0.0f;
    }
}

/* ------------------------------------------------------------------------ */
/* Dequantised GEMM in double                                                */
/* ------------------------------------------------------------------------ */

/*
 * C[m][n] = sum_k dec(A[m][k]) * dec(B[n][k]) * sa(m) * sb(n), A and B both
 * K-contiguous ("TN").  sa_mode/sb_mode: 0 = one scale, 1 = one per row of
 * the operand.  bound[m][n] = the same sum of absolute values.
 * pm/pn: if non-NULL, only the npts points (pm[i], pn[i]) are computed and
 * written to ref[i], bound[i]; else the full M x N result, row-major.
 */
void orc_gemm(const uint8_t *A, int fa, int64_t lda, const uint8_t *B, int fb, int64_t ldb, int64_t M,
              int64_t N, int64_t K, const float *sa, int sa_mode, const float *sb, int sb_mode,
              const int64_t *pm, const int64_t *pn, int64_t npts, double *ref, double *bound)
{
    double da[256], db[256];
    int64_t total = pm ? npts : M * N;
    for (int c = 0; c < 256; c++) {
        da[c] = orc_fp8_decode(c, fa);
        db[c] = orc_fp8_decode(c, fb);
    }
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < total; i++) {
        int64_t m = pm ? pm[i] : i / N, n = pm ? pn[i] : i % N;
        const uint8_t *a = A + m * lda, *b = B + n * ldb;
        double s = 0.0, t = 0.0, scl;
        for (int64_t k = 0; k < K; k++) {
            double p = da[a[k]] * db[b[k]];
            s += p;
            t += fabs(p);
        }
        scl = (double)sa[sa_mode ? m : 0] * (double)sb[sb_mode ? n : 0];
        ref[i] = s * scl;
        bound[i] = t * fabs(scl);
    }
}

/*
 * Grouped GEMM over expert groups; offsets int32 [G+1] (row ranges).
 *
 * mode 0 (M_GROUPED): A [M_total][K] rows of all groups, B [G][N][K];
 *   C[m][n] = sum_k A[m][k] B[e(m)][n][k] sa(m) sb(e(m), n), with
 *   sa_mode 1 -> sa[m], sb_mode 1 -> sb[e*N + n] (0 -> scalar).
 *   Points: (pm[i], pn[i]); pg ignored.
 * mode 1 (K_GROUPED): A [N][ldT], B [K][ldT] in the padded grouped colwise
 *   layout; C[e][n][k] = sum_{r < m_e} A[n][poff_e + r] B[k][poff_e + r]
 *   sa(e, n) sb(e, k); an empty group gives 0.  sa_mode 1 -> sa[e*N + n],
 *   sb_mode 1 -> sb[e*K + k].  Points: (pg[i], pm[i] = n, pn[i] = k).
 */
void orc_grouped_gemm(int mode, const uint8_t *A, int fa, const uint8_t *B, int fb, const int32_t *offsets,
                      int G, int64_t M_total, int64_t N, int64_t K, const float *sa, int sa_mode,
                      const float *sb, int sb_mode, const int64_t *pg, const int64_t *pm,
                      const int64_t *pn, int64_t npts, double *ref, double *bound)
{
    double da[256], db[256];
    int64_t *poff = (int64_t *)malloc(sizeof(int64_t) * (G + 1));
    int64_t ldT = orc_padded_offsets(offsets, G, poff);
    (void)M_total;
    for (int c = 0; c < 256; c++) {
        da[c] = orc_fp8_decode(c, fa);
        db[c] = orc_fp8_decode(c, fb);
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < npts; i++) {
        double s = 0.0, t = 0.0, scl;
        if (mode == 0) {
            int64_t m = pm[i], n = pn[i];
            int e = 0;
            while (e < G - 1 && m >= offsets[e + 1]) e++;
            const uint8_t *a = A + m * K, *b = B + ((int64_t)e * N + n) * K;
            for (int64_t k = 0; k < K; k++) {
                double p = da[a[k]] * db[b[k]];
                s += p;
                t += fabs(p);
            }
            scl = (double)sa[sa_mode ? m : 0] * (double)sb[sb_mode ? (int64_t)e * N + n : 0];
        } else {
            int64_t e = pg[i], n = pm[i], k = pn[i];
            int64_t me = (int64_t)offsets[e + 1] - offsets[e];
            const uint8_t *a = A + n * ldT + poff[e], *b = B + k * ldT + poff[e];
            for (int64_t r = 0; r < me; r++) {
                double p = da[a[r]] * db[b[r]];
                s += p;
                t += fabs(p);
            }
            scl = (double)sa[sa_mode ? e * N + n : 0] * (double)sb[sb_mode ? e * K + k : 0];
        }
        ref[i] = s * scl;
        bound[i] = t * fabs(scl);
    }
    free(poff);
}

/* ------------------------------------------------------------------------ */
/* MXFP8: blocks of 32 elements sharing one power-of-two (E8M0) scale         */
/* ------------------------------------------------------------------------ */
/*
 * "FP8 training for Flux models" (Configuration > Key FP8 Parameters) lists
 * "mxfp8" among the fp8_recipe values, and "FP8 Training on AMD GPUs with
 * TorchTitan and TorchAO" names an MXFP8 grouped GEMM as next work; neither
 * page defines it.  The definition followed here is the public OCP
 * Microscaling Formats (MX) v1.0 specification:
 *   - a block is 32 consecutive elements along the contraction dimension
 *     (rowwise: along a row; colwise: along a column);
 *   - its shared scale is X = 2^e, stored as E8M0 code e + 127 (0 .. 254;
 *     255 is NaN), with e = floor(log2(max_i |V_i|)) - emax_elem, where
 *     emax_elem is the exponent of the element format's largest normal
 *     (8 for E4M3: 448 = 1.75 * 2^8; 15 for E5M2: 57344 = 1.75 * 2^15),
 *     clamped to [-127, 127];
 *   - each element is P_i = sat_rne_fp8(V_i / X) (ties to even, saturating).
 * Readings where the specification leaves a choice: an all-zero block gets
 * code 0; a block holding a NaN or an Inf gets code 255 and every element
 * of it the format's NaN code.  V_i / X is exact in double (X is a power of
 * two), so the element rounding is the single RNE of the encoder.
 *
 * Scales are returned as plain row-major matrices of codes: s[r][b] is the
 * scale of block b of row r (rowwise) or of column r (colwise).
 */
#define ORC_MX_BLOCK 32

int orc_mx_emax(int fmt) { return fmt == ORC_E5M2 ? 15 : 8; }

int orc_mx_scale_code(double amax, int fmt)
{
    int e;
    if (isnan(amax) || isinf(amax)) return 255;
    if (amax == 0.0) return 0;
    (void)frexp(amax, &e); /* amax = f * 2^e with f in [0.5, 1): floor(log2 amax) = e - 1 */
    e = (e - 1) - orc_mx_emax(fmt);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e + 127;
}

double orc_e8m0_decode(int code) { return code == 255 ? NAN : ldexp(1.0, code - 127); }

/* One block: v[0..31] (missing elements are passed as 0), codes to
 * out[i * stride], the scale code returned. */
static int mx_block(const double *v, int fmt, uint8_t *out, int64_t stride)
{
    double amax = 0.0;
    int nonfinite = 0, code;
    for (int i = 0; i < ORC_MX_BLOCK; i++) {
        if (!isfinite(v[i])) nonfinite = 1;
        else if (fabs(v[i]) > amax) amax = fabs(v[i]);
    }
    code = nonfinite ? 255 : orc_mx_scale_code(amax, fmt);
    for (int i = 0; i < ORC_MX_BLOCK; i++) {
        int q = code == 255 ? orc_fp8_nan_code(fmt) : orc_fp8_encode(ldexp(v[i], 127 - code), fmt);
        out[(int64_t)i * stride] = (uint8_t)q;
    }
    return code;
}

/* Group offsets padded to a multiple of `align`; returns the padded total. */
int64_t orc_padded_offsets_align(const int32_t *off, int G, int64_t align, int64_t *poff)
{
    int64_t acc = 0;
    for (int e = 0; e < G; e++) {
        poff[e] = acc;
        acc += ((int64_t)off[e + 1] - off[e] + align - 1) / align * align;
    }
    poff[G] = acc;
    return acc;
}

/*
 * MX quantize of a bf16 matrix x[rows][cols] (cols % 32 == 0).
 *
 * Row layout (layouts & 1): q_row [rows][cols]; s_row [SR][cols / 32] with
 *   SR = rows (ungrouped) or the padded total (grouped): row r of group e is
 *   scale row poff[e] + (r - offsets[e]); scale rows in a group's padding are
 *   all-zero blocks (code 0).
 * Transposed layout (layouts & 2): q_colT [cols][ldT], column c holding the
 *   rows of x (ungrouped: rows % 32 == 0) or group e's rows at poff[e]
 *   followed by zero padding up to poff[e + 1]; blocks run along the rows
 *   of each group (a group's last block is completed with zeros), s_col
 *   [cols][P / 32], P = rows or the padded total.
 * offsets: NULL or int32 [G + 1]; align: the group padding (a multiple of 32).
 */
int orc_mx_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt, int layouts,
                    const int32_t *offsets, int G, int64_t align, uint8_t *q_row, uint8_t *s_row,
                    uint8_t *q_colT, int64_t ldT, uint8_t *s_col)
{
    int ngroups = offsets ? G : 1;
    int64_t *poff = (int64_t *)malloc(sizeof(int64_t) * (ngroups + 1));
    int64_t P, nb = cols / ORC_MX_BLOCK;

    init_tables();
    if (offsets) {
        P = orc_padded_offsets_align(offsets, G, align, poff);
    } else {
        poff[0] = 0;
        poff[1] = rows;
        P = rows;
    }
    if (layouts & ORC_LAYOUT_ROW) {
        if (offsets) memset(s_row, 0, (size_t)(P * nb));
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; r++) {
            int64_t sr = r;
            double v[ORC_MX_BLOCK];
            if (offsets) {
                int e = 0;
                while (e < G - 1 && r >= offsets[e + 1]) e++;
                sr = poff[e] + (r - offsets[e]);
            }
            for (int64_t b = 0; b < nb; b++) {
                for (int i = 0; i < ORC_MX_BLOCK; i++) v[i] = bf16_to_float(x[r * ld_x + b * ORC_MX_BLOCK + i]);
                s_row[sr * nb + b] = (uint8_t)mx_block(v, fmt, q_row + r * cols + b * ORC_MX_BLOCK, 1);
            }
        }
    }
    if (layouts & ORC_LAYOUT_COLT) {
        int64_t pb = P / ORC_MX_BLOCK;
        memset(q_colT, 0, (size_t)(cols * ldT));
        memset(s_col, 0, (size_t)(cols * pb));
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; c++) {
            double v[ORC_MX_BLOCK];
            for (int e = 0; e < ngroups; e++) {
                int64_t r0 = offsets ? offsets[e] : 0, r1 = offsets ? offsets[e + 1] : rows;
                for (int64_t b = 0; r0 + b * ORC_MX_BLOCK < r1; b++) {
                    for (int i = 0; i < ORC_MX_BLOCK; i++) {
                        int64_t r = r0 + b * ORC_MX_BLOCK + i;
                        v[i] = r < r1 ? bf16_to_float(x[r * ld_x + c]) : 0.0;
                    }
                    s_col[c * pb + poff[e] / ORC_MX_BLOCK + b] =
                        (uint8_t)mx_block(v, fmt, q_colT + c * ldT + poff[e] + b * ORC_MX_BLOCK, 1);
                }
            }
        }
    }
    free(poff);
    return 0;
}

/*
 * MX GEMM in double: C[m][n] = sum_k dec(A[m][k]) X_A(m, k / 32)
 * dec(B[n][k]) X_B(n, k / 32), both operands K-contiguous; sA [M][lds_a],
 * sB [N][lds_b] are the E8M0 codes of each row's blocks.  bound = the sum of
 * absolute values.  pm/pn: as orc_gemm (NULL = the full M x N result).
 */
void orc_mx_gemm(const uint8_t *A, int fa, int64_t lda, const uint8_t *sA, int64_t lds_a, const uint8_t *B,
                 int fb, int64_t ldb, const uint8_t *sB, int64_t lds_b, int64_t M, int64_t N, int64_t K,
                 const int64_t *pm, const int64_t *pn, int64_t npts, double *ref, double *bound)
{
    double da[256], db[256];
    int64_t total = pm ? npts : M * N;
    for (int c = 0; c < 256; c++) {
        da[c] = orc_fp8_decode(c, fa);
        db[c] = orc_fp8_decode(c, fb);
    }
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < total; i++) {
        int64_t m = pm ? pm[i] : i / N, n = pm ? pn[i] : i % N;
        const uint8_t *a = A + m * lda, *b = B + n * ldb;
        double s = 0.0, t = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double x = orc_e8m0_decode(sA[m * lds_a + k / ORC_MX_BLOCK]) *
                       orc_e8m0_decode(sB[n * lds_b + k / ORC_MX_BLOCK]);
            double p = da[a[k]] * db[b[k]] * x;
            s += p;
            t += fabs(p);
        }
        ref[i] = s;
        bound[i] = t;
    }
}

/* ------------------------------------------------------------------------ */
/* MoE prologues fused ahead of the quantize: gather (permute) and SwiGLU     */
/* ------------------------------------------------------------------------ */
/*
 * "FP8 Training on AMD GPUs with TorchTitan and TorchAO" (the fused Triton
 * kernels question) replaces a five-kernel eager chain in front of the MoE
 * grouped GEMMs by one fused kernel.  The two element-wise steps that sit
 * in front of the expert GEMMs of a MoE layer are the permutation of token
 * rows into expert order (a gather by routing index) and, between the
 * gate/up and down projections, SwiGLU.  Their definitions here:
 *
 *   gather : row i of the output is row src[i] of the input.
 *   SwiGLU : h = bf16_rne(silu(g) * u) with silu(g) = g * sigma(g),
 *            sigma(g) = 1 / (1 + e^-g): the real-valued result rounded once
 *            to the nearest bf16 (ties to even).  Limits and IEEE
 *            conventions: silu(+Inf) = +Inf, silu(-Inf) = -0 (the limit of
 *            g e^g), NaN in g or u gives NaN, Inf * 0 gives NaN.
 *
 * Evaluation: P = g * u is exact in double (two 8-bit significands), sigma
 * is evaluated in double (libm exp), h_d = P * sigma_d, an error far below
 * half a bf16 ulp.  The one way that error can still move the rounding is
 * h_d landing exactly on a midpoint between two bf16 values while the exact
 * product does not; that happens when sigma_d comes out as exactly 1/2 (|g|
 * tiny) or exactly 1 (g large), and there the side of the exact value is
 * known: sigma(g) > 1/2 for g > 0, < 1/2 for g < 0, and < 1 always.
 */

/* bf16 rounding of a double (nearest; bf16's range: subnormals down to
 * 2^-133, overflow to Inf; NaN gives the quiet NaN 0x7FC0).  An exact
 * midpoint between two bf16 values goes to the larger magnitude when
 * tie > 0, the smaller when tie < 0, the even code when tie == 0. */
static uint16_t bf16_round(double v, int tie)
{
    uint16_t sign;
    double a, q, m, r, h;
    int e, E;
    float f;
    uint32_t u;
    if (isnan(v)) return 0x7FC0;
    sign = signbit(v) ? 0x8000 : 0;
    a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    if (a == 0.0) return sign;
    (void)frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1): floor(log2 a) = e - 1 */
    E = e - 1 < -126 ? -126 : e - 1;
    q = ldexp(1.0, E - 7);       /* the bf16 spacing at a: 8 significant bits */
    m = a / q;                   /* exact (power-of-two scaling) */
    if (m - floor(m) == 0.5 && tie != 0)
        r = tie > 0 ? ceil(m) : floor(m);
    else
        r = nearbyint(m);        /* nearest, ties to even */
    h = r * q;
    if (h >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    f = (float)h;                /* exact: h has at most 8 significant bits */
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

/* bf16 bit pattern of a double rounded once to the nearest bf16 value, ties
 * to even. */
uint16_t orc_bf16_from_double(double v) { return bf16_round(v, 0); }

/* h = bf16_rne(silu(g) * u) for n pairs; g, u and h are bf16 bit patterns. */
void orc_swiglu_bf16(const uint16_t *g, const uint16_t *u, int64_t n, uint16_t *h)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        double gd = bf16_to_float(g[i]), ud = bf16_to_float(u[i]);
        double sig, hd;
        int tie = 0;
        if (isnan(gd) || isnan(ud)) {
            h[i] = 0x7FC0;
            continue;
        }
        if (isinf(gd)) {  /* silu(+Inf) = +Inf, silu(-Inf) = -0 */
            h[i] = bf16_round((gd > 0 ? gd : -0.0) * ud, 0);
            continue;
        }
        sig = 1.0 / (1.0 + exp(-gd));
        hd = (gd * ud) * sig;
        if (sig == 0.5) tie = gd > 0 ? 1 : (gd < 0 ? -1 : 0);
        if (sig == 1.0) tie = -1;
        h[i] = bf16_round(hd, tie);
    }
}

/* ------------------------------------------------------------------------ */
/* Blockwise scaling: 1 x 128 blocks (activations, gradients) or 128 x 128   */
/* blocks (weights), one power-of-two scale per block                         */
/* ------------------------------------------------------------------------ */
/*
 * "FP8 training for Flux models" (Configuration > Key FP8 Parameters) lists
 * a "blockwise" recipe without a definition.  Reading: the contraction
 * dimension is cut into blocks of 128 elements; an activation or gradient
 * block is one row x 128 columns (one column x 128 rows in the transposed
 * layout), a weight block is 128 x 128 and serves both layouts.  Each block
 * takes current scaling with a power-of-two scale: s = the largest 2^e with
 * amax * 2^e <= fp8_max (e clamped to [-127, 127]; amax 0 or non-finite
 * gives s = 1), elements q = sat_rne_fp8(v * s) (no finite element
 * saturates), and the dequantisation factor 1/s = 2^-e is stored as the E8M0
 * code 127 - e, the scale format the MX GEMM consumes.  Codes are returned
 * per 32-element block (each 128-block's code repeated four times), plain
 * row-major like the MX functions, so the MX GEMM oracle applies them.
 */
int orc_blockwise_code(double amax, int fmt)
{
    double fmax = orc_fp8_max_value(fmt);
    int e;
    if (!isfinite(amax) || amax == 0.0) return 127;
    e = -127;
    while (e < 127 && ldexp(amax, e + 1) <= fmax) e++;
    if (ldexp(amax, e) > fmax) e = -127; /* only when even 2^-127 overflows (not for bf16 input) */
    return 127 - e;
}

/*
 * x [rows][cols] bf16 (ld_x); block_rows 1 or 128; cols % 128 == 0 and, for
 * the transposed layout or block_rows 128, rows % 128 == 0.
 * q_row [rows][cols], s_row [rows][cols/32]; q_colT [cols][rows],
 * s_col [cols][rows/32].
 */
int orc_blockwise_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt, int block_rows,
                           int layouts, uint8_t *q_row, uint8_t *s_row, uint8_t *q_colT, uint8_t *s_col)
{
    const int64_t B = 128;
    int64_t nbr = cols / B;
    init_tables();
    if (block_rows == 128) {
        /* one scale per 128 x 128 block, the same for both layouts */
#pragma omp parallel for schedule(static)
        for (int64_t rb = 0; rb < rows / B; rb++)
            for (int64_t cb = 0; cb < nbr; cb++) {
                double amax = 0.0;
                int nonfinite = 0, code;
                double s;
                for (int64_t r = rb * B; r < rb * B + B; r++)
                    for (int64_t c = cb * B; c < cb * B + B; c++) {
                        double v = bf16_to_float(x[r * ld_x + c]);
                        if (!isfinite(v)) nonfinite = 1;
                        else if (fabs(v) > amax) amax = fabs(v);
                    }
                code = orc_blockwise_code(nonfinite ? NAN : amax, fmt);
                s = ldexp(1.0, 127 - code);
                for (int64_t r = rb * B; r < rb * B + B; r++)
                    for (int64_t c = cb * B; c < cb * B + B; c++) {
                        uint8_t q = (uint8_t)orc_fp8_encode(bf16_to_float(x[r * ld_x + c]) * s, fmt);
                        if (layouts & ORC_LAYOUT_ROW) q_row[r * cols + c] = q;
                        if (layouts & ORC_LAYOUT_COLT) q_colT[c * rows + r] = q;
                    }
                for (int64_t r = rb * B; r < rb * B + B; r++)
                    for (int k = 0; k < 4; k++) {
                        if (layouts & ORC_LAYOUT_ROW) s_row[r * (cols / 32) + cb * 4 + k] = (uint8_t)code;
                    }
                for (int64_t c = cb * B; c < cb * B + B; c++)
                    for (int k = 0; k < 4; k++) {
                        if (layouts & ORC_LAYOUT_COLT) s_col[c * (rows / 32) + rb * 4 + k] = (uint8_t)code;
                    }
            }
        return 0;
    }
    /* 1 x 128 blocks along each layout's contraction dimension */
    if (layouts & ORC_LAYOUT_ROW) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; r++)
            for (int64_t cb = 0; cb < nbr; cb++) {
                double amax = 0.0, s;
                int nonfinite = 0, code;
                for (int64_t c = cb * B; c < cb * B + B; c++) {
                    double v = bf16_to_float(x[r * ld_x + c]);
                    if (!isfinite(v)) nonfinite = 1;
                    else if (fabs(v) > amax) amax = fabs(v);
                }
                code = orc_blockwise_code(nonfinite ? NAN : amax, fmt);
                s = ldexp(1.0, 127 - code);
                for (int64_t c = cb * B; c < cb * B + B; c++)
                    q_row[r * cols + c] = (uint8_t)orc_fp8_encode(bf16_to_float(x[r * ld_x + c]) * s, fmt);
                for (int k = 0; k < 4; k++) s_row[r * (cols / 32) + cb * 4 + k] = (uint8_t)code;
            }
    }
    if (layouts & ORC_LAYOUT_COLT) {
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; c++)
            for (int64_t rb = 0; rb < rows / B; rb++) {
                double amax = 0.0, s;
                int nonfinite = 0, code;
                for (int64_t r = rb * B; r < rb * B + B; r++) {
                    double v = bf16_to_float(x[r * ld_x + c]);
                    if (!isfinite(v)) nonfinite = 1;
                    else if (fabs(v) > amax) amax = fabs(v);
                }
                code = orc_blockwise_code(nonfinite ? NAN : amax, fmt);
                s = ldexp(1.0, 127 - code);
                for (int64_t r = rb * B; r < rb * B + B; r++)
                    q_colT[c * rows + r] = (uint8_t)orc_fp8_encode(bf16_to_float(x[r * ld_x + c]) * s, fmt);
                for (int k = 0; k < 4; k++) s_col[c * (rows / 32) + rb * 4 + k] = (uint8_t)code;
            }
    }
    return 0;
}
