/*
 * CPU oracle for the W4A16 group-quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library. The CUDA library never includes,
 * links or calls anything here, and this file includes nothing of it.
 *
 * What it computes (plain loops, written for a reader to check by eye):
 *   - the asymmetric per-group int4 rule named in compressed-tensors PR #269
 *     "Some fixes for AWQ" (opening comment: alignment with AutoAWQ's
 *     pseudo_quantize_tensor): s = (max - min)/15, z = round(-min/s),
 *     q = clamp(round(w/s) + z, 0, 15);
 *   - dequantization (q - z)*s, rounded once to fp16;
 *   - the W4A16 product itself: fp16 inputs times int4-quantized weights
 *     (same PR, the reply defining "w4a16"), accumulated here in fp64 with
 *     the per-element magnitude sum used by the tolerance;
 *   - the packed device layout (a format of this project, specified in the
 *     public header's comment and restated below), and its inverse.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   R-round  every "round" is round-half-to-even (IEEE default);
 *   R-s16    q and z use the stored fp16 scale s16 (converted to fp32), so the
 *            triple (q, s16, z) is self-consistent;
 *   R-eps    if s16 rounds to zero (constant or near-constant group), s16 is
 *            replaced by RNE_fp16(1e-5);
 *   R-zclamp z is clamped to [0, 15] (zeros are uint4);
 *   R-dq     dequant = RNE_fp16((q - z) * s16): one rounding of an exact
 *            product;
 *   R-acc    fp64 accumulation, order free.
 *
 * Arithmetic rules: float operations below are IEEE binary32 with no
 * contraction (built with -ffp-contract=off); fp16 conversions are written
 * out from the binary16 definition, not taken from a compiler type.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* binary16 <-> binary64, from the IEEE 754 binary16 definition            */
/* (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).           */
/* ---------------------------------------------------------------------- */

double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero or subnormal */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even; overflow -> inf. */
uint16_t oracle_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return 0x7e00;
    if (isinf(a))
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);                  /* a in [2^(ex-1), 2^ex) */
    int E = ex - 1;                 /* unbiased exponent of a */
    if (E < -14)
        E = -14;                    /* subnormal range: spacing 2^-24 */
    double spacing = ldexp(1.0, E - 10);
    double r = nearbyint(a / spacing);   /* exact scaling; ties to even */
    double v = r * spacing;              /* the rounded magnitude */
    if (v > 65504.0)                      /* beyond the largest finite half */
        return sign | 0x7c00;
    if (v < ldexp(1.0, -14))             /* subnormal (or zero) */
        return sign | (uint16_t)(v / ldexp(1.0, -24));
    frexp(v, &ex);
    E = ex - 1;
    uint16_t frac = (uint16_t)(v / ldexp(1.0, E - 10) - 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | frac;
}

void oracle_doubles_to_half(const double* x, size_t n, uint16_t* out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = oracle_double_to_half(x[i]);
}

void oracle_halves_to_double(const uint16_t* h, size_t n, double* out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = oracle_half_to_double(h[i]);
}

/* ---------------------------------------------------------------------- */
/* Quantization (offline step).                                            */
/* W: float32 [K][N] row-major; group divides K; G = K / group.            */
/* Outputs q u8 [K][N], s16 fp16 bits [G][N], z u8 [G][N].                 */
/* ---------------------------------------------------------------------- */

static float clamp_0_15(float v)
{
    if (!(v >= 0.0f))   /* also maps NaN to 0 */
        return 0.0f;
    if (v > 15.0f)
        return 15.0f;
    return v;
}

void oracle_quantize(const float* W, int K, int N, int group,
                     uint8_t* q, uint16_t* s16, uint8_t* z)
{
    const int G = K / group;
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int j = 0; j < G; ++j) {
            /* step 1: min and max over the group's k */
            float mn = W[(size_t)(j * group) * N + n];
            float mx = mn;
            for (int k = j * group; k < (j + 1) * group; ++k) {
                float w = W[(size_t)k * N + n];
                if (w < mn) mn = w;
                if (w > mx) mx = w;
            }
            /* step 2: s = (max - min) / 15 in fp32, stored as fp16 */
            float range = mx - mn;
            float s32 = range / 15.0f;
            uint16_t sb = oracle_double_to_half((double)s32);
            if ((sb & 0x7fff) == 0)                       /* R-eps */
                sb = oracle_double_to_half((double)1e-5f);
            float s = (float)oracle_half_to_double(sb);   /* R-s16 */
            /* step 3: z = clamp(round(-min / s), 0, 15) */
            float zf = clamp_0_15(nearbyintf(-mn / s));
            /* step 4: q = clamp(round(w / s) + z, 0, 15) */
            for (int k = j * group; k < (j + 1) * group; ++k) {
                float w = W[(size_t)k * N + n];
                float qf = clamp_0_15(nearbyintf(w / s) + zf);
                q[(size_t)k * N + n] = (uint8_t)qf;
            }
            s16[(size_t)j * N + n] = sb;
            z[(size_t)j * N + n] = (uint8_t)zf;
        }
    }
}

/* deq[k][n] = RNE_fp16((q - z) * s16), one rounding of the exact product. */
void oracle_dequantize(const uint8_t* q, const uint16_t* s16, const uint8_t* z,
                       int K, int N, int group, uint16_t* deq)
{
    #pragma omp parallel for schedule(static)
    for (int k = 0; k < K; ++k) {
        int j = k / group;
        for (int n = 0; n < N; ++n) {
            int d = (int)q[(size_t)k * N + n] - (int)z[(size_t)j * N + n];
            double s = oracle_half_to_double(s16[(size_t)j * N + n]);
            deq[(size_t)k * N + n] = oracle_double_to_half((double)d * s);
        }
    }
}

/* ---------------------------------------------------------------------- */
/* The product.  A: fp16 bits [M][K]; B: fp16 bits [K][N] (the dequantized */
/* weights).  y[m][n] = sum_k a[m][k]*b[k][n] in fp64, and                 */
/* mag[m][n] = sum_k |a[m][k]*b[k][n]| (the tolerance's magnitude term).   */
/* ---------------------------------------------------------------------- */

static double half_table[65536];
static int half_table_ready = 0;

/* Value of every binary16 pattern, computed once from the definition. */
static void fill_half_table(void)
{
    if (half_table_ready)
        return;
    #pragma omp critical(oracle_half_table)
    {
        if (!half_table_ready) {
            for (int h = 0; h < 65536; ++h)
                half_table[h] = oracle_half_to_double((uint16_t)h);
            half_table_ready = 1;
        }
    }
}

void oracle_matmul(const uint16_t* A, const uint16_t* B, int M, int N, int K,
                   double* y, double* mag)
{
    enum { NC = 64 };
    fill_half_table();
    /* Each (m, n) is the sum over k = 0, 1, ..., K-1 in that order; the n
     * loop is innermost only so that rows of B are read contiguously. */
    #pragma omp parallel for schedule(dynamic, 1)
    for (int n0 = 0; n0 < N; n0 += NC) {
        int n1 = n0 + NC < N ? n0 + NC : N;
        double acc[NC], acc_abs[NC];
        for (int m = 0; m < M; ++m) {
            for (int n = n0; n < n1; ++n) {
                acc[n - n0] = 0.0;
                acc_abs[n - n0] = 0.0;
            }
            for (int k = 0; k < K; ++k) {
                double a = half_table[A[(size_t)m * K + k]];
                const uint16_t* brow = B + (size_t)k * N;
                for (int n = n0; n < n1; ++n) {
                    double p = a * half_table[brow[n]];
                    acc[n - n0] += p;
                    acc_abs[n - n0] += fabs(p);
                }
            }
            for (int n = n0; n < n1; ++n) {
                y[(size_t)m * N + n] = acc[n - n0];
                mag[(size_t)m * N + n] = acc_abs[n - n0];
            }
        }
    }
}

/* Tolerance check: ratio[i] = |y_gpu - y_ref| / (2^-9 * mag + 1e-3).      */
/* Returns the maximum ratio; an element passes when its ratio is <= 1.    */
double oracle_check(const uint16_t* y_gpu, const double* y_ref, const double* mag,
                    size_t count, size_t* worst_index)
{
    double worst = 0.0;
    size_t wi = 0;
    for (size_t i = 0; i < count; ++i) {
        double g = oracle_half_to_double(y_gpu[i]);
        double bound = ldexp(mag[i], -9) + 1e-3;
        double r = fabs(g - y_ref[i]) / bound;
        if (!(r <= worst)) {    /* NaN propagates as the worst */
            worst = r;
            wi = i;
            if (isnan(r))
                break;
        }
    }
    if (worst_index)
        *worst_index = wi;
    return worst;
}

/* ---------------------------------------------------------------------- */
/* Packed device layout (format of this project).                           */
/*                                                                          */
/* Weights: uint32 words, 8 nibbles each.  Columns are grouped in strips of */
/* 16 (strip j = columns 16j..16j+15), K in atoms of 64 (atom a = k in      */
/* [64a, 64a+64)).  Word offset = (j*(K/64) + a)*128 + 4*L + i, where       */
/* L in [0,32) and i in [0,4); with g = L>>2, t = L&3, s = i>>1, r = i&1    */
/* the word holds column n = 16j + g + 8r and the 8 values k = 64a + 32s +  */
/* 8t + e, e = 0..7.  Value e sits in nibble p (bits 4p..4p+3), p = the    */
/* 3-bit reversal of e (nibbles 0..7 hold e = 0 4 2 6 1 5 3 7).             */
/* Scales: fp16 at offset (j*G + grp)*16 + 2*(c%8) + c/8 for column 16j+c. */
/* Zeros: bytes; byte (j*G + grp)*8 + c (c < 8) holds the zero of column    */
/* 16j + c in its low nibble and of column 16j + 8 + c in its high nibble.  */
/* ---------------------------------------------------------------------- */

static int nibble_of(int e)
{
    return 4 * (e % 2) + 2 * ((e / 2) % 2) + e / 4;
}

static size_t word_offset(int K, int n, int k)
{
    int j = n / 16, c = n % 16;
    int a = k / 64, kk = k % 64;
    int s = kk / 32, t = (kk % 32) / 8;
    int g = c % 8, r = c / 8;
    int L = 4 * g + t, i = 2 * s + r;
    return ((size_t)j * (K / 64) + a) * 128 + 4 * L + i;
}

void oracle_pack(const uint8_t* q, const uint8_t* z, const uint16_t* s16,
                 int K, int N, int group, uint32_t* Wp, uint16_t* Sp, uint32_t* Zp)
{
    const int G = K / group;
    memset(Wp, 0, (size_t)K * N / 2);
    memset(Zp, 0, (size_t)G * N / 2);
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            uint32_t v = q[(size_t)k * N + n] & 15u;
            Wp[word_offset(K, n, k)] |= v << (4 * nibble_of(k % 8));
        }
    for (int grp = 0; grp < G; ++grp)
        for (int n = 0; n < N; ++n) {
            int j = n / 16, c = n % 16;
            Sp[((size_t)j * G + grp) * 16 + 2 * (c % 8) + c / 8] = s16[(size_t)grp * N + n];
            uint32_t v = z[(size_t)grp * N + n] & 15u;
            /* byte (j*G + grp)*8 + c%8 of the little-endian word array, nibble c/8 */
            Zp[((size_t)j * G + grp) * 2 + (c % 8) / 4] |= v << (8 * ((c % 8) % 4) + 4 * (c / 8));
        }
}

void oracle_unpack(const uint32_t* Wp, const uint16_t* Sp, const uint32_t* Zp,
                   int K, int N, int group, uint8_t* q, uint16_t* s16, uint8_t* z)
{
    const int G = K / group;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n)
            q[(size_t)k * N + n] =
                (uint8_t)((Wp[word_offset(K, n, k)] >> (4 * nibble_of(k % 8))) & 15u);
    for (int grp = 0; grp < G; ++grp)
        for (int n = 0; n < N; ++n) {
            int j = n / 16, c = n % 16;
            s16[(size_t)grp * N + n] = Sp[((size_t)j * G + grp) * 16 + 2 * (c % 8) + c / 8];
            z[(size_t)grp * N + n] =
                (uint8_t)((Zp[((size_t)j * G + grp) * 2 + (c % 8) / 4] >>
                           (8 * ((c % 8) % 4) + 4 * (c / 8))) & 15u);
        }
}

/* ---------------------------------------------------------------------- */
/* Fused gate/up epilogue.                                                  */
/*                                                                          */
/* lmdeploy issue #2274 "[Feature] support qqq(w4a8) for lmdeploy",         */
/* section "Modification": the gate and up weights are fused into one       */
/* weight, and element-wise operations such as SiLU are fused into the      */
/* kernels around the GEMM.  Readings (the pages give no formula):          */
/*   R-gu    the fused weight's N columns are [gate | up], N/2 each; the    */
/*           output is out[m, j] = silu(y[m, j]) * y[m, N/2 + j];            */
/*   R-silu  silu(x) = x * sigmoid(x) = x / (1 + exp(-x)), in fp64.          */
/* bound[m, j] propagates the product's tolerance B = 2^-9 * mag + 1e-3 of  */
/* the two inputs (|silu'| <= 1.1):                                         */
/*   |silu(g)| * Bu + 1.1 * Bg * (|u| + Bu) + 2^-10 * |out| + 1e-3,          */
/* the last two terms for the output's fp16 rounding and the evaluation of  */
/* silu in fp32.                                                            */
/* ---------------------------------------------------------------------- */

double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

void oracle_silu_mul(const double* y, const double* mag, int M, int N, double* out,
                     double* bound)
{
    int H = N / 2;
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < H; ++j) {
            double g = y[(size_t)m * N + j];
            double u = y[(size_t)m * N + H + j];
            double bg = ldexp(mag[(size_t)m * N + j], -9) + 1e-3;
            double bu = ldexp(mag[(size_t)m * N + H + j], -9) + 1e-3;
            double sg = oracle_silu(g);
            double o = sg * u;
            out[(size_t)m * H + j] = o;
            bound[(size_t)m * H + j] =
                fabs(sg) * bu + 1.1 * bg * (fabs(u) + bu) + ldexp(fabs(o), -10) + 1e-3;
        }
}

/* max |Y - ref| / bound over all elements (NaN is the worst), and where. */
double oracle_check_bound(const uint16_t* y_gpu, const double* ref, const double* bound,
                          size_t count, size_t* worst_index)
{
    double worst = 0.0;
    size_t wi = 0;
    for (size_t i = 0; i < count; ++i) {
        double r = fabs(oracle_half_to_double(y_gpu[i]) - ref[i]) / bound[i];
        if (!(r <= worst)) {
            worst = r;
            wi = i;
            if (isnan(r))
                break;
        }
    }
    if (worst_index)
        *worst_index = wi;
    return worst;
}

/* ---------------------------------------------------------------------- */
/* bf16 activations.                                                        */
/*                                                                          */
/* compressed-tensors PR #269 "Some fixes for AWQ": in the naming of the    */
/* preset schemes, the number after "A" is the activations' width, and     */
/* W4A16 keeps them as 16-bit floats, unquantized; a reply in the same      */
/* thread names an API taking fp32, bf16 or fp16 activations.  Readings:    */
/*   R-bf16    the A16 side may be bfloat16 as well as fp16: A and Y are    */
/*             bf16, the quantized weights are the same (q, s16, z);       */
/*   R-dq-bf16 dequant = RNE_bf16((q - z) * s16), one rounding of the exact */
/*             product (both operands of the multiply-accumulate are bf16); */
/*   R-tol-bf16 the fp16 tolerance is four units of fp16 rounding (2^-11)   */
/*             of the magnitude sum; with bf16's unit (2^-8) it becomes     */
/*             |y - y_ref| <= 2^-6 * sum|a*w| + 1e-3.                       */
/* bfloat16 is the upper half of a binary32: 1 sign bit, 8 exponent bits    */
/* with bias 127, 7 fraction bits.                                          */
/* ---------------------------------------------------------------------- */

double oracle_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* zero or subnormal: f * 2^-126 / 128 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a double to the nearest bfloat16, ties to even; overflow -> inf. */
uint16_t oracle_double_to_bf16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return 0x7fc0;
    if (isinf(a))
        return sign | 0x7f80;
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);                  /* a in [2^(ex-1), 2^ex) */
    int E = ex - 1;
    if (E < -126)
        E = -126;                   /* subnormal range: spacing 2^-133 */
    double spacing = ldexp(1.0, E - 7);
    double r = nearbyint(a / spacing);   /* ties to even */
    double v = r * spacing;
    if (v > ldexp(255.0, 120))      /* beyond the largest finite bf16, (2 - 2^-7) * 2^127 */
        return sign | 0x7f80;
    if (v < ldexp(1.0, -126))       /* subnormal (or zero) */
        return sign | (uint16_t)(v / ldexp(1.0, -133));
    frexp(v, &ex);
    E = ex - 1;
    uint16_t frac = (uint16_t)(v / ldexp(1.0, E - 7) - 128.0);
    return sign | (uint16_t)((E + 127) << 7) | frac;
}

void oracle_doubles_to_bf16(const double* x, size_t n, uint16_t* out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = oracle_double_to_bf16(x[i]);
}

void oracle_bf16s_to_double(const uint16_t* h, size_t n, double* out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_to_double(h[i]);
}

/* deq[k][n] = RNE_bf16((q - z) * s16): the exact product, rounded once. */
void oracle_dequantize_bf16(const uint8_t* q, const uint16_t* s16, const uint8_t* z,
                            int K, int N, int group, uint16_t* deq)
{
    #pragma omp parallel for schedule(static)
    for (int k = 0; k < K; ++k) {
        int j = k / group;
        for (int n = 0; n < N; ++n) {
            int d = (int)q[(size_t)k * N + n] - (int)z[(size_t)j * N + n];
            double s = oracle_half_to_double(s16[(size_t)j * N + n]);
            deq[(size_t)k * N + n] = oracle_double_to_bf16((double)d * s);
        }
    }
}

static double bf16_table[65536];
static int bf16_table_ready = 0;

static void fill_bf16_table(void)
{
    if (bf16_table_ready)
        return;
    #pragma omp critical(oracle_bf16_table)
    {
        if (!bf16_table_ready) {
            for (int h = 0; h < 65536; ++h)
                bf16_table[h] = oracle_bf16_to_double((uint16_t)h);
            bf16_table_ready = 1;
        }
    }
}

/* As oracle_matmul for bf16 A [M][K] and bf16 B [K][N]: y and the magnitude */
/* sum in fp64, each (m, n) summed over k in order.                          */
void oracle_matmul_bf16(const uint16_t* A, const uint16_t* B, int M, int N, int K,
                        double* y, double* mag)
{
    enum { NC = 64 };
    fill_bf16_table();
    #pragma omp parallel for schedule(dynamic, 1)
    for (int n0 = 0; n0 < N; n0 += NC) {
        int n1 = n0 + NC < N ? n0 + NC : N;
        double acc[NC], acc_abs[NC];
        for (int m = 0; m < M; ++m) {
            for (int n = n0; n < n1; ++n) {
                acc[n - n0] = 0.0;
                acc_abs[n - n0] = 0.0;
            }
            for (int k = 0; k < K; ++k) {
                double a = bf16_table[A[(size_t)m * K + k]];
                const uint16_t* brow = B + (size_t)k * N;
                for (int n = n0; n < n1; ++n) {
                    double p = a * bf16_table[brow[n]];
                    acc[n - n0] += p;
                    acc_abs[n - n0] += fabs(p);
                }
            }
            for (int n = n0; n < n1; ++n) {
                y[(size_t)m * N + n] = acc[n - n0];
                mag[(size_t)m * N + n] = acc_abs[n - n0];
            }
        }
    }
}

/* R-tol-bf16: ratio[i] = |y_gpu - y_ref| / (2^-6 * mag + 1e-3), y_gpu bf16. */
double oracle_check_bf16(const uint16_t* y_gpu, const double* y_ref, const double* mag,
                         size_t count, size_t* worst_index)
{
    double worst = 0.0;
    size_t wi = 0;
    for (size_t i = 0; i < count; ++i) {
        double g = oracle_bf16_to_double(y_gpu[i]);
        double bound = ldexp(mag[i], -6) + 1e-3;
        double r = fabs(g - y_ref[i]) / bound;
        if (!(r <= worst)) {
            worst = r;
            wi = i;
            if (isnan(r))
                break;
        }
    }
    if (worst_index)
        *worst_index = wi;
    return worst;
}

/* The fused gate/up epilogue of a bf16 product: out as oracle_silu_mul,    */
/* the bound propagated from R-tol-bf16 (B = 2^-6 * mag + 1e-3) with the    */
/* output's bf16 rounding and fp32 evaluation as 2^-7 * |out| + 1e-3.       */
void oracle_silu_mul_bf16(const double* y, const double* mag, int M, int N, double* out,
                          double* bound)
{
    int H = N / 2;
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < H; ++j) {
            double g = y[(size_t)m * N + j];
            double u = y[(size_t)m * N + H + j];
            double bg = ldexp(mag[(size_t)m * N + j], -6) + 1e-3;
            double bu = ldexp(mag[(size_t)m * N + H + j], -6) + 1e-3;
            double sg = oracle_silu(g);
            double o = sg * u;
            out[(size_t)m * H + j] = o;
            bound[(size_t)m * H + j] =
                fabs(sg) * bu + 1.1 * bg * (fabs(u) + bu) + ldexp(fabs(o), -7) + 1e-3;
        }
}

/* max |Y - ref| / bound over bf16 results (NaN is the worst), and where. */
double oracle_check_bound_bf16(const uint16_t* y_gpu, const double* ref, const double* bound,
                               size_t count, size_t* worst_index)
{
    double worst = 0.0;
    size_t wi = 0;
    for (size_t i = 0; i < count; ++i) {
        double r = fabs(oracle_bf16_to_double(y_gpu[i]) - ref[i]) / bound[i];
        if (!(r <= worst)) {
            worst = r;
            wi = i;
            if (isnan(r))
                break;
        }
    }
    if (worst_index)
        *worst_index = wi;
    return worst;
}

/* ---------------------------------------------------------------------- */
/* W4A8: activations quantized to 8 bits inside the operation.             */
/*                                                                          */
/* compressed-tensors PR #269 "Some fixes for AWQ", the Arm contributor's   */
/* example: the operation takes fp16 activations, quantizes them to 8 bits  */
/* internally, multiplies 8-bit activations by the 4-bit weights and        */
/* returns fp16 (lmdeploy issue #2274: W4A8 with online activation          */
/* quantization).  The pages give no formula.  Readings:                    */
/*   R-a8      dynamic, symmetric, per token (row): amax = max_k |a[m,k]|,  */
/*             s_a = amax / 127 and a_q = clamp(round(a / s_a), -127, 127), */
/*             all in IEEE fp32 (the inputs are exact in fp32), round half  */
/*             to even; a row of zeros has s_a = 1 and a_q = 0;             */
/*   R-a8-dot  y[m,n] = s_a[m] * sum_groups s[g,n] * sum_k a_q (q - z): the  */
/*             8-bit by 4-bit products and their group sums are integers,  */
/*             scaled once per group and once per row; fp64 here;           */
/*   R-a8-tol  the result is fp16 (or bf16), checked with the bound of the  */
/*             16-bit product of the same type, with sum |a*w| taken as     */
/*             s_a * sum |a_q (q - z) s|.                                   */
/* ---------------------------------------------------------------------- */

/* A: the activations' values [M][K] (fp16 or bf16, exact as doubles). */
void oracle_quantize_act(const double* A, int M, int K, int8_t* aq, float* s_a)
{
    for (int m = 0; m < M; ++m) {
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) {
            float v = fabsf((float)A[(size_t)m * K + k]);
            if (v > amax)
                amax = v;
        }
        float s = amax > 0.0f ? amax / 127.0f : 1.0f;
        s_a[m] = s;
        for (int k = 0; k < K; ++k) {
            float r = nearbyintf((float)A[(size_t)m * K + k] / s);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            aq[(size_t)m * K + k] = (int8_t)r;
        }
    }
}

/* y[m][n] = s_a[m] * sum_g s16[g][n] * sum_{k in g} aq[m][k] (q[k][n] - z[g][n]) */
/* in fp64, and mag = s_a[m] * sum_k |aq (q - z) s16|.                       */
void oracle_reference_a8(const int8_t* aq, const float* s_a, const uint8_t* q,
                         const uint16_t* s16, const uint8_t* z, int M, int N, int K,
                         int group, double* y, double* mag)
{
    const int G = K / group;
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, acc_abs = 0.0;
            for (int g = 0; g < G; ++g) {
                long long dot = 0, dot_abs = 0;
                int zz = z[(size_t)g * N + n];
                for (int k = g * group; k < (g + 1) * group; ++k) {
                    long long p = (long long)aq[(size_t)m * K + k] *
                                  ((int)q[(size_t)k * N + n] - zz);
                    dot += p;
                    dot_abs += p < 0 ? -p : p;
                }
                double sg = oracle_half_to_double(s16[(size_t)g * N + n]);
                acc += sg * (double)dot;
                acc_abs += sg * (double)dot_abs;
            }
            y[(size_t)m * N + n] = (double)s_a[m] * acc;
            mag[(size_t)m * N + n] = (double)s_a[m] * acc_abs;
        }
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
