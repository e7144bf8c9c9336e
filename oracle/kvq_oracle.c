/*
 * kvq_oracle.c — the CPU oracle of the quantized MLA KV-cache path.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by tests/, by the smoke check and by the benchmark's
 * CPU-baseline leg; never by the product path.  Plain C, one thread, fp64 wherever the
 * method leaves the precision open.  Compile with -ffp-contract=off: every fused
 * multiply-add below is an explicit fmaf() because the method specifies it.
 *
 * Parity status per function (what pins it, in tests/test_oracle_*.py):
 *   orc_e4m3_value / orc_e4m3_rne   exhaustive 256-code table, every midpoint, the
 *                                    library float8_e4m3fn conversion
 *   orc_f16_rne / orc_f16_value     numpy float16 conversion on all 65536 patterns and
 *                                    random doubles
 *   orc_encode_fp8                  brute-force nearest-code search on random rows
 *   orc_tq4_codebook                centroid/threshold conditions in closed form
 *   orc_fwht_*                      Sylvester Hadamard matrix (H·H = nI), scipy.linalg
 *   orc_encode_tq4 / decode         nearest-centroid brute force, rel-L2 ~ 0.096,
 *                                    radius invariance, rotated-domain identities
 *   orc_q4_block / append / gather  all-zero group bits, tie blocks, dequant bound,
 *                                    brute-force page placement
 *   orc_project_rows / _append_q4   exact integer products (numpy int64 matmul), the
 *                                    identity and permutation weights (rows reproduced
 *                                    bit for bit, so the append equals orc_append_q4 of
 *                                    h), the fp32 error bound against an fp64 matmul,
 *                                    bfloat16 widening
 *   orc_mla_decode                  hand-expanded softmax, one-hot and uniform cases,
 *                                    split invariance, a numpy float128-free re-derivation
 */
#include "kvq_oracle.h"
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ===================================================================================
 * Number formats
 * =================================================================================== */

/* Round a non-negative double to the nearest integer, ties to the even integer. */
static double rne_int(double t)
{
    double fl = floor(t);
    double fr = t - fl;
    if (fr > 0.5) return fl + 1.0;
    if (fr < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* e4m3 (OCP FP8 E4M3, "fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; no infinities.  Per the KV8 rebase note of colibri PR #399 (HIP
 * portability item): normals are (1 + M/8) * 2^(E-7), denormals M * 2^-9, and the
 * pattern S.1111.111 reads back as 0.  The encoder below never produces it. */
double orc_e4m3_value(uint8_t code)
{
    int s = code >> 7, E = (code >> 3) & 15, M = code & 7;
    double v;
    if (E == 15 && M == 7)      v = 0.0;
    else if (E == 0)            v = ldexp((double)M, -9);
    else                        v = ldexp(1.0 + M / 8.0, E - 7);
    return s ? -v : v;
}

/* Nearest e4m3 code with ties to even mantissa; magnitudes at or above 448 (the
 * largest finite code) saturate to 448; the sign bit is kept, also for values that
 * round to zero.  Non-finite input is outside the contract. */
uint8_t orc_e4m3_rne(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal spacing 2^-9; an integer n of 8 is exactly the smallest normal */
        double n = rne_int(a * 512.0);
        return sign | (uint8_t)n;
    }
    int e;
    frexp(a, &e);                       /* a in [2^(e-1), 2^e)                  */
    int E = (e - 1) + 7;                /* biased exponent field                */
    double n = rne_int(ldexp(a, 3 - (e - 1)));   /* significand * 8, in [8, 16]  */
    if (n == 16.0) { n = 8.0; E += 1; }
    int code = (E << 3) | ((int)n - 8);
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

/* IEEE 754 binary16, round to nearest, ties to even; overflow to infinity. */
uint16_t orc_f16_rne(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    if (isnan(v)) return sign | 0x7E00;
    if (isinf(v)) return sign | 0x7C00;
    double a = fabs(v);
    if (a < ldexp(1.0, -14)) {
        /* subnormal spacing 2^-24; n = 1024 is exactly the smallest normal */
        double n = rne_int(ldexp(a, 24));
        return sign | (uint16_t)n;
    }
    int e;
    frexp(a, &e);
    int E = (e - 1) + 15;
    if (E >= 31) return sign | 0x7C00;
    double n = rne_int(ldexp(a, 10 - (e - 1)));  /* in [1024, 2048] */
    if (n == 2048.0) { n = 1024.0; E += 1; }
    if (E >= 31) return sign | 0x7C00;
    return sign | (uint16_t)(E << 10) | (uint16_t)((int)n - 1024);
}

double orc_f16_value(uint16_t h)
{
    int s = h >> 15, E = (h >> 10) & 31, M = h & 1023;
    double v;
    if (E == 31)      v = M ? NAN : INFINITY;
    else if (E == 0)  v = ldexp((double)M, -24);
    else              v = ldexp(1.0 + M / 1024.0, E - 15);
    return s ? -v : v;
}

/* ===================================================================================
 * fp8 (KV8) per-row encode — colibri PR #399, Summary and Commit 1: e4m3 codes with
 * one scale per row (amax / 448), nearest-even rounding, and an encoder whose bytes
 * every consumer reads identically.
 * Reading: the scale is amax/448 as an IEEE fp32 division, each element is divided
 * by it (fp32 IEEE division) and rounded to e4m3 with ties to even; a row with
 * amax = 0 stores scale 0 and all-zero codes.
 * =================================================================================== */
void orc_encode_fp8(const float* x, int64_t rows, int dim, int64_t ldx,
                    uint8_t* codes, int64_t ldc, float* scales)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ldx;
        uint8_t* cr = codes + r * ldc;
        float amax = 0.0f;
        for (int i = 0; i < dim; ++i) {
            float a = fabsf(xr[i]);
            if (a > amax) amax = a;
        }
        float s = amax / 448.0f;
        scales[r] = s;
        for (int i = 0; i < dim; ++i)
            cr[i] = (amax == 0.0f) ? 0x00 : orc_e4m3_rne(xr[i] / s);
    }
}

void orc_decode_fp8(const uint8_t* codes, int64_t rows, int dim, int64_t ldc,
                    const float* scales, double* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < dim; ++i)
            out[r * dim + i] = orc_e4m3_value(codes[r * ldc + i]) * (double)scales[r];
}

/* ===================================================================================
 * Rotated-int4 (TQ4) — colibri PR #399, "Why rotated-int4 for the 4-bit tier":
 * a randomized-Hadamard rotation, then a fixed 16-level Lloyd-Max codebook that is
 * optimal for N(0,1) and scaled by radius/sqrt(n); one fp32 radius per row survives
 * the rotation.  The non-power-of-two refusal follows the rebase note ("KV_TQ now
 * refuses non-power-of-two latent row widths").
 * =================================================================================== */

static double std_normal_pdf(double t) { return exp(-0.5 * t * t) / sqrt(2.0 * M_PI); }
static double std_normal_cdf(double t) { return 0.5 * erfc(-t / sqrt(2.0)); }

/* Lloyd-Max for N(0,1) with L = 2^bits levels: the fixed point of "thresholds are the
 * midpoints of adjacent centroids" and "each centroid is the conditional mean of its
 * cell",
 *   c_k = (phi(t_k) - phi(t_{k+1})) / (Phi(t_{k+1}) - Phi(t_k)),  t_k = (c_{k-1} + c_k) / 2,
 * with t_0 = -inf and t_L = +inf.  The stored codebook is each centroid rounded to the
 * nearest binary16 value; the thresholds are the midpoints of the stored centroids
 * (exact in fp32).
 *
 * 16 levels (the 4-bit tier): the plain alternation from a uniform start on [-3, 3]
 * until no centroid moves by 1e-15, or, since the last bits of exp/erfc differ between
 * C libraries and can leave the iterate oscillating at the rounding level, after 20000
 * steps (by then the moves are below 1e-14).
 * 8 and 64 levels: the alternation converges too slowly at 64 levels (its contraction
 * factor is close to 1), so after 500 warm-up steps the same fixed point is solved by
 * Newton's method on c - T(c) = 0.  T_k depends on c_{k-1}, c_k, c_{k+1} only, through
 *   dT_k/dt_k     = phi(t_k) (T_k - t_k) / mass_k,
 *   dT_k/dt_{k+1} = phi(t_{k+1}) (t_{k+1} - T_k) / mass_k,
 * and dt_k/dc_{k-1} = dt_k/dc_k = 1/2, so each step is one tridiagonal solve.  It stops
 * when no centroid moves by 1e-15 (at most 60 steps).
 * The pins check the fixed-point condition to 1e-12 in closed form.  Computed once per
 * process and width. */
#define ORC_TQ_MAXL 64
typedef struct {
    int ready, iters;
    double lloyd[ORC_TQ_MAXL];
    float cb[ORC_TQ_MAXL], thr[ORC_TQ_MAXL];
} tq_codebook_t;
static tq_codebook_t g_tq_cb[7];     /* indexed by bits */

/* Phi(b) - Phi(a) without cancellation in either tail: from the upper tail
 * Q(x) = erfc(x / sqrt 2) / 2 when the cell lies above 0, the lower tail when below. */
static double cell_mass(double a, double b)
{
    const double r = 0.70710678118654752440;
    if (a >= 0.0) return 0.5 * (erfc(a * r) - erfc(b * r));
    if (b <= 0.0) return 0.5 * (erfc(-b * r) - erfc(-a * r));
    return 1.0 - 0.5 * erfc(b * r) - 0.5 * erfc(-a * r);
}

/* one Lloyd step: T(c) into cn; optional tridiagonal Jacobian of T (sub, diag, sup);
 * returns the largest |T_k - c_k|.  `tails`: cell masses from cell_mass (the 4-bit
 * codebook keeps the plain difference of the two CDF values it was computed with) */
static double lloyd_map(const double* c, int L, double* cn, double* sub, double* dia, double* sup,
                        int tails)
{
    double t[ORC_TQ_MAXL + 1];
    t[0] = -INFINITY; t[L] = INFINITY;
    for (int k = 1; k < L; ++k) t[k] = 0.5 * (c[k - 1] + c[k]);
    double move = 0.0;
    for (int k = 0; k < L; ++k) {
        double pa = isinf(t[k]) ? 0.0 : std_normal_pdf(t[k]);
        double pb = isinf(t[k + 1]) ? 0.0 : std_normal_pdf(t[k + 1]);
        double mass = tails ? cell_mass(t[k], t[k + 1]) : std_normal_cdf(t[k + 1]) - std_normal_cdf(t[k]);
        double ck = (pa - pb) / mass;
        if (fabs(ck - c[k]) > move) move = fabs(ck - c[k]);
        cn[k] = ck;
        if (dia) {
            double a = isinf(t[k]) ? 0.0 : pa * (ck - t[k]) / mass;          /* dT_k/dt_k     */
            double b = isinf(t[k + 1]) ? 0.0 : pb * (t[k + 1] - ck) / mass;  /* dT_k/dt_{k+1} */
            sub[k] = 0.5 * a;
            dia[k] = 0.5 * (a + b);
            sup[k] = 0.5 * b;
        }
    }
    return move;
}

static void tq_codebook_compute(int bits)
{
    const int L = 1 << bits;
    tq_codebook_t* cbk = &g_tq_cb[bits];
    double c[ORC_TQ_MAXL], cn[ORC_TQ_MAXL];
    int it = 0;
    if (bits == 4) {
        for (int k = 0; k < L; ++k) c[k] = -3.0 + 6.0 * k / (L - 1);
        for (it = 0; it < 20000; ++it) {
            double move = lloyd_map(c, L, cn, NULL, NULL, NULL, 0);
            memcpy(c, cn, sizeof(double) * L);
            if (move < 1e-15) break;
        }
    } else {
        for (int k = 0; k < L; ++k) c[k] = -3.0 + 6.0 * k / (L - 1);
        for (it = 0; it < 500; ++it) {
            lloyd_map(c, L, cn, NULL, NULL, NULL, 1);
            memcpy(c, cn, sizeof(double) * L);
        }
        double sub[ORC_TQ_MAXL], dia[ORC_TQ_MAXL], sup[ORC_TQ_MAXL];
        for (int n = 0; n < 60; ++n, ++it) {
            /* F(c) = T(c) - c = 0:  (J - I) delta = -F, J tridiagonal */
            lloyd_map(c, L, cn, sub, dia, sup, 1);
            double a[ORC_TQ_MAXL], b[ORC_TQ_MAXL], cc[ORC_TQ_MAXL], d[ORC_TQ_MAXL];
            for (int k = 0; k < L; ++k) {
                a[k] = sub[k];                /* coefficient of delta_{k-1} */
                b[k] = dia[k] - 1.0;          /* of delta_k                 */
                cc[k] = sup[k];               /* of delta_{k+1}             */
                d[k] = -(cn[k] - c[k]);
            }
            for (int k = 1; k < L; ++k) {     /* Thomas algorithm */
                double w = a[k] / b[k - 1];
                b[k] -= w * cc[k - 1];
                d[k] -= w * d[k - 1];
            }
            double delta[ORC_TQ_MAXL], move = 0.0;
            delta[L - 1] = d[L - 1] / b[L - 1];
            for (int k = L - 2; k >= 0; --k) delta[k] = (d[k] - cc[k] * delta[k + 1]) / b[k];
            for (int k = 0; k < L; ++k) {
                c[k] += delta[k];
                if (fabs(delta[k]) > move) move = fabs(delta[k]);
            }
            if (move < 1e-15) break;
        }
    }
    for (int k = 0; k < L; ++k) {
        cbk->lloyd[k] = c[k];
        cbk->cb[k] = (float)orc_f16_value(orc_f16_rne(c[k]));
    }
    for (int k = 0; k < L - 1; ++k) cbk->thr[k] = (cbk->cb[k] + cbk->cb[k + 1]) / 2.0f;
    cbk->iters = it;
    cbk->ready = 1;
}

static int tq_bits_ok(int bits) { return bits == 3 || bits == 4 || bits == 6; }

int orc_tq_codebook(int bits, double* lloyd, float* cb, float* thr, int* iters)
{
    if (!tq_bits_ok(bits)) return -1;
    const int L = 1 << bits;
    if (!g_tq_cb[bits].ready) tq_codebook_compute(bits);
    if (lloyd) memcpy(lloyd, g_tq_cb[bits].lloyd, sizeof(double) * L);
    if (cb) memcpy(cb, g_tq_cb[bits].cb, sizeof(float) * L);
    if (thr) memcpy(thr, g_tq_cb[bits].thr, sizeof(float) * (L - 1));
    if (iters) *iters = g_tq_cb[bits].iters;
    return 0;
}

int orc_tq4_codebook(double lloyd[16], float cb[16], float thr[15], int* iters)
{
    return orc_tq_codebook(4, lloyd, cb, thr, iters);
}

static int is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

/* Unnormalised fast Walsh-Hadamard transform, radix 2, stages h = 1, 2, 4, ... n/2 in
 * that order; each butterfly maps (a, b) to (a + b, a - b) in fp32. */
void orc_fwht_f32(float* w, int n)
{
    for (int h = 1; h < n; h <<= 1)
        for (int i = 0; i < n; ++i)
            if ((i & h) == 0) {
                float a = w[i], b = w[i + h];
                w[i] = a + b;
                w[i + h] = a - b;
            }
}

void orc_fwht_f64(double* w, int n)
{
    for (int h = 1; h < n; h <<= 1)
        for (int i = 0; i < n; ++i)
            if ((i & h) == 0) {
                double a = w[i], b = w[i + h];
                w[i] = a + b;
                w[i + h] = a - b;
            }
}

static int sign_is_negative(const uint32_t* bits, int i)
{
    return (bits[i >> 5] >> (i & 31)) & 1u;
}

/* TQ-b encode of one row (b = 3, 4, 6 bits), step by step:
 *   1. w = s (.) x with s_i = -1 where bit i of sign_bits is set;
 *   2. w = FWHT_n(w) (unnormalised, stages ascending), y = w * c, c = fp32(1/sqrt(n));
 *   3. ss = sum y_i^2 accumulated as 32 partial sums (partial l takes i = l, l+32, ...
 *      ascending, each step one fmaf), then folded by the butterfly
 *      p_l <- p_l + p_(l xor o) for o = 16, 8, 4, 2, 1;
 *   4. radius r = sqrtf(ss) (IEEE), sigma = r * c; a zero radius marks an inert row
 *      (all-zero bytes);
 *   5. u_i = y_i / sigma, code_i = number of thresholds t_k with u_i >= t_k;
 *   6. the codes form a little-endian bit stream: code i occupies bits b*i .. b*i + b - 1
 *      of the row's n*b/8 bytes (bit 0 is the low bit of byte 0).  For b = 4, element 2j
 *      is the low nibble of byte j and element 2j+1 the high nibble.
 * Returns -2 (and writes nothing) for a dimension that is not a power of two, -1 for an
 * unsupported width. */
int orc_encode_tq(int bits, const float* x, int64_t rows, int dim, int64_t ldx,
                  const uint32_t* sign_bits, uint8_t* packed, int64_t ldp, float* radius)
{
    if (!tq_bits_ok(bits)) return -1;
    if (!is_pow2(dim) || dim < 64) return -2;
    const int L = 1 << bits;
    float cb[ORC_TQ_MAXL], thr[ORC_TQ_MAXL];
    orc_tq_codebook(bits, NULL, cb, thr, NULL);
    const float c = (float)(1.0 / sqrt((double)dim));
    const int row_bytes = dim * bits / 8;
    float* y = (float*)malloc(sizeof(float) * (size_t)dim);
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * ldx;
        for (int i = 0; i < dim; ++i)
            y[i] = sign_is_negative(sign_bits, i) ? -xr[i] : xr[i];
        orc_fwht_f32(y, dim);
        for (int i = 0; i < dim; ++i) y[i] = y[i] * c;
        float part[32];
        for (int l = 0; l < 32; ++l) {
            float acc = 0.0f;
            for (int i = l; i < dim; i += 32) acc = fmaf(y[i], y[i], acc);
            part[l] = acc;
        }
        for (int o = 16; o >= 1; o >>= 1) {
            float nxt[32];
            for (int l = 0; l < 32; ++l) nxt[l] = part[l] + part[l ^ o];
            memcpy(part, nxt, sizeof part);
        }
        float rad = sqrtf(part[0]);
        float sigma = rad * c;
        uint8_t* pr = packed + r * ldp;
        radius[r] = rad;
        memset(pr, 0, (size_t)row_bytes);
        if (rad == 0.0f) continue;
        for (int i = 0; i < dim; ++i) {
            float u = y[i] / sigma;
            int n = 0;
            for (int k = 0; k < L - 1; ++k) n += (u >= thr[k]);
            for (int bit = 0; bit < bits; ++bit)
                if ((n >> bit) & 1) {
                    const int pos = bits * i + bit;
                    pr[pos >> 3] |= (uint8_t)(1u << (pos & 7));
                }
        }
    }
    free(y);
    return 0;
}

int orc_encode_tq4(const float* x, int64_t rows, int dim, int64_t ldx,
                   const uint32_t* sign_bits, uint8_t* packed, int64_t ldp,
                   float* radius)
{
    return orc_encode_tq(4, x, rows, dim, ldx, sign_bits, packed, ldp, radius);
}

/* code i of a TQ-b row (the bit stream above) */
static int tq_code(const uint8_t* pr, int bits, int i)
{
    int code = 0;
    for (int bit = 0; bit < bits; ++bit) {
        const int pos = bits * i + bit;
        code |= ((pr[pos >> 3] >> (pos & 7)) & 1) << bit;
    }
    return code;
}

/* TQ-b dequantisation in fp64: yhat_i = cb[code_i] * r / sqrt(n) (the rotated row) and
 * xhat = (1/sqrt(n)) * s (.) FWHT_n(yhat) (the row in the original basis). */
int orc_decode_tq(int bits, const uint8_t* packed, int64_t rows, int dim, int64_t ldp,
                  const float* radius, const uint32_t* sign_bits, double* xhat, double* yhat)
{
    if (!tq_bits_ok(bits)) return -1;
    if (!is_pow2(dim) || dim < 64) return -2;
    float cb[ORC_TQ_MAXL];
    orc_tq_codebook(bits, NULL, cb, NULL, NULL);
    const double inv_sqrt_n = 1.0 / sqrt((double)dim);
    double* w = (double*)malloc(sizeof(double) * (size_t)dim);
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* pr = packed + r * ldp;
        double sigma = (double)radius[r] * inv_sqrt_n;
        for (int i = 0; i < dim; ++i) w[i] = (double)cb[tq_code(pr, bits, i)] * sigma;
        if (yhat) memcpy(yhat + r * dim, w, sizeof(double) * (size_t)dim);
        if (xhat) {
            orc_fwht_f64(w, dim);
            for (int i = 0; i < dim; ++i) {
                double v = w[i] * inv_sqrt_n;
                xhat[r * dim + i] = sign_is_negative(sign_bits, i) ? -v : v;
            }
        }
    }
    free(w);
    return 0;
}

int orc_decode_tq4(const uint8_t* packed, int64_t rows, int dim, int64_t ldp,
                   const float* radius, const uint32_t* sign_bits,
                   double* xhat, double* yhat)
{
    return orc_decode_tq(4, packed, rows, dim, ldp, radius, sign_bits, xhat, yhat);
}

/* ===================================================================================
 * q4_0 paged cache — Strata PR #2533, kv_q4.metal port commit: fwht256 with the
 * orthonormal 1/16 scale; q4_group / q4_store, where of two elements with equal |x|
 * the larger value wins; the fp16 scale rounded to nearest even in software; the codeword
 * int(fma(x, id, 8.5f)) truncating toward zero.  Fixture commit: an all-zero group
 * gives d = -0.0 (scale bits 0x8000), id = 0, code 8, every qs byte 0x88.
 * =================================================================================== */

/* z = FWHT_256(x) * (1/16); stages h = 1 .. 128 ascending, fp32. */
void orc_fwht256_q4(const float* x, float* z)
{
    memcpy(z, x, sizeof(float) * 256);
    orc_fwht_f32(z, 256);
    for (int i = 0; i < 256; ++i) z[i] = z[i] * 0.0625f;
}

/* "a is preferred over b" in the tie rule: larger |.|, then larger value, then +0
 * over -0. */
static int q4_prefer(float a, float b)
{
    float fa = fabsf(a), fb = fabsf(b);
    if (fa != fb) return fa > fb;
    if (a != b) return a > b;
    return !signbit(a) && signbit(b);
}

/* One 32-element block -> 18 bytes: fp16 d (little endian) and 16 bytes whose low
 * nibble holds element j and high nibble element j + 16.
 *   mval = the element of largest magnitude (tie rule above), d = mval / -8,
 *   id = 1/d (0 when d is 0), q_j = trunc(fma(z_j, id, 8.5)) clamped to [0, 15]. */
void orc_q4_block(const float* z, uint8_t out[18])
{
    float mval = z[0];
    for (int j = 1; j < 32; ++j)
        if (q4_prefer(z[j], mval)) mval = z[j];
    float d = mval / -8.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    int q[32];
    for (int j = 0; j < 32; ++j) {
        float t = truncf(fmaf(z[j], id, 8.5f));
        int v = (int)t;
        if (v > 15) v = 15;
        if (v < 0) v = 0;
        q[j] = v;
    }
    uint16_t hb = orc_f16_rne((double)d);
    out[0] = (uint8_t)(hb & 0xFF);
    out[1] = (uint8_t)(hb >> 8);
    for (int j = 0; j < 16; ++j) out[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

static int64_t q4_cell(const int32_t* page_table, int max_pages, int page_size,
                       int seq, int pos, int64_t n_cells)
{
    int page = pos / page_size;
    if (page < 0 || page >= max_pages) return -1;
    int64_t pid = page_table[(int64_t)seq * max_pages + page];
    int64_t cell = pid * page_size + pos % page_size;
    if (pid < 0 || cell >= n_cells) return -1;
    return cell;
}

/* Append n_tok tokens of K and V ([n_seq][n_tok][n_heads][head_dim] fp32) at positions
 * pos0[s] .. pos0[s] + n_tok - 1 of each sequence; each (token, head) row is rotated
 * by fwht256 and stored as 8 blocks (144 bytes) at pool offset
 * (cell * n_heads + head) * 144, cell = page_table[s][pos / page_size] * page_size
 * + pos % page_size.  Returns -1 when a position falls outside the table or pool. */
int orc_append_q4(const float* k, const float* v, int n_seq, const int32_t* pos0,
                  int n_tok, int n_heads, int head_dim, const int32_t* page_table,
                  int max_pages, int page_size, int64_t n_cells,
                  uint8_t* k_pool, uint8_t* v_pool)
{
    if (head_dim != 256) return -2;
    float z[256];
    for (int s = 0; s < n_seq; ++s)
        for (int t = 0; t < n_tok; ++t) {
            int64_t cell = q4_cell(page_table, max_pages, page_size, s, pos0[s] + t, n_cells);
            if (cell < 0) return -1;
            for (int kv = 0; kv < 2; ++kv) {
                const float* src = kv ? v : k;
                uint8_t* pool = kv ? v_pool : k_pool;
                for (int h = 0; h < n_heads; ++h) {
                    const float* row = src + (((int64_t)s * n_tok + t) * n_heads + h) * 256;
                    orc_fwht256_q4(row, z);
                    uint8_t* dst = pool + (cell * n_heads + h) * 144;
                    for (int b = 0; b < 8; ++b) orc_q4_block(z + 32 * b, dst + 18 * b);
                }
            }
        }
    return 0;
}

/* ===================================================================================
 * The q4_0 append with its K/V projection (the producer that computes the rows rotates
 * and quantizes them: Strata PR #2533, the qsa decode commit, fwht_row256 in qsa_prep).
 * The pages leave the projection's arithmetic to the model; this library fixes it as
 * below, and the oracle follows the same steps so that the codes can be compared.
 * =================================================================================== */

/* element i of a weight matrix: fp32, or bfloat16 widened (its bits are the upper half
 * of an fp32 pattern) */
static float weight_at(const void* w, int w_bf16, int64_t i)
{
    if (!w_bf16) return ((const float*)w)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)w)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* y[r][c] = sum_k h[r][k] * w[k][c] (h [rows][d_model], w [d_model][n_out]): the k range
 * in 64 chunks of L = 4 * ceil(d_model / 256) consecutive terms (the last ones short or
 * empty); a chunk's sum is the chain acc = fmaf(h, w, acc) from 0 in ascending k; the 64
 * chunk sums are added in pairs (0+1, 2+3, ...), then the 32 results in pairs, and so on. */
void orc_project_rows(const float* h, int64_t rows, int d_model, const void* w, int w_bf16,
                      int64_t n_out, float* y)
{
    const int L = 4 * ((d_model + 255) / 256);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < n_out; ++c) {
            float part[64];
            for (int j = 0; j < 64; ++j) {
                float acc = 0.0f;
                int k_end = (j + 1) * L < d_model ? (j + 1) * L : d_model;
                for (int k = j * L; k < k_end; ++k)
                    acc = fmaf(h[r * d_model + k], weight_at(w, w_bf16, (int64_t)k * n_out + c), acc);
                part[j] = acc;
            }
            for (int n = 64; n > 1; n /= 2)
                for (int i = 0; i < n / 2; ++i) part[i] = part[2 * i] + part[2 * i + 1];
            y[r * n_out + c] = part[0];
        }
}

/* The projected rows of every new token (K with w_k, V with w_v; [n_seq][n_tok][n_heads
 * * 256]) appended as orc_append_q4 appends them. */
int orc_project_append_q4(const float* h, int n_seq, const int32_t* pos0, int n_tok,
                          int d_model, const void* w_k, const void* w_v, int w_bf16,
                          int n_heads, const int32_t* page_table, int max_pages,
                          int page_size, int64_t n_cells, uint8_t* k_pool, uint8_t* v_pool)
{
    const int64_t rows = (int64_t)n_seq * n_tok, n_out = (int64_t)n_heads * 256;
    float* k = (float*)malloc((size_t)(rows * n_out > 0 ? rows * n_out : 1) * sizeof(float));
    float* v = (float*)malloc((size_t)(rows * n_out > 0 ? rows * n_out : 1) * sizeof(float));
    if (!k || !v) { free(k); free(v); return -3; }
    orc_project_rows(h, rows, d_model, w_k, w_bf16, n_out, k);
    orc_project_rows(h, rows, d_model, w_v, w_bf16, n_out, v);
    int rc = orc_append_q4(k, v, n_seq, pos0, n_tok, n_heads, 256, page_table, max_pages,
                           page_size, n_cells, k_pool, v_pool);
    free(k);
    free(v);
    return rc;
}

/* Gather back to binary16 in the rotated domain: out = f16_rne((q - 8) * f32(d)),
 * out laid out [n_seq][n_tok][n_heads][256]. */
int orc_gather_q4(const uint8_t* pool, int n_seq, const int32_t* pos0, int n_tok,
                  int n_heads, int head_dim, const int32_t* page_table,
                  int max_pages, int page_size, int64_t n_cells, uint16_t* out)
{
    if (head_dim != 256) return -2;
    for (int s = 0; s < n_seq; ++s)
        for (int t = 0; t < n_tok; ++t) {
            int64_t cell = q4_cell(page_table, max_pages, page_size, s, pos0[s] + t, n_cells);
            if (cell < 0) return -1;
            for (int h = 0; h < n_heads; ++h) {
                const uint8_t* src = pool + (cell * n_heads + h) * 144;
                uint16_t* dst = out + (((int64_t)s * n_tok + t) * n_heads + h) * 256;
                for (int b = 0; b < 8; ++b) {
                    const uint8_t* blk = src + 18 * b;
                    uint16_t hb = (uint16_t)(blk[0] | (blk[1] << 8));
                    float d = (float)orc_f16_value(hb);
                    for (int j = 0; j < 32; ++j) {
                        int q = (j < 16) ? (blk[2 + j] & 15) : (blk[2 + j - 16] >> 4);
                        float val = (float)(q - 8) * d;
                        dst[32 * b + j] = orc_f16_rne((double)val);
                    }
                }
            }
        }
    return 0;
}

/* ===================================================================================
 * Absorbed-MLA decode attention in fp64 — colibri PR #399: the MLA latent is both key
 * and value; the decode kernels compute, per query and head,
 *   s_t = tau * (q_lat . c_t + q_rope . k_rope_t)   over the admissible rows t,
 *   out = sum_t softmax(s)_t c_t,     lse = log sum_t exp(s_t);
 * kernels that split T merge per-chunk partial softmax states, and the sparse
 * (DSA-style) gather restricts the rows to a top-k list of absolute row indices.  Rows are dequantised
 * exactly (fp8: code value * scale; TQ4: the fp64 inverse rotation of cb[code] *
 * r / sqrt(n)).  Causal multi-query (draft + verify): query j of a sequence holding L
 * rows sees rows t <= L - n_q + j.
 * =================================================================================== */

static int64_t mla_pool_row(const orc_mla* p, int s, int64_t t)
{
    if (!p->block_table) return (int64_t)s * p->seq_stride_rows + t;
    int64_t page = t / p->page_size;
    if (page >= p->max_pages) return -1;
    int32_t pid = p->block_table[(int64_t)s * p->max_pages + page];
    if (pid < 0) return -1;
    return (int64_t)pid * p->page_size + t % p->page_size;
}

/* dequantise pool row `row` of the tier `fmt` into c[d_lat] and kr[d_rope] (fp64) */
static void mla_dequant(const orc_mla* p, int fmt, int64_t row, double* c, double* kr)
{
    const int DL = p->d_lat, DR = p->d_rope;
    if (fmt == ORC_FMT_FP8) {
        orc_decode_fp8(p->fp8_lat + row * DL, 1, DL, DL, p->fp8_lat_scale + row, c);
        orc_decode_fp8(p->fp8_rope + row * DR, 1, DR, DR, p->fp8_rope_scale + row, kr);
    } else {
        /* the rotated tiers share one set of planes; the format gives the code width */
        const int bits = fmt == ORC_FMT_TQ3 ? 3 : fmt == ORC_FMT_TQ6 ? 6 : 4;
        const int rb = DL * bits / 8;
        orc_decode_tq(bits, p->tq4_lat + row * rb, 1, DL, rb, p->tq4_radius + row,
                      p->tq4_signs, c, NULL);
        orc_decode_fp8(p->tq4_rope + row * DR, 1, DR, DR, p->tq4_rope_scale + row, kr);
    }
}

int orc_mla_decode(const orc_mla* p, double* out, double* lse, uint32_t* bad_index)
{
    const int DL = p->d_lat, DR = p->d_rope, H = p->n_heads, NQ = p->n_q;
    const int D = DL + DR;
    int n_sel = p->seq_sel ? p->n_sel : p->n_seq;
    for (int si = 0; si < n_sel; ++si) {
        int s = p->seq_sel ? p->seq_sel[si] : si;
        int L = p->seq_len[s];
        int fmt = p->seq_fmt[s];
        for (int qi = 0; qi < NQ; ++qi) {
            /* the admissible rows of this query, in order */
            int64_t lim = p->causal ? (int64_t)L - NQ + qi : (int64_t)L - 1;
            int64_t n_cand = p->idx ? p->top_k : (int64_t)L;
            int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_cand > 0 ? n_cand : 1));
            int64_t n_rows = 0;
            for (int64_t j = 0; j < n_cand; ++j) {
                int64_t t = p->idx ? p->idx[((int64_t)s * NQ + qi) * p->top_k + j] : j;
                if (t < 0 || t >= L) { if (bad_index) *bad_index = 1; continue; }
                if (t > lim) continue;
                rows[n_rows++] = t;
            }
            /* dequantise those rows once */
            double* kv = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1) * D);
            for (int64_t j = 0; j < n_rows; ++j) {
                int64_t pr = mla_pool_row(p, s, rows[j]);
                if (pr < 0) { if (bad_index) *bad_index = 1; pr = 0; }
                mla_dequant(p, fmt, pr, kv + j * D, kv + j * D + DL);
            }
            double* sc = (double*)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
            for (int h = p->head_lo; h < p->head_hi; ++h) {
                const float* ql = p->q_lat + (((int64_t)s * NQ + qi) * H + h) * DL;
                const float* qr = p->q_rope + (((int64_t)s * NQ + qi) * H + h) * DR;
                double* o = out + (((int64_t)s * NQ + qi) * H + h) * DL;
                double* ls = lse + ((int64_t)s * NQ + qi) * H + h;
                for (int64_t j = 0; j < n_rows; ++j) {
                    const double* row = kv + j * D;
                    double dot = 0.0;
                    for (int i = 0; i < DL; ++i) dot += (double)ql[i] * row[i];
                    for (int i = 0; i < DR; ++i) dot += (double)qr[i] * row[DL + i];
                    sc[j] = (double)p->sm_scale * dot;
                }
                for (int i = 0; i < DL; ++i) o[i] = 0.0;
                if (n_rows == 0) { *ls = -INFINITY; continue; }
                if (p->n_split <= 0) {
                    /* direct: max-subtracted softmax over all admissible rows */
                    double m = -INFINITY;
                    for (int64_t j = 0; j < n_rows; ++j) if (sc[j] > m) m = sc[j];
                    double l = 0.0;
                    for (int64_t j = 0; j < n_rows; ++j) {
                        double e = exp(sc[j] - m);
                        l += e;
                        for (int i = 0; i < DL; ++i) o[i] += e * kv[j * D + i];
                    }
                    for (int i = 0; i < DL; ++i) o[i] /= l;
                    *ls = m + log(l);
                } else {
                    /* split-T: contiguous chunks of the admissible list, one partial
                     * (m_S, l_S, o_S) each, merged by the log-sum-exp combine
                     *   M = max m_S, L = sum l_S e^(m_S - M),
                     *   out = sum o_S e^(m_S - M) / L, lse = M + log L. */
                    int ns = p->n_split;
                    double* pm = (double*)malloc(sizeof(double) * ns);
                    double* pl = (double*)malloc(sizeof(double) * ns);
                    double* po = (double*)calloc((size_t)ns * DL, sizeof(double));
                    for (int S = 0; S < ns; ++S) {
                        int64_t a = n_rows * S / ns, b = n_rows * (S + 1) / ns;
                        double m = -INFINITY;
                        for (int64_t j = a; j < b; ++j) if (sc[j] > m) m = sc[j];
                        double l = 0.0;
                        for (int64_t j = a; j < b; ++j) {
                            double e = exp(sc[j] - m);
                            l += e;
                            for (int i = 0; i < DL; ++i) po[S * DL + i] += e * kv[j * D + i];
                        }
                        pm[S] = m; pl[S] = l;
                    }
                    double M = -INFINITY;
                    for (int S = 0; S < ns; ++S) if (pm[S] > M) M = pm[S];
                    double Ltot = 0.0;
                    for (int S = 0; S < ns; ++S)
                        if (pl[S] > 0.0) {
                            double w = exp(pm[S] - M);
                            Ltot += pl[S] * w;
                            for (int i = 0; i < DL; ++i) o[i] += po[S * DL + i] * w;
                        }
                    for (int i = 0; i < DL; ++i) o[i] /= Ltot;
                    *ls = M + log(Ltot);
                    free(pm); free(pl); free(po);
                }
            }
            free(sc); free(kv); free(rows);
        }
    }
    return 0;
}

/* ===================================================================================
 * q4_0 paged decode attention in fp64 — Strata PR #2533, the qsa decode commit: the q
 * attention rows pass through the orthonormal 256-point FWHT (as the K and V rows did
 * when they were appended); attention reads the q4 pools with every block dequantised
 * as (nibble - 8) * f32(d); the merged output row o = (sum_t p_t v_t) / L is rotated back
 * (the orthonormal FWHT is its own inverse) BEFORE the optional sigmoid(gate) multiply.
 * Grouped-query attention: query head h reads KV head h / (n_qh / n_kv).  Sequence s
 * holds tokens at positions 0 .. seq_len[s] - 1; a position whose page is missing or
 * outside the pool is skipped and flagged.
 *   q_rot = (1/16) FWHT256(q);  s_t = sm_scale * q_rot . k_t;  p = softmax(s)
 *   out = (1/16) FWHT256(sum_t p_t v_t) [* sigmoid(gate)];  lse = log sum_t exp(s_t)
 * out [n_seq][n_qh][256], lse [n_seq][n_qh] (NULL allowed).  An empty sequence gives
 * out = 0 and lse = -inf.  seq_sel (optional) restricts the sequences computed.
 * =================================================================================== */

/* the 256 values of one dequantised row (exact in fp32, returned in fp64) */
static void q4_row_values(const uint8_t* row, double* x)
{
    for (int b = 0; b < 8; ++b) {
        const uint8_t* blk = row + 18 * b;
        const float d = (float)orc_f16_value((uint16_t)(blk[0] | (blk[1] << 8)));
        for (int j = 0; j < 32; ++j) {
            const int q = (j < 16) ? (blk[2 + j] & 15) : (blk[2 + j - 16] >> 4);
            x[32 * b + j] = (double)((float)(q - 8) * d);
        }
    }
}

int orc_q4_decode(int n_seq, int n_qh, int n_kv, const int32_t* seq_len,
                  const int32_t* page_table, int max_pages, int page_size, int64_t n_cells,
                  const uint8_t* k_pool, const uint8_t* v_pool, const float* q,
                  const float* gate, double sm_scale, const int32_t* seq_sel, int n_sel,
                  double* out, double* lse, uint32_t* bad_page)
{
    if (n_kv <= 0 || n_qh % n_kv != 0) return -1;
    const int grp = n_qh / n_kv;
    double qr[256], kv[256], acc[256];
    const int n_run = seq_sel ? n_sel : n_seq;
    for (int si = 0; si < n_run; ++si) {
        const int s = seq_sel ? seq_sel[si] : si;
        const int L = seq_len[s];
        for (int h = 0; h < n_qh; ++h) {
            const int kvh = h / grp;
            const float* qh = q + ((int64_t)s * n_qh + h) * 256;
            for (int i = 0; i < 256; ++i) qr[i] = qh[i];
            orc_fwht_f64(qr, 256);
            for (int i = 0; i < 256; ++i) qr[i] /= 16.0;
            /* pass 1: the maximum score */
            double m = -INFINITY;
            for (int t = 0; t < L; ++t) {
                const int64_t cell = q4_cell(page_table, max_pages, page_size, s, t, n_cells);
                if (cell < 0) { if (bad_page) *bad_page = 1; continue; }
                q4_row_values(k_pool + (cell * n_kv + kvh) * 144, kv);
                double dot = 0.0;
                for (int i = 0; i < 256; ++i) dot += qr[i] * kv[i];
                const double sc = sm_scale * dot;
                if (sc > m) m = sc;
            }
            /* pass 2: weights and the weighted sum of the V rows */
            double l = 0.0;
            for (int i = 0; i < 256; ++i) acc[i] = 0.0;
            if (m > -INFINITY) {
                for (int t = 0; t < L; ++t) {
                    const int64_t cell = q4_cell(page_table, max_pages, page_size, s, t, n_cells);
                    if (cell < 0) continue;
                    q4_row_values(k_pool + (cell * n_kv + kvh) * 144, kv);
                    double dot = 0.0;
                    for (int i = 0; i < 256; ++i) dot += qr[i] * kv[i];
                    const double pw = exp(sm_scale * dot - m);
                    l += pw;
                    q4_row_values(v_pool + (cell * n_kv + kvh) * 144, kv);
                    for (int i = 0; i < 256; ++i) acc[i] += pw * kv[i];
                }
            }
            double* oh = out + ((int64_t)s * n_qh + h) * 256;
            if (l > 0.0) {
                for (int i = 0; i < 256; ++i) acc[i] /= l;
                orc_fwht_f64(acc, 256);                       /* rotate back ... */
                for (int i = 0; i < 256; ++i) {
                    double o = acc[i] / 16.0;
                    if (gate) {                                /* ... then gate */
                        const double g = gate[((int64_t)s * n_qh + h) * 256 + i];
                        o *= 1.0 / (1.0 + exp(-g));
                    }
                    oh[i] = o;
                }
            } else {
                for (int i = 0; i < 256; ++i) oh[i] = 0.0;
            }
            if (lse) lse[(int64_t)s * n_qh + h] = (l > 0.0) ? m + log(l) : -INFINITY;
        }
    }
    return 0;
}
