/*
 * tahq_oracle.c -- plain, slow, scalar CPU oracle of the TAH-Quant activation codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
 * baseline may build, load or call this file.  The CUDA library shares no code with it.
 *
 * Source: "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over
 * Slow Network" (arXiv 2506.01352v2):
 *   §3.1  tile-wise group quantization: C channels of a token split into G-wide tiles,
 *         each with its own scale and zero-point;
 *   §3.2  eq. (1)-(2) per-tile entropy of the normalised magnitudes, top-p% of the
 *         tiles of every sample get the high bit width, the rest the low one;
 *   §3.3  eq. (3) outlier ratio r = |a(1)| / (|a(2)| + rho), tau = 2.0;
 *         pivot swap P_d (first coordinate <-> arg-max coordinate);
 *         eq. (4) Hadamard transform a P_d H_G / sqrt(G); asymmetric uniform quantizer;
 *         inverse by H^T on the de-quantised values;
 *   §3.4  heterogeneous precisions packed into one contiguous uint8 byte stream of a
 *         fixed shape.
 * Prior-art page "Training Transformers with 4-bit Integers" (summary of arXiv 2306.11987):
 *   "The Hadamard Transform": Sylvester recursion H_k = [[H,H],[H,-H]] and the
 *   block-diagonal Hadamard matrix; "Hardware Implementation Considerations": INT4
 *   packing with element 0 in the low nibble.
 *
 * Readings taken where the pages are silent or garbled (each one is also listed in the
 * design notes):
 *   - eq. (2) is printed without its minus sign; the prose right after it says H is high
 *     for spread-out energy and low for a sharp outlier, so H is Shannon entropy
 *     -sum p log p.  eps, varsigma -> 0 with 0 log 0 = 0, an all-zero tile has H = 0,
 *     log base 2 (the base does not change the ranking).
 *   - With p_k = m_k / L (L = sum m_k), -sum p_k lg p_k = lg L - (sum m_k lg m_k) / L.
 *     That form is evaluated, in fp32, in a fixed order: pairwise sums (the first level
 *     of sum m_k lg m_k as one fused multiply-add per pair), our own table-driven lg.
 *   - rho = 1e-12f, strict r > tau, pivot = lowest index among equal maxima.
 *   - ranking scope: each group of tokens_per_group consecutive tokens (a "sample");
 *     K = floor((budget - lo) * n_g / (hi - lo)) tiles of a group get hi bits, chosen
 *     by (H descending, tile index ascending).
 *   - pivot goes to tile position 0; with hblock h < G the Hadamard is block diagonal.
 *   - Sylvester natural order, FWHT stages len = 1, 2, 4, ..., then x RN(1/sqrt(h)).
 *   - quantizer: min/max affine, float zero-point = min (a zero minimum emitted as +0),
 *     code = the integer nearest (ties to even) to the exact product of the rounded
 *     v - min and the rounded Q / (max - min);
 *     a tile whose range max-min is below 2^-120 (this includes max == min) is
 *     encoded as constant: scale 0, all codes 0, zero = min.
 *   - code k of a tile occupies bits [k*b, k*b+b) of its slot, LSB first within
 *     little-endian bytes; slots follow each other in tile order.
 *   - metadata per tile: fp32 scale, fp32 zero, u8 bit width, u8 pivot (0xFF = no
 *     transform).
 *
 * All fp32 arithmetic below is IEEE binary32 with round-to-nearest-even.  The file must
 * be compiled with -ffp-contract=off and without fast-math: a * b + c is two roundings
 * unless fmaf is written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* ------------------------------------------------------------------------------------ */
/* The canonical base-2 logarithm (table-driven, in the manner of Tang's logarithm).     */
/*                                                                                       */
/* x = 2^e * m with m in [1, 2).  i = the top 7 bits of m's fraction, c_i = 1 + i/128,   */
/* R_i = the float nearest 1/c_i, T_i = the float nearest -log2(R_i) (R_i as stored).    */
/*   r = fmaf(m, R_i, -1)        (m R_i - 1, rounded once; |r| < 2^-7 (1 + 2^-7))        */
/*   lg(x) = e + fmaf(P(r), r, T_i),  P(r) = fmaf(fmaf(k3, r, k2), r, k1)                 */
/* since log2(m) = -log2(R_i) + log2(1 + r).  k_j = (-1)^(j+1) / (j ln 2): the Mercator   */
/* series of log2(1 + r) cut after r^3 (truncation below 2e-9).                           */
/* ------------------------------------------------------------------------------------ */
static float T_tab[128], R_tab[128], P_k[4];
static int tables_ready = 0;

static void init_tables(void)
{
    if (tables_ready) return;
    for (int i = 0; i < 128; i++) {
        double c = 1.0 + (double)i / 128.0;
        R_tab[i] = (float)(1.0 / c);
        T_tab[i] = (float)(-log2((double)R_tab[i]));
    }
    const double ln2 = 0.69314718055994530942;
    for (int j = 1; j <= 3; j++)      /* log2(1+r) = sum_j (-1)^(j+1) r^j / (j ln 2) */
        P_k[j] = (float)(((j % 2) ? 1.0 : -1.0) / ((double)j * ln2));
    tables_ready = 1;
}

void oracle_log2_tables(float *T, float *R, float *k)
{
    init_tables();
    memcpy(T, T_tab, sizeof T_tab);
    memcpy(R, R_tab, sizeof R_tab);
    for (int j = 0; j < 3; j++) k[j] = P_k[j + 1];
}

static uint32_t f2u(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float u2f(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* lg of a positive finite float. */
float oracle_lg(float x)
{
    init_tables();
    uint32_t b = f2u(x);
    int e = (int)(b >> 23) - 127;
    if ((b >> 23) == 0) {                 /* subnormal: scale by 2^24 (exact) first */
        b = f2u(x * 16777216.0f);
        e = (int)(b >> 23) - 127 - 24;
    }
    int i = (int)((b >> 16) & 0x7Fu);
    float m = u2f((b & 0x007FFFFFu) | 0x3F800000u);   /* m in [1, 2) */
    float r = fmaf(m, R_tab[i], -1.0f);
    float p = fmaf(P_k[3], r, P_k[2]);
    p = fmaf(p, r, P_k[1]);
    float t = fmaf(p, r, T_tab[i]);
    return (float)e + t;
}

void oracle_lg_array(const float *x, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_lg(x[i]);
}

/* Pairwise sum of n = 2^k floats: sum(x[0..n)) = sum(x[0..n/2)) + sum(x[n/2..n)). */
float oracle_pairwise_sum(const float *x, int n)
{
    if (n == 1) return x[0];
    return oracle_pairwise_sum(x, n / 2) + oracle_pairwise_sum(x + n / 2, n - n / 2);
}

/* ------------------------------------------------------------------------------------ */
/* Per-tile statistics (§3.2 eq. (1)-(2), §3.3 eq. (3)).                                 */
/* ------------------------------------------------------------------------------------ */

/* Entropy key in bits:  H = lg L - S / L,  L = sum m_k,  S = sum m_k lg m_k.
 * Both sums are pairwise over the tile in natural order.  The first level of S is one
 * fused step per pair: fmaf(m_{2j+1}, lg m_{2j+1}, m_{2j} lg m_{2j}) (the even product
 * rounded, the odd one exact inside the fma); a zero magnitude contributes a zero term. */
float oracle_entropy_key(const float *a, int G)
{
    float m[128], lm[128], L1[64], S1[64];
    for (int k = 0; k < G; k++) {
        m[k] = fabsf(a[k]);
        lm[k] = (m[k] == 0.0f) ? 0.0f : oracle_lg(m[k]);
    }
    for (int j = 0; j < G / 2; j++) {
        L1[j] = m[2 * j] + m[2 * j + 1];
        S1[j] = fmaf(m[2 * j + 1], lm[2 * j + 1], m[2 * j] * lm[2 * j]);
    }
    float L = oracle_pairwise_sum(L1, G / 2);
    float S = oracle_pairwise_sum(S1, G / 2);
    if (L == 0.0f) return 0.0f;
    return oracle_lg(L) - S / L;
}

/* The same key over n values (an allocation tile of n = A channels, §3.2 "Tile
 * decomposition"; n a power of two >= 2), same order: fused first level of S over the
 * pairs (2j, 2j+1), then both sums pairwise in natural order.  NaN if the scratch
 * cannot be allocated. */
float oracle_entropy_key_n(const float *a, int64_t n)
{
    if (n <= 128) return oracle_entropy_key(a, (int)n);
    float *L1 = (float *)malloc((size_t)(n / 2) * sizeof(float));
    float *S1 = (float *)malloc((size_t)(n / 2) * sizeof(float));
    if (!L1 || !S1) { free(L1); free(S1); return NAN; }
    for (int64_t j = 0; j < n / 2; j++) {
        float m0 = fabsf(a[2 * j]), m1 = fabsf(a[2 * j + 1]);
        float l0 = (m0 == 0.0f) ? 0.0f : oracle_lg(m0), l1 = (m1 == 0.0f) ? 0.0f : oracle_lg(m1);
        L1[j] = m0 + m1;
        S1[j] = fmaf(m1, l1, m0 * l0);
    }
    float L = oracle_pairwise_sum(L1, (int)(n / 2));
    float S = oracle_pairwise_sum(S1, (int)(n / 2));
    free(L1);
    free(S1);
    if (L == 0.0f) return 0.0f;
    return oracle_lg(L) - S / L;
}

/* eq. (1)-(2) as printed (with the minus sign restored), in double with natural log:
 * p_k = |a_k| / (||a||_1 + eps),  H = -sum_k p_k log(p_k + vsig).  Diagnostic only. */
double oracle_entropy_literal(const float *a, int G, double eps, double vsig)
{
    double l1 = 0.0;
    for (int k = 0; k < G; k++) l1 += fabs((double)a[k]);
    double h = 0.0;
    for (int k = 0; k < G; k++) {
        double p = fabs((double)a[k]) / (l1 + eps);
        h += p * log(p + vsig);
    }
    return -h;
}

/* Top-2 magnitudes, pivot d (lowest index among equal maxima) and the outlier flag
 * r = m1 / (m2 + 1e-12f) > tau, r an IEEE fp32 division.  Appendix F of the pages varies
 * tau: 0 transforms every tile (every tile whose r is above zero), +inf none. */
void oracle_outlier_tau(const float *a, int G, float tau, int *pivot, int *flag,
                        float *m1_out, float *m2_out)
{
    int d = 0;
    float m1 = fabsf(a[0]);
    for (int k = 1; k < G; k++)
        if (fabsf(a[k]) > m1) { m1 = fabsf(a[k]); d = k; }
    float m2 = -1.0f;
    for (int k = 0; k < G; k++)
        if (k != d && fabsf(a[k]) > m2) m2 = fabsf(a[k]);
    float r = m1 / (m2 + 1e-12f);
    *pivot = d;
    *flag = (r > tau) ? 1 : 0;
    if (m1_out) *m1_out = m1;
    if (m2_out) *m2_out = m2;
}

/* The method's own threshold, tau = 2.0 (§3.3). */
void oracle_outlier(const float *a, int G, int *pivot, int *flag, float *m1_out, float *m2_out)
{
    oracle_outlier_tau(a, G, 2.0f, pivot, flag, m1_out, m2_out);
}

/* ------------------------------------------------------------------------------------ */
/* Hadamard transform with pivot swap (§3.3 eq. (4)).                                    */
/* ------------------------------------------------------------------------------------ */

/* In-place Sylvester FWHT of one block of h = 2^k values, natural order, no scaling:
 * stage len = 1, 2, 4, ..., h/2 maps each pair (j, j+len) to (a+b, a-b). */
void oracle_fwht(float *v, int h)
{
    for (int len = 1; len < h; len *= 2)
        for (int i = 0; i < h; i += 2 * len)
            for (int j = i; j < i + len; j++) {
                float a = v[j], b = v[j + len];
                v[j] = a + b;
                v[j + len] = a - b;
            }
}

static float inv_sqrt_h(int h) { return (float)(1.0 / sqrt((double)h)); }

/* v <- v P_d (H_h blocks) / sqrt(h): swap positions 0 and d, FWHT every h-block, scale. */
void oracle_transform(float *v, int G, int h, int d)
{
    float t = v[0]; v[0] = v[d]; v[d] = t;
    float c = inv_sqrt_h(h);
    for (int blk = 0; blk < G; blk += h) oracle_fwht(v + blk, h);
    for (int k = 0; k < G; k++) v[k] = v[k] * c;
}

/* Inverse: FWHT every h-block, scale, then undo the swap. */
void oracle_inverse_transform(float *v, int G, int h, int d)
{
    float c = inv_sqrt_h(h);
    for (int blk = 0; blk < G; blk += h) oracle_fwht(v + blk, h);
    for (int k = 0; k < G; k++) v[k] = v[k] * c;
    float t = v[0]; v[0] = v[d]; v[d] = t;
}

/* Dense reference in double: y = x H_h / sqrt(h) with H_h[j][k] = (-1)^popcount(j & k),
 * the closed form of the Sylvester recursion.  Diagnostic only. */
void oracle_hadamard_dense(const double *x, double *y, int h)
{
    double c = 1.0 / sqrt((double)h);
    for (int k = 0; k < h; k++) {
        double s = 0.0;
        for (int j = 0; j < h; j++)
            s += (__builtin_popcount((unsigned)(j & k)) & 1) ? -x[j] : x[j];
        y[k] = s * c;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Asymmetric uniform quantizer (§3.3) and bit packing (§3.4).                           */
/* ------------------------------------------------------------------------------------ */

/* Quantise G values to b bits: code_k = round-half-even(u_k), u_k = (v_k - mn) * inv
 * with v_k - mn and inv = Q / D each rounded to float and the product exact (one
 * rounding from the two floats to the code).  near[k] (optional) is set when u_k lies
 * within 1e-5 * max(1, |u_k|) of a .5 rounding boundary. */
void oracle_quantize_tile(const float *v, int G, int b, uint8_t *q, float *scale, float *zero,
                          uint8_t *near)
{
    float mn = v[0], mx = v[0];
    for (int k = 1; k < G; k++) {
        if (v[k] < mn) mn = v[k];
        if (v[k] > mx) mx = v[k];
    }
    int Q = (1 << b) - 1;
    float D = mx - mn;
    *zero = mn + 0.0f;   /* a minimum of zero is emitted as +0 (the set's -0/+0 are equal) */
    if (!(D >= 0x1p-120f)) {
        *scale = 0.0f;
        for (int k = 0; k < G; k++) { q[k] = 0; if (near) near[k] = 0; }
        return;
    }
    *scale = D / (float)Q;
    float inv = (float)Q / D;
    for (int k = 0; k < G; k++) {
        double du = (double)(v[k] - mn) * (double)inv;   /* exact: 24 x 24 bits */
        double r = rint(du);
        if (r < 0.0) r = 0.0;
        if (r > (double)Q) r = (double)Q;
        q[k] = (uint8_t)r;
        if (near) {
            double frac = du - floor(du);
            double tol = 1e-5 * (fabs(du) > 1.0 ? fabs(du) : 1.0);
            near[k] = (fabs(frac - 0.5) <= tol) ? 1 : 0;
        }
    }
}

/* Code k -> bits [k*b, k*b+b) of the slot, least significant bit first. */
void oracle_pack_tile(const uint8_t *q, int G, int b, uint8_t *slot)
{
    memset(slot, 0, (size_t)(G * b / 8));
    for (int k = 0; k < G; k++)
        for (int j = 0; j < b; j++)
            if ((q[k] >> j) & 1) {
                int bit = k * b + j;
                slot[bit >> 3] |= (uint8_t)(1u << (bit & 7));
            }
}

void oracle_unpack_tile(const uint8_t *slot, int G, int b, uint8_t *q)
{
    for (int k = 0; k < G; k++) {
        int val = 0;
        for (int j = 0; j < b; j++) {
            int bit = k * b + j;
            if ((slot[bit >> 3] >> (bit & 7)) & 1) val |= 1 << j;
        }
        q[k] = (uint8_t)val;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Tile-wise bit allocation (§3.2 "Top-p% tile selection").                              */
/* ------------------------------------------------------------------------------------ */

/* Number of tiles of a group that get the high bit width. */
int64_t oracle_hi_count(int64_t n_g, int lo, int hi, float budget)
{
    return (int64_t)floor(((double)budget - (double)lo) * (double)n_g / (double)(hi - lo));
}

typedef struct { float h; int64_t t; } key_t_;

static int cmp_rank(const void *pa, const void *pb)
{
    const key_t_ *a = (const key_t_ *)pa, *b = (const key_t_ *)pb;
    if (a->h > b->h) return -1;          /* higher entropy first */
    if (a->h < b->h) return 1;
    return (a->t < b->t) ? -1 : (a->t > b->t) ? 1 : 0;   /* then lower tile index */
}

/* bits[t] = hi for the K tiles of highest (H, -t), lo for the rest. */
int oracle_allocate(const float *H, int64_t n_g, int64_t K, int lo, int hi, uint8_t *bits)
{
    key_t_ *ord = (key_t_ *)malloc((size_t)(n_g > 0 ? n_g : 1) * sizeof(key_t_));
    if (!ord) return -1;
    for (int64_t t = 0; t < n_g; t++) { ord[t].h = H[t]; ord[t].t = t; }
    qsort(ord, (size_t)n_g, sizeof(key_t_), cmp_rank);
    for (int64_t t = 0; t < n_g; t++) bits[t] = (uint8_t)lo;
    for (int64_t j = 0; j < K && j < n_g; j++) bits[ord[j].t] = (uint8_t)hi;
    free(ord);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Whole-tensor encode / decode.                                                        */
/* ------------------------------------------------------------------------------------ */

static int valid_shape(int64_t T, int64_t C, int G, int h)
{
    if (T < 0 || C <= 0 || G < 8 || G > 128 || (G & (G - 1))) return 0;
    if (C % G) return 0;
    if (h < 2 || h > G || (h & (h - 1))) return 0;
    return 1;
}

static int valid_bits(int lo, int hi, float budget)
{
    if (lo < 1 || hi > 8 || lo >= hi) return 0;
    if (!((double)budget >= (double)lo && (double)budget <= (double)hi)) return 0;
    return 1;
}

/* Payload bytes with allocation tiles of A channels (A = G: the plain codec): K of the
 * n_gA = S C / A allocation tiles of a group get hi, i.e. K A / G quantisation tiles. */
int64_t oracle_payload_size_alloc(int64_t T, int64_t C, int G, int A, int lo, int hi,
                                  float budget, int64_t S)
{
    if (!valid_shape(T, C, G, G) || !valid_bits(lo, hi, budget)) return -1;
    if (A < G || A % G || C % A || ((A / G) & (A / G - 1))) return -1;
    if (S == 0) S = T;
    if (T == 0) return 0;
    if (S <= 0 || T % S) return -1;
    int64_t n_g = S * (C / G), n_ga = S * (C / A);
    int64_t K = oracle_hi_count(n_ga, lo, hi, budget);
    int64_t per_group = n_g * G * lo / 8 + K * (A / G) * G * (hi - lo) / 8;
    return (T / S) * per_group;
}

int64_t oracle_payload_size(int64_t T, int64_t C, int G, int lo, int hi, float budget, int64_t S)
{
    if (!valid_shape(T, C, G, G) || !valid_bits(lo, hi, budget)) return -1;
    if (S == 0) S = T;
    if (T == 0) return 0;
    if (S <= 0 || T % S) return -1;
    int64_t n_g = S * (C / G);
    int64_t K = oracle_hi_count(n_g, lo, hi, budget);
    int64_t per_group = n_g * G * lo / 8 + K * G * (hi - lo) / 8;
    return (T / S) * per_group;
}

static void load_tile(const void *x, int dtype, int64_t off, int G, float *a)
{
    if (dtype == ORACLE_F32) {
        memcpy(a, (const float *)x + off, (size_t)G * sizeof(float));
    } else {
        const uint16_t *xb = (const uint16_t *)x + off;
        for (int k = 0; k < G; k++) a[k] = u2f((uint32_t)xb[k] << 16);   /* exact widening */
    }
}

/* Encode a [T, C] tensor with outlier threshold tau (>= 0, +inf allowed).  keys (n_tiles
 * floats) and near (T*C bytes) are optional outputs for tests.  Returns 0, or -1 on
 * invalid arguments / allocation failure. */
/* Encode with allocation tiles of A channels (§3.2 "Tile decomposition": A a multiple
 * of G aligned with the quantisation tiles, A = C the token-level allocation; here
 * A / G a power of two and A | C): one entropy key per allocation tile over its A values,
 * ranked per group, and every quantisation tile takes its allocation tile's width.  The
 * outlier test, the transform and the quantiser stay per quantisation tile.  keys holds
 * n / (A / G) floats. */
int oracle_encode_alloc(const void *x, int dtype, int64_t T, int64_t C, int G, int h, int lo,
                        int hi, float budget, int64_t S, float tau, int A, uint8_t *codes,
                        float *scales, float *zeros, uint8_t *bits, uint8_t *pivots, float *keys,
                        uint8_t *near)
{
    if (!valid_shape(T, C, G, h) || !valid_bits(lo, hi, budget)) return -1;
    if (!(tau >= 0.0f)) return -1;  /* negative or NaN */
    if (A < G || A % G || C % A || ((A / G) & (A / G - 1))) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16) return -1;
    if (S == 0) S = T;
    if (T == 0) return 0;
    if (S <= 0 || T % S) return -1;
    int64_t W = C / G, n = T * W, m = A / G, na = n / m, n_ga = S * (C / A);
    float *H = keys ? keys : (float *)malloc((size_t)na * sizeof(float));
    int *piv = (int *)malloc((size_t)n * sizeof(int));
    uint8_t *abits = (uint8_t *)malloc((size_t)na);
    float *row = (float *)malloc((size_t)A * sizeof(float));
    if (!H || !piv || !abits || !row) {
        if (!keys) free(H);
        free(piv); free(abits); free(row);
        return -1;
    }
    float a[128];
    uint8_t q[128];

    /* 1. per-tile outlier test on the raw tile; per allocation tile its entropy key */
    for (int64_t t = 0; t < n; t++) {
        load_tile(x, dtype, t * G, G, a);
        int d, flag;
        oracle_outlier_tau(a, G, tau, &d, &flag, NULL, NULL);
        piv[t] = flag ? d : -1;
    }
    for (int64_t i = 0; i < na; i++) {
        for (int64_t k = 0; k < m; k++) load_tile(x, dtype, (i * m + k) * G, G, row + k * G);
        H[i] = oracle_entropy_key_n(row, A);
    }
    /* 2. per-group allocation over the allocation tiles; each tile takes its tile's width */
    int64_t K = oracle_hi_count(n_ga, lo, hi, budget);
    for (int64_t g = 0; g < T / S; g++)
        if (oracle_allocate(H + g * n_ga, n_ga, K, lo, hi, abits + g * n_ga)) {
            if (!keys) free(H);
            free(piv); free(abits); free(row);
            return -1;
        }
    for (int64_t t = 0; t < n; t++) bits[t] = abits[t / m];
    /* 3. transform, quantise and pack, slots in tile order */
    int64_t off = 0;
    for (int64_t t = 0; t < n; t++) {
        load_tile(x, dtype, t * G, G, a);
        if (piv[t] >= 0) oracle_transform(a, G, h, piv[t]);
        int b = bits[t];
        oracle_quantize_tile(a, G, b, q, &scales[t], &zeros[t], near ? near + t * G : NULL);
        oracle_pack_tile(q, G, b, codes + off);
        pivots[t] = (uint8_t)(piv[t] >= 0 ? piv[t] : 0xFF);
        off += G * b / 8;
    }
    if (!keys) free(H);
    free(piv); free(abits); free(row);
    return 0;
}

/* Allocation tile = quantisation tile (the pages' default, A = G), threshold tau. */
int oracle_encode_tau(const void *x, int dtype, int64_t T, int64_t C, int G, int h, int lo,
                      int hi, float budget, int64_t S, float tau, uint8_t *codes, float *scales,
                      float *zeros, uint8_t *bits, uint8_t *pivots, float *keys, uint8_t *near)
{
    return oracle_encode_alloc(x, dtype, T, C, G, h, lo, hi, budget, S, tau, G, codes, scales,
                               zeros, bits, pivots, keys, near);
}

/* The method as the pages state it: tau = 2.0 (§3.3). */
int oracle_encode(const void *x, int dtype, int64_t T, int64_t C, int G, int h, int lo, int hi,
                  float budget, int64_t S, uint8_t *codes, float *scales, float *zeros,
                  uint8_t *bits, uint8_t *pivots, float *keys, uint8_t *near)
{
    return oracle_encode_tau(x, dtype, T, C, G, h, lo, hi, budget, S, 2.0f, codes, scales,
                             zeros, bits, pivots, keys, near);
}

/* Decode into fp32 [T, C].  Returns 0, or -1 on invalid arguments / a bit width outside
 * 1..8 / a pivot outside the tile / a stream shorter than the slots need. */
int oracle_decode(const uint8_t *codes, int64_t codes_bytes, const float *scales, const float *zeros,
                  const uint8_t *bits, const uint8_t *pivots, int64_t T, int64_t C, int G, int h,
                  float *out)
{
    if (!valid_shape(T, C, G, h)) return -1;
    int64_t n = T * (C / G), off = 0;
    uint8_t q[128];
    for (int64_t t = 0; t < n; t++) {
        int b = bits[t];
        if (b < 1 || b > 8) return -1;
        if (pivots[t] != 0xFF && pivots[t] >= G) return -1;
        if (off + G * b / 8 > codes_bytes) return -1;
        oracle_unpack_tile(codes + off, G, b, q);
        float *v = out + t * G;
        for (int k = 0; k < G; k++) v[k] = fmaf((float)q[k], scales[t], zeros[t]);
        if (pivots[t] != 0xFF) oracle_inverse_transform(v, G, h, pivots[t]);
        off += G * b / 8;
    }
    return 0;
}
