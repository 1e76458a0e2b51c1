/*
 * tahq_naive_oracle.c -- plain, slow, scalar CPU oracle of the fixed-point GRADIENT
 * codec of the backward pass.  TEST INFRASTRUCTURE ONLY (see tahq_oracle.c): nothing in
 * the product links or calls it.
 *
 * Source: "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over
 * Slow Network", §3.5 and Algorithm 1 (the second stage sends Q_Naive of the gradient
 * with respect to the activations back to the first, which dequantises it; a simple
 * fixed-point compressor of 6-8 bits, as in AQ-SGD), Appendix H (4-bit stress test; a
 * NaN at 8 bits fixed by going to 10 bits; gradient scaling, eq. (24):
 * g_hat = Q(c g) / c with a constant c).
 *
 * Readings where the pages leave the arithmetic open (this build's own choices):
 *   - Q_Naive is the asymmetric uniform quantizer of §3.3 on the activation codec's tiles
 *     (G consecutive channels of one token), at one width b for every tile, 1 <= b <= 16
 *     (6-10 in the pages), with no bit allocation and no outlier transform.  Per tile:
 *     mn = min, mx = max, D = RN(mx - mn); a range below the cutoff
 *     D_min(b) = max(2^-120, 2^(b - 126)) gives scale 0 and codes 0 (the tile decodes to
 *     its minimum); else scale = RN(D / Q), inv = RN(Q / D), Q = 2^b - 1, and
 *     q_k = RNE(RN(v_k - mn) * inv) (the product exact), clamped to [0, Q].  The cutoff
 *     keeps inv finite and the scale a normal number at every width up to 16 (at 2^-120
 *     alone, widths above 6 could give a subnormal scale or an infinite inv).  Decode:
 *     fmaf(q_k, scale, mn).
 *   - Codes packed least significant bit first at b bits, tile after tile (G * b / 8
 *     bytes a tile); an fp32 scale and zero per tile.
 *   - Gradient scaling: the quantizer sees v = RN(c g) and the decoder returns
 *     RN(fmaf(q, scale, mn) / c).  c must be a power of two, so both steps are exact
 *     unless c g leaves the normal float range; c = 1 is the plain codec.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Bytes of the packed codes of a [T, C] tensor in tiles of G at b bits (0 if invalid). */
size_t oracle_naive_codes_bytes(int64_t T, int64_t C, int G, int b)
{
    if (T < 0 || C <= 0 || G <= 0 || C % G || b < 1 || b > 16 || (G * b) % 8) return 0;
    return (size_t)(T * (C / G)) * (size_t)(G * b / 8);
}

static int naive_args_ok(int64_t T, int64_t C, int G, int b, float c)
{
    if (T < 0 || C <= 0 || G <= 0 || C % G || b < 1 || b > 16 || (G * b) % 8) return 0;
    int e;
    /* a positive finite power of two: frexp gives exactly 0.5 */
    if (!(c > 0.0f) || !isfinite(c) || frexpf(c, &e) != 0.5f) return 0;
    return 1;
}

/* Quantise the G values v to b bits (see the header); near[k] (optional) marks codes
 * whose u_k lies within 1e-5 * max(1, |u_k|) of a .5 rounding boundary. */
static void naive_quantize_tile(const float *v, int G, int b, uint16_t *q, float *scale,
                                float *zero, uint8_t *near)
{
    float mn = v[0], mx = v[0];
    for (int k = 1; k < G; k++) {
        if (v[k] < mn) mn = v[k];
        if (v[k] > mx) mx = v[k];
    }
    const int Q = (1 << b) - 1;
    const float D = mx - mn;
    const float cutoff = ldexpf(1.0f, b - 126 > -120 ? b - 126 : -120);
    *zero = mn + 0.0f;
    if (!(D >= cutoff)) {
        *scale = 0.0f;
        for (int k = 0; k < G; k++) { q[k] = 0; if (near) near[k] = 0; }
        return;
    }
    *scale = D / (float)Q;
    const float inv = (float)Q / D;
    for (int k = 0; k < G; k++) {
        const double u = (double)(v[k] - mn) * (double)inv;  /* exact: 24 x 24 bits */
        double r = rint(u);
        if (r < 0.0) r = 0.0;
        if (r > (double)Q) r = (double)Q;
        q[k] = (uint16_t)r;
        if (near) {
            const double frac = u - floor(u);
            const double tol = 1e-5 * (fabs(u) > 1.0 ? fabs(u) : 1.0);
            near[k] = (fabs(frac - 0.5) <= tol) ? 1 : 0;
        }
    }
}

/* Encode: codes (oracle_naive_codes_bytes), scales and zeros (one per tile), near
 * (optional, one byte per element).  Returns 0, or -1 for invalid arguments. */
int oracle_naive_encode(const float *g, int64_t T, int64_t C, int G, int b, float c,
                        uint8_t *codes, float *scales, float *zeros, uint8_t *near)
{
    if (!naive_args_ok(T, C, G, b, c)) return -1;
    const int64_t n = T * (C / G);
    const size_t slot = (size_t)(G * b / 8);
    float *v = (float *)malloc(sizeof(float) * (size_t)G);
    uint16_t *q = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)G);
    if (!v || !q) { free(v); free(q); return -1; }
    memset(codes, 0, slot * (size_t)n);
    for (int64_t t = 0; t < n; t++) {
        for (int k = 0; k < G; k++) v[k] = c * g[t * G + k];
        naive_quantize_tile(v, G, b, q, &scales[t], &zeros[t], near ? near + t * G : NULL);
        uint8_t *s = codes + (size_t)t * slot;
        for (int k = 0; k < G; k++)
            for (int j = 0; j < b; j++)
                if ((q[k] >> j) & 1u) {
                    const int bit = k * b + j;
                    s[bit >> 3] |= (uint8_t)(1u << (bit & 7));
                }
    }
    free(v);
    free(q);
    return 0;
}

/* Decode into out [T, C] (fp32).  Returns 0, or -1 for invalid arguments. */
int oracle_naive_decode(const uint8_t *codes, const float *scales, const float *zeros,
                        int64_t T, int64_t C, int G, int b, float c, float *out)
{
    if (!naive_args_ok(T, C, G, b, c)) return -1;
    const int64_t n = T * (C / G);
    const size_t slot = (size_t)(G * b / 8);
    for (int64_t t = 0; t < n; t++) {
        const uint8_t *s = codes + (size_t)t * slot;
        for (int k = 0; k < G; k++) {
            unsigned q = 0;
            for (int j = 0; j < b; j++) {
                const int bit = k * b + j;
                q |= (unsigned)((s[bit >> 3] >> (bit & 7)) & 1u) << j;
            }
            out[t * G + k] = fmaf((float)q, scales[t], zeros[t]) / c;
        }
    }
    return 0;
}
