/*
 * tahq_wire_oracle.c -- plain, slow, scalar CPU oracle of the TAH-Quant WIRE FORMAT.
 * TEST INFRASTRUCTURE ONLY (see tahq_oracle.c): nothing in the product links or calls it.
 *
 * Source: "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over
 * Slow Network", §3.2 (the 1-bit per-tile bit map "packed with the quantized payload as
 * metadata"), §3.4 (heterogeneous precisions and their metadata packed into one
 * contiguous uint8 byte stream of fixed size per shape) and its table of communicated
 * bits per element (about 0.61 bits of metadata per element at a tile of 64, 4.41 bits in
 * all for 80% INT4 + 20% INT3).
 *
 * Readings where the pages leave the layout open (all are this build's own choices):
 *   - 39 metadata bits per tile at G = 64 = fp16 scale + fp16 zero + 1-bit width map +
 *     log2(G)-bit pivot.  A scale is never negative, so the sign bit of the fp16 scale
 *     carries the transform flag; an untransformed tile stores pivot 0.
 *   - "round the minimum down, the scale up, quantise with the rounded values": the zero
 *     is the largest fp16 value <= min, the scale the smallest fp16 value s >= 0 with
 *     zero + Q s >= max (exact arithmetic), and the codes are
 *     q_k = RNE((v_k - zero) * inv), inv = RN(1 / s), v_k - zero an fp32 difference,
 *     clamped to [0, Q]; s = 0 (a constant tile whose value is an fp16 number) gives
 *     q = 0.  Decode: v_k = fmaf(q_k, s, zero), then the inverse transform.
 *   - Values outside the fp16 range (|v| > 65504) make the zero or the scale infinite:
 *     undefined, like non-finite input.
 *   - Sections in this order, each at a 16-byte boundary: a 128-byte header, the width
 *     map (bit t = tile t is hi, LSB first), the per-tile (scale, zero) fp16 pairs, the
 *     pivot fields (pb = log2 G bits each, LSB first), the payload (the same packed slots
 *     as the plain codec).
 *
 * Header (little-endian): u32 magic "TAHQ"; u16 version 1; u16 header bytes 128;
 * i64 tokens; i64 channels; i64 tokens per group; u16 tile; u16 hblock; u8 bits_lo;
 * u8 bits_hi; u8 pivot bits; u8 0; f32 budget; f32 tau; u64 tiles; u64 offsets of the
 * width map, the (scale, zero) pairs, the pivots and the payload; u64 payload bytes;
 * u64 total bytes; zeros up to byte 128.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* from tahq_oracle.c */
int oracle_encode_tau(const void *x, int dtype, int64_t T, int64_t C, int G, int h, int lo,
                      int hi, float budget, int64_t S, float tau, uint8_t *codes, float *scales,
                      float *zeros, uint8_t *bits, uint8_t *pivots, float *keys, uint8_t *near);
int64_t oracle_payload_size(int64_t T, int64_t C, int G, int lo, int hi, float budget, int64_t S);
void oracle_transform(float *v, int G, int h, int d);
void oracle_inverse_transform(float *v, int G, int h, int d);
void oracle_pack_tile(const uint8_t *q, int G, int b, uint8_t *slot);
void oracle_unpack_tile(const uint8_t *slot, int G, int b, uint8_t *q);

#define WIRE_MAGIC 0x51484154u   /* bytes 'T' 'A' 'H' 'Q' */
#define WIRE_HEADER 128

/* ---------------------------------------------------------------------- fp16 numbers */

/* Exact value of an fp16 bit pattern (IEEE binary16). */
double oracle_f16_value(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);
    else v = ldexp((double)(1024 + m), e - 25);
    return s ? -v : v;
}

/* The fp16 pattern at position r of the increasing order of values (-inf .. +inf, 0 at 0). */
static uint16_t f16_of_rank(int r) { return r < 0 ? (uint16_t)(0x8000 | -r) : (uint16_t)r; }

/* The largest fp16 value <= x (bisection over the ordered patterns -inf .. +inf). */
uint16_t oracle_f16_round_down(float x)
{
    int lo = -0x7C00, hi = 0x7C00;            /* value(lo) = -inf <= x */
    if (oracle_f16_value(f16_of_rank(hi)) <= (double)x) return f16_of_rank(hi);
    while (hi - lo > 1) {                      /* value(lo) <= x < value(hi) */
        int mid = lo + (hi - lo) / 2;
        if (oracle_f16_value(f16_of_rank(mid)) <= (double)x) lo = mid; else hi = mid;
    }
    return f16_of_rank(lo);
}

/* zero + Q s >= mx, exactly: zero and Q s are multiples of 2^-24 below 2^25 in size, so
 * their sum is exact in double, and so is the comparison with the fp32 mx. */
static int covers(double zero, int Q, double s, float mx)
{
    return zero + (double)Q * s >= (double)mx;
}

/* The smallest fp16 s >= 0 with zero + Q s >= mx (+inf if no finite one does). */
uint16_t oracle_f16_scale_up(float zero, float mx, int Q)
{
    if (covers(zero, Q, 0.0, mx)) return 0;
    int lo = 0, hi = 0x7C00;                  /* not covers(lo); covers(hi) or hi = +inf */
    if (!covers(zero, Q, oracle_f16_value(0x7BFF), mx)) return 0x7C00;
    hi = 0x7BFF;
    while (hi - lo > 1) {
        int mid = lo + (hi - lo) / 2;
        if (covers(zero, Q, oracle_f16_value((uint16_t)mid), mx)) hi = mid; else lo = mid;
    }
    return (uint16_t)hi;
}

/* Quantise one (transformed or raw) tile with fp16 zero and scale, as stated above. */
void oracle_quantize_tile_f16(const float *v, int G, int b, uint8_t *q, uint16_t *scale16,
                              uint16_t *zero16, uint8_t *near)
{
    float mn = v[0], mx = v[0];
    for (int k = 1; k < G; k++) {
        if (v[k] < mn) mn = v[k];
        if (v[k] > mx) mx = v[k];
    }
    int Q = (1 << b) - 1;
    uint16_t z16 = oracle_f16_round_down(mn);
    float z = (float)oracle_f16_value(z16);
    uint16_t s16 = oracle_f16_scale_up(z, mx, Q);
    float s = (float)oracle_f16_value(s16);
    *zero16 = z16;
    *scale16 = s16;
    if (s == 0.0f) {
        for (int k = 0; k < G; k++) { q[k] = 0; if (near) near[k] = 0; }
        return;
    }
    float inv = 1.0f / s;
    for (int k = 0; k < G; k++) {
        double du = (double)(v[k] - z) * (double)inv;   /* exact: 24 x 24 bits */
        double r = rint(du);
        if (!(r >= 0.0)) r = 0.0;              /* also a NaN from out-of-range input */
        if (r > (double)Q) r = (double)Q;
        q[k] = (uint8_t)r;
        if (near) {
            double frac = du - floor(du);
            double tol = 1e-5 * (fabs(du) > 1.0 ? fabs(du) : 1.0);
            near[k] = (fabs(frac - 0.5) <= tol) ? 1 : 0;
        }
    }
}

/* ---------------------------------------------------------------------- layout */

static int64_t up16(int64_t x) { return (x + 15) / 16 * 16; }
static int log2i(int G) { int p = 0; while ((1 << p) < G) p++; return p; }

/* Total bytes of the buffer; off[0..3] = offsets of the width map, the (scale, zero)
 * pairs, the pivots and the payload; off[4] = payload bytes.  -1 on invalid arguments. */
int64_t oracle_wire_layout(int64_t T, int64_t C, int G, int lo, int hi, float budget, int64_t S,
                           int64_t *off)
{
    int64_t pay = oracle_payload_size(T, C, G, lo, hi, budget, S);
    if (pay < 0) return -1;
    int64_t n = T * (C / G);
    int pb = log2i(G);
    off[0] = WIRE_HEADER;
    off[1] = off[0] + up16((n + 7) / 8);
    off[2] = off[1] + up16(4 * n);
    off[3] = off[2] + up16((n * pb + 7) / 8);
    off[4] = pay;
    return off[3] + up16(pay);
}

static void put_u16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put_u32(uint8_t *p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static void put_u64(uint8_t *p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static uint16_t get_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t get_u32(const uint8_t *p) { uint32_t v = 0; for (int i = 3; i >= 0; i--) v = (v << 8) | p[i]; return v; }
static uint64_t get_u64(const uint8_t *p) { uint64_t v = 0; for (int i = 7; i >= 0; i--) v = (v << 8) | p[i]; return v; }

/* ---------------------------------------------------------------------- encode / decode */

/* Encode a [T, C] tensor (dtype as oracle_encode) into wire[0, wire_bytes).  The widths
 * and the transform decisions are the plain codec's (oracle_encode_tau); only the
 * quantiser's zero and scale differ.  near (T*C bytes, optional) flags the elements whose
 * scaled value lies within 1e-5 (relative) of a rounding boundary.  Returns 0, or -1 on
 * invalid arguments or a buffer shorter than oracle_wire_layout says. */
int oracle_encode_wire(const void *x, int dtype, int64_t T, int64_t C, int G, int h, int lo,
                       int hi, float budget, int64_t S, float tau, uint8_t *wire,
                       int64_t wire_bytes, uint8_t *near)
{
    int64_t off[5];
    int64_t total = oracle_wire_layout(T, C, G, lo, hi, budget, S, off);
    if (total < 0 || wire_bytes < total) return -1;
    int64_t n = T * (C / G);
    int pb = log2i(G);
    uint8_t *codes = (uint8_t *)malloc((size_t)(off[4] > 0 ? off[4] : 1));
    float *sc = (float *)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    float *ze = (float *)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    uint8_t *bits = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
    uint8_t *piv = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
    if (!codes || !sc || !ze || !bits || !piv) { free(codes); free(sc); free(ze); free(bits); free(piv); return -1; }
    int rc = oracle_encode_tau(x, dtype, T, C, G, h, lo, hi, budget, S, tau, codes, sc, ze, bits,
                               piv, NULL, NULL);
    if (rc) { free(codes); free(sc); free(ze); free(bits); free(piv); return -1; }

    memset(wire, 0, (size_t)total);
    uint8_t *hd = wire;
    put_u32(hd + 0, WIRE_MAGIC);
    put_u16(hd + 4, 1);
    put_u16(hd + 6, WIRE_HEADER);
    put_u64(hd + 8, (uint64_t)T);
    put_u64(hd + 16, (uint64_t)C);
    put_u64(hd + 24, (uint64_t)(S ? S : T));
    put_u16(hd + 32, (uint16_t)G);
    put_u16(hd + 34, (uint16_t)h);
    hd[36] = (uint8_t)lo;
    hd[37] = (uint8_t)hi;
    hd[38] = (uint8_t)pb;
    memcpy(hd + 40, &budget, 4);
    memcpy(hd + 44, &tau, 4);
    put_u64(hd + 48, (uint64_t)n);
    for (int i = 0; i < 4; i++) put_u64(hd + 56 + 8 * i, (uint64_t)off[i]);
    put_u64(hd + 88, (uint64_t)off[4]);
    put_u64(hd + 96, (uint64_t)total);

    const uint8_t *xb = (const uint8_t *)x;
    size_t esize = dtype == 0 ? 4 : 2;
    float a[128];
    uint8_t q[128];
    int64_t slot = 0;
    for (int64_t t = 0; t < n; t++) {
        /* the raw tile (bf16 widened exactly), transformed where the plain codec did */
        for (int k = 0; k < G; k++) {
            const uint8_t *e = xb + ((size_t)t * G + k) * esize;
            if (dtype == 0) memcpy(&a[k], e, 4);
            else { uint32_t u = (uint32_t)get_u16(e) << 16; memcpy(&a[k], &u, 4); }
        }
        int flag = piv[t] != 0xFF;
        if (flag) oracle_transform(a, G, h, piv[t]);
        int b = bits[t];
        uint16_t s16, z16;
        oracle_quantize_tile_f16(a, G, b, q, &s16, &z16, near ? near + t * G : NULL);
        oracle_pack_tile(q, G, b, wire + off[3] + slot);
        slot += G * b / 8;
        if (b == hi) wire[off[0] + t / 8] |= (uint8_t)(1u << (t % 8));
        put_u16(wire + off[1] + 4 * t, (uint16_t)(s16 | (flag ? 0x8000 : 0)));
        put_u16(wire + off[1] + 4 * t + 2, z16);
        int p = flag ? piv[t] : 0;
        for (int j = 0; j < pb; j++)
            if ((p >> j) & 1) {
                int64_t bit = t * pb + j;
                wire[off[2] + bit / 8] |= (uint8_t)(1u << (bit % 8));
            }
    }
    free(codes); free(sc); free(ze); free(bits); free(piv);
    return 0;
}

/* Header fields, for tests: out = {T, C, S, G, h, lo, hi, pb, n, off x4, payload, total}.
 * Returns 0, or -1 if the header is not a version-1 header. */
int oracle_wire_header(const uint8_t *wire, int64_t wire_bytes, int64_t *out)
{
    if (wire_bytes < WIRE_HEADER || get_u32(wire) != WIRE_MAGIC || get_u16(wire + 4) != 1 ||
        get_u16(wire + 6) != WIRE_HEADER)
        return -1;
    out[0] = (int64_t)get_u64(wire + 8);
    out[1] = (int64_t)get_u64(wire + 16);
    out[2] = (int64_t)get_u64(wire + 24);
    out[3] = get_u16(wire + 32);
    out[4] = get_u16(wire + 34);
    out[5] = wire[36];
    out[6] = wire[37];
    out[7] = wire[38];
    out[8] = (int64_t)get_u64(wire + 48);
    for (int i = 0; i < 4; i++) out[9 + i] = (int64_t)get_u64(wire + 56 + 8 * i);
    out[13] = (int64_t)get_u64(wire + 88);
    out[14] = (int64_t)get_u64(wire + 96);
    return 0;
}

/* Decode a buffer into fp32 [T, C] (the shape the header states; out must hold it).
 * Returns 0, or -1 on a bad header, a buffer shorter than the header says, or fields that
 * do not describe a valid stream. */
int oracle_decode_wire(const uint8_t *wire, int64_t wire_bytes, float *out)
{
    int64_t f[15];
    if (oracle_wire_header(wire, wire_bytes, f)) return -1;
    int64_t T = f[0], C = f[1], n = f[8];
    int G = (int)f[3], h = (int)f[4], lo = (int)f[5], hi = (int)f[6], pb = (int)f[7];
    if (G < 1 || G > 128 || C % G || n != T * (C / G) || f[14] > wire_bytes || pb != log2i(G))
        return -1;
    if (lo < 1 || hi > 8 || lo >= hi || h < 1 || G % h) return -1;
    const uint8_t *map = wire + f[9], *meta = wire + f[10], *pv = wire + f[11], *pay = wire + f[12];
    int64_t slot = 0;
    float a[128];
    uint8_t q[128];
    for (int64_t t = 0; t < n; t++) {
        int b = ((map[t / 8] >> (t % 8)) & 1) ? hi : lo;
        if (slot + G * b / 8 > f[13]) return -1;
        uint16_t s16 = get_u16(meta + 4 * t), z16 = get_u16(meta + 4 * t + 2);
        int flag = s16 >> 15;
        float s = (float)oracle_f16_value((uint16_t)(s16 & 0x7FFF));
        float z = (float)oracle_f16_value(z16);
        int p = 0;
        for (int j = 0; j < pb; j++) {
            int64_t bit = t * pb + j;
            p |= ((pv[bit / 8] >> (bit % 8)) & 1) << j;
        }
        if (p >= G) return -1;
        oracle_unpack_tile(pay + slot, G, b, q);
        slot += G * b / 8;
        for (int k = 0; k < G; k++) a[k] = fmaf((float)q[k], s, z);
        if (flag) oracle_inverse_transform(a, G, h, p);
        memcpy(out + t * G, a, (size_t)G * sizeof(float));
    }
    return 0;
}
