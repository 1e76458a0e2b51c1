// tahq_line.cuh -- the "line" layout of the encode kernels, for tiles of 128 bytes or
// more (fp32 tiles of 32..128 values, bf16 tiles of 64 or 128).
//
// One lane holds one 128-byte line of the staged chunk (32 fp32 or 64 bf16 values); a
// tile spans LPT = 1, 2 or 4 consecutive lines, i.e. that many consecutive lanes.  The
// chunk is staged by a 2-D tensor copy with the 128-byte swizzle: 16-byte unit j of line
// l sits at unit j ^ (l & 7), so the eight lanes of a quarter-warp, reading the same unit
// of eight consecutive lines, touch eight different bank groups.
//
// Arithmetic follows the codec's canonical fp32 order (see tahq_device.cuh): the pairwise
// sums of a line are formed on packed pairs (k, k + 16), which keeps every level of the
// natural-order tree; products that feed an addition are fused (fmaf), as the canonical
// order prescribes, so the packed fma.rn.f32x2 reproduces them bit for bit.
#pragma once

#include "tahq_tile.cuh"

namespace tahq {

template <typename Tin, int G>
struct LineGeom {
  static constexpr int NE = 128 / (int)sizeof(Tin);       // values per line (lane)
  static constexpr int NW = 32;                           // 32-bit words per line
  static constexpr int LPT = G * (int)sizeof(Tin) / 128;  // lines (lanes) per tile
  static constexpr int TPS = 32 / LPT;                    // tiles per warp step
  static_assert(LPT == 1 || LPT == 2 || LPT == 4, "a tile spans 1, 2 or 4 lines");
};

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// The 32 words of line `line` of a swizzled chunk; word k = bytes [4k, 4k + 4).
__device__ __forceinline__ void lds_line(const unsigned char* buf, int line, uint32_t* w) {
  const unsigned char* base = buf + line * 128;
  const int x = (line & 7) << 4;
#pragma unroll
  for (int j = 0; j < 8; j++) {
    const uint4 q = *reinterpret_cast<const uint4*>(base + ((j << 4) ^ x));
    w[4 * j] = q.x;
    w[4 * j + 1] = q.y;
    w[4 * j + 2] = q.z;
    w[4 * j + 3] = q.w;
  }
}

// ------------------------------------------------------------------ entropy sums

// Constant operand pairs of the packed lg, built once in registers by the caller (read
// per use from shared memory they cost more than the arithmetic itself).
struct LgConsts {
  float2 k2, k1, k0;  // polynomial coefficients, both halves
  float2 m1;          // (-1, -1)
  float2 c127;        // -(2^23 + 127): exponent field + 2^23 -> exponent
  uint32_t lane4;     // lane * 4: column of the per-bank tables
};

__device__ __forceinline__ LgConsts lg_consts(const LgTables& tb, int lane) {
  LgConsts c;
  c.k2 = make_float2(tb.k[2], tb.k[2]);
  c.k1 = make_float2(tb.k[1], tb.k[1]);
  c.k0 = make_float2(tb.k[0], tb.k[0]);
  c.m1 = make_float2(-1.0f, -1.0f);
  c.c127 = make_float2(-8388735.0f, -8388735.0f);
  c.lane4 = (uint32_t)lane << 2;
  return c;
}

// lg of a pair of normal (or zero) magnitudes given as bits (tables g_lgT / g_lgR).  A
// zero magnitude gives lg = -127 (its term m lg m is then a zero).
__device__ __forceinline__ float2 lg_pair_f32(uint32_t a, uint32_t b, const LgConsts& c) {
  const uint32_t lane4 = c.lane4;
  const uint32_t oa = ((a >> 9) & 0x3F80u) | lane4, ob = ((b >> 9) & 0x3F80u) | lane4;
  const float2 F = make_float2(__uint_as_float((a >> 23) | 0x4B000000u),
                               __uint_as_float((b >> 23) | 0x4B000000u));
  const float2 mm = make_float2(__uint_as_float((a & 0x007FFFFFu) | 0x3F800000u),
                                __uint_as_float((b & 0x007FFFFFu) | 0x3F800000u));
  const float2 r = fma2(mm, make_float2(lg_tab(g_lgR, oa), lg_tab(g_lgR, ob)), c.m1);
  float2 p = fma2(c.k2, r, c.k1);
  p = fma2(p, r, c.k0);
  const float2 t = fma2(p, r, make_float2(lg_tab(g_lgT, oa), lg_tab(g_lgT, ob)));
  const float2 ef = add2(F, c.c127);  // exponent - 127, exact
  return add2(ef, t);
}

// Half h (16 words, bytes [64 h, 64 h + 64)) of line `line` of a swizzled chunk.
__device__ __forceinline__ void lds_half(const unsigned char* buf, int line, int h, uint32_t* w) {
  const unsigned char* base = buf + line * 128;
  const int x = (line & 7) << 4;
#pragma unroll
  for (int j = 0; j < 4; j++) {
    const uint4 q = *reinterpret_cast<const uint4*>(base + (((4 * h + j) << 4) ^ x));
    w[4 * j] = q.x;
    w[4 * j + 1] = q.y;
    w[4 * j + 2] = q.z;
    w[4 * j + 3] = q.w;
  }
}

// {L, S} of 16 fp32 values: L = pairwise sum of m_k, S = pairwise sum of the fused pairs
// fmaf(m_2j+1, lg m_2j+1, RN(m_2j lg m_2j)); natural order.  Packed pairs (k, k + 8) keep
// every level of the tree.
__device__ __forceinline__ float2 half_sums_f32(const uint32_t* w, const LgTables& tb,
                                                const LgConsts& c) {
  uint32_t mb[16];
#pragma unroll
  for (int k = 0; k < 16; k++) mb[k] = w[k] & 0x7FFFFFFFu;
  // zero or subnormal magnitudes present?  (rare: those take the general lg)
  uint32_t mn = mb[0];
#pragma unroll
  for (int k = 1; k + 1 < 16; k += 2) mn = __vimin3_u32(mn, mb[k], mb[k + 1]);
  mn = min(mn, mb[15]);
  float2 m2[8], l2[8];
  if (mn >= 0x00800000u) {
#pragma unroll
    for (int k = 0; k < 8; k++) {
      m2[k] = make_float2(__uint_as_float(mb[k]), __uint_as_float(mb[k + 8]));
      l2[k] = lg_pair_f32(mb[k], mb[k + 8], c);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const float a = __uint_as_float(mb[k]), b = __uint_as_float(mb[k + 8]);
      m2[k] = make_float2(a, b);
      l2[k] = make_float2(a == 0.0f ? 0.0f : lg_canon<false>(a, tb.T, tb.R, tb.TB, tb.k),
                          b == 0.0f ? 0.0f : lg_canon<false>(b, tb.T, tb.R, tb.TB, tb.k));
    }
  }
  float2 L1[4], S1[4];
#pragma unroll
  for (int j = 0; j < 4; j++) {
    L1[j] = add2(m2[2 * j], m2[2 * j + 1]);
    S1[j] = fma2(m2[2 * j + 1], l2[2 * j + 1], mul2(m2[2 * j], l2[2 * j]));
  }
  const float2 Lt = tree2<4>(L1), St = tree2<4>(S1);
  return make_float2(__fadd_rn(Lt.x, Lt.y), __fadd_rn(St.x, St.y));
}

// {L, S} of 16 words of bf16 (32 values; word k holds values 2k (low half) and 2k + 1).
// The lg of a bf16 magnitude is exact from the table: e + TB[top 7 fraction bits].
__device__ __forceinline__ float2 half_sums_bf16(const uint32_t* w, const LgTables& tb,
                                                 const LgConsts& c) {
  // any half-word with exponent field 0 (zero or subnormal)?  those take the general lg
  uint32_t em = 0xFFFFFFFFu;
#pragma unroll
  for (int k = 0; k < 16; k++) em = __vminu2(em, w[k] & 0x7F807F80u);
  float2 L1[8], S1[8];
  if ((em & 0xFFFFu) != 0u && (em >> 16) != 0u) {
    const uint32_t lane4 = c.lane4;
#pragma unroll
    for (int k = 0; k < 8; k++) {
      const uint32_t a = w[k], b = w[k + 8];
      const float2 mlo = make_float2(__uint_as_float((a << 16) & 0x7FFF0000u),
                                     __uint_as_float((b << 16) & 0x7FFF0000u));
      const float2 mhi = make_float2(__uint_as_float(a & 0x7FFF0000u),
                                     __uint_as_float(b & 0x7FFF0000u));
      const float2 elo = make_float2(__uint_as_float(((a >> 7) & 0xFFu) | 0x4B000000u),
                                     __uint_as_float(((b >> 7) & 0xFFu) | 0x4B000000u));
      const float2 ehi = make_float2(__uint_as_float(((a >> 23) & 0xFFu) | 0x4B000000u),
                                     __uint_as_float(((b >> 23) & 0xFFu) | 0x4B000000u));
      const float2 tlo = make_float2(lg_tab(g_lgTB, ((a << 7) & 0x3F80u) | lane4),
                                     lg_tab(g_lgTB, ((b << 7) & 0x3F80u) | lane4));
      const float2 thi = make_float2(lg_tab(g_lgTB, ((a >> 9) & 0x3F80u) | lane4),
                                     lg_tab(g_lgTB, ((b >> 9) & 0x3F80u) | lane4));
      const float2 llo = add2(add2(elo, c.c127), tlo);
      const float2 lhi = add2(add2(ehi, c.c127), thi);
      L1[k] = add2(mlo, mhi);
      S1[k] = fma2(mhi, lhi, mul2(mlo, llo));
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; k++) {
      float l[2], sm[2];
#pragma unroll
      for (int q = 0; q < 2; q++) {
        const uint32_t x = w[k + 8 * q];
        const float a = __uint_as_float((x << 16) & 0x7FFF0000u);
        const float b = __uint_as_float(x & 0x7FFF0000u);
        const float la = a == 0.0f ? 0.0f : lg_canon<true>(a, tb.T, tb.R, tb.TB, tb.k);
        const float lb = b == 0.0f ? 0.0f : lg_canon<true>(b, tb.T, tb.R, tb.TB, tb.k);
        l[q] = __fadd_rn(a, b);
        sm[q] = __fmaf_rn(b, lb, __fmul_rn(a, la));
      }
      L1[k] = make_float2(l[0], l[1]);
      S1[k] = make_float2(sm[0], sm[1]);
    }
  }
  const float2 Lt = tree2<8>(L1), St = tree2<8>(S1);
  return make_float2(__fadd_rn(Lt.x, Lt.y), __fadd_rn(St.x, St.y));
}

// {L, S} of line `line` of a swizzled chunk, half by half: the line's tree is
// (half 0) + (half 1), each half pairwise in natural order.
template <typename Tin>
__device__ __forceinline__ float2 line_sums(const unsigned char* buf, int line, const LgTables& tb,
                                            const LgConsts& c) {
  float2 r[2];
#pragma unroll
  for (int h = 0; h < 2; h++) {
    uint32_t w[16];
    lds_half(buf, line, h, w);
    if constexpr (InTraits<Tin>::kBf16) {
      r[h] = half_sums_bf16(w, tb, c);
    } else {
      r[h] = half_sums_f32(w, tb, c);
    }
  }
  return add2(r[0], r[1]);
}

// ------------------------------------------------------------------ range and pretest

// min / max of the line, and the largest magnitude of each group of 8 consecutive values
// (ga[g], g < NE / 8) for the two-values pretest.
template <typename Tin>
__device__ __forceinline__ void line_minmax(const uint32_t* w, float& mn, float& mx, float* ga) {
  if constexpr (InTraits<Tin>::kBf16) {
#pragma unroll
    for (int g = 0; g < 8; g++) {
      __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&w[4 * g]);
      __nv_bfloat162 hi = lo;
#pragma unroll
      for (int k = 1; k < 4; k++) {
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[4 * g + k]);
        lo = __hmin2(lo, x);
        hi = __hmax2(hi, x);
      }
      const uint32_t l = *reinterpret_cast<const uint32_t*>(&lo);
      const uint32_t h = *reinterpret_cast<const uint32_t*>(&hi);
      const float gmn = fminf(__uint_as_float(l << 16), __uint_as_float(l & 0xFFFF0000u));
      const float gmx = fmaxf(__uint_as_float(h << 16), __uint_as_float(h & 0xFFFF0000u));
      ga[g] = fmaxf(gmx, -gmn);
      mn = g ? fminf(mn, gmn) : gmn;
      mx = g ? fmaxf(mx, gmx) : gmx;
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; g++) {
      const float* v = reinterpret_cast<const float*>(w + 8 * g);
      const float gmn8 = min3f(min3f(v[0], v[1], v[2]), min3f(v[3], v[4], v[5]), fminf(v[6], v[7]));
      const float gmx8 = max3f(max3f(v[0], v[1], v[2]), max3f(v[3], v[4], v[5]), fmaxf(v[6], v[7]));
      ga[g] = fmaxf(gmx8, -gmn8);
      mn = g ? fminf(mn, gmn8) : gmn8;
      mx = g ? fmaxf(mx, gmx8) : gmx8;
    }
  }
}

// ------------------------------------------------------------------ quantise + pack

// Fields of 8 codes (8b bits each) from the float bits 0x4B400000 + code of 8 values,
// code j at bits [j*b, j*b + b).  b <= 8.
__device__ __forceinline__ unsigned long long pack8(const uint32_t* q, int b) {
  if (b <= 4) {
    uint32_t acc = q[0], pw = 1u, spw = 1u;
#pragma unroll
    for (int j = 1; j < 8; j++) {
      pw <<= b;
      spw += pw;
      acc += q[j] * pw;
    }
    return (unsigned long long)(acc - 0x4B400000u * spw);
  }
  unsigned long long acc = 0ull;
#pragma unroll
  for (int j = 0; j < 8; j++) acc |= (unsigned long long)(q[j] & 0xFFu) << (j * b);
  return acc;
}

// Concatenate two fields of 8b bits into a 16b-bit value (lo, hi) and store its 2b bytes.
__device__ __forceinline__ void sts_two(unsigned char* dst, unsigned long long f0,
                                        unsigned long long f1, int b) {
  const int sh = 8 * b;  // 8..64
  unsigned long long lo = f0, hi = 0ull;
  if (sh < 64) {
    lo |= f1 << sh;
    hi = f1 >> (64 - sh);
  } else {
    hi = f1;
  }
  sts_bytes(dst, lo, hi, 2 * b);
}

// code bits (0x4B400000 + code) of a pair of values: fmaf(v - mn, inv, 1.5 * 2^23)
// (mg = the pair (1.5 * 2^23, 1.5 * 2^23))
__device__ __forceinline__ float2 qpair(float2 v, float2 nmn, float2 inv2, float2 mg) {
  return fma2(add2(v, nmn), inv2, mg);
}

// Quantise the lane's line with (mn, inv) at b bits and store its NE * b / 8 bytes.
template <typename Tin>
__device__ __forceinline__ void line_quant_store(const uint32_t* w, float mn, float inv, int b,
                                                 unsigned char* dst) {
  const float2 nmn = make_float2(-mn, -mn), inv2 = make_float2(inv, inv);
  const float2 mg = make_float2(12582912.0f, 12582912.0f);
  if constexpr (InTraits<Tin>::kBf16) {
    // 64 values: word k -> values 2k, 2k + 1; eight fields of 8 codes (4 words each)
#pragma unroll
    for (int h = 0; h < 4; h++) {
      unsigned long long f[2];
#pragma unroll
      for (int g2 = 0; g2 < 2; g2++) {
        uint32_t q[8];
        const int g = 2 * h + g2;
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const uint32_t x = w[4 * g + k];
          const float2 r = qpair(make_float2(__uint_as_float(x << 16),
                                             __uint_as_float(x & 0xFFFF0000u)), nmn, inv2, mg);
          q[2 * k] = __float_as_uint(r.x);
          q[2 * k + 1] = __float_as_uint(r.y);
        }
        f[g2] = pack8(q, b);
      }
      sts_two(dst + h * 2 * b, f[0], f[1], b);
    }
  } else {
    // 32 values in pairs (k, k + 16): fields of codes 0-7, 8-15, 16-23, 24-31
    uint32_t q[32];
#pragma unroll
    for (int k = 0; k < 16; k++) {
      const float2 r = qpair(make_float2(__uint_as_float(w[k]), __uint_as_float(w[k + 16])),
                             nmn, inv2, mg);
      q[k] = __float_as_uint(r.x);
      q[k + 16] = __float_as_uint(r.y);
    }
    const unsigned long long f0 = pack8(q, b), f1 = pack8(q + 8, b);
    const unsigned long long f2 = pack8(q + 16, b), f3 = pack8(q + 24, b);
    sts_two(dst, f0, f1, b);
    sts_two(dst + 2 * b, f2, f3, b);
  }
}

// ---- the same with the width known at compile time (no width branches; adjacent value
// pairs as loaded; the lane's bytes stored as whole 32-bit words)

template <int B>
__device__ __forceinline__ unsigned long long pack8_ct(const uint32_t* q) {
  if constexpr (B <= 4) {
    uint32_t acc = q[0];
    uint32_t spw = 1u;
#pragma unroll
    for (int j = 1; j < 8; j++) {
      acc += q[j] << (j * B);
      spw += 1u << (j * B);
    }
    return (unsigned long long)(acc - 0x4B400000u * spw);
  } else {
    unsigned long long acc = 0ull;
#pragma unroll
    for (int j = 0; j < 8; j++) acc |= (unsigned long long)(q[j] & 0xFFu) << (j * B);
    return acc;
  }
}

__host__ __device__ constexpr int lowbit_cap16(int n) { return (n & -n) < 16 ? (n & -n) : 16; }

// NF fields of 8 codes (8B bits each), concatenated, stored as NF * B / 4 words at dst
// (aligned to AL bytes).
template <int B, int NF, int AL>
__device__ __forceinline__ void store_fields(unsigned char* dst, const unsigned long long* f) {
  constexpr int NW = NF * B / 4, FB = 8 * B;
  static_assert(NF * B % 4 == 0, "whole words");
  uint32_t word[NW];
#pragma unroll
  for (int k = 0; k < NW; k++) {
    const int bit = 32 * k, fi = bit / FB, off = bit % FB;
    unsigned long long v = f[fi] >> off;
    if (off + 32 > FB && fi + 1 < NF) v |= f[fi + 1] << (FB - off);
    word[k] = (uint32_t)v;
  }
  if constexpr (AL >= 16 && NW % 4 == 0) {
#pragma unroll
    for (int k = 0; k < NW; k += 4)
      *reinterpret_cast<uint4*>(dst + 4 * k) = make_uint4(word[k], word[k + 1], word[k + 2], word[k + 3]);
  } else if constexpr (AL >= 8 && NW % 2 == 0) {
#pragma unroll
    for (int k = 0; k < NW; k += 2)
      *reinterpret_cast<uint2*>(dst + 4 * k) = make_uint2(word[k], word[k + 1]);
  } else {
#pragma unroll
    for (int k = 0; k < NW; k++) *reinterpret_cast<uint32_t*>(dst + 4 * k) = word[k];
  }
}

// Quantise the lane's line at B bits (compile time) and store its NE * B / 8 bytes; dst
// is aligned to the largest power of two (<= 16) dividing NE * B / 8, or to AL bytes if
// AL is smaller (AL = 0: no further limit).
template <typename Tin, int B, int AL = 0>
__device__ __forceinline__ void line_quant_store_ct(const uint32_t* w, float mn, float inv,
                                                    unsigned char* dst) {
  constexpr int NE = 128 / (int)sizeof(Tin), NF = NE / 8;
  const float2 nmn = make_float2(-mn, -mn), inv2 = make_float2(inv, inv);
  const float2 mg = make_float2(12582912.0f, 12582912.0f);
  unsigned long long f[NF];
#pragma unroll
  for (int g = 0; g < NF; g++) {
    uint32_t q[8];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      float2 v;
      if constexpr (InTraits<Tin>::kBf16) {
        const uint32_t x = w[4 * g + k];
        v = make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
      } else {
        v = make_float2(__uint_as_float(w[8 * g + 2 * k]), __uint_as_float(w[8 * g + 2 * k + 1]));
      }
      const float2 r = qpair(v, nmn, inv2, mg);
      q[2 * k] = __float_as_uint(r.x);
      q[2 * k + 1] = __float_as_uint(r.y);
    }
    f[g] = pack8_ct<B>(q);
  }
  constexpr int kNat = lowbit_cap16(NE * B / 8);
  store_fields<B, NF, (AL > 0 && AL < kNat) ? AL : kNat>(dst, f);
}

// Width B known at compile time (B > 0) or not (B == 0, width b); AL as in
// line_quant_store_ct.
template <typename Tin, int B, int AL = 0>
__device__ __forceinline__ void line_quant(const uint32_t* w, float mn, float inv, int b,
                                           unsigned char* dst) {
  if constexpr (B > 0) {
    line_quant_store_ct<Tin, B, AL>(w, mn, inv, dst);
  } else {
    line_quant_store<Tin>(w, mn, inv, b, dst);
  }
}

// ------------------------------------------------------------------ team re-read

// The lane's 32 bytes [sub * 32, sub * 32 + 32) of tile kt of a swizzled chunk, as
// lds_words gives them for an unswizzled one (a team of G * size / 32 lanes per tile).
template <typename Tin, int G>
__device__ __forceinline__ void lds_words_swz(const unsigned char* buf, int kt, int sub, uint32_t* w) {
  const int line = kt * LineGeom<Tin, G>::LPT + (sub >> 2);
  const int u0 = (sub & 3) * 2, x = line & 7;
  const unsigned char* base = buf + line * 128;
  const uint4 a = *reinterpret_cast<const uint4*>(base + ((u0 ^ x) << 4));
  const uint4 b = *reinterpret_cast<const uint4*>(base + (((u0 + 1) ^ x) << 4));
  w[0] = a.x;
  w[1] = a.y;
  w[2] = a.z;
  w[3] = a.w;
  w[4] = b.x;
  w[5] = b.y;
  w[6] = b.z;
  w[7] = b.w;
}

}  // namespace tahq
