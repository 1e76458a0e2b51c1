// tahq_tile.cuh -- per-lane tile arithmetic of the encode kernels.
//
// A tile of G values is held by a team of L = G / V consecutive lanes, V consecutive
// values per lane (32 bytes of input per lane: 16 bf16 or 8 fp32 values, fewer when the
// tile is narrower).  All integer-deciding arithmetic follows the codec's canonical fp32
// order (see tahq_device.cuh); packed fp32x2 adds round each component exactly like the
// scalar add, and bf16x2 min/max/compare are exact.
#pragma once

#include <cuda_bf16.h>

#include "tahq_device.cuh"

namespace tahq {

template <typename Tin>
struct InTraits;
template <>
struct InTraits<float> {
  static constexpr bool kBf16 = false;
  static constexpr bool kNoFraction = false;
};
template <>
struct InTraits<uint16_t> {  // bf16 bit patterns
  static constexpr bool kBf16 = true;
  static constexpr bool kNoFraction = true;
};

template <typename Tin, int G>
struct TileGeom {
  static constexpr int kLaneBytes = 32;
  static constexpr int kPerLane = kLaneBytes / (int)sizeof(Tin);
  static constexpr int V = (G < kPerLane) ? G : kPerLane;  // values per lane
  static constexpr int W = V * (int)sizeof(Tin) / 4;       // 32-bit words per lane
  static constexpr int L = G / V;                          // lanes per tile
  static constexpr int TPW = 32 / L;                       // tiles per warp step
  static_assert(W == 4 || W == 8, "a lane holds 16 or 32 bytes");
};

// Canonical lg tables replicated per bank, in static shared memory of the encode kernels
// (filled by each block at start): entry i for lane l at index i * 32 + l, so the 32 lanes'
// lookups never share a bank.
static __shared__ float g_lgT[128 * 32];   // fp32 input: T
static __shared__ float g_lgR[128 * 32];   // fp32 input: R
static __shared__ float g_lgTB[128 * 32];  // bf16 input: TB

// Byte offset of entry i for `lane` (i < 128): i * 128 + lane * 4.
__device__ __forceinline__ float lg_tab(const float* tab, uint32_t byte_off) {
  return *reinterpret_cast<const float*>(reinterpret_cast<const char*>(tab) + byte_off);
}

// Packed fp32x2 add, each component rounded to nearest even exactly like the scalar
// add.  Products stay scalar (__fmul_rn): a packed multiply followed by an add was
// measured to be fused into a single-rounding multiply-add on this target, which breaks
// the canonical two-rounding order; an add followed by anything cannot be fused.
// The two halves go to the instruction as a register pair (mov.b64 {lo, hi}), so the
// compiler can place them without shifting or moving values around.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// Packed fused multiply-add: a * b + c per component, rounded once (as fmaf).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Lane's words of tile kt from a staged chunk.
template <typename Tin, int G>
__device__ __forceinline__ void lds_words(const unsigned char* buf, int kt, int sub, uint32_t* w) {
  using Gm = TileGeom<Tin, G>;
  const uint4* p = reinterpret_cast<const uint4*>(buf + ((size_t)kt * G + sub * Gm::V) * sizeof(Tin));
#pragma unroll
  for (int i = 0; i < Gm::W / 4; i++) {
    const uint4 q = p[i];
    w[4 * i] = q.x;
    w[4 * i + 1] = q.y;
    w[4 * i + 2] = q.z;
    w[4 * i + 3] = q.w;
  }
}

// Words -> V fp32 values (bf16 widening is exact; element 2k is the low half of word k).
template <typename Tin, int G>
__device__ __forceinline__ void words_to_values(const uint32_t* w, float* v) {
  using Gm = TileGeom<Tin, G>;
  if constexpr (InTraits<Tin>::kBf16) {
#pragma unroll
    for (int k = 0; k < Gm::W; k++) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int k = 0; k < Gm::W; k++) v[k] = __uint_as_float(w[k]);
  }
}

// Pairwise tree over n = 2^k float2 values (both components at once).
template <int N>
__device__ __forceinline__ float2 tree2(const float2* x) {
  if constexpr (N == 1) {
    return x[0];
  } else {
    return add2(tree2<N / 2>(x), tree2<N / 2>(x + N / 2));
  }
}

template <int L>
__device__ __forceinline__ float2 team_sum2(float2 s) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) {
    float2 t;
    t.x = __shfl_xor_sync(kFull, s.x, o);
    t.y = __shfl_xor_sync(kFull, s.y, o);
    s = add2(s, t);
  }
  return s;
}

template <int L>
__device__ __forceinline__ uint32_t team_sum_u(uint32_t s) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) s += __shfl_xor_sync(kFull, s, o);
  return s;
}

// ------------------------------------------------------------------ entropy key

// The two sums of the team's tile that the entropy key needs: L = sum |a_k| and
// S = sum |a_k| lg |a_k|, both pairwise in natural order (returned as {L, S} in every
// lane of the team).  The first level of S is fmaf(m_odd, lg m_odd, RN(m_even lg m_even))
// per pair.  Table lookups go to the per-bank replicated g_lgT / g_lgR / g_lgTB.
template <typename Tin, int G>
__device__ __forceinline__ float2 tile_sums(const uint32_t* w, const LgTables& tb, int lane) {
  using Gm = TileGeom<Tin, G>;
  constexpr int V = Gm::V;
  float2 ls[V / 2];  // level 1: {m_2j + m_2j+1, fused pair of S}
  if constexpr (InTraits<Tin>::kBf16) {
    // bf16 subnormals (exponent 0, mantissa != 0) need the normalising path
    uint32_t subn = 0u;
#pragma unroll
    for (int k = 0; k < Gm::W; k++) {
      const uint32_t m = w[k] & 0x7FFF7FFFu;
      subn |= (m + 0x7FFF7FFFu) & ~(m + 0x7F807F80u);
    }
    if (subn & 0x80008000u) {
      float v[V];
      words_to_values<Tin, G>(w, v);
#pragma unroll
      for (int j = 0; j < V; j += 2) {
        const float m0 = fabsf(v[j]), m1 = fabsf(v[j + 1]);
        const float l0 = m0 == 0.0f ? 0.0f : lg_canon<true>(m0, tb.T, tb.R, tb.TB, tb.k);
        const float l1 = m1 == 0.0f ? 0.0f : lg_canon<true>(m1, tb.T, tb.R, tb.TB, tb.k);
        ls[j / 2] = make_float2(__fadd_rn(m0, m1), __fmaf_rn(m1, l1, __fmul_rn(m0, l0)));
      }
    } else {
      const uint32_t lane4 = (uint32_t)lane << 2;
#pragma unroll
      for (int k = 0; k < Gm::W; k++) {
        const uint32_t x = w[k];
        const float mlo = __uint_as_float((x << 16) & 0x7FFF0000u);
        const float mhi = __uint_as_float(x & 0x7FFF0000u);
        const float elo = __uint_as_float(((x >> 7) & 0xFFu) | 0x4B000000u);
        const float ehi = __uint_as_float(((x >> 23) & 0xFFu) | 0x4B000000u);
        const float tlo = lg_tab(g_lgTB, ((x << 7) & 0x3F80u) | lane4);
        const float thi = lg_tab(g_lgTB, ((x >> 9) & 0x3F80u) | lane4);
        const float2 ef = add2(make_float2(elo, ehi), make_float2(-8388735.0f, -8388735.0f));
        const float2 lg = add2(ef, make_float2(tlo, thi));  // e + TB[i]
        // a zero magnitude gives lg = -127 and a zero term (its sign cannot reach H)
        ls[k] = make_float2(__fadd_rn(mlo, mhi), __fmaf_rn(mhi, lg.y, __fmul_rn(mlo, lg.x)));
      }
    }
  } else {
    float lgv[V], m[V];
    const float k2 = tb.k[2], k1 = tb.k[1], k0 = tb.k[0];  // once, not per value
#pragma unroll
    for (int j = 0; j < V; j++) {
      m[j] = fabsf(__uint_as_float(w[j]));
      const uint32_t b = __float_as_uint(m[j]);
      const uint32_t E = b >> 23;
      if (E == 0u && b != 0u) {
        lgv[j] = lg_canon<false>(m[j], tb.T, tb.R, tb.TB, tb.k);
      } else {  // normal, or zero (lg = -127, a zero term)
        const uint32_t off = ((b >> 9) & 0x3F80u) | ((uint32_t)lane << 2);
        const float ef = __fsub_rn(__uint_as_float(0x4B000000u | E), 8388735.0f);
        const float mm = __uint_as_float((b & 0x007FFFFFu) | 0x3F800000u);
        const float r = __fmaf_rn(mm, lg_tab(g_lgR, off), -1.0f);
        float p = __fmaf_rn(k2, r, k1);
        p = __fmaf_rn(p, r, k0);
        lgv[j] = __fadd_rn(ef, __fmaf_rn(p, r, lg_tab(g_lgT, off)));
      }
    }
#pragma unroll
    for (int j = 0; j < V; j += 2)
      ls[j / 2] = make_float2(__fadd_rn(m[j], m[j + 1]),
                              __fmaf_rn(m[j + 1], lgv[j + 1], __fmul_rn(m[j], lgv[j])));
  }
  return team_sum2<Gm::L>(tree2<V / 2>(ls));
}

// Entropy key in bits from the two sums: H = lg L - S / L (0 for an all-zero tile).
__device__ __forceinline__ float entropy_key(float Ls, float Ss, const LgTables& tb) {
  return (Ls == 0.0f) ? 0.0f
                      : __fsub_rn(lg_canon<false>(Ls, tb.T, tb.R, tb.TB, tb.k), __fdiv_rn(Ss, Ls));
}

// ------------------------------------------------------------------ quantizer

// min / max of the lane's raw values (exact; bf16 via packed bf16x2 min/max).
template <typename Tin, int G>
__device__ __forceinline__ void lane_minmax_raw(const uint32_t* w, float& mn, float& mx) {
  using Gm = TileGeom<Tin, G>;
  if constexpr (InTraits<Tin>::kBf16) {
    __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&w[0]);
    __nv_bfloat162 hi = lo;
#pragma unroll
    for (int k = 1; k < Gm::W; k++) {
      const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
      lo = __hmin2(lo, x);
      hi = __hmax2(hi, x);
    }
    const uint32_t l = *reinterpret_cast<const uint32_t*>(&lo);
    const uint32_t h = *reinterpret_cast<const uint32_t*>(&hi);
    mn = fminf(__uint_as_float(l << 16), __uint_as_float(l & 0xFFFF0000u));
    mx = fmaxf(__uint_as_float(h << 16), __uint_as_float(h & 0xFFFF0000u));
  } else {
    mn = mx = __uint_as_float(w[0]);
#pragma unroll
    for (int k = 1; k < Gm::W; k++) {
      mn = fminf(mn, __uint_as_float(w[k]));
      mx = fmaxf(mx, __uint_as_float(w[k]));
    }
  }
}

// Whether two or more values of the team's tile have |v| >= thr, from a lane-level test
// (for L >= 2: two lanes whose own max |v| reaches thr; one lane alone is inconclusive
// and returns false).  `lane_amax` is the lane's own max |v|.
template <int L>
__device__ __forceinline__ bool team_two_ge(float lane_amax, float thr, int team) {
  const unsigned m = __ballot_sync(kFull, lane_amax >= thr);
  const unsigned mine = (m >> (team * L)) & ((L == 32) ? 0xFFFFFFFFu : ((1u << L) - 1u));
  return __popc(mine) >= 2;
}

// Number of lane values with |v| >= thr (thr = m1 / 2, exact).
template <typename Tin, int G>
__device__ __forceinline__ uint32_t lane_count_ge(const uint32_t* w, float thr) {
  using Gm = TileGeom<Tin, G>;
  uint32_t c = 0;
  if constexpr (InTraits<Tin>::kBf16) {
    const uint32_t t16 = __float_as_uint(thr) >> 16;  // thr is a bf16 value
    const uint32_t tt = t16 | (t16 << 16);
    const __nv_bfloat162 t2 = *reinterpret_cast<const __nv_bfloat162*>(&tt);
    __nv_bfloat162 acc = __float2bfloat162_rn(0.0f);
#pragma unroll
    for (int k = 0; k < Gm::W; k++) {
      const uint32_t a = w[k] & 0x7FFF7FFFu;
      acc = __hadd2(acc, __hge2(*reinterpret_cast<const __nv_bfloat162*>(&a), t2));
    }
    c = (uint32_t)__bfloat162float(acc.x) + (uint32_t)__bfloat162float(acc.y);
  } else {
#pragma unroll
    for (int k = 0; k < Gm::W; k++) c += (fabsf(__uint_as_float(w[k])) >= thr) ? 1u : 0u;
  }
  return c;
}

// Quantise 8 values to b bits with the tile's (mn, inv); code j at bits [j*b, j*b+b).
//   code = the integer nearest (v - mn) * inv, the difference rounded and the product
//   exact: fmaf(v - mn, inv, 1.5*2^23) rounds at integer spacing (ties to even), and the
//   float bits are then 0x4B400000 + code.  The product lies in [0, Q (1 + 2^-24)], so
//   the code never exceeds Q and no clamp is needed.  Returns the 8b-bit field (b <= 8).
__device__ __forceinline__ unsigned long long quant8(const float* v, float mn, float inv, int b) {
  const float2 nmn = make_float2(-mn, -mn);
  const float2 mg = make_float2(12582912.0f, 12582912.0f);
  const float2 inv2 = make_float2(inv, inv);
  uint32_t bits[8];
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float2 a = add2(make_float2(v[j], v[j + 1]), nmn);
    const float2 r = fma2(a, inv2, mg);
    bits[j] = __float_as_uint(r.x);
    bits[j + 1] = __float_as_uint(r.y);
  }
  if (b <= 4) {
    // sum of bits_j * 2^(j b) = sum code_j 2^(j b) + 0x4B400000 * sum 2^(j b)  (mod 2^32)
    uint32_t acc = bits[0], pw = 1u, spw = 1u;
#pragma unroll
    for (int j = 1; j < 8; j++) {
      pw <<= b;
      spw += pw;
      acc += bits[j] * pw;
    }
    return (unsigned long long)(acc - 0x4B400000u * spw);
  }
  unsigned long long acc = 0ull;
#pragma unroll
  for (int j = 0; j < 8; j++) acc |= (unsigned long long)(bits[j] & 0xFFu) << (j * b);
  return acc;
}

// Store n (<= 16) bytes, given as a little-endian 128-bit value (lo, hi), at a shared
// memory address, with the widest naturally aligned stores the address and n allow.
__device__ __forceinline__ void sts_bytes(unsigned char* dst, unsigned long long lo,
                                          unsigned long long hi, int n) {
  const uint32_t a = (uint32_t)(uintptr_t)dst;
  if (((a | (uint32_t)n) & 7u) == 0u) {
    unsigned long long* d = reinterpret_cast<unsigned long long*>(dst);
    d[0] = lo;
    if (n == 16) d[1] = hi;
  } else if (((a | (uint32_t)n) & 3u) == 0u) {
    uint32_t* d = reinterpret_cast<uint32_t*>(dst);
#pragma unroll 1
    for (int k = 0; k < n / 4; k++) d[k] = (uint32_t)((k < 2 ? lo : hi) >> (32 * (k & 1)));
  } else if (((a | (uint32_t)n) & 1u) == 0u) {
    uint16_t* d = reinterpret_cast<uint16_t*>(dst);
#pragma unroll 1
    for (int k = 0; k < n / 2; k++) d[k] = (uint16_t)((k < 4 ? lo : hi) >> (16 * (k & 3)));
  } else {
#pragma unroll 1
    for (int k = 0; k < n; k++) dst[k] = (unsigned char)((k < 8 ? lo : hi) >> (8 * (k & 7)));
  }
}

// Quantise and pack the lane's V values (8 or 16) into its V*b/8 bytes at dst.
template <int V>
__device__ __forceinline__ void quant_store(const float* v, float mn, float inv, int b,
                                            unsigned char* dst) {
  unsigned long long lo = quant8(v, mn, inv, b), hi = 0ull;
  if constexpr (V == 16) {
    const unsigned long long q1 = quant8(v + 8, mn, inv, b);
    const int sh = 8 * b;  // 24..64 bits
    if (sh < 64) {
      lo |= q1 << sh;
      hi = q1 >> (64 - sh);
    } else {
      hi = q1;
    }
  }
  sts_bytes(dst, lo, hi, V * b / 8);
}

// scale = D / Q and inv = Q / D for the team (one division per lane; lanes of a pair
// exchange results).  Degenerate range (D < 2^-120, incl. D = 0): scale = inv = 0.
// `mask` holds every lane that calls this together (both lanes of each pair).
template <int L>
__device__ __forceinline__ void scale_inv(float D, int b, int sub, float& scale, float& inv,
                                          unsigned mask = kFull) {
  const float qf = __fsub_rn(__uint_as_float(0x4B000000u | ((1u << b) - 1u)), 8388608.0f);
  const bool degenerate = !(D >= 0x1p-120f);
  if constexpr (L >= 2) {
    const bool odd = sub & 1;
    const float r = __fdiv_rn(odd ? qf : D, odd ? D : qf);
    const float o = __shfl_xor_sync(mask, r, 1);
    scale = odd ? o : r;
    inv = odd ? r : o;
  } else {
    scale = __fdiv_rn(D, qf);
    inv = __fdiv_rn(qf, D);
  }
  if (degenerate) {
    scale = 0.0f;
    inv = 0.0f;
  }
}

}  // namespace tahq
