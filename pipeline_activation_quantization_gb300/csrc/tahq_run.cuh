// tahq_run.cuh -- the streaming encoder of the TAH-Quant activation codec for widths
// {3, 4} (or one width of 3 or 4 bits), one key per quantisation tile (A = G), any tau,
// fp32 or wire metadata, on tiles of 32, 64 or 128 values (included by tahq_encode.cuh,
// after the work-queue items it reuses).
//
// "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over Slow
// Network" (arXiv 2506.01352v2): §3.2 eq. (1)-(2) entropy keys and "Top-p% tile
// selection"; §3.3 eq. (3) outlier ratio, pivot swap, eq. (4) Hadamard, the asymmetric
// quantizer; §3.4 the contiguous uint8 stream.
//
// Layout: a lane holds a "run" of 32 consecutive values of a 32 KB input chunk (128
// bytes of fp32, 64 of bf16), staged by a 2-D tensor copy with the 128-byte swizzle; a
// tile is LPT = G / 32 consecutive runs (lanes).  Per lane the whole per-tile computation
// is a handful of instructions per value:
//   range and group maxima (the two-values pretest of eq. (3));
//   an approximate entropy key from the hardware base-2 logarithm on the tile scaled by a
//     power of two to a maximum in [1, 2) -- within kKeyErr of the codec's canonical key
//     (the bound is derived below);
//   the codes at both candidate widths (work-queue encoder: two scratch streams) or at
//     the one width every tile gets (straight into the stream).
// Tiles the pretest cannot clear go to one block-wide list and get the exact test, and
// where it holds the pivot swap, Hadamard and new codes (teams of 8 values a lane).
//
// The allocation stays exactly the canonical one: the select of a group finds the
// histogram bucket of its K-th approximate key, and every tile whose approximate key
// lies within kWinBins buckets of it gets its canonical key recomputed from the input
// (k_run_select); all other tiles are at least 2 kKeyErr away from the K-th canonical
// key, so their approximate keys rank them on the right side of it, and the select gives
// them their widths at once.  Three launches: k_run_tiles, k_run_select, k_run_compact.
#pragma once

#include "tahq_encode.cuh"

namespace tahq {

template <typename Tin, int G>
struct RunGeom {
  static constexpr bool kBf = InTraits<Tin>::kBf16;
  static constexpr int ES = (int)sizeof(Tin);
  static constexpr int LPT = G / 32;                   // runs (lanes) per tile
  static constexpr int RPC = kChunkBytes / (32 * ES);  // runs per chunk: 256 f32, 512 bf16
  static constexpr int RPT = RPC / kThreads;           // runs per thread
  static constexpr int CH = RPC / LPT;                 // tiles per chunk
  static_assert(LPT == 1 || LPT == 2 || LPT == 4, "tiles of 32, 64 or 128 values");
  static_assert(CH == Cfg<Tin, G>::CH, "same chunks as the work queue");
};

// Error bound of the approximate key against the canonical one, and the select window.
//
// Both keys estimate H = lg L - S / L (L = sum m_k, S = sum m_k lg m_k, m_k = |a_k|) of
// the same tile.  The approximate one works on m'_k = m_k 2^-E + 2^-100 with 2^E <= max
// m_k < 2^(E+1) (the scaling is exact and H is invariant under it; the 2^-100 shifts H by
// less than 2^-90), so L' lies in [1, G (2 + 2^-99)] and every m'_k in (0, 2].  With
// u = 2^-24, lg2.approx's absolute error below 2^-21.5 on (0, 2] (2^-22.6 on [0.5, 2],
// two units in the last place of |lg x| < 100 elsewhere, i.e. below 2^-22 |lg x| + 2^-22.6;
// terms with m'_k < 2^-30 L' weigh less than 2^-30 each and change the key by under
// 2^-50), and A = sum p_k |lg m'_k| <= lg L' + H <= 2 lg G + 1 <= 15 (p_k = m'_k / L',
// m'_k <= L'):
//   lg terms in S'/L'              <= 2^-21.5 + 2^-22 A            < 2^-17.9
//   sums of at most 32 + 2 levels  <= 34 u (A + 15)                < 2^-14.0
//   lg L', S' / L', the difference <= 2^-21.5 + 2^-22 lg L' + 3 u 15 < 2^-18.6
// so the approximate key is within 2^-13.8 of the exact entropy of the scaled tile, and
// the canonical key (table logarithm within 2^-23 + 2 u |lg m|, pairwise sums of 8
// levels, exact scaling invariance up to those roundings: |lg m| < 140 with weights as
// above, L from 2^-149 to 2^136) within 2^-15.2 of it for tiles with 2^-100 <= max
// m_k <= 2^100 (the others get the canonical key in the main pass).  kKeyErr = 2^-13
// covers both.
constexpr float kKeyErr = 0x1p-13f;
// Buckets of 2^-13 (scale 8192: tiles of up to 256 values): a window of kWinBins buckets
// either side of the K-th key's bucket is 2 kKeyErr wide.
constexpr int kWinBins = 2;
static_assert(kWinBins * 0x1p-13f >= 2 * kKeyErr, "window covers twice the key error");

// Base-2 logarithm of the special-function unit (denormal inputs flushed; every input
// here is a normal number).
__device__ __forceinline__ float lg2_approx(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Run r (32 values) of a swizzled chunk (rows of 128 bytes, 16-byte unit j of row q at
// j ^ (q & 7)): fp32 runs are whole rows, bf16 runs half rows.  Values widened to fp32.
template <typename Tin>
__device__ __forceinline__ void lds_run(const unsigned char* buf, int r, float* v) {
  if constexpr (!InTraits<Tin>::kBf16) {
    const unsigned char* base = buf + r * 128;
    const int x = r & 7;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const uint4 q = *reinterpret_cast<const uint4*>(base + ((j ^ x) << 4));
      v[4 * j] = __uint_as_float(q.x);
      v[4 * j + 1] = __uint_as_float(q.y);
      v[4 * j + 2] = __uint_as_float(q.z);
      v[4 * j + 3] = __uint_as_float(q.w);
    }
  } else {
    const int row = r >> 1, x = row & 7, u0 = (r & 1) * 4;
    const unsigned char* base = buf + row * 128;
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const uint4 q = *reinterpret_cast<const uint4*>(base + (((u0 + j) ^ x) << 4));
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; e++) {
        v[8 * j + 2 * e] = __uint_as_float(w[e] << 16);
        v[8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
  }
}

// The input value x as the codec sees it when the caller asks for RN(c x) (the gradient
// codec; c a power of two): bf16 inputs rounded back to bf16 (nearest, ties to even), as a
// scaled bf16 copy of the input would hold them.
template <bool kBf>
__device__ __forceinline__ float scaled_in(float x, float c) {
  const float y = __fmul_rn(x, c);
  if constexpr (!kBf) {
    return y;
  } else {
    const uint32_t u = __float_as_uint(y);
    return __uint_as_float(((u + ((u >> 16) & 1u) + 0x7FFFu) >> 16) << 16);
  }
}

template <typename Tin, int N, bool kS>
__device__ __forceinline__ void scale_values(const EncParams& p, float* v) {
  if constexpr (kS) {
#pragma unroll
    for (int j = 0; j < N; j++) v[j] = scaled_in<InTraits<Tin>::kBf16>(v[j], p.scale_c);
  }
}

// min / max of the run and the largest magnitude of each group of 8 values.
__device__ __forceinline__ void run_minmax(const float* v, float& mn, float& mx, float* ga) {
#pragma unroll
  for (int g = 0; g < 4; g++) {
    const float* w = v + 8 * g;
    const float gmn = min3f(min3f(w[0], w[1], w[2]), min3f(w[3], w[4], w[5]), fminf(w[6], w[7]));
    const float gmx = max3f(max3f(w[0], w[1], w[2]), max3f(w[3], w[4], w[5]), fmaxf(w[6], w[7]));
    ga[g] = fmaxf(gmx, -gmn);
    mn = g ? fminf(mn, gmn) : gmn;
    mx = g ? fmaxf(mx, gmx) : gmx;
  }
}

// {L', S'} of the run's magnitudes scaled by f (a power of two) plus 2^-100: the sums of
// the approximate key (any order: four packed accumulators).
__device__ __forceinline__ float2 run_sums_approx(const float* v, float f) {
  const float2 f2 = make_float2(f, f), g2 = make_float2(0x1p-100f, 0x1p-100f);
  float2 L[4], S[4];
#pragma unroll
  for (int j = 0; j < 16; j++) {
    const float2 m = fma2(make_float2(fabsf(v[j]), fabsf(v[j + 16])), f2, g2);
    const float2 l = make_float2(lg2_approx(m.x), lg2_approx(m.y));
    if (j < 4) {
      L[j] = m;
      S[j] = mul2(m, l);
    } else {
      L[j & 3] = add2(L[j & 3], m);
      S[j & 3] = fma2(m, l, S[j & 3]);
    }
  }
  const float2 Lt = add2(add2(L[0], L[1]), add2(L[2], L[3]));
  const float2 St = add2(add2(S[0], S[1]), add2(S[2], S[3]));
  return make_float2(Lt.x + Lt.y, St.x + St.y);
}

// The canonical {L, S} of the run's 32 values (pairwise in natural order, first level of
// S fused as fmaf(m_odd, lg m_odd, RN(m_even lg m_even)), zero magnitudes contributing
// zero terms), with the canonical logarithm from the shared tables.  Rare path.
template <typename Tin>
__device__ __forceinline__ float2 run_sums_exact(const float* v, const LgTables& tb) {
  float2 x[16];
#pragma unroll
  for (int j = 0; j < 16; j++) {
    const float a = fabsf(v[2 * j]), b = fabsf(v[2 * j + 1]);
    const float la = a == 0.0f ? 0.0f : lg_canon<InTraits<Tin>::kNoFraction>(a, tb.T, tb.R, tb.TB, tb.k);
    const float lb = b == 0.0f ? 0.0f : lg_canon<InTraits<Tin>::kNoFraction>(b, tb.T, tb.R, tb.TB, tb.k);
    x[j] = make_float2(__fadd_rn(a, b), __fmaf_rn(b, lb, __fmul_rn(a, la)));
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
    for (int j = 0; j < w; j++) x[j] = make_float2(__fadd_rn(x[2 * j].x, x[2 * j + 1].x),
                                                   __fadd_rn(x[2 * j].y, x[2 * j + 1].y));
  }
  return x[0];
}

// The lane's 32 codes at width B from u = RN(v - min) and inv: B words (code k at bits
// [k B, k B + B) of the run's field), stored at dst (aligned to AL bytes).
template <int B, int AL>
__device__ __forceinline__ void quant_run(const float2* u, float inv, unsigned char* dst) {
  const float2 inv2 = make_float2(inv, inv), mg = make_float2(12582912.0f, 12582912.0f);
  unsigned long long f[4];
#pragma unroll
  for (int g = 0; g < 4; g++) {
    uint32_t q[8];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const float2 r = fma2(u[4 * g + k], inv2, mg);
      q[2 * k] = __float_as_uint(r.x);
      q[2 * k + 1] = __float_as_uint(r.y);
    }
    f[g] = pack8_ct<B>(q);
  }
  store_fields<B, 4, AL>(dst, f);
}


// ------------------------------------------------------------------ shared state

template <typename Tin, int G>
struct alignas(1024) RunSmem {
  unsigned char buf[2][kChunkBytes];      // staged input chunks (128-byte swizzle)
  uint16_t dl[RunGeom<Tin, G>::CH];       // the chunk's deferred tiles
  uint32_t hist[2][kCoarseBins];          // coarse key counts of the last two chunks
  LgTables tabs;
  unsigned long long bar[2];
  long long cur[2];                       // the chunk in each stage (-1: none)
  uint32_t ndef[2];                       // deferred counts, by chunk parity
};

template <typename Tin, int G>
__device__ __forceinline__ RunSmem<Tin, G>& run_smem(unsigned char* raw) {
  const uint32_t a = smem_u32(raw);
  return *reinterpret_cast<RunSmem<Tin, G>*>(raw + ((1024u - (a & 1023u)) & 1023u));
}

// ------------------------------------------------------------------ exact path

// Values a lane in the exact path (a tile is a team of G / V lanes): 16 for bf16 tiles of
// 64 or 128 values (fewer lane exchanges and less per-lane bookkeeping a value: measured
// 3-7% faster on those shapes), else 8 (fp32 chunks hold a quarter as many deferred
// tiles, and 16 a lane leaves fewer, longer team steps for the block barrier to wait on:
// measured 3.5% slower at fp32 G = 128, 5% at bf16 G = 32).
template <typename Tin, int G>
__host__ __device__ constexpr int pass_v() {
  return (InTraits<Tin>::kBf16 && G >= 64) ? 16 : 8;
}

// Deferred tiles list[first .. n) of a staged chunk (the pretest could not rule out
// r > tau), teams of L = G / V lanes, V = pass_v values a lane, several teams a warp and
// the list spread over the block's warps.  The main pass has written every tile's codes and
// metadata as untransformed; here the exact ratio test of eq. (3) runs (kT2, tau = 2,
// without a division: RN(m1 / d) > 2 iff m1 / 2 - d > d 2^-24, d = RN(m2 + 1e-12), exact
// by Sterbenz's lemma; else RN(m1 / d) > tau), and the tiles it flags get the pivot swap, the Hadamard of eq. (4),
// a new range and new codes: at both widths into out_lo / out_hi (kFlat false: scales
// keep the range D) or at width kB into out_lo (kFlat: the final scale).  kW: the wire
// format's quantiser (zero = the fp16 value below the minimum, the smallest covering fp16
// scale of each width); ranked, the scales field keeps the maximum.
template <typename Tin, int G, bool kFlat, int kB, bool kW, bool kS, bool kT2>
__device__ __forceinline__ void pass2_run(const EncParams& p, const unsigned char* src,
                                          const uint16_t* list, int first, int n, long long t0,
                                          unsigned char* out_lo, unsigned char* out_hi) {
  constexpr int V = pass_v<Tin, G>(), L = G / V, TPW = 32 / L;
  static_assert(V == 8 || V == 16, "8 or 16 values a lane");
  static_assert(L >= 2, "a pair of lanes shares the two divisions");
  constexpr int ES = (int)sizeof(Tin), NU = V * ES / 16, UPT = G * ES / 16;
  constexpr bool kBf = InTraits<Tin>::kBf16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L, base = lane - sub;
#pragma unroll 1
  for (int j0 = first + warp * TPW; j0 < n; j0 += kWarps * TPW) {
    const int ci = j0 + team;
    const bool valid = ci < n;
    const int cj = valid ? ci : first;
    const int kt = (int)list[cj];
    float v[V];
#pragma unroll
    for (int k = 0; k < NU; k++) {
      // 16-byte unit U of the chunk, in the swizzled layout
      const int U = kt * UPT + sub * NU + k, row = U >> 3;
      const uint4 q = *reinterpret_cast<const uint4*>(src + row * 128 + (((U & 7) ^ (row & 7)) << 4));
      const uint32_t wq[4] = {q.x, q.y, q.z, q.w};
      if constexpr (kBf) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
          v[8 * k + 2 * e] = __uint_as_float(wq[e] << 16);
          v[8 * k + 2 * e + 1] = __uint_as_float(wq[e] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; e++) v[4 * k + e] = __uint_as_float(wq[e]);
      }
    }
    scale_values<Tin, V, kS>(p, v);
    float m1, m2;
    int i1;
    team_top2_values<V, L>(v, sub, m1, i1, m2);
    const float d = __fadd_rn(m2, 1e-12f);
    const bool flag = valid && (kT2 ? __fsub_rn(__fmul_rn(m1, 0.5f), d) > __fmul_rn(d, 0x1p-24f)
                                    : __fdiv_rn(m1, d) > p.tau);
    if (!__any_sync(kFull, flag)) continue;  // the main pass's codes stand
    float t[V];
#pragma unroll
    for (int j = 0; j < V; j++) t[j] = v[j];
    team_swap0<V>(t, flag ? i1 : 0, sub, base);
    team_fwht<V, L>(t, p.h, sub);
#pragma unroll
    for (int j = 0; j < V; j++) v[j] = __fmul_rn(t[j], p.c_h);
    float mn = v[0], mx = v[0];
#pragma unroll
    for (int j = 1; j < V; j++) {
      mn = fminf(mn, v[j]);
      mx = fmaxf(mx, v[j]);
    }
    mn = team_min<L>(mn);
    mx = team_max<L>(mx);
    const float D = __fsub_rn(mx, mn);
    const float qa = qmax_f(kFlat ? kB : 3), qb = qmax_f(kFlat ? kB : 4);
    float inv0, r1d, qz = mn, meta = D;
    if constexpr (kW) {
      qz = wire_zero(mn);
      const float sa = wire_scale(qz, mx, qa);
      inv0 = wire_inv(sa);
      r1d = kFlat ? sa : wire_inv(wire_scale(qz, mx, qb));
      meta = kFlat ? sa : mx;
    } else {
      // lane 0 of the team: Q_lo / D (flat: Q / D); lane 1: Q_hi / D (flat: D / Q)
      const bool one = sub == 1;
      const float r = kFlat ? __fdiv_rn(one ? D : qa, one ? qa : D) : __fdiv_rn(one ? qb : qa, D);
      const float r0 = __shfl_sync(kFull, r, base), r1 = __shfl_sync(kFull, r, base + 1);
      const bool degenerate = !(D >= 0x1p-120f);
      inv0 = degenerate ? 0.0f : r0;
      r1d = degenerate ? 0.0f : r1;
      if (kFlat) meta = r1d;
    }
    const float2 nmn = make_float2(-qz, -qz), mg = make_float2(12582912.0f, 12582912.0f);
    float2 u[V / 2];
#pragma unroll
    for (int j = 0; j < V / 2; j++) u[j] = add2(make_float2(v[2 * j], v[2 * j + 1]), nmn);
#pragma unroll
    for (int w2 = 0; w2 < (kFlat ? 1 : 2); w2++) {
      const int b = kFlat ? kB : (w2 ? 4 : 3);
      const float inv = w2 ? r1d : inv0;
      const float2 inv2 = make_float2(inv, inv);
      unsigned char* slot = (w2 ? out_hi : out_lo) + (size_t)kt * (G * b / 8);
      if constexpr (V == 8) {
        uint32_t f = 0u;
#pragma unroll
        for (int j = 0; j < V / 2; j++) {
          const float2 c = fma2(u[j], inv2, mg);
          f |= (__float_as_uint(c.x) - 0x4B400000u) << (2 * j * b);
          f |= (__float_as_uint(c.y) - 0x4B400000u) << ((2 * j + 1) * b);
        }
        // eight codes a lane: one word at b = 4; at b = 3 the fields of four lanes make
        // three words (slots start on 4-byte boundaries)
        const uint32_t f1 = __shfl_down_sync(kFull, f, 1), f2 = __shfl_down_sync(kFull, f, 2);
        const uint32_t f3 = __shfl_down_sync(kFull, f, 3);
        if (flag && b == 4) {
          *reinterpret_cast<uint32_t*>(slot + 4 * sub) = f;
        } else if (flag && (sub & 3) == 0) {
          uint32_t* dw = reinterpret_cast<uint32_t*>(slot + 3 * sub);
          dw[0] = f | (f1 << 24);
          dw[1] = (f1 >> 8) | (f2 << 16);
          dw[2] = (f2 >> 16) | (f3 << 8);
        }
      } else {
        unsigned long long f = 0ull;
#pragma unroll
        for (int j = 0; j < V / 2; j++) {
          const float2 c = fma2(u[j], inv2, mg);
          f |= (unsigned long long)(__float_as_uint(c.x) - 0x4B400000u) << (2 * j * b);
          f |= (unsigned long long)(__float_as_uint(c.y) - 0x4B400000u) << ((2 * j + 1) * b);
        }
        // sixteen codes a lane: two words at b = 4 (slots start on 8-byte boundaries); at
        // b = 3 the 48-bit fields of a pair of lanes make three words (4-byte boundaries)
        const unsigned long long f1 = __shfl_down_sync(kFull, f, 1);
        if (flag && b == 4) {
          *reinterpret_cast<uint2*>(slot + 8 * sub) = make_uint2((uint32_t)f, (uint32_t)(f >> 32));
        } else if (flag && (sub & 1) == 0) {
          uint32_t* dw = reinterpret_cast<uint32_t*>(slot + 6 * sub);
          dw[0] = (uint32_t)f;
          dw[1] = (uint32_t)(f >> 32) | ((uint32_t)f1 << 16);
          dw[2] = (uint32_t)(f1 >> 16);
        }
      }
    }
    if (flag && sub == 0) put_meta(p, t0 + kt, qz, (uint8_t)i1, meta, kFlat);
  }
}

// ------------------------------------------------------------------ main pass

// One staged chunk (tiles t0 .. t0 + nt of group g), chunk number k of the block.  kFlat:
// every tile at width kB, codes straight into the stream at out_lo (slot t G kB / 8);
// else keys, histograms and both widths into the scratch streams out_lo / out_hi.
// Deferred tiles go to the list s.dl (s.ndef[k & 1] of them).  kW: the wire format's
// quantiser (see pass2_run).
template <typename Tin, int G, bool kFlat, int kB, bool kW, bool kS, bool kT2>
__device__ __forceinline__ void main_run(RunSmem<Tin, G>& s, const EncParams& p, long long g,
                                         long long t0, int nt, int k, unsigned char* out_lo,
                                         unsigned char* out_hi) {
  using RG = RunGeom<Tin, G>;
  constexpr int LPT = RG::LPT;
  const int sl = k & 1;
  const unsigned char* buf = s.buf[sl];
#pragma unroll 1
  for (int rr = 0; rr < RG::RPT; rr++) {
    const int r = rr * kThreads + threadIdx.x;  // the lane's run
    const int kt = r / LPT, sub = r % LPT;
    const bool valid = kt < nt;
    float v[32];
    lds_run<Tin>(buf, r, v);
    scale_values<Tin, 32, kS>(p, v);
    float mn, mx, ga[4];
    run_minmax(v, mn, mx, ga);
    mn = team_min<LPT>(mn);
    mx = team_max<LPT>(mx);
    const float m1 = fmaxf(mx, -mn);
    // two values of at least m1 / tau rule out r > tau (tau = 2: an exact halving for
    // m1 >= 2^-120; else m1 / tau rounded up)
    const float thr = kT2 ? __fmul_rn(m1, 0.5f) : __fdiv_ru(m1, p.tau);
    uint32_t cnt = 0;
#pragma unroll
    for (int q = 0; q < 4; q++) cnt += ga[q] >= thr ? 1u : 0u;
    cnt = team_sum_u<LPT>(cnt);
    // below 2^-120 the ratio cannot exceed a tau >= 1 (m2 + 1e-12 > m1 / tau); a maximum
    // that is not finite goes to the exact test
    const bool small = (kT2 || p.tau >= 1.0f) && m1 < 0x1p-120f;
    const bool deferred = valid && !small && (!(m1 <= FLT_MAX) || cnt < 2u);
    if constexpr (!kFlat) {
      // entropy key: approximate on tiles of moderate magnitude, canonical otherwise
      const bool special = !(m1 >= 0x1p-100f && m1 <= 0x1p100f);
      // f = 2^-E with 2^E <= m1 < 2^(E+1)
      const float f = __uint_as_float((254u - (__float_as_uint(m1) >> 23)) << 23);
      float2 ls = run_sums_approx(v, special ? 1.0f : f);
      ls = team_sum2<LPT>(ls);
      float H = __fsub_rn(lg2_approx(ls.x), __fmul_rn(ls.y, rcp_approx(ls.x)));
      if (__any_sync(kFull, special)) {
        float2 ex = run_sums_exact<Tin>(v, s.tabs);
        ex = team_sum2<LPT>(ex);
        if (special) {
          H = entropy_key(ex.x, ex.y, s.tabs);
          if (valid && sub == 0 &&
              (!(ex.x <= FLT_MAX) || !(fabsf(ex.y) <= FLT_MAX) || !(fabsf(H) <= FLT_MAX)))
            set_status(p.status, kStNonFinite);
        }
      }
      if (valid && sub == 0) {
        p.keys[t0 + kt] = H;
        const int b = fine_bin(H, p.fscale);
        atomicAdd(&p.hist_fine[g * (long long)kFineBins + b], 1u);
        atomicAdd(&s.hist[sl][b >> 8], 1u);  // the chunk's coarse counts
      }
    } else {
      if (valid && sub == 0 && !(m1 <= FLT_MAX)) set_status(p.status, kStNonFinite);
    }
    const float D = __fsub_rn(mx, mn);
    // kFlat: inv = Q / D and the scale D / Q; else Q_lo / D and Q_hi / D (a pair of lanes
    // shares the two divisions)
    float r0, r1;
    const float qa = qmax_f(kFlat ? kB : 3), qb = qmax_f(kFlat ? kB : 4);
    float qz = mn, meta = D;  // the quantiser's zero; the scales field (ranked)
    if constexpr (kW) {
      // wire: zero = the fp16 value below the minimum; the smallest covering fp16 scale of
      // each width (a pair of lanes shares the two); ranked, the scales field keeps the
      // maximum (the select derives the scale of the tile's width from zero and maximum)
      qz = wire_zero(mn);
      if constexpr (kFlat) {
        r1 = wire_scale(qz, mx, qa);
        r0 = wire_inv(r1);
      } else if constexpr (LPT >= 2) {
        const bool odd = sub & 1;
        const float iv = wire_inv(wire_scale(qz, mx, odd ? qb : qa));
        const float o = __shfl_xor_sync(kFull, iv, 1);
        r0 = odd ? o : iv;
        r1 = odd ? iv : o;
      } else {
        r0 = wire_inv(wire_scale(qz, mx, qa));
        r1 = wire_inv(wire_scale(qz, mx, qb));
      }
      meta = mx;
    } else {
      if constexpr (LPT >= 2) {
        const bool odd = sub & 1;
        const float rv = kFlat ? __fdiv_rn(odd ? D : qa, odd ? qa : D) : __fdiv_rn(odd ? qb : qa, D);
        const float o = __shfl_xor_sync(kFull, rv, 1);
        r0 = odd ? o : rv;
        r1 = odd ? rv : o;
      } else {
        r0 = __fdiv_rn(qa, D);
        r1 = kFlat ? __fdiv_rn(D, qa) : __fdiv_rn(qb, D);
      }
      if (!(D >= 0x1p-120f)) r0 = r1 = 0.0f;
    }
    float2 u[16];
    const float2 nmn = make_float2(-qz, -qz);
#pragma unroll
    for (int j = 0; j < 16; j++) u[j] = add2(make_float2(v[2 * j], v[2 * j + 1]), nmn);
    if (valid) {
      if constexpr (kFlat) {
        unsigned char* dst = out_lo + (size_t)kt * (G * kB / 8) + sub * (4 * kB);
        quant_run<kB, kB == 4 ? 16 : 4>(u, r0, dst);
        if (sub == 0) put_meta(p, t0 + kt, qz, (uint8_t)0xFF, r1, true);
      } else {
        quant_run<3, 4>(u, r0, out_lo + (size_t)kt * (G * 3 / 8) + sub * 12);
        quant_run<4, 16>(u, r1, out_hi + (size_t)kt * (G / 2) + sub * 16);
        if (sub == 0) put_meta(p, t0 + kt, qz, (uint8_t)0xFF, meta, false);
      }
    }
    if (deferred && sub == 0) s.dl[atomicAdd(&s.ndef[sl], 1u)] = (uint16_t)kt;
  }
}

// ------------------------------------------------------------------ the streaming loop

// Tensor copy of the chunk starting at tile t0 (rows t0 G size / 128 .. + 256).
template <typename Tin, int G>
__device__ __forceinline__ void issue_run_chunk(RunSmem<Tin, G>& s, const EncParams& p,
                                                long long t0, int slot, unsigned long long pol) {
  mbar_expect_tx(&s.bar[slot], (uint32_t)kChunkBytes);
  const int row = (int)(t0 * G * (long long)sizeof(Tin) / 128);
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(s.buf[slot])),
      "l"(reinterpret_cast<unsigned long long>(&p.tmap)), "r"(0), "r"(row),
      "r"(smem_u32(&s.bar[slot])), "l"(pol)
      : "memory");
}

// The chunks blockIdx.x, + gridDim.x, ... of the input, each copied in while the one
// before is processed: the main pass, one block barrier, the exact path of the chunk's
// deferred tiles (spread over the block's warps).
template <typename Tin, int G, bool kFlat, int kB, bool kW, bool kS, bool kT2>
__device__ __forceinline__ void run_chunks(RunSmem<Tin, G>& s, const EncParams& p,
                                           long long n_chunks) {
  constexpr int CH = RunGeom<Tin, G>::CH;
  const unsigned long long pol = policy_evict_first();  // the input is read once
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_barrier_init();
    s.ndef[0] = s.ndef[1] = 0u;
  }
  for (int i = threadIdx.x; i < 2 * kCoarseBins; i += kThreads) (&s.hist[0][0])[i] = 0u;
  if (!kFlat) {
    const float* src = reinterpret_cast<const float*>(&p.tabs);
    float* dst = reinterpret_cast<float*>(&s.tabs);
    for (int i = threadIdx.x; i < (int)(sizeof(LgTables) / 4); i += kThreads) dst[i] = src[i];
  }
  const int slot_a = kFlat ? G * kB / 8 : G * 3 / 8, slot_b = G / 2;
  long long c = blockIdx.x;
  if (threadIdx.x == 0 && c < n_chunks) issue_run_chunk<Tin, G>(s, p, c * CH, 0, pol);
  uint32_t parity = 0u;
  long long gp = 0;  // group of the previous chunk
  int k = 0;
  for (; c < n_chunks; c += gridDim.x, ++k) {
    const int sl = k & 1;
    csync();  // chunk k - 1 is done: its buffer, list and counts are free
    if (threadIdx.x == 0) {
      s.ndef[sl ^ 1] = 0u;
      if (c + gridDim.x < n_chunks)
        issue_run_chunk<Tin, G>(s, p, (c + gridDim.x) * CH, sl ^ 1, pol);
    }
    if constexpr (!kFlat) {  // coarse counts of chunk k - 1, one global add per bin
      static_assert(kThreads == kCoarseBins, "one coarse bin per thread");
      const uint32_t cb = s.hist[sl ^ 1][threadIdx.x];
      if (cb) {
        atomicAdd(&p.hist_coarse[gp * kCoarseBins + threadIdx.x], cb);
        s.hist[sl ^ 1][threadIdx.x] = 0u;
      }
    }
    const long long t0 = c * CH;
    const int nt = (int)min((long long)CH, p.n_tiles - t0);
    const long long g = kFlat ? 0 : t0 / p.n_g;  // chunks never straddle groups here
    unsigned char* lo = (kFlat ? p.codes : p.scratch_lo) + t0 * slot_a;
    unsigned char* hi = kFlat ? lo : p.scratch_hi + t0 * slot_b;
    mbar_wait(&s.bar[sl], (parity >> sl) & 1u, p.status, p.wait_ns);
    parity ^= 1u << sl;
    main_run<Tin, G, kFlat, kB, kW, kS, kT2>(s, p, g, t0, nt, k, lo, hi);
    csync();  // the list is complete, and the codes written before the exact path's
    pass2_run<Tin, G, kFlat, kB, kW, kS, kT2>(p, s.buf[sl], s.dl, 0, (int)s.ndef[sl], t0, lo, hi);
    gp = g;
  }
  if (!kFlat && k) {  // the last chunk's coarse counts
    csync();
    const uint32_t cb = s.hist[(k - 1) & 1][threadIdx.x];
    if (cb) atomicAdd(&p.hist_coarse[gp * kCoarseBins + threadIdx.x], cb);
  }
}

// The chunks of the input, each copied in while the one before is processed: the main
// pass, one block barrier, the exact path of the chunk's deferred tiles (spread over the
// block's warps).  kDyn: chunks handed out in increasing order by an atomic ticket
// (faster blocks take more); else blockIdx.x, + gridDim.x, ... (measured faster for the
// ranked pass, whose blocks all write the same group's histograms).
template <typename Tin, int G, bool kFlat, int kB, bool kDyn, bool kW, bool kS, bool kT2>
__device__ __forceinline__ void run_chunks_dyn(RunSmem<Tin, G>& s, const EncParams& p,
                                           long long n_chunks) {
  constexpr int CH = RunGeom<Tin, G>::CH;
  const unsigned long long pol = policy_evict_first();  // the input is read once
  for (int i = threadIdx.x; i < 2 * kCoarseBins; i += kThreads) (&s.hist[0][0])[i] = 0u;
  if (!kFlat) {
    const float* src = reinterpret_cast<const float*>(&p.tabs);
    float* dst = reinterpret_cast<float*>(&s.tabs);
    for (int i = threadIdx.x; i < (int)(sizeof(LgTables) / 4); i += kThreads) dst[i] = src[i];
  }
  const int slot_a = kFlat ? G * kB / 8 : G * 3 / 8, slot_b = G / 2;
  long long nxt = -1;  // thread 0: the chunk after the staged ones
  auto next_chunk = [&](long long cur) -> long long {
    if constexpr (kDyn) {
      return (long long)atomicAdd(p.ticket, 1u);
    } else {
      return cur + gridDim.x;
    }
  };
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_barrier_init();
    s.ndef[0] = s.ndef[1] = 0u;
    const long long c0 = kDyn ? next_chunk(0) : (long long)blockIdx.x;
    s.cur[0] = c0 < n_chunks ? c0 : -1;
    if (c0 < n_chunks) issue_run_chunk<Tin, G>(s, p, c0 * CH, 0, pol);
    nxt = c0 < n_chunks ? next_chunk(c0) : n_chunks;
  }
  uint32_t parity = 0u;
  long long gp = 0;  // group of the previous chunk
  int k = 0;
  for (;; ++k) {
    const int sl = k & 1;
    csync();  // chunk k - 1 is done: its buffer, list and counts are free
    const long long c = s.cur[sl];
    if (c < 0) break;  // block-uniform
    if (threadIdx.x == 0) {
      s.ndef[sl ^ 1] = 0u;
      s.cur[sl ^ 1] = nxt < n_chunks ? nxt : -1;
      if (nxt < n_chunks) {
        issue_run_chunk<Tin, G>(s, p, nxt * CH, sl ^ 1, pol);
        nxt = next_chunk(nxt);
      }
    }
    if constexpr (!kFlat) {  // coarse counts of chunk k - 1, one global add per bin
      static_assert(kThreads == kCoarseBins, "one coarse bin per thread");
      const uint32_t cb = s.hist[sl ^ 1][threadIdx.x];
      if (cb) {
        atomicAdd(&p.hist_coarse[gp * kCoarseBins + threadIdx.x], cb);
        s.hist[sl ^ 1][threadIdx.x] = 0u;
      }
    }
    const long long t0 = c * CH;
    const int nt = (int)min((long long)CH, p.n_tiles - t0);
    const long long g = kFlat ? 0 : t0 / p.n_g;  // chunks never straddle groups here
    unsigned char* lo = (kFlat ? p.codes : p.scratch_lo) + t0 * slot_a;
    unsigned char* hi = kFlat ? lo : p.scratch_hi + t0 * slot_b;
    mbar_wait(&s.bar[sl], (parity >> sl) & 1u, p.status, p.wait_ns);
    parity ^= 1u << sl;
    main_run<Tin, G, kFlat, kB, kW, kS, kT2>(s, p, g, t0, nt, k, lo, hi);
    csync();  // the list is complete, and the codes written before the exact path's
    pass2_run<Tin, G, kFlat, kB, kW, kS, kT2>(p, s.buf[sl], s.dl, 0, (int)s.ndef[sl], t0, lo, hi);
    gp = g;
  }
  if (!kFlat && k) {  // the last chunk's coarse counts (the loop ended after a barrier)
    const uint32_t cb = s.hist[(k - 1) & 1][threadIdx.x];
    if (cb) atomicAdd(&p.hist_coarse[gp * kCoarseBins + threadIdx.x], cb);
  }
}

// Every tile gets the same width kB (K = 0 or K = n_g): codes at t G kB / 8.  kW: the
// wire format's quantiser; kS: the input read as RN(c x) (scaled_in); kT2: tau = 2 (else
// p.tau, the pretest's threshold rounded up and the exact test by a division).
template <typename Tin, int G, int kB, bool kW, bool kS, bool kT2>
__global__ void __launch_bounds__(kThreads, 3) k_run_flat(const __grid_constant__ EncParams p,
                                                          long long n_chunks) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  run_chunks_dyn<Tin, G, true, kB, true, kW, kS, kT2>(run_smem<Tin, G>(smem_raw), p, n_chunks);
}

// Stage 1 of widths {3, 4} ranked per group: keys, histograms, both widths into scratch.
// kW: the wire format's quantiser; kS: the input read as RN(c x) (scaled_in); kT2: tau = 2
// (else p.tau).
template <typename Tin, int G, bool kW, bool kS, bool kT2>
__global__ void __launch_bounds__(kThreads, 3) k_run_tiles(const __grid_constant__ EncParams p,
                                                           long long n_chunks) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  dep_launch();
  run_chunks<Tin, G, false, 0, kW, kS, kT2>(run_smem<Tin, G>(smem_raw), p, n_chunks);
}

// ------------------------------------------------------------------ stage 2: the select

// The canonical entropy key of a tile, computed by one warp: lane l holds values
// [l V, l V + V), V = G / 32, from its raw input bytes (canonical pairwise tree: the
// lane's own levels, then lanes xor 1, 2, ..., 16).
template <typename Tin, int G>
__device__ __forceinline__ float warp_exact_key(const uint4& raw, const LgTables& tb) {
  constexpr int V = G / 32;
  constexpr bool kBf = InTraits<Tin>::kBf16;
  float m[4];
  if constexpr (kBf) {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int k = 0; k < V; k++)
      m[k] = __uint_as_float(((k & 1) ? (w[k >> 1] & 0xFFFF0000u) : (w[k >> 1] << 16)) & 0x7FFFFFFFu);
  } else {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < V; k++) m[k] = __uint_as_float(w[k] & 0x7FFFFFFFu);
  }
  float l[4];
#pragma unroll
  for (int k = 0; k < V; k++)
    l[k] = m[k] == 0.0f ? 0.0f : lg_canon<InTraits<Tin>::kNoFraction>(m[k], tb.T, tb.R, tb.TB, tb.k);
  float Ls, Ss;
  const int lane = threadIdx.x & 31;
  if constexpr (V == 1) {
    // level 1 pairs lanes (2j, 2j + 1): the odd value is the fused one
    const float mo = __shfl_xor_sync(kFull, m[0], 1), lo = __shfl_xor_sync(kFull, l[0], 1);
    const bool odd = lane & 1;
    const float me = odd ? mo : m[0], le = odd ? lo : l[0];
    const float mod = odd ? m[0] : mo, lod = odd ? l[0] : lo;
    Ls = __fadd_rn(me, mod);
    Ss = __fmaf_rn(mod, lod, __fmul_rn(me, le));
#pragma unroll
    for (int o = 2; o < 32; o <<= 1) {
      Ls = __fadd_rn(Ls, __shfl_xor_sync(kFull, Ls, o));
      Ss = __fadd_rn(Ss, __shfl_xor_sync(kFull, Ss, o));
    }
  } else {
    float x[2], y[2];
#pragma unroll
    for (int j = 0; j < V / 2; j++) {
      x[j] = __fadd_rn(m[2 * j], m[2 * j + 1]);
      y[j] = __fmaf_rn(m[2 * j + 1], l[2 * j + 1], __fmul_rn(m[2 * j], l[2 * j]));
    }
    Ls = x[0];
    Ss = y[0];
    if constexpr (V == 4) {
      Ls = __fadd_rn(x[0], x[1]);
      Ss = __fadd_rn(y[0], y[1]);
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      Ls = __fadd_rn(Ls, __shfl_xor_sync(kFull, Ls, o));
      Ss = __fadd_rn(Ss, __shfl_xor_sync(kFull, Ss, o));
    }
  }
  return entropy_key(Ls, Ss, tb);
}

// The lane's raw bytes of tile t for warp_exact_key (G * size / 32 bytes: 2 to 16).
template <typename Tin, int G>
__device__ __forceinline__ uint4 warp_tile_raw(const EncParams& p, long long t) {
  constexpr int LB = G * (int)sizeof(Tin) / 32;
  const int lane = threadIdx.x & 31;
  const unsigned char* src = static_cast<const unsigned char*>(p.x) + (t * G * (long long)sizeof(Tin)) + lane * LB;
  uint4 r = make_uint4(0u, 0u, 0u, 0u);
  if constexpr (LB == 16) {
    r = __ldg(reinterpret_cast<const uint4*>(src));
  } else if constexpr (LB == 8) {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(src));
    r.x = a.x;
    r.y = a.y;
  } else if constexpr (LB == 4) {
    r.x = __ldg(reinterpret_cast<const unsigned int*>(src));
  } else {
    static_assert(LB == 2, "2 to 16 bytes a lane");
    r.x = __ldg(reinterpret_cast<const unsigned short*>(src));
  }
  return r;
}

// Tiles of a select part: kSelPart (8 a thread), or kSelPartWide (12 a thread) when
// parts of kSelPart would need a second wave of select blocks; candidates ranked through
// a histogram when they are at most kRankHist (their rank keys and 4096 bins fill 32 KB).
constexpr int kSelPart = 2048;
constexpr int kSelPartWide = 3072;
constexpr uint32_t kRankHist = 2048;

// A lane's raw input bytes (warp_tile_raw) read as RN(c x) (scaled_in).
template <typename Tin>
__device__ __forceinline__ uint4 scale_raw(uint4 r, float c) {
  uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int k = 0; k < 4; k++) {
    if constexpr (!InTraits<Tin>::kBf16) {
      w[k] = __float_as_uint(scaled_in<false>(__uint_as_float(w[k]), c));
    } else {
      const uint32_t lo = __float_as_uint(scaled_in<true>(__uint_as_float(w[k] << 16), c));
      const uint32_t hi = __float_as_uint(scaled_in<true>(__uint_as_float(w[k] & 0xFFFF0000u), c));
      w[k] = (lo >> 16) | (hi & 0xFFFF0000u);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

struct SelSmem {
  unsigned char buf[kChunkBytes];  // window tiles, then candidate rank keys
  LgTables tabs;
  uint32_t bins[256];
  uint32_t scan[16];
  uint32_t wscan[kWarps + 4];
  unsigned long long theta;
  uint32_t last;
};

// Width b of tile t and its scale: D / Q_b (D is what the tiles pass left in scales), or
// kW: the smallest fp16 scale covering [zero, x] at Q_b steps (x the tile's maximum).
template <bool kW>
__device__ __forceinline__ void put_width(const EncParams& p, long long t, bool hi, float D,
                                          float zero) {
  const int b = hi ? 4 : 3;
  p.bits[t] = (uint8_t)b;
  if constexpr (kW) {
    p.scales[t] = wire_scale(zero, D, qmax_f(b));
  } else {
    p.scales[t] = (D >= 0x1p-120f) ? __fdiv_rn(D, qmax_f(b)) : 0.0f;
  }
}

// Stage 2, blocks (group g, j): part j of the group, `per` tiles (a multiple of 32, at
// most kB kThreads).  The group's K-th approximate key lies in fine bucket b*; every tile
// whose approximate key lies within kWinBins buckets of b* is a candidate: it gets its
// canonical key (written over the approximate one and appended, as a rank key, to the
// group's candidates).  Every other tile lies at least 2 kKeyErr from the K-th canonical
// key, so its side of it is known now: hi above the window, lo below; its width, scale,
// bit of its segment's hi mask and its chunk's hi count are written here.  The group's
// last block ranks the candidates (the r-th largest rank key, r = K - tiles above the
// window, is the group's threshold), gives them their widths, and turns the chunks' hi
// counts into their byte offsets in the stream.
template <typename Tin, int G, bool kW, int kB>
__global__ void __launch_bounds__(kThreads, 5) k_run_select(const __grid_constant__ EncParams p,
                                                         int J, long long per) {
  __shared__ __align__(16) SelSmem s;
  const long long g = blockIdx.x / J, jb = blockIdx.x % J;
  const uint32_t K = (uint32_t)p.K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    const float* src = reinterpret_cast<const float*>(&p.tabs);
    float* dst = reinterpret_cast<float*>(&s.tabs);
    for (int i = threadIdx.x; i < (int)(sizeof(LgTables) / 4); i += kThreads) dst[i] = src[i];
  }
  const long long lo = jb * per, hi = min(p.n_g, lo + per);
  dep_wait();
  dep_launch();
  // the part's keys and ranges, loaded while warp 0 finds the window
  static_assert(kB * kThreads <= kChunkBytes / 4, "the part's list fits the buffer");
  const float* kg = p.keys + g * p.n_g;
  const float* dg = p.scales + g * p.n_g;
  float hv[kB], dv[kB], zv[kB];
#pragma unroll
  for (int u = 0; u < kB; u++) {
    const long long i = lo + u * kThreads + threadIdx.x;
    hv[u] = i < hi ? __ldcg(&kg[i]) : 0.0f;
    dv[u] = i < hi ? __ldcg(&dg[i]) : 0.0f;
    zv[u] = (kW && i < hi) ? __ldcg(&p.zeros[g * p.n_g + i]) : 0.0f;
  }
  const uint32_t* hf = p.hist_fine + g * (long long)kFineBins;
  if (warp == 0) {
    for (int i = lane; i < 256; i += 32) s.bins[i] = __ldcg(&p.hist_coarse[g * kCoarseBins + i]);
    __syncwarp();
    int cb;
    uint32_t above_c;
    warp_find_from_top(s.bins, K, cb, above_c);
    __syncwarp();
    for (int i = lane; i < 256; i += 32) s.bins[i] = __ldcg(&hf[cb * 256 + i]);
    __syncwarp();
    int fb;
    uint32_t above_f;
    warp_find_from_top(s.bins, K - above_c, fb, above_f);
    const int bstar = cb * 256 + fb;
    const int blo = max(0, bstar - kWinBins), bhi = min(kFineBins - 1, bstar + kWinBins);
    uint32_t upper = 0, inwin = 0;  // tiles above bstar in the window; in the window
    const int b = blo + lane;
    if (b <= bhi) {
      const uint32_t cnt = (b >> 8) == cb ? s.bins[b & 255] : __ldcg(&hf[b]);
      inwin = cnt;
      upper = b > bstar ? cnt : 0u;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      upper += __shfl_xor_sync(kFull, upper, o);
      inwin += __shfl_xor_sync(kFull, inwin, o);
    }
    __syncwarp();
    for (int i = lane; i < 256; i += 32) s.bins[i] = 0u;
    if (lane == 0) {
      s.scan[0] = (uint32_t)blo;
      s.scan[1] = (uint32_t)bhi;
      s.scan[2] = above_c + above_f - upper;  // tiles above the window
      s.scan[3] = inwin;
      s.scan[4] = 0u;  // list length
    }
  }
  __syncthreads();
  const int blo = (int)s.scan[0], bhi = (int)s.scan[1];
  uint32_t* list = reinterpret_cast<uint32_t*>(s.buf);
  uint32_t* segmask = p.segmask + g * ((p.n_g + 31) / 32);
  unsigned long long* words = p.lookback + g * p.nC;
#pragma unroll
  for (int u = 0; u < kB; u++) {
    const long long iw = lo + u * kThreads + warp * 32;  // the warp's segment
    const long long i = iw + lane;
    const int fbin = fine_bin(hv[u], p.fscale);
    const bool in = i < hi;
    const bool hit = in && fbin >= blo && fbin <= bhi;
    const bool above = in && fbin > bhi;
    if (in && !hit) put_width<kW>(p, g * p.n_g + i, above, dv[u], zv[u]);
    const unsigned hm = __ballot_sync(kFull, above);
    if (lane == 0 && iw < hi) {
      segmask[iw >> 5] = hm;  // the candidates' bits follow in the last block
      if (hm) atomicAdd(&words[iw / p.CHC], (unsigned long long)__popc(hm));
    }
    const unsigned mask = __ballot_sync(kFull, hit);
    if (mask) {
      uint32_t pos0 = 0;
      const int leader = __ffs(mask) - 1;
      if (lane == leader) pos0 = atomicAdd(&s.scan[4], (uint32_t)__popc(mask));
      pos0 = __shfl_sync(kFull, pos0, leader);
      if (hit) list[pos0 + __popc(mask & ((1u << lane) - 1u))] = (uint32_t)i;
    }
  }
  __syncthreads();
  {
    // canonical keys, one warp a tile, eight tiles' loads in flight a warp (four of 16
    // bytes a lane)
    const int n = (int)s.scan[4];
    constexpr int kF = G * (int)sizeof(Tin) >= 512 ? 4 : 8;
#pragma unroll 1
    for (int i0 = warp * kF; i0 < n; i0 += kWarps * kF) {
      uint4 raw[kF];
#pragma unroll
      for (int q = 0; q < kF; q++) {
        const int i = i0 + q;
        raw[q] = i < n ? warp_tile_raw<Tin, G>(p, g * p.n_g + list[i]) : make_uint4(0u, 0u, 0u, 0u);
        if (p.scale_c != 1.0f) raw[q] = scale_raw<Tin>(raw[q], p.scale_c);
      }
      uint32_t tl_mine = 0u;
      float h_mine = 0.0f;
#pragma unroll
      for (int q = 0; q < kF; q++) {
        if (i0 + q >= n) break;  // warp-uniform
        const float H = warp_exact_key<Tin, G>(raw[q], s.tabs);
        if (lane == q) {
          tl_mine = list[i0 + q];
          h_mine = H;
        }
      }
      const int nk = min(kF, n - i0);
      uint32_t pos0 = 0;
      if (lane == 0) pos0 = atomicAdd(&p.cand_cnt[g], (uint32_t)nk);
      pos0 = __shfl_sync(kFull, pos0, 0);
      if (lane < nk) {
        p.keys[g * p.n_g + tl_mine] = h_mine;
        p.cand[g * p.n_g + pos0 + lane] = rank_key(h_mine, tl_mine);
        if (!(fabsf(h_mine) <= FLT_MAX)) set_status(p.status, kStNonFinite);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&p.doneB[g], 1u);
    __threadfence();
    s.last = (prev == (uint32_t)J - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (!s.last) return;
  const unsigned long long* cg = p.cand + g * p.n_g;
  const uint32_t cnt = __ldcg(&p.cand_cnt[g]);
  if (threadIdx.x == 0 && cnt != s.scan[3]) set_status(p.status, kStSelectMismatch);
  const uint32_t r = max(1u, min(K - s.scan[2], cnt));  // rank (from 1) among them
  // the r-th largest rank key (they are distinct): through a histogram when the
  // candidates are at most kRankHist, else a radix select (8 passes of 8 bits); from
  // shared memory when they fit
  constexpr uint32_t kStage = kChunkBytes / 8;
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(s.buf);
  const bool staged = cnt <= kStage;
  if (staged)
    for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) ck[i] = __ldcg(&cg[i]);
  if (threadIdx.x == 0) {
    s.theta = ~0ull;  // no candidate: none of them is hi
    s.scan[7] = 0xFFFFFFFFu;
    s.scan[8] = 0u;
  }
  __syncthreads();
  if (cnt > 0u && cnt <= kRankHist) {
    // the top words (entropy order) of the candidates' rank keys span a narrow range:
    // a 4096-bin histogram of them, shifted to fit, finds the bin of the r-th largest;
    // within it, counting among its members (rank keys are distinct)
    uint32_t* hb = reinterpret_cast<uint32_t*>(s.buf + 8 * kRankHist);
    for (int i = threadIdx.x; i < 4096; i += kThreads) hb[i] = 0u;
    uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
    for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
      const uint32_t h = (uint32_t)(ck[i] >> 32);
      kmn = min(kmn, h);
      kmx = max(kmx, h);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      kmn = min(kmn, __shfl_xor_sync(kFull, kmn, o));
      kmx = max(kmx, __shfl_xor_sync(kFull, kmx, o));
    }
    if (lane == 0) {
      atomicMin(&s.scan[7], kmn);
      atomicMax(&s.scan[8], kmx);
    }
    __syncthreads();
    kmn = s.scan[7];
    const uint32_t span = s.scan[8] - kmn;
    const int sh = max(0, 20 - __clz(span));  // (span >> sh) < 4096
    for (uint32_t i = threadIdx.x; i < cnt; i += kThreads)
      atomicAdd(&hb[((uint32_t)(ck[i] >> 32) - kmn) >> sh], 1u);
    __syncthreads();
    // thread t holds bins 4095 - 16 t - j, j = 0..15 (from the top)
    uint32_t c16[16], sum = 0;
#pragma unroll
    for (int j = 0; j < 16; j++) {
      c16[j] = hb[4095 - 16 * threadIdx.x - j];
      sum += c16[j];
    }
    uint32_t tot;
    uint32_t above = block_exclusive_scan<kThreads>(sum, tot, s.wscan);
    if (above < r && above + sum >= r) {
#pragma unroll
      for (int j = 0; j < 16; j++) {
        if (above < r && above + c16[j] >= r) {
          s.scan[9] = 4095u - 16u * threadIdx.x - (uint32_t)j;
          s.scan[10] = above;
        }
        above += c16[j];
      }
    }
    if (threadIdx.x == 0) s.scan[11] = 0u;
    __syncthreads();
    const uint32_t bstar_r = s.scan[9], rr = r - s.scan[10];
    unsigned long long* mem = reinterpret_cast<unsigned long long*>(hb);  // the bin's members
    for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
      const unsigned long long v = ck[i];
      if ((((uint32_t)(v >> 32) - kmn) >> sh) == bstar_r) mem[atomicAdd(&s.scan[11], 1u)] = v;
    }
    __syncthreads();
    const uint32_t m = s.scan[11];
    for (uint32_t i = threadIdx.x; i < m; i += kThreads) {
      const unsigned long long ki = mem[i];
      uint32_t larger = 0;
      for (uint32_t j = 0; j < m; j++) larger += mem[j] > ki ? 1u : 0u;
      if (larger == rr - 1u) s.theta = ki;
    }
  } else if (cnt > 0u) {
    uint32_t rr = r;
    unsigned long long prefix = 0ull, mask = 0ull;
    for (int pass = 7; pass >= 0; --pass) {
      const int shift = pass * 8;
      for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
        const unsigned long long v = staged ? ck[i] : __ldcg(&cg[i]);
        if ((v & mask) == prefix) atomicAdd(&s.bins[(v >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        int d;
        uint32_t ab;
        warp_find_from_top(s.bins, rr, d, ab);
        if (lane == 0) {
          s.scan[5] = (uint32_t)d;
          s.scan[6] = ab;
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)s.scan[5] << shift;
      rr -= s.scan[6];
      mask |= 0xFFull << shift;
      for (int i = threadIdx.x; i < 256; i += kThreads) s.bins[i] = 0u;
      __syncthreads();
    }
    if (threadIdx.x == 0) s.theta = prefix;
  }
  __syncthreads();
  const unsigned long long theta = s.theta;
  if (threadIdx.x == 0) p.sel[g] = SelResult{theta, cnt ? kSelThreshold : kSelNone, 0u};
  // the candidates' widths, mask bits and chunk counts
  for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
    const unsigned long long v = staged ? ck[i] : __ldcg(&cg[i]);
    const uint32_t tl = 0xFFFFFFFFu - (uint32_t)v;
    const bool ishi = v >= theta;
    put_width<kW>(p, g * p.n_g + tl, ishi, __ldcg(&p.scales[g * p.n_g + tl]),
                  kW ? __ldcg(&p.zeros[g * p.n_g + tl]) : 0.0f);
    if (ishi) {
      atomicOr(&segmask[tl >> 5], 1u << (tl & 31));
      atomicAdd(&words[tl / p.CHC], 1ull);
    }
  }
  __syncthreads();
  // exclusive prefix of the nC counts: each thread sums a contiguous run, one block scan
  const long long run = (p.nC + kThreads - 1) / kThreads;
  const long long r0 = min(p.nC, (long long)threadIdx.x * run), r1 = min(p.nC, r0 + run);
  unsigned long long mine = 0;
  for (long long c = r0; c < r1; c++) mine += __ldcg(&words[c]);
  uint32_t tot;
  unsigned long long acc = block_exclusive_scan<kThreads>((uint32_t)mine, tot, s.wscan);
  for (long long c = r0; c < r1; c++) {
    const unsigned long long v = __ldcg(&words[c]);
    words[c] = acc;
    acc += v;
  }
}

// ------------------------------------------------------------------ stage 3: compaction

// Block (group g, chunk cc): every warp owns whole 32-tile segments of the chunk; the
// segment masks and a warp scan of their counts give every tile's place.  Widths {3, 4}
// on tiles of G values: a lo slot is three units of U = G / 8 bytes, a hi slot four
// (slots, group stride and chunk offsets are multiples of U).  A warp copies two
// segments at a time, lane l unit l & 3 of tiles l / 4 + 8 q, q = 0..7: eight loads a
// lane in flight.
template <int G>
__global__ void __launch_bounds__(kThreads, 4) k_run_compact(const __grid_constant__ EncParams p) {
  constexpr int U = G / 8;
  using Unit = std::conditional_t<U == 16, uint4, std::conditional_t<U == 8, uint2, uint32_t>>;
  const long long g = blockIdx.x / p.nC, cc = blockIdx.x % p.nC;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  dep_wait();
  dep_launch();
  const long long tl0 = cc * p.CHC;
  const int nt = (int)min(p.CHC, p.n_g - tl0);
  const int nseg = (nt + 31) >> 5;
  if (2 * warp >= nseg) return;
  const long long t0 = g * p.n_g + tl0;
  const uint32_t* sm = p.segmask + g * ((p.n_g + 31) / 32) + (tl0 >> 5);
  const uint32_t m0 = lane < nseg ? __ldcg(sm + lane) : 0u;
  const uint32_t m1 = lane + 32 < nseg ? __ldcg(sm + lane + 32) : 0u;
  const unsigned long long prefix = __ldcg(&p.lookback[g * p.nC + cc]);
  const uint32_t c0 = (uint32_t)__popc(m0), c1 = (uint32_t)__popc(m1);
  uint32_t e0 = c0, e1 = c1;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t a = __shfl_up_sync(kFull, e0, d), b = __shfl_up_sync(kFull, e1, d);
    if (lane >= d) {
      e0 += a;
      e1 += b;
    }
  }
  e1 += __shfl_sync(kFull, e0, 31) - c1;
  e0 -= c0;
  // units within the group's stream (a group's stream is below 2^31 bytes)
  Unit* gout = reinterpret_cast<Unit*>(p.codes + g * p.group_bytes);
  const uint32_t gunits = (uint32_t)(p.group_bytes / U);
  const uint32_t base = (uint32_t)(3 * tl0 + (long long)prefix);
  const Unit* slo = reinterpret_cast<const Unit*>(p.scratch_lo) + 3 * t0;
  const Unit* shi = reinterpret_cast<const Unit*>(p.scratch_hi) + 4 * t0;
  const int u = lane & 3, kl = lane >> 2;
  for (int sb = 2 * warp; sb < nseg; sb += 2 * kWarps) {
    uint32_t mk[2], ob[2];
    int nv[2];
#pragma unroll
    for (int j = 0; j < 2; j++) {
      const int seg = sb + j;  // segments sb, sb + 1 lie in the same half of the chunk
      mk[j] = __shfl_sync(kFull, seg < 32 ? m0 : m1, seg & 31);
      const uint32_t before = __shfl_sync(kFull, seg < 32 ? e0 : e1, seg & 31);
      nv[j] = seg < nseg ? min(32, nt - 32 * seg) : 0;
      ob[j] = base + 96u * seg + before;  // the segment's first unit
    }
    Unit val[8];
    uint32_t dst[8];  // 0xFFFFFFFF: no unit
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const int j = q >> 2, kt = kl + 8 * (q & 3);  // tile kt of segment sb + j
      const bool ishi = (mk[j] >> kt) & 1u;
      dst[q] = 0xFFFFFFFFu;
      if (kt < nv[j] && (ishi || u < 3)) {
        const int tile = 32 * (sb + j) + kt;  // within the chunk
        val[q] = __ldcg(ishi ? shi + 4 * tile + u : slo + 3 * tile + u);
        dst[q] = ob[j] + 3u * kt + (uint32_t)__popc(mk[j] & ((1u << kt) - 1u)) + u;
      }
    }
#pragma unroll
    for (int q = 0; q < 8; q++) {
      if (dst[q] == 0xFFFFFFFFu) continue;
      if (dst[q] < gunits) {
        gout[dst[q]] = val[q];
      } else {
        set_status(p.status, kStSelectMismatch);  // only if the select went wrong
      }
    }
  }
}

}  // namespace tahq
