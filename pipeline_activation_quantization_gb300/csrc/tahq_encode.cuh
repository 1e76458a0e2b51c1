// tahq_encode.cuh -- encode kernels of the TAH-Quant activation codec for sm_103a
// (instantiated per input type by tahq_encode_f32.cu and tahq_encode_bf16.cu).
//
// "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over Slow
// Network" (arXiv 2506.01352v2):
//   §3.2 eq. (1)-(2): entropy key of every tile and the per-group key histograms;
//   §3.2 "Top-p% tile selection": the K tiles of highest (key, -index) of each group get
//        the high bit width -- histogram bucket, then an exact selection among the
//        candidates of that bucket;
//   §3.3 eq. (3) outlier ratio and pivot, pivot swap + eq. (4) Hadamard, the asymmetric
//        quantizer; §3.4's contiguous uint8 stream.
//
// The input is read from HBM once.  k_encode runs four kinds of work item in one
// persistent kernel:
//   tiles    (per 32 KB input chunk) entropy key + histograms, range, pretest, the exact
//            outlier test / pivot swap / Hadamard where needed, and the tile quantised at
//            BOTH candidate widths into two scratch streams with fixed slots;
//   select   (per group) the K-th ranked key: candidates of the histogram bucket that
//            holds it, then their exact rank;
//   offsets  (per group) every tile's width, hi counts per compaction chunk, their
//            exclusive prefix;
//   compact  (per compaction chunk) copy each tile's slot of its width from scratch to
//            its place in the stream, and its scale; the scratch lines are then dropped
//            from L2 without being written back.
// Items are handed out in increasing order by an atomic ticket and only wait for earlier
// items, so every wait ends (and each is bounded anyway).  The ticket order interleaves
// one group's tiles items with the compaction of the group two (or one) before, so the
// scratch a compaction reads is still in L2.
//
// k_encode_flat covers allocations that do not depend on the ranking (K = 0 or K = n_g:
// every tile gets the same width): one pass straight into the stream, no keys.
//
// Two data layouts, chosen per (input type, tile width):
//   line   (tiles of >= 128 bytes) one lane = one 128-byte line, chunks staged by 2-D
//          tensor copies with the 128-byte swizzle (tahq_line.cuh);
//   narrow (smaller tiles) a team of L lanes holds a tile, 32 bytes per lane, chunks
//          staged by 1-D bulk copies (tahq_tile.cuh).
// In both, a tile that fails the cheap two-values pretest (two values of magnitude
// >= max / 2 rule out r > tau) is handled again exactly, with the whole team or warp.
#pragma once

#include <algorithm>
#include <cfloat>
#include <cstring>
#include <mutex>
#include <type_traits>

#include <cuda.h>

#include "tahq_device.cuh"
#include "tahq_launch.h"
#include "tahq_line.cuh"
#include "tahq_tile.cuh"

namespace tahq {

constexpr int kChunkBytes = kEncChunkBytes;
constexpr uint8_t kDeferred = 0xFE;  // narrow layout: pass-1 marker of a tile left to pass 2
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kDirectCC = 1024;  // tiles per compaction chunk of the direct path (<= 64 segments)
constexpr int kMaxCC = kEncMaxCC;     // tiles per compaction chunk, at most
constexpr int kRankMax = 2048;        // candidates ranked in one pass (else radix select)

template <typename Tin, int G>
struct Cfg {
  static constexpr bool kBf16 = InTraits<Tin>::kBf16;
  static constexpr bool kLine = G * (int)sizeof(Tin) >= 128;
  static constexpr int CH = kChunkBytes / (G * (int)sizeof(Tin));  // tiles per input chunk
  // narrow layout: a team of L lanes per tile, V values per lane
  using Gm = TileGeom<Tin, G>;
  static constexpr int V = Gm::V, W = Gm::W, L = Gm::L, TPW = Gm::TPW;
  static constexpr int kSteps = CH / (kWarps * TPW);  // warp steps per chunk
  static constexpr int NS = CH / kWarps;              // tiles owned by a warp
  static constexpr int kArr = kLine ? 1 : CH;         // per-tile arrays of the narrow layout
  static constexpr int kAlloc = kLine ? CH : 1;       // line layout: per-tile sums (A != G)
  static_assert(kLine || kSteps * kWarps * TPW == CH, "chunk must be whole warp steps");
};

// A 2-D tensor-copy descriptor (the driver's CUtensorMap, opaque here).
struct alignas(64) TmaDesc {
  unsigned char bytes[128];
};

// Barrier of the block's 256 threads (named barrier 1).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

struct Item {
  int type;  // kItemTiles, kItemSelect, kItemOffsets, kItemCompact
  long long g, idx;
};
constexpr int kItemTiles = 0, kItemSelect = 1, kItemOffsets = 2, kItemCompact = 3;

template <typename Tin, int G>
struct alignas(128) EncSmem {  // placed on a 1024-byte boundary (enc_smem)
  using C = Cfg<Tin, G>;
  unsigned char buf[2][kChunkBytes];  // input chunks (a compaction uses its slot's as stage)
  LgTables tabs;
  // narrow layout, per tile of the input chunk: (L, S) in stats, then (min, max) and
  // (inv_lo, inv_hi or scale); deferred lists
  float ta[C::kArr], tb[C::kArr], tc[C::kArr];
  float aL[C::kAlloc], aS[C::kAlloc];  // line layout: each tile's (L, S) when A != G
  uint16_t qoff[C::kAlloc];  // k_quant: each tile's slot offset in its chunk's run
  uint8_t qb[C::kAlloc];     // k_quant: each tile's width
  uint8_t piv[C::kArr];
  uint16_t dl[C::CH];  // deferred tiles (line: one list per block; narrow: per warp)
  uint32_t ndef[2];    // line layout: length of dl, one counter per item parity
  uint32_t hist[kCoarseBins];
  uint32_t scan[kWarps + 4];
  unsigned long long bar[2];  // the slot's input chunk has landed
  Item item[2];
  uint32_t last;
};

struct EncParams {
  TmaDesc tmap;  // line layout: the input as [rows of 128 bytes]
  unsigned long long wait_ns;  // bound of every wait (see mbar_wait / wait_counter)
  float scale_c;               // streaming encoder: the input is read as RN(c x) (1: as it is)
  const void* x;
  long long n_tiles, n_g, n_groups, K, group_bytes, codes_bytes;
  long long nA, nC, CHC, J, lag, pre1, pre2, n_items;
  uint32_t seg_n;
  uint32_t seg[5][8];
  int lo, hi, h, flat_b;
  int direct;  // compaction copies slots straight from scratch (16-byte aligned throughout)
  int slot_lo, slot_hi;
  float c_h;
  float tau;  // outlier threshold (§3.3 eq. (3): transform where r > tau)
  int wire;   // quantise with the wire format's fp16 zero and scales
  int mlog;         // allocation tiles of 2^mlog tiles (§3.2 "Tile decomposition")
  long long n_ga;   // allocation tiles per group (one key each)
  float fscale;     // key -> fine histogram bucket scale (fine_bin)
  uint8_t* codes;
  float* scales;
  float* zeros;
  uint8_t* bits;
  uint8_t* pivots;
  uint8_t* scratch_lo;
  uint8_t* scratch_hi;
  float* keys;
  unsigned long long* cand;
  uint32_t* segmask;  // per group, per 32-tile segment: bit k = tile k is hi
  uint32_t* cand_cnt;
  uint32_t* hist_coarse;
  uint32_t* hist_fine;
  uint32_t* doneA;
  uint32_t* doneB;
  uint32_t* doneB2;
  uint32_t* selready;  // 1 once sel[g] is published, 2 once the compaction offsets are
  SelResult* sel;
  unsigned long long* lookback;  // per group: hi count, then offset, of each compaction chunk
  uint32_t* ticket;
  uint32_t* status;
  unsigned long long* items;  // [n_items] the decoded queue
  LgTables tabs;
};

// ====================================================================== helpers

template <typename Tin, int G>
__device__ __forceinline__ void init_tables(EncSmem<Tin, G>& sm, const LgTables& tabs) {
  for (int i = threadIdx.x; i < 128 * 32; i += kThreads) {
    if constexpr (Cfg<Tin, G>::kBf16) {
      g_lgTB[i] = tabs.TB[i >> 5];
    } else {
      g_lgT[i] = tabs.T[i >> 5];
      g_lgR[i] = tabs.R[i >> 5];
    }
  }
  for (int i = threadIdx.x; i < 128; i += kThreads) {
    sm.tabs.T[i] = tabs.T[i];
    sm.tabs.R[i] = tabs.R[i];
    sm.tabs.TB[i] = tabs.TB[i];
  }
  if (threadIdx.x < 3) sm.tabs.k[threadIdx.x] = tabs.k[threadIdx.x];
}

template <int kN>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t& total,
                                                         uint32_t* s_warp) {
  constexpr int kW = kN / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  csync();
  if (warp == 0) {
    const uint32_t w = lane < kW ? s_warp[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += y;
    }
    __syncwarp();
    if (lane < kW) s_warp[lane] = wi - w;
    if (lane == kW - 1) s_warp[kW] = wi;
  }
  csync();
  total = s_warp[kW];
  const uint32_t r = s_warp[warp] + incl - v;
  csync();
  return r;
}

// One warp: bins[0..255] in shared memory, 1 <= k <= sum(bins).  Walking the bins from
// the top (255 down to 0) with a running count, returns the bin at which the count first
// reaches k and the count strictly above that bin.
__device__ __forceinline__ void warp_find_from_top(const uint32_t* bins, uint32_t k, int& bin,
                                                   uint32_t& above) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8], s = 0;
#pragma unroll
  for (int j = 0; j < 8; j++) {
    c[j] = bins[255 - (lane * 8 + j)];
    s += c[j];
  }
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t excl = incl - s;
  const unsigned hit = __ballot_sync(kFull, incl >= k);
  const int src = hit ? (__ffs(hit) - 1) : 31;
  int my_bin = 0;
  uint32_t my_above = 0;
  if (lane == src) {
    uint32_t cum = excl;
    my_bin = 255 - (lane * 8 + 7);
    my_above = cum;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      if (cum + c[j] >= k) {
        my_bin = 255 - (lane * 8 + j);
        my_above = cum;
        break;
      }
      cum += c[j];
    }
  }
  bin = __shfl_sync(kFull, my_bin, src);
  above = __shfl_sync(kFull, my_above, src);
}

__device__ __forceinline__ float qmax_f(int b) {
  return __fsub_rn(__uint_as_float(0x4B000000u | ((1u << b) - 1u)), 8388608.0f);
}

// The wire format's quantiser for a tile of range [mn, mx]: off = the fp16 zero,
// inv_lo / inv_hi = RN(1 / s_b) of the fp16 scales; meta = what the tile's scale slot
// keeps: the scale of the one width (flat; inv_hi is then that scale too, like the fp32
// path's), else mx, from which the offsets items take the scale of the chosen width.
__device__ __forceinline__ void wire_params(float mn, float mx, int lo, int hi, bool flat,
                                            float& off, float& inv_lo, float& inv_hi,
                                            float& meta) {
  off = wire_zero(mn);
  const float s_lo = wire_scale(off, mx, qmax_f(lo));
  inv_lo = wire_inv(s_lo);
  if (flat) {
    inv_hi = s_lo;
    meta = s_lo;
  } else {
    inv_hi = wire_inv(wire_scale(off, mx, qmax_f(hi)));
    meta = mx;
  }
}

// Per-tile results of the tiles pass that do not depend on the width chosen later:
// zero-point, pivot, and the range D (in `scales` until the compaction turns it into
// D / Q).  In the one-width pass the scale and width are final at once.
__device__ __forceinline__ void put_meta(const EncParams& p, long long t, float mn, uint8_t piv,
                                         float d_or_scale, bool flat) {
  p.zeros[t] = __fadd_rn(mn, 0.0f);
  p.pivots[t] = piv;
  p.scales[t] = d_or_scale;
  if (flat) p.bits[t] = (uint8_t)p.flat_b;
}

// ====================================================================== tiles: line layout

// Deferred tiles of the narrow layout, a team of L lanes (V values each) per tile: list[j] for j = first +
// team, first + TPW + team, ... while j < n (first / step warp-uniform): the exact ratio
// test (eq. (3)), pivot swap and Hadamard (eq. (4)) where it holds, range, both widths.
template <typename Tin, int G>
__device__ __forceinline__ void pass2_teams(const EncParams& p, const unsigned char* buf,
                                            const uint16_t* list, int n, int first, int step,
                                            long long t0, bool flat, unsigned char* stage_lo,
                                            unsigned char* stage_hi) {
  using C = Cfg<Tin, G>;
  constexpr int V = C::V, W = C::W, L = C::L;
  const int lane = threadIdx.x & 31;
  const int team = lane / L, sub = lane % L;
  const int lo = flat ? p.flat_b : p.lo, hi = p.hi;
  const int slot_lo = G * lo / 8;
#pragma unroll 1
  for (int j0 = first; j0 < n; j0 += step) {
    const int ci = j0 + team;
    const bool valid = ci < n;
    const int kt = valid ? (int)list[ci] : 0;
    uint32_t w[W];
    if (valid) {
      lds_words<Tin, G>(buf, kt, sub, w);
    } else {
#pragma unroll
      for (int k = 0; k < W; k++) w[k] = 0u;
    }
    float v[V];
    words_to_values<Tin, G>(w, v);
    float m1, m2;
    int i1;
    team_top2_values<V, L>(v, sub, m1, i1, m2);
    const bool flag = valid && __fdiv_rn(m1, __fadd_rn(m2, 1e-12f)) > p.tau;
    if (__any_sync(kFull, flag)) {
      float t[V];
#pragma unroll
      for (int j = 0; j < V; j++) t[j] = v[j];
      team_swap0<V>(t, flag ? i1 : 0, sub, lane - sub);
      team_fwht<V, L>(t, p.h, sub);
      if (flag) {
#pragma unroll
        for (int j = 0; j < V; j++) v[j] = __fmul_rn(t[j], p.c_h);
      }
    }
    float mn = v[0], mx = v[0];
#pragma unroll
    for (int j = 1; j < V; j++) {
      mn = fminf(mn, v[j]);
      mx = fmaxf(mx, v[j]);
    }
    mn = team_min<L>(mn);
    mx = team_max<L>(mx);
    const float D = __fsub_rn(mx, mn);
    float scale_lo, inv_lo, scale_hi, inv_hi;
    scale_inv<L>(D, valid ? lo : 1, sub, scale_lo, inv_lo);
    scale_inv<L>(D, valid ? hi : 1, sub, scale_hi, inv_hi);
    float qoff = mn, meta = flat ? scale_lo : D;
    if (p.wire) wire_params(mn, mx, lo, hi, flat, qoff, inv_lo, inv_hi, meta);
    if (valid) {
      quant_store<V>(v, qoff, inv_lo, lo, stage_lo + kt * slot_lo + sub * (V * lo / 8));
      if (!flat) quant_store<V>(v, qoff, inv_hi, hi, stage_hi + kt * p.slot_hi + sub * (V * hi / 8));
      if (sub == 0) put_meta(p, t0 + kt, qoff, flag ? (uint8_t)i1 : (uint8_t)0xFF, meta, flat);
    }
  }
}

// Warp-wide reductions of the redux unit (one instruction per warp).
__device__ __forceinline__ float warp_max_abs(float x) {
  float r;
  asm("redux.sync.max.abs.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float warp_max_f(float x) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float warp_min_f(float x) {
  float r;
  asm("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

// Keys of the chunk's allocation tiles (2^mlog consecutive tiles each; §3.2 "Tile
// decomposition"): the block adds the tiles' (L, S) pairwise in place, level by level
// (pairs (j, j + w) for j a multiple of 2w: the natural-order pairwise sum over each
// allocation tile's A values, whose halves are whole tiles), then one thread per
// allocation tile forms the key and counts it in the group's histograms.  The chunk
// starts on an allocation-tile boundary and holds whole allocation tiles.  Called by the
// whole block.
template <typename Tin, int G>
__device__ __noinline__ void alloc_keys(EncSmem<Tin, G>& s, const EncParams& p, long long g,
                                        long long t0, int nt, float* Ls, float* Ss) {
  const int m = 1 << p.mlog;
  for (int w = 1; w < m; w <<= 1) {
    for (int j = threadIdx.x * 2 * w; j < nt; j += kThreads * 2 * w) {
      Ls[j] = __fadd_rn(Ls[j], Ls[j + w]);
      Ss[j] = __fadd_rn(Ss[j], Ss[j + w]);
    }
    csync();
  }
  for (int i = threadIdx.x; i < (nt >> p.mlog); i += kThreads) {
    const float L = Ls[i * m], S = Ss[i * m];
    const float H = entropy_key(L, S, s.tabs);
    p.keys[(t0 >> p.mlog) + i] = H;
    if (!(L <= FLT_MAX) || !(fabsf(S) <= FLT_MAX) || !(fabsf(H) <= FLT_MAX))
      set_status(p.status, kStNonFinite);
    const int b = fine_bin(H, p.fscale);
    atomicAdd(&p.hist_fine[g * (long long)kFineBins + b], 1u);
    atomicAdd(&p.hist_coarse[g * kCoarseBins + (b >> 8)], 1u);
  }
}

// Values a lane takes in the exact path of the line layout: more values a lane means
// fewer shuffle stages and team reductions per tile and 32 / (G / V) tiles per warp step.
// One lane's codes at the wider width must fit 64 bits (widths known at compile time,
// else up to 8 bits), and a team has at least two lanes.
constexpr int kP2Target = 8;
template <typename Tin, int G, int kLo, int kHi>
__host__ __device__ constexpr int p2_values() {
  const int vpu = InTraits<Tin>::kBf16 ? 8 : 4;
  const int bmax = (kLo > 0 && kHi > 0) ? (kLo > kHi ? kLo : kHi) : 8;
  int v = kP2Target < vpu ? vpu : kP2Target;
  while (v > vpu && (v * bmax > 64 || G / v < 2)) v /= 2;
  return v;
}

// Deferred tiles of the line layout (the pretest could not rule out r > tau), one
// block-wide list: teams of L = G / V lanes (V consecutive values a lane, in 16-byte
// units of the line) take list entries warp * TPW + team, + kWarps * TPW, ...  The main
// pass has already written every tile's slots and metadata as untransformed; here the
// exact ratio test (eq. (3)) runs, and only the tiles it flags get the pivot swap and
// Hadamard (eq. (4)), a new range and new slots of both widths.  V * bits <= 64 (one
// lane's codes in one 64-bit word); for V < 8, 8 / V lanes gather each group of 8 codes.
//
// The ratio test RN(m1 / d) > tau, d = RN(m2 + 1e-12) >= 1e-12.  For the method's
// tau = 2 it needs no division: it holds iff m1 / d > 2 + 2^-23 (ties round to 2), i.e.
// m1 / 2 - d > d 2^-24.  m1 / 2 is exact, m1 / 2 - d is exact by Sterbenz's lemma where it
// matters (d <= m1 <= 4 d; below, it is negative; above, it rounds to at least d), and
// d 2^-24 is a normal number.  Other thresholds take the IEEE division.
template <typename Tin, int G, int V, bool kGen>
__device__ __forceinline__ void pass2_line(const EncParams& p, const unsigned char* buf,
                                           const uint16_t* list, int n, long long t0, bool flat,
                                           int lo, int hi, unsigned char* stage_lo,
                                           unsigned char* stage_hi) {
  constexpr bool kBf = InTraits<Tin>::kBf16;
  constexpr int VPU = kBf ? 8 : 4;  // values per 16-byte unit
  constexpr int NU = V / VPU;       // units per lane
  constexpr int L = G / V, TPW = 32 / L, LPT = LineGeom<Tin, G>::LPT;
  constexpr int kGrp = V < 8 ? 8 / V : 1;  // lanes per group of 8 codes
  static_assert(NU >= 1 && 8 % NU == 0, "whole 16-byte units of one line");
  static_assert(L >= 2 && L <= 32, "team of 2..32 lanes");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L, base = lane - sub;
#pragma unroll 1
  for (int j0 = warp * TPW; j0 < n; j0 += kWarps * TPW) {
    const int ci = j0 + team;
    const bool valid = ci < n;
    const int kt = valid ? (int)list[ci] : 0;
    const int u0 = sub * NU;  // the lane's first unit in the tile
    const int line = kt * LPT + (u0 >> 3);
    float v[V];
#pragma unroll
    for (int k = 0; k < NU; k++) {
      const int ju = (u0 & 7) + k;
      const uint4 q = *reinterpret_cast<const uint4*>(buf + line * 128 + ((ju ^ (line & 7)) << 4));
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
    // top two magnitudes and the first arg-max of the tile
    float m1, m2;
    int i1;
    if constexpr (L == 32) {
      float la = fabsf(v[0]);
#pragma unroll
      for (int j = 1; j < V; j++) la = fmaxf(la, fabsf(v[j]));
      m1 = warp_max_abs(la);
      int jj = V;
#pragma unroll
      for (int j = V - 1; j >= 0; j--)
        if (fabsf(v[j]) == m1) jj = j;
      const unsigned hit = __ballot_sync(kFull, jj < V);
      const int src = hit ? __ffs(hit) - 1 : 0;
      i1 = __shfl_sync(kFull, lane * V + (jj < V ? jj : 0), src);
      float l2 = 0.0f;
#pragma unroll
      for (int j = 0; j < V; j++)
        if (lane * V + j != i1) l2 = fmaxf(l2, fabsf(v[j]));
      m2 = warp_max_f(l2);
    } else {
      team_top2_values<V, L>(v, sub, m1, i1, m2);
    }
    const float d = __fadd_rn(m2, 1e-12f);
    const bool flag =
        valid && ((!kGen || p.tau == 2.0f)
                      ? __fsub_rn(__fmul_rn(m1, 0.5f), d) > __fmul_rn(d, 0x1p-24f)
                      : __fdiv_rn(m1, d) > p.tau);
    if (!__any_sync(kFull, flag)) continue;  // the main pass's slots stand
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
    if constexpr (L == 32) {
      mn = warp_min_f(mn);
      mx = warp_max_f(mx);
    } else {
      mn = team_min<L>(mn);
      mx = team_max<L>(mx);
    }
    const float D = __fsub_rn(mx, mn);
    // lane 0 of the team: Q_lo / D; lane 1: Q_hi / D (or D / Q_b in the one-width pass)
    const float num = sub == 1 ? (flat ? D : qmax_f(hi)) : qmax_f(lo);
    const float den = sub == 1 ? (flat ? qmax_f(lo) : D) : D;
    const float r = __fdiv_rn(num, den);
    const float r0 = __shfl_sync(kFull, r, base), r1s = __shfl_sync(kFull, r, base + 1);
    const bool degenerate = !(D >= 0x1p-120f);
    float inv_lo = degenerate ? 0.0f : r0, r1 = degenerate ? 0.0f : r1s;
    float qoff = mn, meta = flat ? r1 : D;
    if (kGen && p.wire) {
      // lane 0 of the team searches the scale of bits_lo, the others that of bits_hi
      qoff = wire_zero(mn);
      const float sm = wire_scale(qoff, mx, qmax_f(sub != 0 && !flat ? hi : lo));
      const float s_lo = __shfl_sync(kFull, sm, base), s_hi = __shfl_sync(kFull, sm, base + 1);
      inv_lo = wire_inv(s_lo);
      r1 = flat ? s_lo : wire_inv(s_hi);
      meta = flat ? s_lo : mx;
    }
#pragma unroll
    for (int w2 = 0; w2 < 2; w2++) {
      if (w2 == 1 && flat) break;
      const int b = w2 ? hi : lo;
      const float inv = w2 ? r1 : inv_lo;
      unsigned long long f = 0ull;
#pragma unroll
      for (int j = 0; j < V; j++) {
        const float c = __fmaf_rn(__fsub_rn(v[j], qoff), inv, 12582912.0f);
        f |= (unsigned long long)(__float_as_uint(c) - 0x4B400000u) << (j * b);
      }
      unsigned char* slot = (w2 ? stage_hi : stage_lo) + kt * (G * b / 8);
      if constexpr (kGrp > 1) {
        f |= __shfl_down_sync(kFull, f, 1) << (V * b);
        if (flag && sub % kGrp == 0) sts_bytes(slot + (sub / kGrp) * b, f, 0ull, b);
      } else {
        if (flag) sts_bytes(slot + sub * (V * b / 8), f, 0ull, V * b / 8);
      }
    }
    if (flag && sub == 0) put_meta(p, t0 + kt, qoff, (uint8_t)i1, meta, flat);
  }
}

// Tiles pass over one staged chunk, line layout: each warp takes 32 consecutive lines.
// kLo / kHi: the two widths when known at compile time (0: from p).
template <typename Tin, int G, int kLo, int kHi, bool kGen>
__device__ __forceinline__ void tiles_line(EncSmem<Tin, G>& s, const EncParams& p, long long g,
                                           long long t0, int nt, const unsigned char* buf,
                                           bool flat, unsigned char* stage_lo,
                                           unsigned char* stage_hi, uint32_t* ndef) {
  using LG = LineGeom<Tin, G>;
  constexpr int LPT = LG::LPT, NE = LG::NE;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int line = warp * 32 + lane;
  const int kt = line / LPT, sub = line % LPT;
  const bool valid = kt < nt;
  // entropy key and histograms (§3.2)
  if (!flat) {
    float2 ls = line_sums<Tin>(buf, line, s.tabs, lg_consts(s.tabs, lane));
    ls = team_sum2<LPT>(ls);
    if (valid && sub == 0) {
      if (kGen && p.mlog > 0) {  // the allocation tiles' keys follow the block barrier below
        s.aL[kt] = ls.x;
        s.aS[kt] = ls.y;
      } else {
        const float H = entropy_key(ls.x, ls.y, s.tabs);
        p.keys[t0 + kt] = H;
        if (!(ls.x <= FLT_MAX) || !(fabsf(ls.y) <= FLT_MAX) || !(fabsf(H) <= FLT_MAX))
          set_status(p.status, kStNonFinite);
        const int b = fine_bin(H, p.fscale);
        atomicAdd(&p.hist_fine[g * (long long)kFineBins + b], 1u);
        // the coarse bins of a group's tiles are few (similar entropies): count them in
        // the block first, one global add per bin and item below
        atomicAdd(&s.hist[b >> 8], 1u);
      }
    }
  }

  // range and the two-values pretest
  uint32_t w[32];
  lds_line(buf, line, w);
  float mn, mx, ga[NE / 8];
  line_minmax<Tin>(w, mn, mx, ga);
  mn = team_min<LPT>(mn);
  mx = team_max<LPT>(mx);
  const float m1 = fmaxf(mx, -mn);
  // two values of at least m1 / tau give m2 >= m1 / tau, so r < tau: the threshold is
  // rounded up to keep the test on the safe side (m1 / 2 is exact for m1 >= 2^-120)
  const float thr = (!kGen || p.tau == 2.0f) ? __fmul_rn(m1, 0.5f) : __fdiv_ru(m1, p.tau);
  uint32_t cnt = 0;
#pragma unroll
  for (int q = 0; q < NE / 8; q++) cnt += ga[q] >= thr ? 1u : 0u;
  cnt = team_sum_u<LPT>(cnt);
  // for tau >= 1 a maximum below 2^-120 can never give r > tau (the ratio is below 1e-24);
  // a tile whose maximum is not finite goes to the exact test
  const bool small = m1 < 0x1p-120f && (!kGen || p.tau >= 1.0f);
  const bool deferred = !small && (!(m1 <= FLT_MAX) || cnt < 2u);

  // widths: Q_lo / D and Q_hi / D (or D / Q_b), split over the team's lanes
  const int lo = kLo ? kLo : (flat ? p.flat_b : p.lo);
  const int hi = kHi ? kHi : p.hi;
  const float D = __fsub_rn(mx, mn);
  float inv_lo, r1;
  if constexpr (LPT >= 2) {
    const bool odd = sub & 1;
    const float num = odd ? (flat ? D : qmax_f(hi)) : qmax_f(lo);
    const float den = odd ? (flat ? qmax_f(lo) : D) : D;
    const float r = __fdiv_rn(num, den);
    const float o = __shfl_xor_sync(kFull, r, 1);
    inv_lo = odd ? o : r;
    r1 = odd ? r : o;
  } else {
    inv_lo = __fdiv_rn(qmax_f(lo), D);
    r1 = flat ? __fdiv_rn(D, qmax_f(lo)) : __fdiv_rn(qmax_f(hi), D);
  }
  if (!(D >= 0x1p-120f)) inv_lo = r1 = 0.0f;
  float qoff = mn, meta = flat ? r1 : D;
  if (kGen && p.wire) {
    if constexpr (LPT >= 2) {
      // the tile's even lanes search the scale of bits_lo, its odd lanes that of bits_hi
      qoff = wire_zero(mn);
      const bool odd = sub & 1;
      const float sm = wire_scale(qoff, mx, qmax_f(odd && !flat ? hi : lo));
      const float so = __shfl_xor_sync(kFull, sm, 1);
      const float s_lo = odd ? so : sm, s_hi = odd ? sm : so;
      inv_lo = wire_inv(s_lo);
      r1 = flat ? s_lo : wire_inv(s_hi);
      meta = flat ? s_lo : mx;
    } else {
      wire_params(mn, mx, lo, hi, flat, qoff, inv_lo, r1, meta);
    }
  }
  // every tile as untransformed; the exact test below redoes the ones it flags
  if (valid) {
    line_quant<Tin, kLo>(w, qoff, inv_lo, lo, stage_lo + kt * (G * lo / 8) + sub * (NE * lo / 8));
    if (!flat)
      line_quant<Tin, kHi>(w, qoff, r1, hi, stage_hi + kt * (G * hi / 8) + sub * (NE * hi / 8));
    if (sub == 0) put_meta(p, t0 + kt, qoff, (uint8_t)0xFF, meta, flat);
  }
  // tiles the pretest could not clear: one list for the block, teams of the whole block
  // take them in turn (outlier channels sit at fixed tile positions, so per-warp lists
  // would load some warps far more than others).  The barrier also orders the main
  // pass's slot writes before the exact path overwrites flagged slots.
  if (valid && deferred && sub == 0) s.dl[atomicAdd(ndef, 1u)] = (uint16_t)kt;
  csync();
  if (kGen && !flat && p.mlog > 0) alloc_keys(s, p, g, t0, nt, s.aL, s.aS);
  if (!flat) {
    static_assert(kThreads == kCoarseBins, "one coarse bin per thread");
    const uint32_t c = s.hist[threadIdx.x];
    if (c) {
      atomicAdd(&p.hist_coarse[g * kCoarseBins + threadIdx.x], c);
      s.hist[threadIdx.x] = 0u;  // bins are all zero between items
    }
  }
  pass2_line<Tin, G, p2_values<Tin, G, kLo, kHi>(), kGen>(p, buf, s.dl, (int)*ndef, t0, flat, lo, hi,
                                                    stage_lo, stage_hi);
}

// ====================================================================== tiles: narrow layout

// Tile `l` (0 <= l < NS) of warp `warp`: the tiles a warp handles over all its steps.
template <typename Tin, int G>
__device__ __forceinline__ int warp_tile(int l, int warp) {
  using C = Cfg<Tin, G>;
  return ((l / C::TPW) * kWarps + warp) * C::TPW + (l % C::TPW);
}

// Tiles pass over one staged chunk, narrow layout (a team of L lanes per tile, V values
// per lane; each warp handles its own NS tiles with no block-wide barrier):
//   stats    per warp step the team's two sums; then one lane per tile forms the key;
//   phase 1  per warp step the tile's min / max and the two-values test (two lanes whose
//            own max |v| reaches max / 2); tiles that fail it are deferred;
//   phase 2  one lane per tile: the two divisions and the tile's metadata;
//   phase 3  per warp step: quantise and pack the tiles that were not deferred;
//   pass 2   the deferred tiles, compacted: exact ratio test (eq. (3)), pivot swap and
//            Hadamard (eq. (4)) where it holds, then the quantizer.
template <typename Tin, int G>
__device__ __forceinline__ void tiles_narrow(EncSmem<Tin, G>& s, const EncParams& p, long long g,
                                             long long t0, int nt, const unsigned char* buf,
                                             bool flat, unsigned char* stage_lo,
                                             unsigned char* stage_hi) {
  using C = Cfg<Tin, G>;
  constexpr int V = C::V, W = C::W, L = C::L, TPW = C::TPW, NS = C::NS;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L;
  const int lo = flat ? p.flat_b : p.lo, hi = p.hi;
  const int slot_lo = G * lo / 8;

  if (!flat) {
#pragma unroll 1
    for (int st = 0; st < C::kSteps; st++) {
      const int kt = (st * kWarps + warp) * TPW + team;
      const bool valid = kt < nt;
      uint32_t w[W];
      if (valid) {
        lds_words<Tin, G>(buf, kt, sub, w);
      } else {
#pragma unroll
        for (int k = 0; k < W; k++) w[k] = 0u;
      }
      const float2 ls = tile_sums<Tin, G>(w, s.tabs, lane);
      if (valid && sub == 0) {
        s.ta[kt] = ls.x;
        s.tb[kt] = ls.y;
      }
    }
    __syncwarp();
    uint32_t* hf = p.hist_fine + g * (long long)kFineBins;
    uint32_t* hc = p.hist_coarse + g * kCoarseBins;
    if (p.mlog > 0) {
      // allocation tiles span warps: every tile's sums in place, then their keys, before
      // phase 1 reuses the arrays
      csync();
      alloc_keys(s, p, g, t0, nt, s.ta, s.tb);
      csync();
    }
#pragma unroll 1
    for (int l0 = 0; l0 < (p.mlog > 0 ? 0 : NS); l0 += 32) {
      const int l = l0 + lane;
      const int kt = warp_tile<Tin, G>(l, warp);
      const bool valid = l < NS && kt < nt;
      int cb = -1;
      if (valid) {
        const float Ls = s.ta[kt], Ss = s.tb[kt];
        const float H = entropy_key(Ls, Ss, s.tabs);
        p.keys[t0 + kt] = H;
        if (!(Ls <= FLT_MAX) || !(fabsf(Ss) <= FLT_MAX) || !(fabsf(H) <= FLT_MAX))
          set_status(p.status, kStNonFinite);
        const int b = fine_bin(H, p.fscale);
        atomicAdd(&hf[b], 1u);
        cb = b >> 8;
      }
      const unsigned same = __match_any_sync(kFull, cb);
      if (cb >= 0 && lane == __ffs(same) - 1) atomicAdd(&hc[cb], (uint32_t)__popc(same));
    }
    __syncwarp();
  }
  // phase 1
#pragma unroll 1
  for (int st = 0; st < C::kSteps; st++) {
    const int kt = (st * kWarps + warp) * TPW + team;
    const bool valid = kt < nt;
    uint32_t w[W];
    if (valid) {
      lds_words<Tin, G>(buf, kt, sub, w);
    } else {
#pragma unroll
      for (int k = 0; k < W; k++) w[k] = 0u;
    }
    float mn, mx;
    lane_minmax_raw<Tin, G>(w, mn, mx);
    const float lane_amax = fmaxf(mx, -mn);
    mn = team_min<L>(mn);
    mx = team_max<L>(mx);
    const float m1 = fmaxf(mx, -mn);
    const float thr = p.tau == 2.0f ? __fmul_rn(m1, 0.5f) : __fdiv_ru(m1, p.tau);
    bool two;
    if constexpr (L >= 2) {
      two = team_two_ge<L>(lane_amax, thr, team);
    } else {
      two = lane_count_ge<Tin, G>(w, thr) >= 2u;
    }
    const bool tiny = !(m1 >= 0x1p-120f) || !(m1 <= FLT_MAX);
    if (valid && sub == 0) {
      s.piv[kt] = (tiny || !two) ? kDeferred : (uint8_t)0xFF;
      s.ta[kt] = mn;
      s.tb[kt] = mx;
    }
  }
  __syncwarp();
  // phase 2 (and the list of deferred tiles, kept in this warp's part of s.dl)
  uint16_t* dl = s.dl + warp * NS;
  int ndef = 0;
#pragma unroll 1
  for (int l0 = 0; l0 < NS; l0 += 32) {
    const int l = l0 + lane;
    const int kt = warp_tile<Tin, G>(l, warp);
    const bool valid = l < NS && kt < nt;
    const bool def = valid && s.piv[kt] == kDeferred;
    const unsigned dm = __ballot_sync(kFull, def);
    if (def) dl[ndef + __popc(dm & ((1u << lane) - 1u))] = (uint16_t)kt;
    ndef += __popc(dm);
    if (valid && !def) {
      const float mn = s.ta[kt], mx = s.tb[kt];
      const float D = __fsub_rn(mx, mn);
      const bool degenerate = !(D >= 0x1p-120f);
      const float inv_lo = degenerate ? 0.0f : __fdiv_rn(qmax_f(lo), D);
      float r1 =
          degenerate ? 0.0f : (flat ? __fdiv_rn(D, qmax_f(lo)) : __fdiv_rn(qmax_f(hi), D));
      float il = inv_lo, qoff = mn, meta = flat ? r1 : D;
      if (p.wire) wire_params(mn, mx, lo, hi, flat, qoff, il, r1, meta);
      s.ta[kt] = qoff;  // phase 3 quantises from the offset
      s.tb[kt] = il;
      s.tc[kt] = r1;
      put_meta(p, t0 + kt, qoff, (uint8_t)0xFF, meta, flat);
    }
  }
  __syncwarp();
  // phase 3
#pragma unroll 1
  for (int st = 0; st < C::kSteps; st++) {
    const int kt = (st * kWarps + warp) * TPW + team;
    if (kt >= nt || s.piv[kt] == kDeferred) continue;
    const float mn = s.ta[kt];
    uint32_t w[W];
    lds_words<Tin, G>(buf, kt, sub, w);
    float v[V];
    words_to_values<Tin, G>(w, v);
    quant_store<V>(v, mn, s.tb[kt], lo, stage_lo + kt * slot_lo + sub * (V * lo / 8));
    if (!flat) quant_store<V>(v, mn, s.tc[kt], hi, stage_hi + kt * p.slot_hi + sub * (V * hi / 8));
  }
  // pass 2
  pass2_teams<Tin, G>(p, buf, dl, ndef, 0, TPW, t0, flat, stage_lo, stage_hi);
}

// ====================================================================== stores

// Copy stage[0, nbytes) to dst[base, base + nbytes): 16-byte stores for the aligned
// middle (realigned from shared memory with funnel shifts), byte stores at the two ends.
__device__ __forceinline__ void store_stage(const unsigned char* stage, uint8_t* dst,
                                            long long base, int nbytes) {
  const int head = (int)((16 - (base & 15)) & 15);
  const int h = min(head, nbytes);
  const int n16 = (nbytes - h) / 16;
  const int tail0 = h + 16 * n16;
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(stage);
  const int sh = (h & 3) * 8;
  for (int i = threadIdx.x; i < n16; i += kThreads) {
    const int o = h + 16 * i;  // stage byte offset of this global 16-byte word
    const int q = o >> 2;
    uint32_t a[5];
#pragma unroll
    for (int k = 0; k < 5; k++) a[k] = sw[q + k];
    uint4 out;
    out.x = __funnelshift_r(a[0], a[1], sh);
    out.y = __funnelshift_r(a[1], a[2], sh);
    out.z = __funnelshift_r(a[2], a[3], sh);
    out.w = __funnelshift_r(a[3], a[4], sh);
    *reinterpret_cast<uint4*>(dst + base + o) = out;
  }
  const int nb = h + (nbytes - tail0);
  for (int i = threadIdx.x; i < nb; i += kThreads) {
    const int o = (i < h) ? i : tail0 + (i - h);
    dst[base + o] = stage[o];
  }
}

// ====================================================================== work items

// Round r (0 <= r < NG + lag) of the work queue:
//   the first pre1 tiles items of group r  (if r < NG)
//   the J select items of group r-1        (if 1 <= r <= NG)
//   the next pre2 tiles items of group r
//   the J offsets items of group r-1       (if 1 <= r <= NG)
//   the other tiles items of group r spread evenly among the compaction items of group
//   r-lag.
// A group's select items come after all its tiles items, its offsets items after its
// select items, and its compaction items (round >= r+1) after its offsets items.  The
// tiles items in front of the select and offsets items give the ones they wait for time
// to finish.  32-bit arithmetic: the host keeps the item count below 2^31 (and
// pos * nC below 2^32).
__device__ __forceinline__ Item decode_item(const EncParams& p, uint32_t q) {
  // segments of rounds with the same make-up (host-computed, see queue_segments)
  for (uint32_t i = 0; i < p.seg_n; i++) {
    const uint32_t* sg = p.seg[i];
    if (q >= sg[7]) continue;
    const uint32_t len = sg[5], nB = sg[2], nAr = sg[3], nCr = sg[4];
    const uint32_t r = sg[0] + (q - sg[6]) / len;
    uint32_t pos = (q - sg[6]) % len;
    const uint32_t pre1 = min((uint32_t)p.pre1, nAr);
    const uint32_t pre2 = min((uint32_t)p.pre2, nAr - pre1);
    if (pos < pre1) return Item{kItemTiles, (long long)r, (long long)pos};
    pos -= pre1;
    if (pos < nB) return Item{kItemSelect, (long long)r - 1, (long long)pos};
    pos -= nB;
    if (pos < pre2) return Item{kItemTiles, (long long)r, (long long)(pre1 + pos)};
    pos -= pre2;
    if (pos < nB) return Item{kItemOffsets, (long long)r - 1, (long long)pos};
    pos -= nB;
    // the remaining na tiles items and nCr compaction items, compaction evenly spread:
    // position pos holds a compaction item iff floor((pos+1) nCr / n) > floor(pos nCr / n)
    const uint32_t na = nAr - pre1 - pre2, n = na + nCr;
    const uint32_t before = pos * nCr / n, upto = (pos + 1u) * nCr / n;
    if (upto > before) return Item{kItemCompact, (long long)(r - (uint32_t)p.lag), (long long)before};
    return Item{kItemTiles, (long long)r, (long long)(pre1 + pre2 + pos - before)};
  }
  return Item{-1, 0, 0};
}

// Rounds r in [r0, r1) have the same items: the breakpoints 0, 1, lag, NG, NG + 1,
// NG + lag cut the rounds into at most 5 such segments.  seg[i] = {r0, r1, nB, nA, nC,
// len, first item, end item}.
static void queue_segments(EncParams& p) {
  const long long NG = p.n_groups, lag = p.lag;
  long long bp[6] = {0, 1, lag, NG, NG + 1, NG + lag};
  std::sort(bp, bp + 6);
  const long long rmax = NG + lag;
  long long cum = 0;
  p.seg_n = 0;
  for (int k = 0; k < 5; k++) {
    const long long r0 = bp[k], r1 = std::min(bp[k + 1], rmax);
    if (r1 <= r0) continue;
    const bool hasB = r0 >= 1 && r0 <= NG, hasA = r0 < NG, hasC = r0 >= lag && r0 < NG + lag;
    const long long nB = hasB ? p.J : 0, nA = hasA ? p.nA : 0, nC = hasC ? p.nC : 0;
    const long long len = 2 * nB + nA + nC;
    if (len == 0) continue;
    const long long span = (r1 - r0) * len;
    uint32_t* sg = p.seg[p.seg_n++];
    sg[0] = (uint32_t)r0;
    sg[1] = (uint32_t)r1;
    sg[2] = (uint32_t)nB;
    sg[3] = (uint32_t)nA;
    sg[4] = (uint32_t)nC;
    sg[5] = (uint32_t)len;
    sg[6] = (uint32_t)cum;
    sg[7] = (uint32_t)(cum + span);
    cum += span;
  }
}

template <typename Tin, int G>
__device__ __forceinline__ void tiles_range(const EncParams& p, const Item& it, long long& t0,
                                            int& nt) {
  constexpr int CH = Cfg<Tin, G>::CH;
  t0 = it.g * p.n_g + it.idx * CH;
  nt = (int)min((long long)CH, p.n_g - it.idx * CH);
}

// ---- tiles item: the whole per-tile computation of one input chunk, both widths into
// the scratch streams.
template <typename Tin, int G, int kLo, int kHi, bool kGen>
__device__ void do_tiles(EncSmem<Tin, G>& s, const EncParams& p, const Item& it,
                         const unsigned char* buf, uint32_t* ndef) {
  long long t0;
  int nt;
  tiles_range<Tin, G>(p, it, t0, nt);
  // slots go straight to the scratch streams (L2-resident; every warp writes whole
  // contiguous runs); the caller publishes the item after its next barrier
  unsigned char* out_lo = p.scratch_lo + t0 * p.slot_lo;
  unsigned char* out_hi = p.scratch_hi + t0 * p.slot_hi;
  if constexpr (Cfg<Tin, G>::kLine) {
    tiles_line<Tin, G, kLo, kHi, kGen>(s, p, it.g, t0, nt, buf, false, out_lo, out_hi, ndef);
  } else {
    tiles_narrow<Tin, G>(s, p, it.g, t0, nt, buf, false, out_lo, out_hi);
  }
}

// ---- select item: gather the candidates of the threshold bucket; the last select item
// of the group resolves the K-th ranked tile exactly.
template <typename Tin, int G>
__device__ void do_select(EncSmem<Tin, G>& s, const EncParams& p, const Item& it,
                          unsigned char* scratch) {
  const long long g = it.g;
  const uint32_t K = (uint32_t)p.K;
  if (threadIdx.x == 0) wait_counter(&p.doneA[g], (uint32_t)p.nA, p.status, p.wait_ns);
  csync();
  uint32_t* bins = s.hist;  // all zero between items; left zero below
  if (threadIdx.x < 32) {
    for (int i = threadIdx.x; i < 256; i += 32) bins[i] = __ldcg(&p.hist_coarse[g * kCoarseBins + i]);
    __syncwarp();
    int cb;
    uint32_t above_c;
    warp_find_from_top(bins, K, cb, above_c);
    __syncwarp();
    for (int i = threadIdx.x; i < 256; i += 32)
      bins[i] = __ldcg(&p.hist_fine[g * (long long)kFineBins + cb * 256 + i]);
    __syncwarp();
    int fb;
    uint32_t above_f;
    warp_find_from_top(bins, K - above_c, fb, above_f);
    if (threadIdx.x == 0) {
      s.scan[0] = (uint32_t)(cb * 256 + fb);
      s.scan[1] = above_c + above_f;
    }
  }
  csync();
  const int bstar = (int)s.scan[0];
  const uint32_t above = s.scan[1];
  // candidates of this item's slice of the group
  // the group's n_ga keys (one per allocation tile)
  const long long per = (p.n_ga + p.J - 1) / p.J;
  const long long lo = it.idx * per, hi = min(p.n_ga, lo + per);
  const float* kg = p.keys + g * p.n_ga;
  unsigned long long* cg = p.cand + g * p.n_ga;
  const int lane = threadIdx.x & 31;
  constexpr int kB = 8;  // keys in flight per thread
  for (long long base = lo; base < hi; base += kB * kThreads) {
    float hv[kB];
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const long long i = base + u * kThreads + threadIdx.x;
      hv[u] = i < hi ? __ldcg(&kg[i]) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const long long i = base + u * kThreads + threadIdx.x;
      const bool hit = i < hi && fine_bin(hv[u], p.fscale) == bstar;
      const unsigned mask = __ballot_sync(kFull, hit);
      if (mask) {
        uint32_t pos0 = 0;
        const int leader = __ffs(mask) - 1;
        if (lane == leader) pos0 = atomicAdd(&p.cand_cnt[g], (uint32_t)__popc(mask));
        pos0 = __shfl_sync(kFull, pos0, leader);
        if (hit) cg[pos0 + __popc(mask & ((1u << lane) - 1u))] = rank_key(hv[u], (uint32_t)i);
      }
    }
  }
  csync();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&p.doneB[g], 1u);
    __threadfence();
    s.last = (prev == (uint32_t)p.J - 1u) ? 1u : 0u;
  }
  csync();
  if (s.last) {
    const uint32_t cnt = __ldcg(&p.cand_cnt[g]);
    const uint32_t expect = __ldcg(&p.hist_fine[g * (long long)kFineBins + bstar]);
    if (threadIdx.x == 0 && cnt != expect) set_status(p.status, kStSelectMismatch);
    const uint32_t r = max(1u, min(K - above, cnt));  // rank (from 1) inside the bucket
    unsigned long long theta = 0ull;
    if (cnt > 0u && cnt <= (uint32_t)kRankMax) {
      // one pass: the candidate with exactly r - 1 larger keys (rank keys are distinct)
      unsigned long long* ck = reinterpret_cast<unsigned long long*>(scratch);
      for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) ck[i] = __ldcg(&cg[i]);
      if (threadIdx.x == 0) s.scan[2] = 0u;
      csync();
      for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
        const unsigned long long ki = ck[i];
        uint32_t larger = 0;
        for (uint32_t j = 0; j < cnt; j++) larger += ck[j] > ki ? 1u : 0u;
        if (larger == r - 1u) s.scan[2] = i;
      }
      csync();
      theta = ck[s.scan[2]];
      csync();
    } else if (cnt > 0u) {
      // radix select (8 passes of 8 bits) of the r-th largest candidate key
      uint32_t rr = r;
      unsigned long long prefix = 0ull, mask = 0ull;
      for (int pass = 7; pass >= 0; --pass) {
        const int shift = pass * 8;
        for (int i = threadIdx.x; i < 256; i += kThreads) bins[i] = 0u;
        csync();
        for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
          const unsigned long long v = __ldcg(&cg[i]);
          if ((v & mask) == prefix) atomicAdd(&bins[(v >> shift) & 255u], 1u);
        }
        csync();
        if (threadIdx.x < 32) {
          int d;
          uint32_t ab;
          warp_find_from_top(bins, rr, d, ab);
          if (threadIdx.x == 0) {
            s.scan[2] = (uint32_t)d;
            s.scan[3] = ab;
          }
        }
        csync();
        prefix |= (unsigned long long)s.scan[2] << shift;
        rr -= s.scan[3];
        mask |= 0xFFull << shift;
        csync();
      }
      theta = prefix;
    }
    if (threadIdx.x == 0) {
      p.sel[g] = SelResult{theta, cnt ? kSelThreshold : kSelNone, 0u};
      __threadfence();
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&p.selready[g]), "r"(1u) : "memory");
    }
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) bins[i] = 0u;
  csync();
}

// ---- offsets item: the width and the scale of every tile of its compaction chunks and
// their hi counts; the last offsets item of the group turns the counts into exclusive
// prefixes.
template <typename Tin, int G, bool kGen>
__device__ void do_offsets(EncSmem<Tin, G>& s, const EncParams& p, const Item& it) {
  const long long g = it.g;
  if (threadIdx.x == 0) wait_counter(&p.selready[g], 1u, p.status, p.wait_ns);
  csync();
  const unsigned long long theta = __ldcg(&p.sel[g].theta);
  const uint32_t mode = __ldcg(&p.sel[g].mode);
  unsigned long long* words = p.lookback + g * p.nC;
  const long long per = (p.nC + p.J - 1) / p.J;
  const long long c0 = it.idx * per, c1 = min(p.nC, c0 + per);
  // every thread one tile at a time, eight tiles' loads in flight; a warp's 32 tiles are
  // one segment of one compaction chunk (chunks hold a multiple of 32 tiles): its hi mask
  // goes to segmask, its hi count to the chunk's count in s.hist[c - c0]
  const long long tl_begin = c0 * p.CHC, tl_end = min(p.n_g, c1 * p.CHC);
  const int lane = threadIdx.x & 31;
  const uint32_t chc = (uint32_t)p.CHC;
  const int mlog = kGen ? p.mlog : 0;
  uint32_t* segmask = p.segmask + g * ((p.n_g + 31) / 32);
  constexpr int kB = 8;
  for (long long tb = tl_begin; tb < tl_end; tb += kB * kThreads) {
    float key[kB], Dv[kB], Zv[kB];
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const long long tl = tb + u * kThreads + threadIdx.x;
      key[u] = 0.0f;
      Dv[u] = 0.0f;
      Zv[u] = 0.0f;
      if (tl < tl_end) {
        const long long t = g * p.n_g + tl;
        if (mode == kSelThreshold) key[u] = __ldcg(&p.keys[t >> mlog]);  // its allocation tile's
        Dv[u] = __ldcg(&p.scales[t]);
        if (kGen && p.wire) Zv[u] = __ldcg(&p.zeros[t]);
      }
    }
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const long long tw = tb + u * kThreads + (threadIdx.x & ~31);  // the warp's segment
      const long long tl = tw + lane;
      bool ishi = false;
      if (tl < tl_end) {
        const long long t = g * p.n_g + tl;
        ishi = mode == kSelAll ||
               (mode == kSelThreshold && rank_key(key[u], (uint32_t)(tl >> mlog)) >= theta);
        const int b = ishi ? p.hi : p.lo;
        p.bits[t] = (uint8_t)b;
        // the range D left by the tiles pass becomes the scale D / Q (wire format: the
        // maximum left there gives the fp16 scale of this width)
        p.scales[t] = (kGen && p.wire) ? wire_scale(Zv[u], Dv[u], qmax_f(b))
                             : ((Dv[u] >= 0x1p-120f) ? __fdiv_rn(Dv[u], qmax_f(b)) : 0.0f);
      }
      const unsigned hm = __ballot_sync(kFull, ishi);
      if (lane == 0 && tw < tl_end) {
        segmask[tw >> 5] = hm;
        if (hm) atomicAdd(&s.hist[(uint32_t)(tw - tl_begin) / chc], (uint32_t)__popc(hm));
      }
    }
  }
  csync();
  for (long long c = c0 + threadIdx.x; c < c1; c += kThreads) {
    words[c] = s.hist[c - c0];
    s.hist[c - c0] = 0u;  // bins are all zero between items
  }
  csync();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&p.doneB2[g], 1u);
    __threadfence();
    s.last = (prev == (uint32_t)p.J - 1u) ? 1u : 0u;
  }
  csync();
  if (s.last) {
    // exclusive prefix of the nC counts: each thread sums a contiguous run, one block scan
    const long long run = (p.nC + kThreads - 1) / kThreads;
    const long long r0 = min(p.nC, (long long)threadIdx.x * run), r1 = min(p.nC, r0 + run);
    unsigned long long mine = 0;
    for (long long c = r0; c < r1; c++) mine += __ldcg(&words[c]);
    uint32_t tot;
    unsigned long long acc = block_exclusive_scan<kThreads>((uint32_t)mine, tot, s.scan);
    for (long long c = r0; c < r1; c++) {
      const unsigned long long v = __ldcg(&words[c]);
      words[c] = acc;
      acc += v;
    }
    csync();
    if (threadIdx.x == 0) {
      __threadfence();
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&p.selready[g]), "r"(2u) : "memory");
    }
  }
}

// Copy every tile's slot of its width from scratch into the stage, in units of Unit.
template <typename Unit>
__device__ __forceinline__ void gather_units(const uint16_t* off, const uint8_t* cbits,
                                             const EncParams& p, long long t0, int nt,
                                             unsigned char* stage) {
  constexpr int U = (int)sizeof(Unit);
  const int uph = p.slot_hi / U, upl = p.slot_lo / U;
  const int total = nt * uph;
  for (int i = threadIdx.x; i < total; i += kThreads) {
    const int k = i / uph, u = i - k * uph;
    const bool ishi = cbits[k] == (uint8_t)p.hi;
    if (!ishi && u >= upl) continue;
    const Unit* src = ishi ? reinterpret_cast<const Unit*>(p.scratch_hi + (t0 + k) * p.slot_hi)
                           : reinterpret_cast<const Unit*>(p.scratch_lo + (t0 + k) * p.slot_lo);
    *reinterpret_cast<Unit*>(stage + off[k] + u * U) = __ldcg(src + u);
  }
}

// Drop the whole 128-byte lines of [a, b) from L2 without writing them back.
__device__ __forceinline__ void discard_lines(const uint8_t* base, long long a, long long b) {
  const long long first = (a + 127) / 128, last = b / 128;
  for (long long l = first + threadIdx.x; l < last; l += kThreads)
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(base + l * 128) : "memory");
}

// Compaction with 16-byte slots and stream (the common case): every warp owns whole
// segments of 32 tiles of the chunk and needs no other warp.  The offsets items left
// each segment's hi mask; one load of the chunk's masks (two per lane, at most 64
// segments) and a warp scan of their counts give every segment's place, the mask every
// tile's.  Each lane then has up to eight 16-byte loads (two segments) in flight before
// its stores, and the warp drops its segments' scratch lines from L2.
static __device__ void compact_direct(const EncParams& p, long long g, long long cc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long tl0 = cc * p.CHC;
  const int nt = (int)min(p.CHC, p.n_g - tl0);
  const int nseg = (nt + 31) >> 5;
  if (warp >= nseg) return;
  if (lane == 0) wait_counter(&p.selready[g], 2u, p.status, p.wait_ns);
  __syncwarp();
  const long long t0 = g * p.n_g + tl0;
  const uint32_t* sm = p.segmask + g * ((p.n_g + 31) / 32) + (tl0 >> 5);
  const uint32_t m0 = lane < nseg ? __ldcg(sm + lane) : 0u;
  const uint32_t m1 = lane + 32 < nseg ? __ldcg(sm + lane + 32) : 0u;
  const unsigned long long prefix = __ldcg(&p.lookback[g * p.nC + cc]);
  // hi tiles of the chunk before segment lane (e0) and lane + 32 (e1)
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
  const int slot_lo = p.slot_lo, slot_hi = p.slot_hi, slot_d = slot_hi - slot_lo;
  const int UH = slot_hi >> 4, UL = slot_lo >> 4;
  const long long base = g * p.group_bytes + tl0 * slot_lo + (long long)prefix * slot_d;
  for (int sa = warp; sa < nseg; sa += 2 * kWarps) {
    uint32_t mask[2];
    long long ob[2], st0[2];
    int nv[2];
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const int seg = sa + h * kWarps;           // warp-uniform
      const int sx = seg < nseg ? seg : sa;
      mask[h] = __shfl_sync(kFull, sx < 32 ? m0 : m1, sx & 31);
      const uint32_t before = __shfl_sync(kFull, sx < 32 ? e0 : e1, sx & 31);
      nv[h] = seg < nseg ? min(32, nt - 32 * seg) : 0;
      st0[h] = t0 + 32 * seg;  // the segment's first tile
      ob[h] = base + 32ll * seg * slot_lo + (long long)before * slot_d;
    }
    for (int r0 = 0; r0 < UH; r0 += 4) {
      uint4 val[2][4];
      long long dst[2][4];
#pragma unroll
      for (int h = 0; h < 2; h++) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const int i = lane + 32 * (r0 + q);
          const int kt = i / UH, u = i - kt * UH;  // kt < 32 whenever r0 + q < UH
          const bool in = r0 + q < UH && kt < nv[h];
          const bool ishi = in && ((mask[h] >> (kt & 31)) & 1u);
          dst[h][q] = -1;
          if (in && (ishi || u < UL)) {
            const uint4* src = reinterpret_cast<const uint4*>(
                ishi ? p.scratch_hi + (st0[h] + kt) * slot_hi : p.scratch_lo + (st0[h] + kt) * slot_lo);
            val[h][q] = __ldcg(src + u);
            dst[h][q] = ob[h] + (long long)kt * slot_lo +
                        (long long)__popc(mask[h] & ((1u << kt) - 1u)) * slot_d + 16 * u;
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; h++) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
          if (dst[h][q] < 0) continue;
          if (dst[h][q] + 16 <= p.codes_bytes) {
            *reinterpret_cast<uint4*>(p.codes + dst[h][q]) = val[h][q];
          } else {
            set_status(p.status, kStSelectMismatch);  // only if the select went wrong
          }
        }
      }
    }
    __syncwarp();
    // 32 slots of 16-byte multiples are whole 128-byte lines
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const long long a = st0[h], b = st0[h] + nv[h];
      for (long long l = (a * slot_lo + 127) / 128 + lane; l < b * slot_lo / 128; l += 32)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(p.scratch_lo + l * 128) : "memory");
      for (long long l = (a * slot_hi + 127) / 128 + lane; l < b * slot_hi / 128; l += 32)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(p.scratch_hi + l * 128) : "memory");
    }
  }
}

// ---- compaction item: widths from the offsets items, slots from scratch, the chunk's
// place in the stream from the prefix of hi counts.  `stage` holds
// the chunk's bytes, `off` / `cbits` (CHC entries each) every tile's place and width.
template <typename Tin, int G>
__device__ void do_compact(EncSmem<Tin, G>& s, const EncParams& p, const Item& it,
                           unsigned char* stage, uint16_t* off, uint8_t* cbits) {
  const long long g = it.g, cc = it.idx;
  if (p.direct) {
    compact_direct(p, g, cc);
    return;
  }
  if (threadIdx.x == 0) wait_counter(&p.selready[g], 2u, p.status, p.wait_ns);
  csync();
  const long long tl0 = cc * p.CHC;
  const int nt = (int)min(p.CHC, p.n_g - tl0);
  const long long t0 = g * p.n_g + tl0;
  const unsigned long long prefix = __ldcg(&p.lookback[g * p.nC + cc]);
  const int slot_lo = p.slot_lo, slot_d = p.slot_hi - p.slot_lo;
  const long long base = g * p.group_bytes + tl0 * slot_lo + (long long)prefix * slot_d;
  // each thread takes `per` consecutive tiles; a block scan gives their places
  constexpr int kPer = kMaxCC / kThreads;
  const int per = (nt + kThreads - 1) / kThreads;
  uint32_t hiflags = 0u, cnt = 0u;
  uint8_t bl[kPer];
#pragma unroll
  for (int j = 0; j < kPer; j++) {
    const int k = threadIdx.x * per + j;
    bl[j] = 0;
    if (j < per && k < nt) {
      bl[j] = __ldcg(&p.bits[t0 + k]);
      if (bl[j] == (uint8_t)p.hi) {
        hiflags |= 1u << j;
        ++cnt;
      }
    }
  }
  uint32_t chunk_hi;
  uint32_t before = block_exclusive_scan<kThreads>(cnt, chunk_hi, s.scan);
#pragma unroll
  for (int j = 0; j < kPer; j++) {
    const int k = threadIdx.x * per + j;
    if (j < per && k < nt) {
      cbits[k] = bl[j];
      off[k] = (uint16_t)(k * slot_lo + before * slot_d);
      before += (hiflags >> j) & 1u;
    }
  }
  csync();
  const int u = __ffs(p.slot_lo | p.slot_hi | 16) - 1;  // log2 of the largest common unit
  if (u >= 4) {
    gather_units<uint4>(off, cbits, p, t0, nt, stage);
  } else if (u == 3) {
    gather_units<unsigned long long>(off, cbits, p, t0, nt, stage);
  } else if (u == 2) {
    gather_units<unsigned int>(off, cbits, p, t0, nt, stage);
  } else if (u == 1) {
    gather_units<unsigned short>(off, cbits, p, t0, nt, stage);
  } else {
    gather_units<unsigned char>(off, cbits, p, t0, nt, stage);
  }
  csync();
  int nbytes = nt * slot_lo + (int)chunk_hi * slot_d;
  if (base + nbytes > p.codes_bytes) {  // only if the select went wrong: never write past
    if (threadIdx.x == 0) set_status(p.status, kStSelectMismatch);
    nbytes = (int)max(0ll, p.codes_bytes - base);
  }
  store_stage(stage, p.codes, base, nbytes);
  discard_lines(p.scratch_lo, t0 * slot_lo, (t0 + nt) * slot_lo);
  discard_lines(p.scratch_hi, t0 * p.slot_hi, (t0 + nt) * p.slot_hi);
}

// ====================================================================== kernels

template <typename Tin, int G>
__device__ __forceinline__ void issue_chunk(EncSmem<Tin, G>& s, const EncParams& p, long long t0,
                                            int nt, int slot, unsigned long long pol) {
  if constexpr (Cfg<Tin, G>::kLine) {
    // the whole box (256 rows); rows past the tensor are zero-filled and still counted
    mbar_expect_tx(&s.bar[slot], (uint32_t)kChunkBytes);
    const int row = (int)(t0 * G * (long long)sizeof(Tin) / 128);
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(s.buf[slot])),
        "l"(reinterpret_cast<unsigned long long>(&p.tmap)), "r"(0), "r"(row),
        "r"(smem_u32(&s.bar[slot])), "l"(pol)
        : "memory");
  } else {
    const uint32_t bytes = (uint32_t)nt * G * (uint32_t)sizeof(Tin);
    mbar_expect_tx(&s.bar[slot], bytes);
    bulk_load(s.buf[slot], static_cast<const Tin*>(p.x) + t0 * G, bytes, &s.bar[slot], pol);
  }
}

template <typename Tin, int G>
__device__ __forceinline__ EncSmem<Tin, G>& enc_smem(unsigned char* raw) {
  const uint32_t a = smem_u32(raw);
  return *reinterpret_cast<EncSmem<Tin, G>*>(raw + ((1024u - (a & 1023u)) & 1023u));
}

// The queue, decoded once per call: one 64-bit record per ticket (type in bits 62-63,
// group in bits 40-61, index in bits 0-39).
__device__ __forceinline__ unsigned long long pack_item(const Item& it) {
  return ((unsigned long long)(it.type & 3) << 62) | ((unsigned long long)it.g << 40) |
         (unsigned long long)it.idx;
}
__device__ __forceinline__ Item unpack_item(unsigned long long r) {
  return Item{(int)(r >> 62), (long long)((r >> 40) & 0x3FFFFFull), (long long)(r & 0xFFFFFFFFFFull)};
}

static __global__ void __launch_bounds__(256) k_items(const __grid_constant__ EncParams p) {
  const long long q = (long long)blockIdx.x * 256 + threadIdx.x;
  if (q < p.n_items) p.items[q] = pack_item(decode_item(p, (uint32_t)q));
}

// kGen: the general kernel (any tau, the wire format's quantiser, allocation tiles);
// without it, the method's defaults (tau = 2, fp32 metadata, A = G) with their runtime
// checks compiled out.
template <typename Tin, int G, int kLo, int kHi, bool kGen>
__global__ void __launch_bounds__(kThreads, 2) k_encode(const __grid_constant__ EncParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  EncSmem<Tin, G>& s = enc_smem<Tin, G>(smem_raw);
  unsigned char* stage_lo = reinterpret_cast<unsigned char*>(&s) + sizeof(EncSmem<Tin, G>);
  init_tables<Tin, G>(s, p.tabs);
  for (int i = threadIdx.x; i < kCoarseBins; i += kThreads) s.hist[i] = 0u;
  const unsigned long long pol = policy_evict_first();  // the input is read once
  const uint32_t n_items = (uint32_t)p.n_items;
  // Thread 0 runs the queue two items ahead: ticket tk2 (item i + 2) and the record
  // rec1 of item i + 1 are requested one item before they are used.
  uint32_t tk1 = 0u, tk2 = 0u;
  unsigned long long rec1 = 0ull;
  auto record = [&](uint32_t t) { return t < n_items ? __ldcg(p.items + t) : ~0ull; };
  auto start = [&](unsigned long long r, int slot) {  // publish the item, start its copy
    const Item it = r == ~0ull ? Item{-1, 0, 0} : unpack_item(r);
    s.item[slot] = it;
    if (it.type == kItemTiles) {
      long long t0;
      int nt;
      tiles_range<Tin, G>(p, it, t0, nt);
      issue_chunk<Tin, G>(s, p, t0, nt, slot, pol);
    }
  };
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_barrier_init();
    s.ndef[0] = s.ndef[1] = 0u;
    start(record(atomicAdd(p.ticket, 1u)), 0);
    tk1 = atomicAdd(p.ticket, 1u);
    rec1 = record(tk1);
    tk2 = atomicAdd(p.ticket, 1u);
  }
  uint32_t parity = 0u;  // bit s = phase parity of buffer s
  long long done_g = -1;  // thread 0: group of a tiles item not yet published
  for (int slot = 0;; slot ^= 1) {
    csync();  // everyone is done with the previous item, its buffer and shared state
    if (threadIdx.x == 0) {
      if (done_g >= 0) {
        // the block's slot and metadata writes, ordered by the barrier, are published by
        // one gpu-scope fence
        __threadfence();
        atomicAdd(&p.doneA[done_g], 1u);
        done_g = -1;
      }
      s.ndef[slot ^ 1] = 0u;  // the previous item's list is consumed
      // a block holds up to four tickets and works through them in order; items only
      // wait for smaller tickets, so the smallest item in work never waits for an item
      // that has not started
      start(rec1, slot ^ 1);
      if (tk1 < n_items) {
        tk1 = tk2;
        rec1 = record(tk1);
        if (tk1 < n_items) tk2 = atomicAdd(p.ticket, 1u);
      }
    }
    const Item it = s.item[slot];
    if (it.type < 0) break;
    if (it.type == kItemTiles) {
      mbar_wait(&s.bar[slot], (parity >> slot) & 1u, p.status, p.wait_ns);
      parity ^= 1u << slot;
      do_tiles<Tin, G, kLo, kHi, kGen>(s, p, it, s.buf[slot], &s.ndef[slot]);
      done_g = it.g;
    } else if (it.type == kItemCompact) {
      do_compact<Tin, G>(s, p, it, s.buf[slot], reinterpret_cast<uint16_t*>(stage_lo),
                         stage_lo + 2 * kMaxCC);
    } else if (it.type == kItemSelect) {
      do_select<Tin, G>(s, p, it, s.buf[slot]);
    } else if (it.type == kItemOffsets) {
      do_offsets<Tin, G, kGen>(s, p, it);
    }
  }
}

// Every tile gets the same width b (K = 0 or K = n_g): slot offsets are t * G * b / 8.
template <typename Tin, int G, int kB>
__global__ void __launch_bounds__(kThreads, 2) k_encode_flat(const __grid_constant__ EncParams p,
                                                             long long n_chunks) {
  using C = Cfg<Tin, G>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  EncSmem<Tin, G>& s = enc_smem<Tin, G>(smem_raw);
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_barrier_init();
    s.ndef[0] = s.ndef[1] = 0u;
  }
  const unsigned long long pol = policy_evict_first();
  uint32_t parity = 0u;
  const int slot_b = G * p.flat_b / 8;
  long long c = blockIdx.x;
  int slot = 0;
  if (threadIdx.x == 0 && c < n_chunks)
    issue_chunk<Tin, G>(s, p, c * C::CH, (int)min((long long)C::CH, p.n_tiles - c * C::CH), 0, pol);
  for (; c < n_chunks; c += gridDim.x) {
    // everyone is done with the previous chunk: its buffer and list are free
    csync();
    const long long nx = c + gridDim.x;
    if (threadIdx.x == 0) {
      s.ndef[slot ^ 1] = 0u;
      if (nx < n_chunks)
        issue_chunk<Tin, G>(s, p, nx * C::CH, (int)min((long long)C::CH, p.n_tiles - nx * C::CH),
                            slot ^ 1, pol);
    }
    const long long t0 = c * C::CH;
    const int nt = (int)min((long long)C::CH, p.n_tiles - t0);
    mbar_wait(&s.bar[slot], (parity >> slot) & 1u, p.status, p.wait_ns);
    parity ^= 1u << slot;
    // one width: tile t's slot is at t * slot_b in the stream
    unsigned char* out = p.codes + t0 * slot_b;
    if constexpr (C::kLine) {
      tiles_line<Tin, G, kB, 0, true>(s, p, 0, t0, nt, s.buf[slot], true, out, out, &s.ndef[slot]);
    } else {
      tiles_narrow<Tin, G>(s, p, 0, t0, nt, s.buf[slot], true, out, out);
    }
    slot ^= 1;
  }
}

// ====================================================================== three-stage encoder
//
// The method's defaults on the line layout (widths {3, 4}, tau = 2, A = G, fp32
// metadata, token groups of whole 32 KB chunks) in three streaming stages instead of the
// work queue: k_stats (every tile's entropy key and its group's histograms), then the
// select (k_select_groups: the K-th key of each group), the widths and each chunk's hi
// count (k_widths) and the chunks' places in the stream (k_chunk_scan), then k_quant
// (every tile quantised once, at its width, straight into its slot).  The input is read
// twice, but each stage is a plain stream over 32 KB chunks without waits between blocks.
// The stages after the first are dependent launches (launch_dependent): each starts while
// the one before drains (k_quant with its first input copy) and waits for it with
// dep_wait before it reads what that one wrote.

// Stage 1: entropy keys and the per-group key histograms.
template <typename Tin, int G>
__global__ void __launch_bounds__(kThreads, 2) k_stats(const __grid_constant__ EncParams p,
                                                       long long n_chunks) {
  using C = Cfg<Tin, G>;
  constexpr int LPT = LineGeom<Tin, G>::LPT;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  EncSmem<Tin, G>& s = enc_smem<Tin, G>(smem_raw);
  init_tables<Tin, G>(s, p.tabs);
  for (int i = threadIdx.x; i < kCoarseBins; i += kThreads) s.hist[i] = 0u;
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_barrier_init();
  }
  const unsigned long long pol = policy_evict_normal();  // k_quant reads the last chunks again
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int line = warp * 32 + lane, kt = line / LPT, sub = line % LPT;
  dep_launch();
  uint32_t parity = 0u;
  int slot = 0;
  long long c = blockIdx.x;
  if (threadIdx.x == 0 && c < n_chunks)
    issue_chunk<Tin, G>(s, p, c * C::CH, (int)min((long long)C::CH, p.n_tiles - c * C::CH), 0, pol);
  for (; c < n_chunks; c += gridDim.x) {
    csync();  // the previous chunk's buffer and bins are free
    const long long nx = c + gridDim.x;
    if (threadIdx.x == 0 && nx < n_chunks)
      issue_chunk<Tin, G>(s, p, nx * C::CH, (int)min((long long)C::CH, p.n_tiles - nx * C::CH),
                          slot ^ 1, pol);
    const long long t0 = c * C::CH;
    const int nt = (int)min((long long)C::CH, p.n_tiles - t0);
    const long long g = t0 / p.n_g;  // chunks never straddle groups here
    mbar_wait(&s.bar[slot], (parity >> slot) & 1u, p.status, p.wait_ns);
    parity ^= 1u << slot;
    float2 ls = line_sums<Tin>(s.buf[slot], line, s.tabs, lg_consts(s.tabs, lane));
    ls = team_sum2<LPT>(ls);
    if (kt < nt && sub == 0) {
      const float H = entropy_key(ls.x, ls.y, s.tabs);
      p.keys[t0 + kt] = H;
      if (!(ls.x <= FLT_MAX) || !(fabsf(ls.y) <= FLT_MAX) || !(fabsf(H) <= FLT_MAX))
        set_status(p.status, kStNonFinite);
      const int b = fine_bin(H, p.fscale);
      atomicAdd(&p.hist_fine[g * (long long)kFineBins + b], 1u);
      atomicAdd(&s.hist[b >> 8], 1u);  // the chunk's coarse counts, one global add per bin
    }
    csync();
    const uint32_t cnt = s.hist[threadIdx.x];
    if (cnt) {
      atomicAdd(&p.hist_coarse[g * kCoarseBins + threadIdx.x], cnt);
      s.hist[threadIdx.x] = 0u;
    }
    slot ^= 1;
  }
}

// The fine bucket that holds a group's K-th ranked key and the keys ranked above that
// bucket (warp 0 of the calling block; bins = 256 words of shared memory).
__device__ __forceinline__ void find_bucket(const EncParams& p, long long g, uint32_t* bins,
                                            int& bstar, uint32_t& above) {
  const int lane = threadIdx.x & 31;
  const uint32_t K = (uint32_t)p.K;
  for (int i = lane; i < 256; i += 32) bins[i] = __ldcg(&p.hist_coarse[g * kCoarseBins + i]);
  __syncwarp();
  int cb;
  uint32_t above_c;
  warp_find_from_top(bins, K, cb, above_c);
  __syncwarp();
  for (int i = lane; i < 256; i += 32)
    bins[i] = __ldcg(&p.hist_fine[g * (long long)kFineBins + cb * 256 + i]);
  __syncwarp();
  int fb;
  uint32_t above_f;
  warp_find_from_top(bins, K - above_c, fb, above_f);
  bstar = cb * 256 + fb;
  above = above_c + above_f;
}

// Stage 2a: blocks (group, j) gather the rank keys of the group's keys in the bucket that
// holds its K-th ranked key (rank = key descending, then tile index ascending), each from
// its own slice of the group.
static __global__ void __launch_bounds__(kThreads) k_gather(const __grid_constant__ EncParams p,
                                                            int J) {
  __shared__ uint32_t bins[256];
  __shared__ int s_b;
  const long long g = blockIdx.x / J, j = blockIdx.x % J;
  const int lane = threadIdx.x & 31;
  dep_wait();
  dep_launch();
  if (threadIdx.x < 32) {
    int bstar;
    uint32_t above;
    find_bucket(p, g, bins, bstar, above);
    if (lane == 0) s_b = bstar;
  }
  __syncthreads();
  const int bstar = s_b;
  const long long per = (p.n_g + J - 1) / J;
  const long long lo = j * per, hi = min(p.n_g, lo + per);
  const float* kg = p.keys + g * p.n_g;
  unsigned long long* cg = p.cand + g * p.n_g;
  constexpr int kB = 8;
  for (long long base = lo; base < hi; base += kB * kThreads) {
    float hv[kB];
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const long long i = base + u * kThreads + threadIdx.x;
      hv[u] = i < hi ? __ldcg(&kg[i]) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kB; u++) {
      const long long i = base + u * kThreads + threadIdx.x;
      const bool hit = i < hi && fine_bin(hv[u], p.fscale) == bstar;
      const unsigned mask = __ballot_sync(kFull, hit);
      if (mask) {
        uint32_t pos0 = 0;
        const int leader = __ffs(mask) - 1;
        if (lane == leader) pos0 = atomicAdd(&p.cand_cnt[g], (uint32_t)__popc(mask));
        pos0 = __shfl_sync(kFull, pos0, leader);
        if (hit) cg[pos0 + __popc(mask & ((1u << lane) - 1u))] = rank_key(hv[u], (uint32_t)i);
      }
    }
  }
}

// Stage 2a': one block per group ranks the gathered candidates exactly (one pass up to
// kRankMax of them, else an 8-pass radix select over their 64-bit rank keys).
static __global__ void __launch_bounds__(kThreads) k_rank(const __grid_constant__ EncParams p) {
  __shared__ uint32_t bins[256];
  __shared__ uint32_t sc[8];
  __shared__ unsigned long long ck[kRankMax];
  const long long g = blockIdx.x;
  dep_wait();
  dep_launch();
  if (threadIdx.x < 32) {
    int bstar;
    uint32_t above;
    find_bucket(p, g, bins, bstar, above);
    if (threadIdx.x == 0) {
      sc[0] = (uint32_t)bstar;
      sc[1] = above;
    }
  }
  __syncthreads();
  const int bstar = (int)sc[0];
  const uint32_t above = sc[1];
  const uint32_t K = (uint32_t)p.K;
  const unsigned long long* cg = p.cand + g * p.n_g;
  const uint32_t cnt = __ldcg(&p.cand_cnt[g]);
  const uint32_t expect = __ldcg(&p.hist_fine[g * (long long)kFineBins + bstar]);
  if (threadIdx.x == 0 && cnt != expect) set_status(p.status, kStSelectMismatch);
  const uint32_t r = max(1u, min(K - above, cnt));  // rank (from 1) inside the bucket
  unsigned long long theta = 0ull;
  if (cnt > 0u && cnt <= (uint32_t)kRankMax) {
    for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) ck[i] = __ldcg(&cg[i]);
    __syncthreads();
    // one pass: the candidate with exactly r - 1 larger rank keys (they are distinct)
    for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
      const unsigned long long ki = ck[i];
      uint32_t larger = 0;
      for (uint32_t j = 0; j < cnt; j++) larger += ck[j] > ki ? 1u : 0u;
      if (larger == r - 1u) sc[3] = i;
    }
    __syncthreads();
    theta = ck[sc[3]];
  } else if (cnt > 0u) {
    uint32_t rr = r;
    unsigned long long prefix = 0ull, mask = 0ull;
    for (int pass = 7; pass >= 0; --pass) {
      const int shift = pass * 8;
      for (int i = threadIdx.x; i < 256; i += kThreads) bins[i] = 0u;
      __syncthreads();
      for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
        const unsigned long long v = __ldcg(&cg[i]);
        if ((v & mask) == prefix) atomicAdd(&bins[(v >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        int d;
        uint32_t ab;
        warp_find_from_top(bins, rr, d, ab);
        if (threadIdx.x == 0) {
          sc[4] = (uint32_t)d;
          sc[5] = ab;
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)sc[4] << shift;
      rr -= sc[5];
      mask |= 0xFFull << shift;
      __syncthreads();
    }
    theta = prefix;
  }
  if (threadIdx.x == 0) p.sel[g] = SelResult{theta, cnt ? kSelThreshold : kSelNone, 0u};
}

// Stage 2b: every tile's width, each chunk's hi count, and per chunk its tiles in width
// order (bits_lo first) as descriptors k | hi << 8 | (slot offset in the chunk's run)
// << 16, so that stage 3 gives a warp tiles of one width (a block covers 256 tiles =
// whole chunks of CH <= 256 tiles; chunks never straddle groups).
template <int CH>
__global__ void __launch_bounds__(kThreads) k_widths(const __grid_constant__ EncParams p,
                                                     uint32_t* chunk_hi, uint32_t* desc) {
  __shared__ uint32_t wcnt[kWarps];
  const long long t = (long long)blockIdx.x * kThreads + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  dep_wait();
  dep_launch();
  bool ishi = false;
  if (t < p.n_tiles) {
    // group and tile within it (32-bit: the host keeps n_tiles below 2^31 here)
    const uint32_t g = (uint32_t)t / (uint32_t)p.n_g, tl = (uint32_t)t - g * (uint32_t)p.n_g;
    const SelResult sr = p.sel[g];
    ishi = sr.mode == kSelAll ||
           (sr.mode == kSelThreshold && rank_key(__ldcg(&p.keys[t]), tl) >= sr.theta);
    p.bits[t] = (uint8_t)(ishi ? p.hi : p.lo);
  }
  const unsigned m = __ballot_sync(kFull, ishi);
  if (lane == 0) wcnt[warp] = (uint32_t)__popc(m);
  __syncthreads();
  constexpr int kWpc = CH / 32;  // warps a chunk
  const int wc = warp - warp % kWpc;  // the chunk's first warp
  uint32_t pre = (uint32_t)__popc(m & ((1u << lane) - 1u)), tot = 0;
  for (int w = wc; w < warp; w++) pre += wcnt[w];
  for (int w = wc; w < wc + kWpc; w++) tot += wcnt[w];
  if (t < p.n_tiles) {
    const long long c0 = t - t % CH;
    const int k = (int)(t - c0), nt = (int)min((long long)CH, p.n_tiles - c0);
    const int qo = k * p.slot_lo + (int)pre * (p.slot_hi - p.slot_lo);
    const int pos = ishi ? nt - (int)tot + (int)pre : k - (int)pre;
    desc[c0 + pos] = (uint32_t)k | (ishi ? 0x100u : 0u) | ((uint32_t)qo << 16);
  }
  if (threadIdx.x < kThreads / CH) {
    uint32_t sum = 0;
    for (int w = 0; w < kWpc; w++) sum += wcnt[threadIdx.x * kWpc + w];
    const long long c = (long long)blockIdx.x * (kThreads / CH) + threadIdx.x;
    if (c * CH < p.n_tiles) chunk_hi[c] = sum;
  }
}

// Stage 2c: one block per group turns its chunks' hi counts into their byte offsets in
// the stream (chunk c of the group starts at g * group_bytes + c CH slot_lo + (hi tiles
// before it) (slot_hi - slot_lo)).
template <int CH>
__global__ void __launch_bounds__(kThreads) k_chunk_scan(const __grid_constant__ EncParams p,
                                                         const uint32_t* chunk_hi,
                                                         unsigned long long* chunk_off) {
  __shared__ uint32_t s_warp[kWarps + 4];
  const long long g = blockIdx.x;
  dep_wait();
  dep_launch();
  const long long nc = p.n_g / CH, c0 = g * nc;
  const long long run = (nc + kThreads - 1) / kThreads;
  const long long r0 = min(nc, (long long)threadIdx.x * run), r1 = min(nc, r0 + run);
  uint32_t mine = 0;
  for (long long c = r0; c < r1; c++) mine += __ldcg(&chunk_hi[c0 + c]);
  uint32_t tot;
  unsigned long long acc = block_exclusive_scan<kThreads>(mine, tot, s_warp);
  const long long slot_lo = p.slot_lo, slot_d = p.slot_hi - p.slot_lo;
  for (long long c = r0; c < r1; c++) {
    const uint32_t v = __ldcg(&chunk_hi[c0 + c]);
    chunk_off[c0 + c] = (unsigned long long)(g * p.group_bytes + c * CH * slot_lo + (long long)acc * slot_d);
    acc += v;
  }
}

// Stage 3's exact path for the tiles the pretest could not clear (as pass2_line, one
// width: the tile's own, into its slot at out + qoff[kt]); kTau2: tau = 2, tested without
// a division; kWire: the wire format's quantiser (fp16 zero and scale).
template <typename Tin, int G, int V, bool kTau2, bool kWire>
__device__ __forceinline__ void pass2_k3(const EncParams& p, const unsigned char* buf,
                                         const uint16_t* list, int n, long long t0,
                                         unsigned char* out, const uint16_t* qoff,
                                         const uint8_t* qb) {
  constexpr bool kBf = InTraits<Tin>::kBf16;
  constexpr int VPU = kBf ? 8 : 4, NU = V / VPU;
  constexpr int L = G / V, TPW = 32 / L, LPT = LineGeom<Tin, G>::LPT;
  constexpr int kGrp = V < 8 ? 8 / V : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L, base = lane - sub;
#pragma unroll 1
  for (int j0 = warp * TPW; j0 < n; j0 += kWarps * TPW) {
    const int ci = j0 + team;
    const bool valid = ci < n;
    const int kt = valid ? (int)list[ci] : 0;
    const int u0 = sub * NU;
    const int line = kt * LPT + (u0 >> 3);
    float v[V];
#pragma unroll
    for (int k = 0; k < NU; k++) {
      const int ju = (u0 & 7) + k;
      const uint4 q = *reinterpret_cast<const uint4*>(buf + line * 128 + ((ju ^ (line & 7)) << 4));
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
    float m1, m2;
    int i1;
    if constexpr (L == 32) {
      float la = fabsf(v[0]);
#pragma unroll
      for (int j = 1; j < V; j++) la = fmaxf(la, fabsf(v[j]));
      m1 = warp_max_abs(la);
      int jj = V;
#pragma unroll
      for (int j = V - 1; j >= 0; j--)
        if (fabsf(v[j]) == m1) jj = j;
      const unsigned hit = __ballot_sync(kFull, jj < V);
      const int src = hit ? __ffs(hit) - 1 : 0;
      i1 = __shfl_sync(kFull, lane * V + (jj < V ? jj : 0), src);
      float l2 = 0.0f;
#pragma unroll
      for (int j = 0; j < V; j++)
        if (lane * V + j != i1) l2 = fmaxf(l2, fabsf(v[j]));
      m2 = warp_max_f(l2);
    } else {
      team_top2_values<V, L>(v, sub, m1, i1, m2);
    }
    // the ratio test (at tau = 2 without a division, see pass2_line)
    const float d = __fadd_rn(m2, 1e-12f);
    const bool flag =
        valid && (kTau2 ? __fsub_rn(__fmul_rn(m1, 0.5f), d) > __fmul_rn(d, 0x1p-24f)
                        : __fdiv_rn(m1, d) > p.tau);
    if (!__any_sync(kFull, flag)) continue;  // the main pass's slot stands
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
    if constexpr (L == 32) {
      mn = warp_min_f(mn);
      mx = warp_max_f(mx);
    } else {
      mn = team_min<L>(mn);
      mx = team_max<L>(mx);
    }
    const int b = valid ? (int)qb[kt] : 3;
    const float D = __fsub_rn(mx, mn);
    // lane 0 of the team: Q_b / D; lane 1: D / Q_b (the tile's scale)
    const float r = sub == 1 ? __fdiv_rn(D, qmax_f(b)) : __fdiv_rn(qmax_f(b), D);
    const float r0 = __shfl_sync(kFull, r, base), r1 = __shfl_sync(kFull, r, base + 1);
    const bool degenerate = !(D >= 0x1p-120f);
    float inv = degenerate ? 0.0f : r0, scale = degenerate ? 0.0f : r1;
    float qz = mn;  // the quantiser's zero
    if constexpr (kWire) {  // fp16 zero rounded down, smallest fp16 scale that covers max
      qz = wire_zero(mn);
      scale = wire_scale(qz, mx, qmax_f(b));
      inv = wire_inv(scale);
    }
    // the lane's field of V codes (one word for V = 8, b <= 4)
    using Field = std::conditional_t<V == 8, uint32_t, unsigned long long>;
    Field f = 0;
#pragma unroll
    for (int j = 0; j < V; j++) {
      const float c = __fmaf_rn(__fsub_rn(v[j], qz), inv, 12582912.0f);
      f |= (Field)(__float_as_uint(c) - 0x4B400000u) << (j * b);
    }
    unsigned char* slot = out + (valid ? (int)qoff[kt] : 0);
    if constexpr (V == 8) {
      // eight codes a lane: one word at b = 4; at b = 3 (the only other width of the
      // three-stage encoder) the fields of four lanes make three words (slots start on
      // 16-byte boundaries)
      const uint32_t f0 = (uint32_t)f;
      const uint32_t f1 = __shfl_down_sync(kFull, f0, 1), f2 = __shfl_down_sync(kFull, f0, 2);
      const uint32_t f3 = __shfl_down_sync(kFull, f0, 3);
      if (flag && b == 4) {
        *reinterpret_cast<uint32_t*>(slot + 4 * sub) = f0;
      } else if (flag && (sub & 3) == 0) {
        uint32_t* d = reinterpret_cast<uint32_t*>(slot + 3 * sub);
        d[0] = f0 | (f1 << 24);
        d[1] = (f1 >> 8) | (f2 << 16);
        d[2] = (f2 >> 16) | (f3 << 8);
      }
    } else if constexpr (kGrp > 1) {
      f |= __shfl_down_sync(kFull, f, 1) << (V * b);
      if (flag && sub % kGrp == 0) sts_bytes(slot + (sub / kGrp) * b, f, 0ull, b);
    } else {
      if (flag) sts_bytes(slot + sub * (V * b / 8), f, 0ull, V * b / 8);
    }
    if (flag && sub == 0) put_meta(p, t0 + kt, qz, (uint8_t)i1, scale, false);
  }
}

// Stage 3: every tile quantised once, at its width, straight into its slot; the range,
// the two-values pretest and the exact path as in the single-pass kernel.  Chunks in
// reverse order: the first ones are the last that stage 1 read, partly still in L2.
// Three blocks per SM (no lg tables, <= 80 registers): while one block's warps wait at a
// barrier for the exact path of its deferred tiles, the others issue.
// kTau2: tau = 2 (the pretest's threshold by an exact halving, the exact test without a
// division); else the threshold is m1 / tau rounded up and the test divides.  kWire: the
// wire format's quantiser (fp16 zero rounded down, the smallest fp16 scale that covers the
// maximum, codes from those).
// kAL: the alignment of the slots (16 when every slot size and the group stride are
// multiples of 16 bytes, else 4: widths 3 and 4 of tiles of 32 values or more).
constexpr int kQuantBlocks = 3;
template <typename Tin, int G, int kAL, bool kTau2, bool kWire>
__global__ void __launch_bounds__(kThreads, kQuantBlocks) k_quant(const __grid_constant__ EncParams p,
                                                       long long n_chunks,
                                                       const unsigned long long* chunk_off,
                                                       const uint32_t* desc) {
  using C = Cfg<Tin, G>;
  using LG = LineGeom<Tin, G>;
  constexpr int LPT = LG::LPT, NE = LG::NE;
  static_assert(C::CH <= kThreads, "one thread per tile of a chunk");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  EncSmem<Tin, G>& s = enc_smem<Tin, G>(smem_raw);
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_barrier_init();
    s.ndef[0] = s.ndef[1] = 0u;
  }
  const unsigned long long pol = policy_evict_first();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int line = warp * 32 + lane, pos = line / LPT, sub = line % LPT;
  uint32_t parity = 0u;
  int slot = 0;
  auto chunk_of = [&](long long i) { return n_chunks - 1 - i; };
  long long i = blockIdx.x;
  // this lane's descriptor (its place `pos` in the chunk's width order), a chunk ahead
  auto load_desc = [&](long long ii) -> uint32_t {
    if (ii >= n_chunks) return 0u;
    const long long cc = chunk_of(ii);
    return pos < (int)min((long long)C::CH, p.n_tiles - cc * C::CH) ? __ldcg(&desc[cc * C::CH + pos])
                                                                     : 0u;
  };
  if (threadIdx.x == 0 && i < n_chunks) {
    const long long c = chunk_of(i);
    issue_chunk<Tin, G>(s, p, c * C::CH, (int)min((long long)C::CH, p.n_tiles - c * C::CH), 0, pol);
  }
  dep_wait();  // descriptors and chunk offsets of the stages before
  uint32_t dnext = load_desc(i);
  for (; i < n_chunks; i += gridDim.x) {
    const uint32_t dcur = dnext;
    dnext = load_desc(i + gridDim.x);
    csync();  // the previous chunk's buffer, list and arrays are free
    const long long nx = i + gridDim.x;
    if (threadIdx.x == 0) {
      s.ndef[slot ^ 1] = 0u;
      if (nx < n_chunks) {
        const long long cn = chunk_of(nx);
        issue_chunk<Tin, G>(s, p, cn * C::CH, (int)min((long long)C::CH, p.n_tiles - cn * C::CH),
                            slot ^ 1, pol);
      }
    }
    const long long c = chunk_of(i);
    const long long t0 = c * C::CH;
    const int nt = (int)min((long long)C::CH, p.n_tiles - t0);
    unsigned char* out = p.codes + __ldcg(&chunk_off[c]);
    // the chunk's tiles in width order (k_widths), so that a warp's tiles share one width
    const bool valid = pos < nt;
    const int kt = (int)(dcur & 0xFFu);
    const int b = (dcur & 0x100u) ? 4 : 3;
    const int qo = (int)(dcur >> 16);
    mbar_wait(&s.bar[slot], (parity >> slot) & 1u, p.status, p.wait_ns);
    parity ^= 1u << slot;
    const unsigned char* buf = s.buf[slot];
    const int tline = kt * LPT + sub;  // this lane's line of the chunk
    uint32_t w[32];
    lds_line(buf, tline, w);
    float mn, mx, ga[NE / 8];
    line_minmax<Tin>(w, mn, mx, ga);
    mn = team_min<LPT>(mn);
    mx = team_max<LPT>(mx);
    const float m1 = fmaxf(mx, -mn);
    // two values of at least m1 / tau rule out r > tau (for tau = 2 an exact halving,
    // m1 >= 2^-120 here)
    const float thr = kTau2 ? __fmul_rn(m1, 0.5f) : __fdiv_ru(m1, p.tau);
    uint32_t cnt = 0;
#pragma unroll
    for (int q = 0; q < NE / 8; q++) cnt += ga[q] >= thr ? 1u : 0u;
    cnt = team_sum_u<LPT>(cnt);
    // below 2^-120 the ratio cannot exceed a tau >= 1 (m2 + 1e-12 > m1 / tau)
    const bool small = (kTau2 || p.tau >= 1.0f) && m1 < 0x1p-120f;
    const bool deferred = !small && (!(m1 <= FLT_MAX) || cnt < 2u);
    const float D = __fsub_rn(mx, mn);
    float inv, scale;
    if constexpr (LPT >= 2) {
      const bool odd = sub & 1;
      const float r = odd ? __fdiv_rn(D, qmax_f(b)) : __fdiv_rn(qmax_f(b), D);
      const float o = __shfl_xor_sync(kFull, r, 1);
      inv = odd ? o : r;
      scale = odd ? r : o;
    } else {
      inv = __fdiv_rn(qmax_f(b), D);
      scale = __fdiv_rn(D, qmax_f(b));
    }
    if (!(D >= 0x1p-120f)) inv = scale = 0.0f;
    float qz = mn;  // the quantiser's zero
    if constexpr (kWire) {  // fp16 zero rounded down, smallest fp16 scale that covers max
      qz = wire_zero(mn);
      scale = wire_scale(qz, mx, qmax_f(b));
      inv = wire_inv(scale);
    }
    if (valid) {
      if (b == 3) {
        line_quant<Tin, 3, kAL>(w, qz, inv, 3, out + qo + sub * (NE * 3 / 8));
      } else {
        line_quant<Tin, 4, kAL>(w, qz, inv, 4, out + qo + sub * (NE * 4 / 8));
      }
      if (sub == 0) put_meta(p, t0 + kt, qz, (uint8_t)0xFF, scale, false);
    }
    if (valid && sub == 0) {
      s.qoff[kt] = (uint16_t)qo;
      s.qb[kt] = (uint8_t)b;
      if (deferred) s.dl[atomicAdd(&s.ndef[slot], 1u)] = (uint16_t)kt;
    }
    csync();
    pass2_k3<Tin, G, p2_values<Tin, G, 3, 4>(), kTau2, kWire>(p, buf, s.dl, (int)s.ndef[slot], t0, out,
                                                s.qoff, s.qb);
    slot ^= 1;
  }
}

}  // namespace tahq

#include "tahq_run.cuh"

namespace tahq {

// ====================================================================== launchers

using QuantFn = void (*)(EncParams, long long, const unsigned long long*, const uint32_t*);

// The three-stage quantiser for tau = 2 or not, plain or wire, 16-byte or word slots.
template <typename Tin, int G, bool kTau2, bool kWire>
static QuantFn quant_kernel(bool direct) {
  return direct ? k_quant<Tin, G, 16, kTau2, kWire> : k_quant<Tin, G, 4, kTau2, kWire>;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// The input viewed as [rows][128 bytes], boxes of 256 rows (one 32 KB chunk), 128-byte
// swizzle.
static cudaError_t make_line_map(TmaDesc* d, const void* x, bool bf16, long long n_tiles, int G) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  const int esize = bf16 ? 2 : 4;
  const long long rows = n_tiles * G * esize / 128;
  CUtensorMap m;
  const cuuint64_t dims[2] = {(cuuint64_t)(128 / esize), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / esize), 256u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = fn(&m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        2, const_cast<void*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  static_assert(sizeof(CUtensorMap) == sizeof(TmaDesc), "descriptor size");
  std::memcpy(d->bytes, &m, sizeof m);
  return cudaSuccess;
}

template <typename Tin, int G>
static cudaError_t run_encode(const EncodeArgs& a, cudaStream_t st) {
  using C = Cfg<Tin, G>;
  EncParams p{};
  p.x = a.x;
  p.n_tiles = a.n_tiles;
  p.n_g = a.n_g;
  p.n_groups = a.n_groups;
  p.K = a.K;
  p.group_bytes = a.group_bytes;
  p.codes_bytes = a.n_groups * a.group_bytes;
  p.lo = a.lo;
  p.hi = a.hi;
  p.h = a.h;
  p.c_h = a.c_h;
  p.tau = a.tau;
  p.wire = a.wire ? 1 : 0;
  p.mlog = a.mlog;
  p.n_ga = a.n_g >> a.mlog;
  // keys of A = 2^mlog G values lie in [0, log2 A]
  p.fscale = ((long long)G << a.mlog) <= 256 ? 8192.0f : 4096.0f;
  p.slot_lo = G * a.lo / 8;
  p.slot_hi = G * a.hi / 8;
  p.direct = (p.slot_lo % 16 == 0 && p.slot_hi % 16 == 0 && a.group_bytes % 16 == 0) ? 1 : 0;
  p.codes = a.codes;
  p.scales = a.scales;
  p.zeros = a.zeros;
  p.bits = a.bits;
  p.pivots = a.pivots;
  p.scratch_lo = a.scratch_lo;
  p.scratch_hi = a.scratch_hi;
  p.keys = a.keys;
  p.cand = a.cand;
  p.cand_cnt = a.cand_cnt;
  p.segmask = a.segmask;
  p.hist_coarse = a.hist_coarse;
  p.hist_fine = a.hist_fine;
  p.doneA = a.doneA;
  p.doneB = a.doneB;
  p.doneB2 = a.doneB2;
  p.selready = a.selready;
  p.sel = a.sel;
  p.lookback = a.lookback;
  p.ticket = a.ticket;
  p.items = a.items;
  p.status = a.status;
  p.tabs = *a.tabs;
  p.wait_ns = a.wait_ns ? a.wait_ns : kWaitNs;
  p.scale_c = a.scale_c;
  if constexpr (C::kLine) {
    const cudaError_t e = make_line_map(&p.tmap, a.x, C::kBf16, a.n_tiles, G);
    if (e != cudaSuccess) return e;
  }
  const int grid_cap = a.num_sms * 2;
  const bool flat = a.K == 0 || a.K == (a.n_g >> a.mlog);
  p.flat_b = a.K == 0 ? a.lo : a.hi;
  if constexpr (G >= 32 && G <= 128) {
    // the streaming encoder: A = G, any tau (compiled for tau = 2 and for the rest), fp32
    // metadata or the wire format's quantiser, one width of 3 or 4 bits, or widths {3, 4}
    // ranked per group of whole input chunks; the input in 128-byte rows
    const long long esz = (long long)sizeof(Tin);
    const bool rows = (a.n_tiles * G * esz) % 128 == 0 && (a.n_g * G) % 128 == 0 &&
                      a.n_tiles < (1ll << 31);
    const bool plain = a.mlog == 0 && rows;
    const bool t2 = a.tau == 2.0f;
    // the scaled read is compiled for tau = 2 without the wire quantiser
    const bool ok_mode = a.scale_c == 1.0f || (t2 && !a.wire);
    const size_t smem_r = sizeof(RunSmem<Tin, G>) + 1024;
    const long long n_chunks = (a.n_tiles + C::CH - 1) / C::CH;
    // three blocks an SM (<= 80 registers, two 32 KB stages each)
    const int grid_r = (int)std::max<long long>(1, std::min<long long>(3ll * a.num_sms, n_chunks));
    if (plain && ok_mode && flat && (p.flat_b == 3 || p.flat_b == 4)) {
      cudaError_t e = make_line_map(&p.tmap, a.x, C::kBf16, a.n_tiles, G);
      if (e != cudaSuccess) return e;
      // modes (wire, scaled, tau = 2): plain, wire, scaled at tau = 2; plain, wire at any tau
      using FlatFn = void (*)(EncParams, long long);
      static const FlatFn fl[2][5] = {
          {k_run_flat<Tin, G, 3, false, false, true>, k_run_flat<Tin, G, 3, true, false, true>,
           k_run_flat<Tin, G, 3, false, true, true>, k_run_flat<Tin, G, 3, false, false, false>,
           k_run_flat<Tin, G, 3, true, false, false>},
          {k_run_flat<Tin, G, 4, false, false, true>, k_run_flat<Tin, G, 4, true, false, true>,
           k_run_flat<Tin, G, 4, false, true, true>, k_run_flat<Tin, G, 4, false, false, false>,
           k_run_flat<Tin, G, 4, true, false, false>}};
      const int mode = t2 ? (a.wire ? 1 : a.scale_c != 1.0f ? 2 : 0) : (a.wire ? 4 : 3);
      FlatFn kern = fl[p.flat_b == 3 ? 0 : 1][mode];
      static const cudaError_t e_attr = [smem_r] {
        for (const auto& row : fl)
          for (FlatFn k : row) {
            const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_r);
            if (e != cudaSuccess) return e;
          }
        return cudaSuccess;
      }();
      if (e_attr != cudaSuccess) return e_attr;
      kern<<<grid_r, kThreads, smem_r, st>>>(p, n_chunks);
      return cudaGetLastError();
    }
    // compaction chunks: the largest power of two of tiles up to kEncMaxCC that still
    // gives four blocks an SM (small tensors), and no smaller than the chunks the
    // workspace holds counts for
    long long chc = kEncMaxCC;
    const long long min_chc = encode_cchunk_tiles(C::kBf16 ? 1 : 0, G, a.hi);
    while (chc / 2 >= min_chc && chc / 2 >= 32 && a.n_tiles / chc < 4ll * a.num_sms) chc /= 2;
    if (plain && ok_mode && !flat && a.lo == 3 && a.hi == 4 && a.n_g % C::CH == 0 &&
        (a.n_g + chc - 1) / chc <= 64 * 256 && a.group_bytes < (1ll << 31)) {
      cudaError_t e = make_line_map(&p.tmap, a.x, C::kBf16, a.n_tiles, G);
      if (e != cudaSuccess) return e;
      p.CHC = chc;
      p.nC = (a.n_g + p.CHC - 1) / p.CHC;
      // select parts a group: of kSelPart tiles, or of kSelPartWide when the narrow parts
      // would need a second wave of select blocks (five an SM)
      const bool wide = a.n_groups * ((a.n_g + kSelPart - 1) / kSelPart) > 5ll * a.num_sms;
      const int part = wide ? kSelPartWide : kSelPart;
      const int J2 = (int)((a.n_g + part - 1) / part);
      // modes as for the one-width pass
      using TilesFn = void (*)(EncParams, long long);
      static const TilesFn tl[5] = {k_run_tiles<Tin, G, false, false, true>, k_run_tiles<Tin, G, true, false, true>,
                                    k_run_tiles<Tin, G, false, true, true>, k_run_tiles<Tin, G, false, false, false>,
                                    k_run_tiles<Tin, G, true, false, false>};
      static const cudaError_t e_attr = [smem_r] {
        for (TilesFn k : tl) {
          const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_r);
          if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
      }();
      if (e_attr != cudaSuccess) return e_attr;
      const int mode = t2 ? (a.wire ? 1 : a.scale_c != 1.0f ? 2 : 0) : (a.wire ? 4 : 3);
      tl[mode]<<<grid_r, kThreads, smem_r, st>>>(p, n_chunks);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      constexpr int kN = kSelPart / kThreads, kWd = kSelPartWide / kThreads;
      e = launch_dependent(wide ? (a.wire ? k_run_select<Tin, G, true, kWd> : k_run_select<Tin, G, false, kWd>)
                                : (a.wire ? k_run_select<Tin, G, true, kN> : k_run_select<Tin, G, false, kN>),
                           (unsigned)(a.n_groups * J2), kThreads, 0, st, p, J2, (long long)part);
      if (e != cudaSuccess) return e;
      // slots of 3 and 4 units of G / 8 bytes: group strides are whole units
      static_assert(G % 32 == 0, "units of G / 8 bytes");
      return launch_dependent(k_run_compact<G>, (unsigned)(a.n_groups * p.nC), kThreads, 0, st, p);
    }
  }
  // only the streaming encoder reads its input scaled (the caller scales a copy for the rest)
  if (a.scale_c != 1.0f) return cudaErrorNotYetImplemented;
  // a compaction chunk's per-tile arrays (3 bytes per tile) follow the shared state
  const size_t stages = flat ? 0 : 3 * kMaxCC;
  const size_t smem = sizeof(EncSmem<Tin, G>) + 1024 + stages;
  if (flat) {
    void (*kern)(EncParams, long long) = k_encode_flat<Tin, G, 0>;
    if constexpr (C::kLine) {  // the common widths, compiled with the width known
      if (p.flat_b == 3) kern = k_encode_flat<Tin, G, 3>;
      if (p.flat_b == 4) kern = k_encode_flat<Tin, G, 4>;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long n_chunks = (a.n_tiles + C::CH - 1) / C::CH;
    const int grid = (int)std::max<long long>(1, std::min<long long>(grid_cap, n_chunks));
    kern<<<grid, kThreads, smem, st>>>(p, n_chunks);
    return cudaGetLastError();
  }
  if constexpr (C::kLine) {
    // the method's defaults with widths {3, 4} and groups of whole chunks: the three-stage
    // encoder (its quantiser stores whole 16-byte units where every slot starts on a
    // 16-byte boundary, else words)
    if (a.mlog == 0 && a.lo == 3 && a.hi == 4 && a.n_g % C::CH == 0) {
      static_assert(C::CH >= 64 && C::CH <= kThreads && (kThreads % C::CH) == 0,
                    "chunks of 64..256 tiles");
      const long long n_chunks = a.n_tiles / C::CH;
      const int grid = (int)std::max<long long>(1, std::min<long long>(grid_cap, n_chunks));
      // the candidates array is free once the select has run: each chunk's hi count; the
      // offsets go where the work queue keeps its segment masks (n / CH words of 8 bytes
      // fit in n / 32 words of 4)
      uint32_t* chunk_hi = reinterpret_cast<uint32_t*>(a.cand);
      uint32_t* desc = reinterpret_cast<uint32_t*>(a.cand + (n_chunks + 1) / 2 + 1);
      unsigned long long* chunk_off = reinterpret_cast<unsigned long long*>(a.segmask);
      if (a.n_tiles >= (1ll << 31)) return cudaErrorInvalidValue;
      const int J = (int)std::max<long long>(1, std::min<long long>(64, a.n_g / 4096));
      // neither stage uses the compaction's per-tile arrays
      const size_t smem3 = sizeof(EncSmem<Tin, G>) + 1024;
      const int grid_q = (int)std::max<long long>(1, std::min<long long>(a.num_sms * kQuantBlocks, n_chunks));
      QuantFn quant = a.wire ? (a.tau == 2.0f ? quant_kernel<Tin, G, true, true>(p.direct)
                                              : quant_kernel<Tin, G, false, true>(p.direct))
                             : (a.tau == 2.0f ? quant_kernel<Tin, G, true, false>(p.direct)
                                              : quant_kernel<Tin, G, false, false>(p.direct));
      cudaError_t e = cudaFuncSetAttribute(k_stats<Tin, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem3);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(quant, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem3);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(quant, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      k_stats<Tin, G><<<grid, kThreads, smem3, st>>>(p, n_chunks);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      e = launch_dependent(k_gather, (unsigned)(a.n_groups * J), kThreads, 0, st, p, J);
      if (e != cudaSuccess) return e;
      e = launch_dependent(k_rank, (unsigned)a.n_groups, kThreads, 0, st, p);
      if (e != cudaSuccess) return e;
      e = launch_dependent(k_widths<C::CH>, (unsigned)((a.n_tiles + kThreads - 1) / kThreads),
                           kThreads, 0, st, p, chunk_hi, desc);
      if (e != cudaSuccess) return e;
      e = launch_dependent(k_chunk_scan<C::CH>, (unsigned)a.n_groups, kThreads, 0, st, p,
                           (const uint32_t*)chunk_hi, chunk_off);
      if (e != cudaSuccess) return e;
      return launch_dependent(quant, (unsigned)grid_q, kThreads, smem3, st, p, n_chunks,
                              (const unsigned long long*)chunk_off, (const uint32_t*)desc);
    }
  }
  p.nA = (a.n_g + C::CH - 1) / C::CH;
  p.CHC = encode_cchunk_tiles(C::kBf16, G, a.hi);
  // the direct compaction needs no stage: larger chunks, fewer items (never more chunks
  // than the workspace sizing assumes)
  if (p.direct) p.CHC = std::max<long long>(p.CHC, kDirectCC);
  p.nC = (a.n_g + p.CHC - 1) / p.CHC;
  // keep the scratch of three (or, for big groups, two) groups in L2 between a group's
  // tiles pass and its compaction
  const long long group_scratch = a.n_g * (long long)(p.slot_lo + p.slot_hi);
  p.lag = (3 * group_scratch <= (64ll << 20)) ? 2 : 1;
  // one tiles item per block before the select items (the group's last tiles items
  // finish meanwhile), an eighth of the group before the offsets items
  p.pre1 = std::min<long long>(p.nA, grid_cap);
  p.pre2 = std::min<long long>(p.nA - p.pre1, p.nA / 8);
  p.J = encode_sel_items(p.nA, p.nC);
  p.n_items = a.n_groups * (p.nA + 2 * p.J + p.nC);
  if (p.n_items > a.items_cap) return cudaErrorInvalidValue;
  if (p.n_items >= (1ll << 31) || (p.nA + 2 * p.J + p.nC) * p.nC >= (1ll << 32))
    return cudaErrorInvalidValue;
  queue_segments(p);
  void (*kern)(EncParams) = k_encode<Tin, G, 0, 0, true>;
  if constexpr (C::kLine) {
    // the method's defaults with widths {3, 4}: the specialised kernel
    const bool plain = a.tau == 2.0f && !a.wire && a.mlog == 0;
    if (a.lo == 3 && a.hi == 4) kern = plain ? k_encode<Tin, G, 3, 4, false> : k_encode<Tin, G, 3, 4, true>;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::max<long long>(1, std::min<long long>(grid_cap, p.n_items));
  k_items<<<(unsigned)((p.n_items + 255) / 256), 256, 0, st>>>(p);
  kern<<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tahq
