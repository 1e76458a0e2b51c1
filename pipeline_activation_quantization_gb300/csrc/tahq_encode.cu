// tahq_encode.cu -- encode kernels of the TAH-Quant activation codec for sm_103a.
//
// "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over Slow
// Network" (arXiv 2506.01352v2):
//   stats    §3.2 eq. (1)-(2): entropy key of every tile, plus the per-group key
//            histograms the allocator selects from;
//   select   §3.2 "Top-p% tile selection": the K tiles of highest (key, -index) of each
//            group get the high bit width -- histogram bucket, then an exact radix
//            select among the candidates of that bucket;
//   quant    §3.3 eq. (3) outlier ratio and pivot, pivot swap + eq. (4) Hadamard, the
//            asymmetric quantizer, and §3.4's contiguous uint8 stream.
//
// k_encode runs the three as work items of one persistent kernel.  Items are handed out
// in increasing order by an atomic ticket and only ever wait for earlier items, so every
// wait ends.  The order keeps a group's input in L2 between its stats pass and its
// quantize pass (see decode_item for the round layout).  Each block double-buffers 32 KB
// input chunks in shared memory with bulk (TMA) copies.  Offsets items count the hi
// tiles of every chunk once the group's threshold is known and scan the counts into
// the chunks' offsets in the stream, so a quantize item never waits on another chunk.
//
// k_encode_flat covers allocations that do not depend on the ranking (K = 0 or K = n_g,
// every tile gets the same width): one streaming pass, fixed slot offsets.
//
// Within a chunk, pass 1 quantises every tile that provably needs no transform (two or
// more values with |v| >= max|v| / 2 give r <= tau); pass 2 takes the remaining tiles,
// compacted, and applies the exact ratio test, pivot swap and Hadamard transform.
#include <algorithm>
#include <cfloat>

#include "tahq_device.cuh"
#include "tahq_launch.h"
#include "tahq_tile.cuh"

namespace tahq {

constexpr int kChunkBytes = 32768;
constexpr uint8_t kDeferred = 0xFE;  // pass-1 marker of a tile left to pass 2
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename Tin, int G>
struct Cfg {
  using Gm = TileGeom<Tin, G>;
  static constexpr int V = Gm::V, W = Gm::W, L = Gm::L, TPW = Gm::TPW;
  static constexpr int CH = kChunkBytes / (G * (int)sizeof(Tin));  // tiles per chunk
  static constexpr int kSteps = CH / (kWarps * TPW);               // warp steps per chunk
  static constexpr int kPer = (CH + kThreads - 1) / kThreads;      // tiles per thread (scan)
  static constexpr int kStage = CH * G + 64;                       // b <= 8, plus slack
  static constexpr int NS = CH / kWarps;                           // tiles owned by a warp
  static_assert(kSteps * kWarps * TPW == CH, "chunk must be whole warp steps");
  static_assert(kPer <= 32, "hi flags are kept in one word per thread");
};

struct Item {
  int type;  // kItemStats, kItemSelect, kItemOffsets, kItemQuant
  long long g, idx;
};
constexpr int kItemStats = 0, kItemSelect = 1, kItemOffsets = 2, kItemQuant = 3;

template <typename Tin, int G>
struct alignas(128) EncSmem {
  using C = Cfg<Tin, G>;
  unsigned char buf[2][kChunkBytes];
  unsigned char stage[C::kStage];
  float Trep[128 * 32];  // lg tables replicated per bank: entry i of lane l at i*32 + l
  float Rrep[InTraits<Tin>::kNoFraction ? 4 : 128 * 32];
  LgTables tabs;
  float scale[C::CH], zero[C::CH];
  float ta[C::CH], tb[C::CH];  // per-tile pairs: (L, S) in stats, (min, max) then inv in quant
  uint16_t off[C::CH];
  uint16_t cand[C::CH];
  uint8_t bits[C::CH], piv[C::CH];
  uint32_t hist[kCoarseBins];
  uint32_t scan[kWarps + 4];
  unsigned long long bar[2];
  Item item[2];
  long long next, base;
  uint32_t last, ncand;
};

struct EncParams {
  const void* x;
  long long n_tiles, n_g, n_groups, K, group_bytes, codes_bytes;
  long long nA, J, lag, pre, n_items;
  int lo, hi, h;
  float c_h;
  uint8_t* codes;
  float* scales;
  float* zeros;
  uint8_t* bits;
  uint8_t* pivots;
  float* keys;
  unsigned long long* cand;
  uint32_t* cand_cnt;
  uint32_t* hist_coarse;
  uint32_t* hist_fine;
  uint32_t* doneA;
  uint32_t* doneB;
  uint32_t* doneB2;
  uint32_t* selready;  // 1 once sel[g] is published, 2 once the chunk offsets are
  SelResult* sel;
  unsigned long long* lookback;
  uint32_t* ticket;
  uint32_t* status;
  LgTables tabs;
};

// ====================================================================== helpers

template <typename Tin, int G>
__device__ __forceinline__ void init_tables(EncSmem<Tin, G>& sm, const LgTables& tabs) {
  for (int i = threadIdx.x; i < 128 * 32; i += kThreads) {
    if constexpr (InTraits<Tin>::kNoFraction) {
      sm.Trep[i] = tabs.TB[i >> 5];
    } else {
      sm.Trep[i] = tabs.T[i >> 5];
      sm.Rrep[i] = tabs.R[i >> 5];
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
  __syncthreads();
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
  __syncthreads();
  total = s_warp[kW];
  const uint32_t r = s_warp[warp] + incl - v;
  __syncthreads();
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

// ====================================================================== quantize a chunk

// Tile `l` (0 <= l < NS) of warp `warp`: the tiles a warp handles over all its steps.
template <typename Tin, int G>
__device__ __forceinline__ int warp_tile(int l, int warp) {
  using C = Cfg<Tin, G>;
  return ((l / C::TPW) * kWarps + warp) * C::TPW + (l % C::TPW);
}

// Quantise and pack the chunk's tiles into s.stage (s.bits / s.off must be ready).  Each
// warp handles its own NS tiles with no block-wide barrier:
//   phase 1, per warp step: the tile's min / max and the two-values test -- two values
//            with |v| >= max|v|/2 give r <= tau, so no transform; tiles that fail it
//            (or are below 2^-120) are deferred;
//   phase 2, one lane per tile: scale = D/Q, inv = Q/D, zero-point;
//   phase 3, per warp step: quantise and pack the tiles that were not deferred;
//   pass 2:  the deferred tiles, compacted: exact ratio test (eq. (3)), pivot swap and
//            Hadamard (eq. (4)) where it holds, then the quantizer.
template <typename Tin, int G>
__device__ __forceinline__ void quant_chunk(EncSmem<Tin, G>& s, const unsigned char* buf, int nt,
                                            int h, float c_h) {
  using C = Cfg<Tin, G>;
  constexpr int V = C::V, W = C::W, L = C::L, TPW = C::TPW, NS = C::NS;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L;
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
    const float thr = __fmul_rn(m1, 0.5f);  // exact halving for m1 >= 2^-120
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
  // phase 2 (and the list of deferred tiles, kept in this warp's part of s.cand)
  uint16_t* dl = s.cand + warp * NS;
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
      const int b = s.bits[kt];
      const float qf = __fsub_rn(__uint_as_float(0x4B000000u | ((1u << b) - 1u)), 8388608.0f);
      const float D = __fsub_rn(mx, mn);
      const bool degenerate = !(D >= 0x1p-120f);
      s.scale[kt] = degenerate ? 0.0f : __fdiv_rn(D, qf);
      s.tb[kt] = degenerate ? 0.0f : __fdiv_rn(qf, D);  // inv
      s.zero[kt] = __fadd_rn(mn, 0.0f);
    }
  }
  __syncwarp();
  // phase 3
#pragma unroll 1
  for (int st = 0; st < C::kSteps; st++) {
    const int kt = (st * kWarps + warp) * TPW + team;
    if (kt >= nt || s.piv[kt] == kDeferred) continue;
    const float mn = s.ta[kt];
    const float inv = s.tb[kt];
    const int b = s.bits[kt];
    uint32_t w[W];
    lds_words<Tin, G>(buf, kt, sub, w);
    float v[V];
    words_to_values<Tin, G>(w, v);
    quant_store<V>(v, mn, inv, b, s.stage + s.off[kt] + sub * (V * b / 8));
  }
  // pass 2
#pragma unroll 1
  for (int j0 = 0; j0 < ndef; j0 += TPW) {
    const int ci = j0 + team;
    const bool valid = ci < ndef;
    const int kt = valid ? (int)dl[ci] : 0;
    uint32_t w[W];
    if (valid) {
      lds_words<Tin, G>(buf, kt, sub, w);
    } else {
#pragma unroll
      for (int k = 0; k < W; k++) w[k] = 0u;
    }
    float v[V];
    words_to_values<Tin, G>(w, v);
    float m1 = fabsf(v[0]), m2 = -1.0f;
    int i1 = sub * V;
#pragma unroll
    for (int j = 1; j < V; j++) {
      const float m = fabsf(v[j]);
      if (m > m1) {
        m2 = m1;
        m1 = m;
        i1 = sub * V + j;
      } else if (m > m2) {
        m2 = m;
      }
    }
    team_top2<L>(m1, i1, m2);
    const bool flag = valid && __fdiv_rn(m1, __fadd_rn(m2, 1e-12f)) > 2.0f;
    if (__any_sync(kFull, flag)) {
      float t[V];
#pragma unroll
      for (int j = 0; j < V; j++) t[j] = v[j];
      team_swap0<V>(t, flag ? i1 : 0, sub, lane - sub);
      team_fwht<V, L>(t, h, sub);
      if (flag) {
#pragma unroll
        for (int j = 0; j < V; j++) v[j] = __fmul_rn(t[j], c_h);
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
    const int b = valid ? (int)s.bits[kt] : 1;
    float scale, inv;
    scale_inv<L>(__fsub_rn(mx, mn), b, sub, scale, inv);
    if (valid) {
      quant_store<V>(v, mn, inv, b, s.stage + s.off[kt] + sub * (V * b / 8));
      if (sub == 0) {
        s.scale[kt] = scale;
        s.zero[kt] = __fadd_rn(mn, 0.0f);
        s.piv[kt] = flag ? (uint8_t)i1 : (uint8_t)0xFF;
      }
    }
  }
}

// Copy s.stage[0, nbytes) to codes[base, base + nbytes): 16-byte stores for the aligned
// middle (realigned from shared memory with funnel shifts), byte stores at the two ends.
template <typename Tin, int G>
__device__ __forceinline__ void store_stage(const EncSmem<Tin, G>& s, uint8_t* codes,
                                            long long base, int nbytes) {
  const int head = (int)((16 - (base & 15)) & 15);
  const int h = min(head, nbytes);
  const int n16 = (nbytes - h) / 16;
  const int tail0 = h + 16 * n16;
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(s.stage);
  const int sh = (h & 3) * 8;
  for (int i = threadIdx.x; i < n16; i += kThreads) {
    const int o = h + 16 * i;          // stage byte offset of this global 16-byte word
    const int q = o >> 2;
    uint32_t a[5];
#pragma unroll
    for (int k = 0; k < 5; k++) a[k] = sw[q + k];
    uint4 out;
    out.x = __funnelshift_r(a[0], a[1], sh);
    out.y = __funnelshift_r(a[1], a[2], sh);
    out.z = __funnelshift_r(a[2], a[3], sh);
    out.w = __funnelshift_r(a[3], a[4], sh);
    *reinterpret_cast<uint4*>(codes + base + o) = out;
  }
  const int nb = h + (nbytes - tail0);
  for (int i = threadIdx.x; i < nb; i += kThreads) {
    const int o = (i < h) ? i : tail0 + (i - h);
    codes[base + o] = s.stage[o];
  }
}

template <typename Tin, int G>
__device__ __forceinline__ void store_meta(const EncSmem<Tin, G>& s, const EncParams& p,
                                           long long t0, int nt) {
  for (int k = threadIdx.x; k < nt; k += kThreads) {
    p.scales[t0 + k] = s.scale[k];
    p.zeros[t0 + k] = s.zero[k];
    p.bits[t0 + k] = s.bits[k];
    p.pivots[t0 + k] = s.piv[k];
  }
}

// ====================================================================== work items


// Round r (0 <= r < NG + lag) of the work queue:
//   the J select items of group r-1        (if 1 <= r <= NG)
//   the first `pre` stats items of group r (if r < NG)
//   the J offset items of group r-1        (if 1 <= r <= NG)
//   the other stats items of group r interleaved with the quantize items of group r-lag.
// A group's select items come after all its stats items, its offset items after its
// select items, and its quantize items (round >= r+1) after its offset items.
__device__ __forceinline__ Item decode_item(const EncParams& p, long long q) {
  const long long NG = p.n_groups, lag = p.lag, nA = p.nA, J = p.J;
  long long bp[6] = {0, 1, lag, NG, NG + 1, NG + lag};
#pragma unroll
  for (int i = 1; i < 6; i++)
#pragma unroll
    for (int j = i; j > 0; j--)
      if (bp[j] < bp[j - 1]) {
        const long long t = bp[j];
        bp[j] = bp[j - 1];
        bp[j - 1] = t;
      }
  const long long rmax = NG + lag;
  long long cum = 0;
  for (int seg = 0; seg < 5; seg++) {
    const long long r0 = bp[seg], r1 = min(bp[seg + 1], rmax);
    if (r1 <= r0) continue;
    const bool hasB = r0 >= 1 && r0 <= NG, hasA = r0 < NG, hasC = r0 >= lag && r0 < NG + lag;
    const long long nB = hasB ? J : 0, nAr = hasA ? nA : 0, nCr = hasC ? nA : 0;
    const long long len = 2 * nB + nAr + nCr;
    if (len == 0) continue;
    const long long span = (r1 - r0) * len;
    if (q < cum + span) {
      const long long r = r0 + (q - cum) / len;
      long long pos = (q - cum) % len;
      if (pos < nB) return Item{kItemSelect, r - 1, pos};
      pos -= nB;
      const long long pre = min(p.pre, nAr);
      if (pos < pre) return Item{kItemStats, r, pos};
      pos -= pre;
      if (pos < nB) return Item{kItemOffsets, r - 1, pos};
      pos -= nB;
      const long long na = nAr - pre, m = min(na, nCr);
      if (pos < 2 * m)
        return (pos & 1) ? Item{kItemQuant, r - lag, pos >> 1} : Item{kItemStats, r, pre + (pos >> 1)};
      const long long rest = pos - 2 * m;
      return (na > nCr) ? Item{kItemStats, r, pre + m + rest} : Item{kItemQuant, r - lag, m + rest};
    }
    cum += span;
  }
  return Item{-1, 0, 0};
}

template <typename Tin, int G>
__device__ __forceinline__ void item_range(const EncParams& p, const Item& it, long long& t0,
                                           int& nt) {
  constexpr int CH = Cfg<Tin, G>::CH;
  t0 = it.g * p.n_g + it.idx * CH;
  nt = (int)min((long long)CH, p.n_g - it.idx * CH);
}

// ---- stats item: entropy keys and histograms of one chunk.  Per warp step the team
// reduces its tile's two sums (lane 0 keeps them); then one lane per tile of the warp
// forms the key, writes it and adds it to the group's histograms.
template <typename Tin, int G>
__device__ void do_stats(EncSmem<Tin, G>& s, const EncParams& p, const Item& it,
                         const unsigned char* buf) {
  using C = Cfg<Tin, G>;
  constexpr int W = C::W, L = C::L, TPW = C::TPW, NS = C::NS;
  long long t0;
  int nt;
  item_range<Tin, G>(p, it, t0, nt);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L;
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
    const float2 ls = tile_sums<Tin, G>(w, s.Trep, s.Rrep, s.tabs, lane);
    if (valid && sub == 0) {
      s.ta[kt] = ls.x;
      s.tb[kt] = ls.y;
    }
  }
  __syncwarp();
  uint32_t* hf = p.hist_fine + it.g * (long long)kFineBins;
  uint32_t* hc = p.hist_coarse + it.g * kCoarseBins;
#pragma unroll 1
  for (int l0 = 0; l0 < NS; l0 += 32) {
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
      const int b = fine_bin(H);
      atomicAdd(&hf[b], 1u);
      cb = b >> 8;
    }
    // coarse bins: one atomic per distinct bin in the warp
    const unsigned same = __match_any_sync(kFull, cb);
    if (cb >= 0 && lane == __ffs(same) - 1) atomicAdd(&hc[cb], (uint32_t)__popc(same));
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(&p.doneA[it.g], 1u);
}

// ---- select item: gather the candidates of the threshold bucket; the last select item
// of the group resolves the K-th ranked tile exactly.
template <typename Tin, int G>
__device__ void do_select(EncSmem<Tin, G>& s, const EncParams& p, const Item& it) {
  const long long g = it.g;
  const uint32_t K = (uint32_t)p.K;
  if (threadIdx.x == 0) wait_counter(&p.doneA[g], (uint32_t)p.nA, p.status);
  __syncthreads();
  uint32_t* bins = s.hist;  // all zero between stats items; left zero below
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
  __syncthreads();
  const int bstar = (int)s.scan[0];
  const uint32_t above = s.scan[1];
  // candidates of this item's slice of the group
  const long long per = (p.n_g + p.J - 1) / p.J;
  const long long lo = it.idx * per, hi = min(p.n_g, lo + per);
  const float* kg = p.keys + g * p.n_g;
  unsigned long long* cg = p.cand + g * p.n_g;
  const int lane = threadIdx.x & 31;
  for (long long base = lo; base < hi; base += kThreads) {
    const long long i = base + threadIdx.x;
    float hv = 0.0f;
    bool hit = false;
    if (i < hi) {
      hv = __ldcg(&kg[i]);
      hit = fine_bin(hv) == bstar;
    }
    const unsigned mask = __ballot_sync(kFull, hit);
    if (mask) {
      uint32_t pos0 = 0;
      const int leader = __ffs(mask) - 1;
      if (lane == leader) pos0 = atomicAdd(&p.cand_cnt[g], (uint32_t)__popc(mask));
      pos0 = __shfl_sync(kFull, pos0, leader);
      if (hit) cg[pos0 + __popc(mask & ((1u << lane) - 1u))] = rank_key(hv, (uint32_t)i);
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(&p.doneB[g], 1u);
    __threadfence();
    s.last = (prev == (uint32_t)p.J - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (s.last) {
    // radix select (8 passes of 8 bits) of the r-th largest candidate key, r from 1
    const uint32_t cnt = __ldcg(&p.cand_cnt[g]);
    const uint32_t expect = __ldcg(&p.hist_fine[g * (long long)kFineBins + bstar]);
    if (threadIdx.x == 0 && cnt != expect) set_status(p.status, kStSelectMismatch);
    uint32_t r = max(1u, min(K - above, cnt));
    unsigned long long prefix = 0ull, mask = 0ull;
    for (int pass = 7; pass >= 0 && cnt > 0u; --pass) {
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
        warp_find_from_top(bins, r, d, ab);
        if (threadIdx.x == 0) {
          s.scan[2] = (uint32_t)d;
          s.scan[3] = ab;
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)s.scan[2] << shift;
      r -= s.scan[3];
      mask |= 0xFFull << shift;
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      p.sel[g] = SelResult{prefix, cnt ? kSelThreshold : kSelNone, 0u};
      __threadfence();
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&p.selready[g]), "r"(1u) : "memory");
    }
  }
  for (int i = threadIdx.x; i < 256; i += kThreads) bins[i] = 0u;
  __syncthreads();
}

// ---- offsets item: hi-tile count of each of its chunks; the last offsets item of the
// group turns the counts into exclusive prefixes (chunk offsets in the stream).
template <typename Tin, int G>
__device__ void do_offsets(EncSmem<Tin, G>& s, const EncParams& p, const Item& it) {
  constexpr int CH = Cfg<Tin, G>::CH;
  const long long g = it.g;
  if (threadIdx.x == 0) wait_counter(&p.selready[g], 1u, p.status);
  __syncthreads();
  const unsigned long long theta = __ldcg(&p.sel[g].theta);
  const uint32_t mode = __ldcg(&p.sel[g].mode);
  unsigned long long* words = p.lookback + g * p.nA;
  const long long per = (p.nA + p.J - 1) / p.J;
  const long long c0 = it.idx * per, c1 = min(p.nA, c0 + per);
  // one warp per chunk: count the chunk's hi tiles
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (long long c = c0 + warp; c < c1; c += kWarps) {
    const long long t0 = g * p.n_g + c * CH;
    const int nt = (int)min((long long)CH, p.n_g - c * CH);
    uint32_t cnt = 0;
    for (int k = lane; k < nt; k += 32) {
      bool ishi = mode == kSelAll;
      if (mode == kSelThreshold)
        ishi = rank_key(__ldcg(&p.keys[t0 + k]), (uint32_t)(t0 + k - g * p.n_g)) >= theta;
      cnt += ishi ? 1u : 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    if (lane == 0) words[c] = cnt;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(&p.doneB2[g], 1u);
    __threadfence();
    s.last = (prev == (uint32_t)p.J - 1u) ? 1u : 0u;
  }
  __syncthreads();
  if (s.last) {
    // exclusive prefix of the nA counts: each thread sums a contiguous run, one block scan
    const long long run = (p.nA + kThreads - 1) / kThreads;
    const long long r0 = min(p.nA, (long long)threadIdx.x * run), r1 = min(p.nA, r0 + run);
    unsigned long long mine = 0;
    for (long long c = r0; c < r1; c++) mine += __ldcg(&words[c]);
    uint32_t tot;
    unsigned long long acc = block_exclusive_scan<kThreads>((uint32_t)mine, tot, s.scan);
    for (long long c = r0; c < r1; c++) {
      const unsigned long long v = __ldcg(&words[c]);
      words[c] = acc;
      acc += v;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&p.selready[g]), "r"(2u) : "memory");
  }
}

// ---- quantize item: bit widths from the group's threshold, the chunk's stream offset
// from the offsets items, then quantize + pack the chunk and write it out.
template <typename Tin, int G>
__device__ void do_quant(EncSmem<Tin, G>& s, const EncParams& p, const Item& it,
                         const unsigned char* buf, unsigned long long* bar, uint32_t parity) {
  using C = Cfg<Tin, G>;
  long long t0;
  int nt;
  item_range<Tin, G>(p, it, t0, nt);
  const long long g = it.g, lc = it.idx;
  if (threadIdx.x == 0) wait_counter(&p.selready[g], 2u, p.status);
  __syncthreads();
  const unsigned long long theta = __ldcg(&p.sel[g].theta);
  const uint32_t mode = __ldcg(&p.sel[g].mode);
  const unsigned long long prefix = __ldcg(&p.lookback[g * p.nA + lc]);
  const int slot_lo = G * p.lo / 8, slot_d = G * (p.hi - p.lo) / 8;
  // widths and exclusive hi counts inside the chunk
  uint32_t hiflags = 0u, cnt = 0u;
#pragma unroll
  for (int j = 0; j < C::kPer; j++) {
    const int k = threadIdx.x * C::kPer + j;
    if (k < nt) {
      const long long t = t0 + k;
      bool ishi = mode == kSelAll;
      if (mode == kSelThreshold)
        ishi = rank_key(__ldcg(&p.keys[t]), (uint32_t)(t - g * p.n_g)) >= theta;
      if (ishi) {
        hiflags |= 1u << j;
        ++cnt;
      }
    }
  }
  uint32_t chunk_hi;
  uint32_t before = block_exclusive_scan<kThreads>(cnt, chunk_hi, s.scan);
#pragma unroll
  for (int j = 0; j < C::kPer; j++) {
    const int k = threadIdx.x * C::kPer + j;
    if (k < nt) {
      const bool ishi = (hiflags >> j) & 1u;
      s.bits[k] = (uint8_t)(ishi ? p.hi : p.lo);
      s.off[k] = (uint16_t)(k * slot_lo + before * slot_d);
      before += ishi ? 1u : 0u;
    }
  }
  mbar_wait(bar, parity, p.status);
  __syncthreads();
  quant_chunk<Tin, G>(s, buf, nt, p.h, p.c_h);
  __syncthreads();
  const long long base = g * p.group_bytes + lc * (long long)C::CH * slot_lo + (long long)prefix * slot_d;
  int nbytes = nt * slot_lo + (int)chunk_hi * slot_d;
  if (base + nbytes > p.codes_bytes) {  // only if the select went wrong: never write past
    if (threadIdx.x == 0) set_status(p.status, kStSelectMismatch);
    nbytes = (int)max(0ll, p.codes_bytes - base);
  }
  store_stage<Tin, G>(s, p.codes, base, nbytes);
  store_meta<Tin, G>(s, p, t0, nt);
}

template <typename Tin, int G>
__global__ void __launch_bounds__(kThreads, 2) k_encode(const __grid_constant__ EncParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  EncSmem<Tin, G>& s = *reinterpret_cast<EncSmem<Tin, G>*>(smem_raw);
  init_tables<Tin, G>(s, p.tabs);
  for (int i = threadIdx.x; i < kCoarseBins; i += kThreads) s.hist[i] = 0u;
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_barrier_init();
    s.next = (long long)atomicAdd(p.ticket, 1u);
  }
  __syncthreads();
  const unsigned long long pol_keep = policy_evict_last(), pol_drop = policy_evict_first();
  const Tin* x = static_cast<const Tin*>(p.x);
  uint32_t parity = 0u;  // bit s = phase parity of buffer s

  // Thread 0 starts the bulk copy of item `it`'s input chunk into buffer `slot`.
  auto issue = [&](const Item& it, int slot) {
    if (it.type != kItemStats && it.type != kItemQuant) return;
    long long t0;
    int nt;
    item_range<Tin, G>(p, it, t0, nt);
    const uint32_t bytes = (uint32_t)nt * G * (uint32_t)sizeof(Tin);
    mbar_expect_tx(&s.bar[slot], bytes);
    bulk_load(s.buf[slot], x + t0 * G, bytes, &s.bar[slot],
              it.type == kItemStats ? pol_keep : pol_drop);
  };

  // Thread 0 decodes each item once (s.item[slot]) when it dequeues it.
  long long cur = s.next;
  int slot = 0;
  if (threadIdx.x == 0 && cur < p.n_items) {
    s.item[0] = decode_item(p, cur);
    issue(s.item[0], 0);
  }
  while (cur < p.n_items) {
    __syncthreads();  // everyone is done with the previous item and its buffer
    if (threadIdx.x == 0) {
      const long long nxt = (long long)atomicAdd(p.ticket, 1u);
      s.next = nxt;
      if (nxt < p.n_items) {
        s.item[slot ^ 1] = decode_item(p, nxt);
        issue(s.item[slot ^ 1], slot ^ 1);
      }
    }
    const Item it = s.item[slot];
    if (it.type == kItemStats) {
      mbar_wait(&s.bar[slot], (parity >> slot) & 1u, p.status);
      parity ^= 1u << slot;
      do_stats<Tin, G>(s, p, it, s.buf[slot]);
    } else if (it.type == kItemQuant) {
      do_quant<Tin, G>(s, p, it, s.buf[slot], &s.bar[slot], (parity >> slot) & 1u);
      parity ^= 1u << slot;
    } else if (it.type == kItemSelect) {
      do_select<Tin, G>(s, p, it);
    } else if (it.type == kItemOffsets) {
      do_offsets<Tin, G>(s, p, it);
    }
    __syncthreads();
    cur = s.next;
    slot ^= 1;
  }
}

// ====================================================================== one-pass kernel

// Every tile gets the same width b (K = 0 or K = n_g): slot offsets are t * G * b / 8.
template <typename Tin, int G>
__global__ void __launch_bounds__(kThreads, 2) k_encode_flat(const __grid_constant__ EncParams p,
                                                             int b, long long n_chunks) {
  using C = Cfg<Tin, G>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  EncSmem<Tin, G>& s = *reinterpret_cast<EncSmem<Tin, G>*>(smem_raw);
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_barrier_init();
  }
  for (int k = threadIdx.x; k < C::CH; k += kThreads) {
    s.bits[k] = (uint8_t)b;
    s.off[k] = (uint16_t)(k * G * b / 8);
  }
  __syncthreads();
  const unsigned long long pol = policy_evict_first();
  const Tin* x = static_cast<const Tin*>(p.x);
  uint32_t parity = 0u;
  auto issue = [&](long long c, int slot) {
    const long long t0 = c * C::CH;
    const int nt = (int)min((long long)C::CH, p.n_tiles - t0);
    const uint32_t bytes = (uint32_t)nt * G * (uint32_t)sizeof(Tin);
    mbar_expect_tx(&s.bar[slot], bytes);
    bulk_load(s.buf[slot], x + t0 * G, bytes, &s.bar[slot], pol);
  };
  long long c = blockIdx.x;
  int slot = 0;
  if (threadIdx.x == 0 && c < n_chunks) issue(c, 0);
  for (; c < n_chunks; c += gridDim.x) {
    const long long nx = c + gridDim.x;
    if (threadIdx.x == 0 && nx < n_chunks) issue(nx, slot ^ 1);
    const long long t0 = c * C::CH;
    const int nt = (int)min((long long)C::CH, p.n_tiles - t0);
    mbar_wait(&s.bar[slot], (parity >> slot) & 1u, p.status);
    parity ^= 1u << slot;
    __syncthreads();
    quant_chunk<Tin, G>(s, s.buf[slot], nt, p.h, p.c_h);
    __syncthreads();
    store_stage<Tin, G>(s, p.codes, t0 * G * b / 8, nt * G * b / 8);
    store_meta<Tin, G>(s, p, t0, nt);
    __syncthreads();
    slot ^= 1;
  }
}

// ====================================================================== launchers

template <typename Tin, int G>
static cudaError_t run_encode(const EncodeArgs& a, cudaStream_t st) {
  using C = Cfg<Tin, G>;
  const size_t smem = sizeof(EncSmem<Tin, G>);
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
  p.codes = a.codes;
  p.scales = a.scales;
  p.zeros = a.zeros;
  p.bits = a.bits;
  p.pivots = a.pivots;
  p.keys = a.keys;
  p.cand = a.cand;
  p.cand_cnt = a.cand_cnt;
  p.hist_coarse = a.hist_coarse;
  p.hist_fine = a.hist_fine;
  p.doneA = a.doneA;
  p.doneB = a.doneB;
  p.doneB2 = a.doneB2;
  p.selready = a.selready;
  p.sel = a.sel;
  p.lookback = a.lookback;
  p.ticket = a.ticket;
  p.status = a.status;
  p.tabs = *a.tabs;
  p.nA = (a.n_g + C::CH - 1) / C::CH;
  const int grid_cap = a.num_sms * 2;
  if (a.K == 0 || a.K == a.n_g) {
    cudaError_t e = cudaFuncSetAttribute(k_encode_flat<Tin, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long n_chunks = (a.n_tiles + C::CH - 1) / C::CH;
    const int grid = (int)std::max<long long>(1, std::min<long long>(grid_cap, n_chunks));
    k_encode_flat<Tin, G><<<grid, kThreads, smem, st>>>(p, a.K == 0 ? a.lo : a.hi, n_chunks);
    return cudaGetLastError();
  }
  // keep two (or, for big groups, one) groups' input in L2 between a group's stats pass
  // and its quantize pass
  const long long group_in = a.n_g * G * (long long)sizeof(Tin);
  p.lag = (3 * group_in <= (72ll << 20)) ? 2 : 1;
  p.pre = (p.lag == 1) ? p.nA / 4 : p.nA / 8;
  p.J = std::max<long long>(1, std::min<long long>(256, p.nA / 8));
  p.n_items = a.n_groups * (2 * p.nA + 2 * p.J);
  cudaError_t e = cudaFuncSetAttribute(k_encode<Tin, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::max<long long>(1, std::min<long long>(grid_cap, p.n_items));
  k_encode<Tin, G><<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

long long encode_chunks(int bf16, int G, long long n_g, long long n_groups) {
  const long long ch = kChunkBytes / (G * (bf16 ? 2 : 4));
  return n_groups * ((n_g + ch - 1) / ch);
}

cudaError_t launch_encode(const EncodeArgs& a, cudaStream_t st) {
#define TAHQ_G_CASE(T, GG) \
  case GG:                 \
    return run_encode<T, GG>(a, st);
  if (a.bf16) {
    switch (a.G) {
      TAHQ_G_CASE(uint16_t, 8)
      TAHQ_G_CASE(uint16_t, 16)
      TAHQ_G_CASE(uint16_t, 32)
      TAHQ_G_CASE(uint16_t, 64)
      TAHQ_G_CASE(uint16_t, 128)
    }
  } else {
    switch (a.G) {
      TAHQ_G_CASE(float, 8)
      TAHQ_G_CASE(float, 16)
      TAHQ_G_CASE(float, 32)
      TAHQ_G_CASE(float, 64)
      TAHQ_G_CASE(float, 128)
    }
  }
#undef TAHQ_G_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tahq
