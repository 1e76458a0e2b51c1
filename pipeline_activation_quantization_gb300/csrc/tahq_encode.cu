// tahq_encode.cu -- encode kernels of the TAH-Quant activation codec for sm_103a.
//
// "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over Slow
// Network" (arXiv 2506.01352v2):
//   k_stats          §3.2 eq. (1)-(2) entropy key, §3.3 eq. (3) outlier ratio + pivot,
//                    plus the per-group key histograms the allocator selects from;
//   k_select_collect §3.2 "Top-p% tile selection": locate the histogram bucket that holds
//   k_select_final   the K-th ranked tile of each group and resolve it exactly;
//   k_quant          §3.3 pivot swap + eq. (4) Hadamard, asymmetric quantizer, and the
//                    §3.4 contiguous uint8 stream (slot offsets by a decoupled look-back).
#include <algorithm>
#include <cfloat>

#include "tahq_device.cuh"
#include "tahq_launch.h"

namespace tahq {

template <typename Tin>
struct InTraits;
template <>
struct InTraits<float> {
  static constexpr int V = 4;
  static constexpr bool kNoFraction = false;
};
template <>
struct InTraits<uint16_t> {  // bf16 bit patterns
  static constexpr int V = 8;
  static constexpr bool kNoFraction = true;
};

// One 16-byte streaming load of a lane's V consecutive values, widened to fp32.
template <typename Tin>
__device__ __forceinline__ void load_lane(const Tin* __restrict__ x, long long elem, float* v) {
  uint4 w;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
               : "l"(x + elem));
  if constexpr (sizeof(Tin) == 4) {
    v[0] = __uint_as_float(w.x);
    v[1] = __uint_as_float(w.y);
    v[2] = __uint_as_float(w.z);
    v[3] = __uint_as_float(w.w);
  } else {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      v[2 * j] = __uint_as_float(ws[j] << 16);            // element 2j: low half
      v[2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u); // element 2j+1: high half
    }
  }
}

__device__ __forceinline__ void load_tables(const LgTables& tabs, float* sT, float* sR, float* sk) {
  for (int i = threadIdx.x; i < 128; i += blockDim.x) {
    sT[i] = tabs.T[i];
    sR[i] = tabs.R[i];
  }
  if (threadIdx.x < 4) sk[threadIdx.x] = tabs.k[threadIdx.x];
}

// ====================================================================== tile statistics

template <typename Tin, int G>
__global__ void __launch_bounds__(256) k_stats(const Tin* __restrict__ x, long long n_tiles,
                                               long long n_g, LgTables tabs,
                                               float* __restrict__ keys,
                                               uint8_t* __restrict__ pivots,
                                               uint32_t* __restrict__ hist_coarse,
                                               uint32_t* __restrict__ hist_fine,
                                               uint32_t* __restrict__ status) {
  constexpr int V = InTraits<Tin>::V;
  using Gm = Geom<V, G>;
  constexpr int L = Gm::L;
  __shared__ float sT[128], sR[128], sk[4];
  load_tables(tabs, sT, sR, sk);
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int team = lane / L, sub = lane % L;
  const long long n_steps = (n_tiles + Gm::TPW - 1) / Gm::TPW;
  const long long n_warps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long step = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; step < n_steps;
       step += n_warps) {
    const long long t = step * Gm::TPW + team;
    const bool valid = t < n_tiles;
    float v[V];
    if (valid) {
      load_lane<Tin>(x, t * G + sub * V, v);
    } else {
#pragma unroll
      for (int j = 0; j < V; j++) v[j] = 0.0f;
    }
    float m[V];
#pragma unroll
    for (int j = 0; j < V; j++) m[j] = fabsf(v[j]);

    // top-2 magnitudes and the first arg-max (eq. (3))
    float m1 = m[0], m2 = -1.0f;
    int i1 = sub * V;
#pragma unroll
    for (int j = 1; j < V; j++) {
      if (m[j] > m1) {
        m2 = m1;
        m1 = m[j];
        i1 = sub * V + j;
      } else if (m[j] > m2) {
        m2 = m[j];
      }
    }
    team_top2<L>(m1, i1, m2);

    // entropy key (eq. (1)-(2)): H = lg L - S / L
    float term[V];
#pragma unroll
    for (int j = 0; j < V; j++)
      term[j] = (m[j] == 0.0f)
                    ? 0.0f
                    : __fmul_rn(m[j], lg_canon<InTraits<Tin>::kNoFraction>(m[j], sT, sR, sk));
    const float Ls = team_sum<L>(lane_pairwise<V>(m));
    const float Ss = team_sum<L>(lane_pairwise<V>(term));
    const float H =
        (Ls == 0.0f) ? 0.0f : __fsub_rn(lg_canon<false>(Ls, sT, sR, sk), __fdiv_rn(Ss, Ls));
    const bool flag = __fdiv_rn(m1, __fadd_rn(m2, 1e-12f)) > 2.0f;

    if (valid && sub == 0) {
      keys[t] = H;
      pivots[t] = flag ? (uint8_t)i1 : (uint8_t)0xFF;
      if (!(Ls <= FLT_MAX) || !(fabsf(Ss) <= FLT_MAX) || !(fabsf(H) <= FLT_MAX))
        set_status(status, kStNonFinite);
      const long long g = t / n_g;
      const int b = fine_bin(H);
      atomicAdd(&hist_fine[g * kFineBins + b], 1u);
      atomicAdd(&hist_coarse[g * kCoarseBins + (b >> 8)], 1u);
    }
  }
}

// ====================================================================== exact select

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

// Threshold bucket of one group: b* and the count of tiles in buckets above it.  Run by
// warp 0 of a block; results left in shared memory.
__device__ __forceinline__ void find_threshold_bucket(const uint32_t* hist_coarse,
                                                      const uint32_t* hist_fine, uint32_t K,
                                                      uint32_t* s_bins, int* s_bstar,
                                                      uint32_t* s_above) {
  if (threadIdx.x < 32) {
    for (int i = threadIdx.x; i < 256; i += 32) s_bins[i] = hist_coarse[i];
    __syncwarp();
    int cb;
    uint32_t above_c;
    warp_find_from_top(s_bins, K, cb, above_c);
    __syncwarp();
    for (int i = threadIdx.x; i < 256; i += 32) s_bins[i] = hist_fine[cb * 256 + i];
    __syncwarp();
    int fb;
    uint32_t above_f;
    warp_find_from_top(s_bins, K - above_c, fb, above_f);
    if (threadIdx.x == 0) {
      *s_bstar = cb * 256 + fb;
      *s_above = above_c + above_f;
    }
  }
}

__global__ void __launch_bounds__(256) k_select_collect(
    const float* __restrict__ keys, long long n_g, uint32_t K,
    const uint32_t* __restrict__ hist_coarse, const uint32_t* __restrict__ hist_fine,
    unsigned long long* __restrict__ cand, uint32_t* __restrict__ cand_cnt) {
  __shared__ uint32_t s_bins[256];
  __shared__ int s_bstar;
  __shared__ uint32_t s_above;
  const long long g = blockIdx.y;
  find_threshold_bucket(hist_coarse + g * kCoarseBins, hist_fine + g * (long long)kFineBins, K,
                        s_bins, &s_bstar, &s_above);
  __syncthreads();
  const int bstar = s_bstar;
  const long long per = (n_g + gridDim.x - 1) / gridDim.x;
  const long long lo = (long long)blockIdx.x * per;
  const long long hi = min(n_g, lo + per);
  const float* kg = keys + g * n_g;
  unsigned long long* cg = cand + g * n_g;
  const int lane = threadIdx.x & 31;
  for (long long base = lo; base < hi; base += blockDim.x) {
    const long long i = base + threadIdx.x;
    float h = 0.0f;
    bool hit = false;
    if (i < hi) {
      h = kg[i];
      hit = fine_bin(h) == bstar;
    }
    const unsigned mask = __ballot_sync(kFull, hit);
    if (mask) {
      uint32_t pos0 = 0;
      const int leader = __ffs(mask) - 1;
      if (lane == leader) pos0 = atomicAdd(&cand_cnt[g], (uint32_t)__popc(mask));
      pos0 = __shfl_sync(kFull, pos0, leader);
      if (hit) cg[pos0 + __popc(mask & ((1u << lane) - 1u))] = rank_key(h, (uint32_t)i);
    }
  }
}

// Radix select (8 passes of 8 bits) of the r-th largest composite key among the
// candidates of the threshold bucket; r counts from 1.
__global__ void __launch_bounds__(1024) k_select_final(
    long long n_g, uint32_t K, const uint32_t* __restrict__ hist_coarse,
    const uint32_t* __restrict__ hist_fine, const unsigned long long* __restrict__ cand,
    const uint32_t* __restrict__ cand_cnt, SelResult* __restrict__ sel,
    uint32_t* __restrict__ status) {
  __shared__ uint32_t s_bins[256];
  __shared__ int s_bstar;
  __shared__ uint32_t s_above;
  __shared__ unsigned long long s_prefix;
  __shared__ uint32_t s_r;
  const long long g = blockIdx.x;
  if (K == 0u || (long long)K == n_g) {
    if (threadIdx.x == 0) sel[g] = SelResult{0ull, K == 0u ? kSelNone : kSelAll, 0u};
    return;
  }
  const uint32_t* hc = hist_coarse + g * kCoarseBins;
  const uint32_t* hf = hist_fine + g * (long long)kFineBins;
  find_threshold_bucket(hc, hf, K, s_bins, &s_bstar, &s_above);
  __syncthreads();
  const uint32_t expect = hf[s_bstar];
  const uint32_t cnt = cand_cnt[g];
  if (threadIdx.x == 0) {
    if (cnt != expect) set_status(status, kStSelectMismatch);
    uint32_t r = K - s_above;
    if (r < 1u) r = 1u;
    if (r > cnt) r = cnt;
    s_r = r;
    s_prefix = 0ull;
  }
  __syncthreads();
  const unsigned long long* cg = cand + g * n_g;
  unsigned long long mask = 0ull;
  for (int pass = 7; pass >= 0 && cnt > 0u; --pass) {
    const int shift = pass * 8;
    if (threadIdx.x < 256) s_bins[threadIdx.x] = 0u;
    __syncthreads();
    const unsigned long long prefix = s_prefix;
    for (uint32_t i = threadIdx.x; i < cnt; i += blockDim.x) {
      const unsigned long long v = cg[i];
      if ((v & mask) == prefix) atomicAdd(&s_bins[(v >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      int d;
      uint32_t above;
      warp_find_from_top(s_bins, s_r, d, above);
      if (threadIdx.x == 0) {
        s_r -= above;
        s_prefix = prefix | ((unsigned long long)d << shift);
      }
    }
    mask |= 0xFFull << shift;
    __syncthreads();
  }
  if (threadIdx.x == 0) sel[g] = SelResult{s_prefix, cnt ? kSelThreshold : kSelNone, 0u};
}

// ====================================================================== quantize + pack

template <int kThreads>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t& total,
                                                         uint32_t* s_warp) {
  constexpr int kWarps = kThreads / 32;
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
    const uint32_t w = lane < kWarps ? s_warp[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += y;
    }
    __syncwarp();
    if (lane < kWarps) s_warp[lane] = wi - w;
    if (lane == kWarps - 1) s_warp[kWarps] = wi;
  }
  __syncthreads();
  total = s_warp[kWarps];
  const uint32_t r = s_warp[warp] + incl - v;
  __syncthreads();
  return r;
}

template <typename Tin, int G>
struct QuantCfg {
  static constexpr int V = InTraits<Tin>::V;
  using Gm = Geom<V, G>;
  static constexpr int kThreads = 256;
  static constexpr int CH = 32768 / (G * (int)sizeof(Tin));   // tiles per chunk (32 KB in)
  static constexpr int kSteps = CH / (8 * Gm::TPW);            // warp steps per chunk
  static constexpr int kPer = (CH + kThreads - 1) / kThreads;  // tiles per thread (scan)
  static constexpr int kStageBytes = CH * G + 48;              // b <= 8, plus alignment pad
  static_assert(kSteps * 8 * Gm::TPW == CH, "chunk must be whole warp steps");
  static_assert(kPer <= 32, "hi flags are kept in one 32-bit word per thread");
};

template <typename Tin, int G>
__global__ void __launch_bounds__(256) k_quant(
    const Tin* __restrict__ x, long long n_g, long long group_bytes, long long codes_bytes,
    int lo, int hi, int h,
    float c_h, const float* __restrict__ keys, const uint8_t* __restrict__ piv_in,
    const SelResult* __restrict__ sel, uint8_t* __restrict__ codes, float* __restrict__ scales,
    float* __restrict__ zeros, uint8_t* __restrict__ bits,
    unsigned long long* __restrict__ lookback, uint32_t* __restrict__ ticket,
    uint32_t* __restrict__ status, long long n_chunks) {
  using Cf = QuantCfg<Tin, G>;
  constexpr int V = Cf::V, L = Cf::Gm::L, TPW = Cf::Gm::TPW, CH = Cf::CH;
  __shared__ __align__(16) uint32_t s_stage[Cf::kStageBytes / 4];
  __shared__ uint16_t s_off[CH];
  __shared__ uint8_t s_bits[CH];
  __shared__ uint32_t s_warp[9];
  __shared__ long long s_c;
  __shared__ long long s_base;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L;
  const long long cpg = (n_g + CH - 1) / CH;
  const int slot_lo = G * lo / 8, slot_d = G * (hi - lo) / 8;

  for (;;) {
    if (threadIdx.x == 0) s_c = (long long)atomicAdd(ticket, 1u);
    __syncthreads();
    const long long c = s_c;
    if (c >= n_chunks) break;
    const long long g = c / cpg, lc = c % cpg;
    const long long t0 = g * n_g + lc * CH;
    const int nt = (int)min((long long)CH, n_g - lc * CH);
    const SelResult sg = sel[g];

    // 1. bit widths of this chunk's tiles and their exclusive hi counts
    uint32_t hiflags = 0u, cnt = 0u;
#pragma unroll
    for (int j = 0; j < Cf::kPer; j++) {
      const int k = threadIdx.x * Cf::kPer + j;
      if (k < nt) {
        const long long t = t0 + k;
        bool ishi = sg.mode == kSelAll;
        if (sg.mode == kSelThreshold)
          ishi = rank_key(keys[t], (uint32_t)(t - g * n_g)) >= sg.theta;
        if (ishi) {
          hiflags |= 1u << j;
          ++cnt;
        }
      }
    }
    uint32_t chunk_hi;
    uint32_t before = block_exclusive_scan<256>(cnt, chunk_hi, s_warp);
#pragma unroll
    for (int j = 0; j < Cf::kPer; j++) {
      const int k = threadIdx.x * Cf::kPer + j;
      if (k < nt) {
        const bool ishi = (hiflags >> j) & 1u;
        s_bits[k] = (uint8_t)(ishi ? hi : lo);
        s_off[k] = (uint16_t)(k * slot_lo + before * slot_d);
        bits[t0 + k] = (uint8_t)(ishi ? hi : lo);
        before += ishi ? 1u : 0u;
      }
    }

    // 2. chunk offset in the stream: look-back over the earlier chunks of this group
    if (threadIdx.x == 0) {
      unsigned long long prefix = 0ull;
      if (lc == 0) {
        st_release_u64(&lookback[c], kLbPre | (unsigned long long)chunk_hi);
      } else {
        st_release_u64(&lookback[c], kLbAgg | (unsigned long long)chunk_hi);
        prefix = lookback_prefix(lookback, c, g * cpg, status);
        st_release_u64(&lookback[c], kLbPre | (prefix + chunk_hi));
      }
      s_base = g * group_bytes + lc * (long long)CH * slot_lo + (long long)prefix * slot_d;
    }
    int chunk_bytes = nt * slot_lo + (int)chunk_hi * slot_d;
    __syncthreads();
    const long long base = s_base;
    if (base + chunk_bytes > codes_bytes) {  // only if the select went wrong: never write past
      if (threadIdx.x == 0) set_status(status, kStSelectMismatch);
      chunk_bytes = (int)max(0ll, codes_bytes - base);
    }
    const int pad = (int)(base & 15);
    const int stage_words = (pad + chunk_bytes + 15) / 16 * 4;
    for (int i = threadIdx.x; i < stage_words; i += Cf::kThreads) s_stage[i] = 0u;
    __syncthreads();

    // 3. per tile: pivot swap + Hadamard (flagged tiles), quantise, pack
#pragma unroll 1
    for (int s = 0; s < Cf::kSteps; s++) {
      const int kt = (s * 8 + warp) * TPW + team;
      const bool valid = kt < nt;
      const long long t = t0 + kt;
      float v[V];
      if (valid) {
        load_lane<Tin>(x, t * G + sub * V, v);
      } else {
#pragma unroll
        for (int j = 0; j < V; j++) v[j] = 0.0f;
      }
      const int piv = valid ? (int)piv_in[t] : 0xFF;
      const bool flag = piv != 0xFF;
      if (__any_sync(kFull, flag)) {
        float w[V];
#pragma unroll
        for (int j = 0; j < V; j++) w[j] = v[j];
        team_swap0<V>(w, flag ? piv : 0, sub, lane - sub);
        team_fwht<V, L>(w, h, sub);
        if (flag) {
#pragma unroll
          for (int j = 0; j < V; j++) v[j] = __fmul_rn(w[j], c_h);
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
      const int b = valid ? (int)s_bits[kt] : lo;
      const uint32_t Q = (1u << b) - 1u;
      const float D = __fsub_rn(mx, mn);
      const bool degenerate = !(D >= 0x1p-120f);
      const float qf = (float)Q;
      const float scale = degenerate ? 0.0f : __fdiv_rn(D, qf);
      const float inv = degenerate ? 0.0f : __fdiv_rn(qf, D);
      unsigned long long acc = 0ull;
#pragma unroll
      for (int j = 0; j < V; j++) {
        const float u = __fmul_rn(__fsub_rn(v[j], mn), inv);
        // round to nearest even: for 0 <= u < 2^22, u + 1.5*2^23 lands on an integer
        uint32_t q = __float_as_uint(__fadd_rn(u, 12582912.0f)) - 0x4B400000u;
        q = min(q, Q);
        if (degenerate) q = 0u;
        acc |= (unsigned long long)q << (j * b);
      }
      if (valid && (int)s_off[kt] + G * b / 8 <= chunk_bytes) {
        const int pos = 8 * (pad + (int)s_off[kt]) + sub * V * b;
        const int wi = pos >> 5, sh = pos & 31;
        const unsigned long long lo64 = acc << sh;
        const uint32_t w0 = (uint32_t)lo64, w1 = (uint32_t)(lo64 >> 32);
        const uint32_t w2 = sh ? (uint32_t)(acc >> (64 - sh)) : 0u;
        if (w0) atomicOr(&s_stage[wi], w0);
        if (w1) atomicOr(&s_stage[wi + 1], w1);
        if (w2) atomicOr(&s_stage[wi + 2], w2);
        if (sub == 0) {
          scales[t] = scale;
          zeros[t] = mn;
        }
      }
    }
    __syncthreads();

    // 4. copy the staged bytes to codes[base, base + chunk_bytes)
    const uint8_t* sb = reinterpret_cast<const uint8_t*>(s_stage);
    const long long a0 = base - pad;
    const int n16 = (pad + chunk_bytes + 15) / 16;
    for (int w16 = threadIdx.x; w16 < n16; w16 += Cf::kThreads) {
      const long long gb = a0 + 16ll * w16;
      if (gb >= base && gb + 16 <= base + chunk_bytes) {
        *reinterpret_cast<uint4*>(codes + gb) = reinterpret_cast<const uint4*>(s_stage)[w16];
      } else {
#pragma unroll
        for (int k = 0; k < 16; k++) {
          const long long p = gb + k;
          if (p >= base && p < base + chunk_bytes) codes[p] = sb[16 * w16 + k];
        }
      }
    }
    __syncthreads();
  }
}

// ====================================================================== launchers

template <typename Tin, int G>
static cudaError_t run_encode(const EncodeArgs& a, cudaStream_t st) {
  using Cf = QuantCfg<Tin, G>;
  const Tin* x = static_cast<const Tin*>(a.x);
  const long long stats_need = (a.n_tiles + 8 * Cf::Gm::TPW - 1) / (8 * Cf::Gm::TPW);
  const int stats_blocks = (int)std::max<long long>(1, std::min<long long>((long long)a.num_sms * 8, stats_need));
  k_stats<Tin, G><<<stats_blocks, 256, 0, st>>>(x, a.n_tiles, a.n_g, *a.tabs, a.keys, a.pivots,
                                                 a.hist_coarse, a.hist_fine, a.status);
  if (a.K > 0 && a.K < a.n_g) {
    const int per_group = (int)std::max<long long>(1, std::min<long long>(64, a.n_g / 4096));
    k_select_collect<<<dim3(per_group, (unsigned)a.n_groups), 256, 0, st>>>(
        a.keys, a.n_g, (uint32_t)a.K, a.hist_coarse, a.hist_fine, a.cand, a.cand_cnt);
  }
  k_select_final<<<(unsigned)a.n_groups, 1024, 0, st>>>(a.n_g, (uint32_t)a.K, a.hist_coarse,
                                                         a.hist_fine, a.cand, a.cand_cnt, a.sel,
                                                         a.status);
  const long long n_chunks = encode_chunks(a.bf16, G, a.n_g, a.n_groups);
  const int quant_blocks = (int)std::max<long long>(1, std::min<long long>((long long)a.num_sms * 6, n_chunks));
  k_quant<Tin, G><<<quant_blocks, 256, 0, st>>>(
      x, a.n_g, a.group_bytes, a.n_groups * a.group_bytes, a.lo, a.hi, a.h, a.c_h, a.keys,
      a.pivots, a.sel, a.codes,
      a.scales, a.zeros, a.bits, a.lookback, a.ticket, a.status, n_chunks);
  return cudaGetLastError();
}

long long encode_chunks(int bf16, int G, long long n_g, long long n_groups) {
  const long long ch = 32768 / (G * (bf16 ? 2 : 4));
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
