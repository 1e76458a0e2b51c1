// tahq_device.cuh -- device building blocks of the sm_103a TAH-Quant codec.
//
// Arithmetic that decides an integer (the entropy key that ranks tiles, the outlier
// flag, the quantised codes) is spelled out with explicit round-to-nearest intrinsics
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fmaf_rn), so that no contraction or reordering
// can change a result.  The evaluation order is the canonical one of the codec:
//   - pairwise sums: sum(x[0..n)) = sum(x[0..n/2)) + sum(x[n/2..n)), the first level of
//     S fused: fmaf(m_odd, lg m_odd, RN(m_even lg m_even)),
//   - lg(x) = e + fmaf(P(r), r, T[i]), r = fmaf(m, R[i], -1) for x = 2^e m, i the top 7
//     fraction bits, P(r) = fmaf(fmaf(k3, r, k2), r, k1) (Tang-style table logarithm),
//   - entropy key H = lg(L) - S / L, L = sum |a|, S = sum |a| lg |a|,
//   - Hadamard stages len = 1, 2, 4, ... then x RN(1/sqrt(h)),
//   - code = the integer nearest (ties to even) to RN(v - min) * RN(Q / (max - min)),
//     one rounding (fmaf(v - min, inv, 1.5 * 2^23)); it never exceeds Q, so no clamp.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tahq {

constexpr unsigned kFull = 0xffffffffu;

// Device status word bits (mirror the TAHQ_DEV_* macros of tahq.h).
constexpr uint32_t kStNonFinite = 0x1u;
constexpr uint32_t kStWaitTimeout = 0x2u;
constexpr uint32_t kStSelectMismatch = 0x4u;
constexpr uint32_t kStBadBits = 0x8u;
constexpr uint32_t kStOverrun = 0x10u;
constexpr uint32_t kStBadWire = 0x20u;

// Tables of the canonical logarithm, passed to kernels by value and copied to shared
// memory (indexed loads from the parameter bank would serialise).
//   T[i] = RN(-log2 R[i]), R[i] = RN(1 / c_i), c_i = 1 + i/128, k = Mercator coefficients
//   (1/ln2, -1/(2 ln2), 1/(3 ln2)); TB[i] = the fraction part of lg(c_i) as the general
//   path computes it (fmaf(P(r), r, T[i]) with r = fmaf(c_i, R[i], -1)), for inputs whose
//   mantissa has no bits below the top 7 (every bf16 value).
struct LgTables {
  float T[128];
  float R[128];
  float TB[128];
  float k[3];
};

// One group's threshold: a tile is hi iff mode == kSelAll, or mode == kSelThreshold and
// its composite rank key >= theta.
struct SelResult {
  unsigned long long theta;
  uint32_t mode;
  uint32_t pad;
};
constexpr uint32_t kSelNone = 0, kSelAll = 1, kSelThreshold = 2;

// Fine-histogram geometry: bucket = floor(H * 8192) clamped to [0, 65535] (H is in bits,
// 0 <= H <= log2(tile) <= 7), coarse bucket = bucket >> 8.
constexpr int kFineBins = 65536;
constexpr int kCoarseBins = 256;

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

// ------------------------------------------------------------------ dependent launches

// A kernel launched by launch_dependent may start while the kernel before it on the
// stream is still running: dep_wait blocks until that kernel has finished and its writes
// are visible (a no-op for a kernel launched the ordinary way), dep_launch lets the next
// kernel on the stream start once every block of this one has called it or exited.  A
// dependent kernel calls dep_wait before it reads anything the kernels before it wrote,
// and before it ends, so that it also finishes after all of them.
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ------------------------------------------------------------------ canonical logarithm

// The canonical base-2 logarithm of a positive finite float: x = 2^e m, m in [1, 2),
// i = top 7 fraction bits, r = fmaf(m, R[i], -1), lg = e + fmaf(P(r), r, T[i]) with
// P(r) = fmaf(fmaf(k3, r, k2), r, k1).  kNoFraction: the caller guarantees that x has no
// mantissa bits below the top 7 (true for every bf16 value, normal or subnormal), so
// m = c_i and the fraction part is the precomputed TB[i] -- the same value.
template <bool kNoFraction>
__device__ __forceinline__ float lg_canon(float x, const float* sT, const float* sR,
                                          const float* sTB, const float* sk) {
  uint32_t b = __float_as_uint(x);
  int e = (int)(b >> 23) - 127;
  if ((b >> 23) == 0u) {  // subnormal: normalise by 2^24, exactly
    b = __float_as_uint(__fmul_rn(x, 16777216.0f));
    e = (int)(b >> 23) - 151;
  }
  const int i = (int)((b >> 16) & 0x7Fu);
  float t;
  if (kNoFraction) {
    t = sTB[i];
  } else {
    const float m = __uint_as_float((b & 0x007FFFFFu) | 0x3F800000u);
    const float r = __fmaf_rn(m, sR[i], -1.0f);
    float p = __fmaf_rn(sk[2], r, sk[1]);
    p = __fmaf_rn(p, r, sk[0]);
    t = __fmaf_rn(p, r, sT[i]);
  }
  return __fadd_rn((float)e, t);
}

// Order-preserving 32-bit image of a float key (-0 is folded onto +0 first).  NaN (only
// from non-finite input) maps to the lowest rank, as fine_bin puts it in bucket 0, so
// the histogram and the rank keys always agree and a group never gets more than K hi
// tiles.
__device__ __forceinline__ uint32_t order_key(float h) {
  if (h != h) return 0u;
  const uint32_t b = __float_as_uint(__fadd_rn(h, 0.0f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Composite rank key of tile t_local of a group: larger = ranked earlier
// (higher entropy first, then lower tile index).
__device__ __forceinline__ unsigned long long rank_key(float h, uint32_t t_local) {
  return ((unsigned long long)order_key(h) << 32) | (unsigned long long)(0xFFFFFFFFu - t_local);
}

// Bucket of a key: keys of tiles of up to 256 values lie in [0, 8] bits (scale 8192),
// of allocation tiles of up to 65536 values in [0, 16] (scale 4096); the scale is a power
// of two, so h * scale is exact and the buckets keep the keys' order.
__device__ __forceinline__ int fine_bin(float h, float scale) {
  if (!(h >= 0.0f)) return 0;          // negative rounding residue or NaN
  const float x = __fmul_rn(h, scale);
  if (!(x < (float)kFineBins)) return kFineBins - 1;
  return (int)x;                       // truncation == floor for x >= 0
}

// ------------------------------------------------------------------ tile geometry

// A tile of G values is spread over L = G / V consecutive lanes of a warp ("team"),
// each lane holding V consecutive values.
template <int kV, int kG>
struct Geom {
  static constexpr int V = kV;
  static constexpr int G = kG;
  static constexpr int L = kG / kV;
  static constexpr int TPW = 32 / L;  // tiles per warp per step
  static_assert(kG % kV == 0 && L >= 1 && L <= 32, "tile must span 1..32 lanes");
};

// Pairwise sum of the lane's V values.
template <int V>
__device__ __forceinline__ float lane_pairwise(const float* v) {
  if constexpr (V == 8) {
    return __fadd_rn(__fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3])),
                     __fadd_rn(__fadd_rn(v[4], v[5]), __fadd_rn(v[6], v[7])));
  } else {
    static_assert(V == 4, "V is 4 or 8");
    return __fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3]));
  }
}

// Continue the pairwise tree across the L lanes of a team (xor 1, 2, ..., L/2).
template <int L>
__device__ __forceinline__ float team_sum(float s) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) s = __fadd_rn(s, __shfl_xor_sync(kFull, s, o));
  return s;
}

template <int L>
__device__ __forceinline__ float team_min(float s) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) s = fminf(s, __shfl_xor_sync(kFull, s, o));
  return s;
}

template <int L>
__device__ __forceinline__ float team_max(float s) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) s = fmaxf(s, __shfl_xor_sync(kFull, s, o));
  return s;
}

template <int L>
__device__ __forceinline__ int team_min_i(int s) {
#pragma unroll
  for (int o = 1; o < L; o <<= 1) s = min(s, __shfl_xor_sync(kFull, s, o));
  return s;
}

// Top-2 of a tile spread over a team of L lanes, V values a lane (position sub * V + j):
// m1 = the largest magnitude, i1 = the first position holding it, m2 = the largest
// magnitude of the other positions.  No branches: three team reductions.
template <int V, int L>
__device__ __forceinline__ void team_top2_values(const float* v, int sub, float& m1, int& i1,
                                                 float& m2) {
  float a[V], la = 0.0f;
#pragma unroll
  for (int j = 0; j < V; j++) {
    a[j] = fabsf(v[j]);
    la = fmaxf(la, a[j]);
  }
  m1 = team_max<L>(la);
  int jj = V;
#pragma unroll
  for (int j = V - 1; j >= 0; j--) jj = a[j] == m1 ? j : jj;
  i1 = team_min_i<L>(jj < V ? sub * V + jj : V * L);
  float l2 = 0.0f;
#pragma unroll
  for (int j = 0; j < V; j++) l2 = fmaxf(l2, sub * V + j == i1 ? 0.0f : a[j]);
  m2 = team_max<L>(l2);
}

// In-register Sylvester FWHT of every h-block of the team's tile (h | G, h a power of
// two), stages len = 1, 2, ..., h/2 in that order; the pair (j, j+len) -> (a+b, a-b).
// Stages with len < V stay in the lane (indices are compile-time after unrolling);
// stages with len >= V pair lane sub with lane sub ^ (len / V).  h is warp-uniform.
template <int V, int L>
__device__ __forceinline__ void team_fwht(float* v, int h, int sub) {
#pragma unroll
  for (int s = 0; (1 << s) < V; s++) {
    const int len = 1 << s;
    if (len < h) {
#pragma unroll
      for (int j = 0; j < V; j++) {
        if ((j & len) == 0) {
          const float a = v[j], b = v[j | len];
          v[j] = __fadd_rn(a, b);
          v[j | len] = __fsub_rn(a, b);
        }
      }
    }
  }
#pragma unroll
  for (int s = 0; (1 << s) < L; s++) {
    const int lanes = 1 << s;
    if (lanes * V < h) {
      // lower lane: v + o; upper lane: o - v.  fma(+-1, v, o) rounds exactly once, like
      // the add / subtract it stands for.
      const float sg = (sub & lanes) ? -1.0f : 1.0f;
#pragma unroll
      for (int j = 0; j < V; j++) {
        const float o = __shfl_xor_sync(kFull, v[j], lanes);
        v[j] = __fmaf_rn(sg, v[j], o);
      }
    }
  }
}

// Swap tile positions 0 and d (d < G) across the team: lane 0 of the team holds
// position 0, lane d / V holds position d.  All lanes of the warp must call this.
template <int V>
__device__ __forceinline__ void team_swap0(float* v, int d, int sub, int team_base_lane) {
  const int dl = d / V, dj = d % V;
  float vd = v[0];
#pragma unroll
  for (int j = 0; j < V; j++)
    if (j == dj) vd = v[j];
  const float x0 = __shfl_sync(kFull, v[0], team_base_lane);
  const float xd = __shfl_sync(kFull, vd, team_base_lane + dl);
  if (d != 0) {
    if (sub == 0) v[0] = xd;
#pragma unroll
    for (int j = 0; j < V; j++)
      if (sub == dl && j == dj) v[j] = x0;
  }
}

// ------------------------------------------------------------------ bounded waits

// Every wait of a kernel on another block or on a bulk copy is bounded in time: it gives
// up after a limit in nanoseconds of the global timer (the kernel parameters carry it;
// kWaitNs by default), sets kStWaitTimeout in the status word and returns, and a wait
// that finds that bit already set returns at once, so that one lost publication costs a
// call one limit, not one limit per later wait.
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool timed_out(const uint32_t* status) {
  return (*reinterpret_cast<const volatile uint32_t*>(status) & kStWaitTimeout) != 0u;
}

// ------------------------------------------------------------------ bulk copies (TMA)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// L2 eviction-priority policies for bulk loads.
__device__ __forceinline__ unsigned long long policy_evict_last() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ unsigned long long policy_evict_normal() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ unsigned long long policy_evict_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// One-dimensional bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          unsigned long long* bar, unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Plain arrival (release at cta scope) on a barrier.
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete.  A bulk copy always completes unless the
// device has faulted; the bound (limit_ns) only keeps a broken device from spinning
// forever.  The clock and the status word are looked at every 256 polls.
__device__ __forceinline__ void mbar_wait(unsigned long long* bar, uint32_t parity,
                                          uint32_t* status, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_ns();
  for (uint32_t n = 1;; n++) {
    if (mbar_try_wait(bar, parity)) return;
    if ((n & 255u) == 0u && (timed_out(status) || global_ns() - t0 > limit_ns)) {
      set_status(status, kStWaitTimeout);
      return;
    }
  }
}

// Wait until *flag >= target (flag written by other blocks with release semantics), at
// most limit_ns; returns false (status bit set) if it gave up or another wait already had.
__device__ __forceinline__ bool wait_counter(const uint32_t* flag, uint32_t target,
                                             uint32_t* status, unsigned long long limit_ns) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v >= target) return true;
    if (timed_out(status) || global_ns() - t0 > limit_ns) {
      set_status(status, kStWaitTimeout);
      return false;
    }
    __nanosleep(64);
  }
}

// ------------------------------------------------------------------ wire-format quantiser
// ("TAH-Quant" §3.4: fixed-size buffer with fp16 metadata.)  The zero is the largest fp16
// value <= the tile minimum, the scale of width b the smallest fp16 value s >= 0 with
// zero + Q_b s >= max (Q_b = 2^b - 1), and the codes use inv = RN(1 / s) (0 when s = 0).

// The largest fp16 value <= mn, as fp32 (exact).
__device__ __forceinline__ float wire_zero(float mn) {
  return __half2float(__float2half_rd(mn));
}

// zero + Q s >= mx, decided exactly in fp32: Q s is exact (8 x 11 bits), TwoSum gives
// zero + Q s = sum + err exactly with sum = RN(zero + Q s) and |err| <= ulp(sum) / 2, and
// since sum and mx are floats the inequality holds iff sum > mx, or sum == mx and
// err >= 0.  (An infinite zero gives NaN terms: not covered, as no finite scale covers.)
__device__ __forceinline__ bool wire_covers(float zero, float Q, float s, float mx) {
  const float a = __fmul_rn(Q, s);
  const float sum = __fadd_rn(a, zero);
  const float bb = __fsub_rn(sum, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(sum, bb)), __fsub_rn(zero, bb));
  return sum > mx || (sum == mx && err >= 0.0f);
}

// The smallest fp16 scale covering [zero, mx] at Q steps, as fp32 (exact; +inf when no
// finite fp16 value does).  RU(RU(mx - zero) / Q) rounded up to fp16 is never below the
// answer and at most one fp16 step above it (the fp32 over-estimate is under 2^-22
// relative, the fp16 spacing 2^-10 relative or 2^-24 absolute), so an exact test of the
// fp16 value below settles it.
__device__ __forceinline__ float wire_scale(float zero, float mx, float Q) {
  if (!(mx > zero)) return 0.0f;
  uint16_t c = __half_as_ushort(__float2half_ru(__fdiv_ru(__fsub_ru(mx, zero), Q)));
  if (c > 0x7C00u) c = 0x7C00u;  // NaN from out-of-range input: treated as +inf
#pragma unroll
  for (int step = 0; step < 2; step++) {
    const uint16_t below = (uint16_t)(c - 1u);
    if (c > 0u && wire_covers(zero, Q, __half2float(__ushort_as_half(below)), mx)) c = below;
  }
  return __half2float(__ushort_as_half(c));
}

// RN(1 / s), or 0 for a zero scale.
__device__ __forceinline__ float wire_inv(float s) { return s > 0.0f ? __frcp_rn(s) : 0.0f; }

}  // namespace tahq
