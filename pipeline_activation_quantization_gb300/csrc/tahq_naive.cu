// tahq_naive.cu -- the backward pass's fixed-point gradient codec and its C entry points.
//
// "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over Slow
// Network", §3.5 and Algorithm 1: the second stage sends a fixed-point quantisation of
// the gradient with respect to the activations back to the first (6-8 bits; 10 after the
// NaN event of Appendix H); Appendix H eq. (24): g_hat = Q(c g) / c.  The quantiser is
// the §3.3 asymmetric uniform one at a single width b (1..16) on tiles of G consecutive
// channels of a token, with no bit allocation and no outlier transform: per tile
// mn = min, mx = max, D = RN(mx - mn), inv = RN(Q / D), scale = RN(D / Q) (both 0 when
// D < max(2^-120, 2^(b - 126))), q = RNE(RN(v - mn) * inv) with the product exact,
// v = RN(c g); codes
// packed least significant bit first at b bits; decode RN(fma(q, scale, mn) / c).  c is a
// power of two, so the scaling is exact unless c g leaves the normal float range.
//
// Encode: a warp takes eight consecutive tiles at a time (G = 32, 64 or 128: V = G / 32
// values a lane, positions lane * V ...), every load in flight first; it stores a lane's
// codes straight from registers when they make whole bytes, else composes the slot's
// words in shared memory.  Decode: a thread takes groups of 4 consecutive values, a warp
// 32 consecutive groups.  Both are streams bound by HBM (4 bytes read and b / 8 written an
// element, or the reverse).
#include <algorithm>
#include <cmath>

#include "../../include/tahq.h"
#include "tahq_device.cuh"
#include "tahq_tile.cuh"

namespace tahq {
namespace {

constexpr int kNaiveWarps = 8;
constexpr int kNaiveTiles = 8;  // tiles a warp has in flight

// The range below which a tile quantises to its minimum: max(2^-120, 2^(b - 126)), so that
// Q / D stays finite and D / Q a normal float at every width up to 16.
__device__ __forceinline__ float naive_cutoff(int b) {
  return __uint_as_float((uint32_t)(127 + max(-120, b - 126)) << 23);
}

__device__ __forceinline__ float warp_min(float x) {
  float r;
  asm("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

template <int V>
__device__ __forceinline__ void load_v(const float* src, float* v) {
  if constexpr (V == 4) {
    const float4 q = __ldcs(reinterpret_cast<const float4*>(src));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  } else if constexpr (V == 2) {
    const float2 q = __ldcs(reinterpret_cast<const float2*>(src));
    v[0] = q.x; v[1] = q.y;
  } else {
    v[0] = __ldcs(src);
  }
}

// One warp takes kNaiveTiles consecutive tiles at a time (every load of the group in
// flight before any arithmetic), lane l holding values l V .. l V + V - 1 of each tile.
// The codes of a tile are staged in shared memory; lane w then writes word w of the slot
// (bits [32 w, 32 w + 32)) from the codes it covers.
template <int G>
__global__ void __launch_bounds__(32 * kNaiveWarps) k_naive_encode(const float* __restrict__ g,
                                                                   long long n_tiles, int b,
                                                                   float c, uint8_t* codes,
                                                                   float* scales, float* zeros) {
  constexpr int V = G / 32;
  __shared__ uint16_t sq[kNaiveWarps][kNaiveTiles][G];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t Q = (1u << b) - 1u;
  const float Qf = (float)Q, cut = naive_cutoff(b);
  const int words = G * b / 32;  // the tile's slot, whole 32-bit words (G >= 32)
  // a lane's V codes fill 1, 2, 4 or 8 whole bytes: stored straight from registers
  const int fbytes = V * b / 8;
  const bool direct = (V * b) % 8 == 0 && (fbytes == 1 || fbytes == 2 || fbytes == 4 || fbytes == 8);
  const long long stride = (long long)gridDim.x * kNaiveWarps * kNaiveTiles;
  for (long long t0 = ((long long)blockIdx.x * kNaiveWarps + warp) * kNaiveTiles; t0 < n_tiles;
       t0 += stride) {
    const int nu = (int)min((long long)kNaiveTiles, n_tiles - t0);
    float v[kNaiveTiles][V];
#pragma unroll
    for (int u = 0; u < kNaiveTiles; u++)
      if (u < nu) load_v<V>(g + (t0 + u) * G + lane * V, v[u]);
#pragma unroll
    for (int u = 0; u < kNaiveTiles; u++) {
      if (u >= nu) break;  // warp-uniform
      float mn, mx;
#pragma unroll
      for (int j = 0; j < V; j++) {
        v[u][j] = __fmul_rn(c, v[u][j]);
        mn = j ? fminf(mn, v[u][j]) : v[u][j];
        mx = j ? fmaxf(mx, v[u][j]) : v[u][j];
      }
      mn = warp_min(mn);
      mx = warp_max(mx);
      const float D = __fsub_rn(mx, mn);
      const bool live = D >= cut;
      const float inv = live ? __fdiv_rn(Qf, D) : 0.0f;
      unsigned long long field = 0ull;
#pragma unroll
      for (int j = 0; j < V; j++) {
        uint32_t q = __float_as_uint(__fmaf_rn(__fsub_rn(v[u][j], mn), inv, 12582912.0f)) - 0x4B400000u;
        q = live ? min(q, Q) : 0u;
        if (direct) {
          field |= (unsigned long long)q << (j * b);
        } else {
          sq[warp][u][lane * V + j] = (uint16_t)q;
        }
      }
      if (direct) {  // the lane's V codes are whole bytes: one store
        unsigned char* dst = codes + (t0 + u) * (long long)(G * b / 8) + lane * fbytes;
        if (fbytes == 8) *reinterpret_cast<unsigned long long*>(dst) = field;
        else if (fbytes == 4) *reinterpret_cast<uint32_t*>(dst) = (uint32_t)field;
        else if (fbytes == 2) *reinterpret_cast<uint16_t*>(dst) = (uint16_t)field;
        else *dst = (unsigned char)field;
      }
      if (lane == 0) {
        scales[t0 + u] = live ? __fdiv_rn(D, Qf) : 0.0f;
        zeros[t0 + u] = __fadd_rn(mn, 0.0f);  // a zero minimum as +0
      }
    }
    if (direct) continue;  // warp-uniform
    __syncwarp();
#pragma unroll
    for (int u = 0; u < kNaiveTiles; u++) {
      if (u >= nu) break;
      uint32_t* dst = reinterpret_cast<uint32_t*>(codes + (t0 + u) * (long long)(G * b / 8));
      for (int w = lane; w < words; w += 32) {
        int k = (32 * w) / b;
        int off = k * b - 32 * w;  // where code k starts, relative to the word (<= 0)
        uint32_t acc = 0u;
        for (; off < 32; ++k, off += b) {
          const uint32_t q = sq[warp][u][k];
          acc |= off >= 0 ? (q << off) : (q >> (-off));
        }
        dst[w] = acc;
      }
    }
    __syncwarp();
  }
}

// Encode at widths B = 4, 8, 16, where 16 codes make whole 8-, 16- or 32-byte fields:
// thread i takes groups of 16 consecutive values (group i, i + S, ...; kEncGroups in
// flight), a tile is G / 16 consecutive lanes (team reductions for its range), and a
// lane stores its 16 codes with one or two vector stores.
constexpr int kEncGroups = 2;
constexpr int kEncBlockThreads = 256;

template <int G, int B>
__global__ void __launch_bounds__(kEncBlockThreads) k_naive_encode16(const float* __restrict__ g,
                                                                     long long n_tiles, float c,
                                                                     uint8_t* codes, float* scales,
                                                                     float* zeros) {
  constexpr int L = G / 16;  // lanes a tile
  constexpr uint32_t Q = (1u << B) - 1u;
  const float Qf = (float)Q, cut = naive_cutoff(B);
  const int lane = threadIdx.x & 31, sub = lane % L;
  const long long n16 = n_tiles * L;  // groups of 16 values
  const long long S = (long long)gridDim.x * kEncBlockThreads;  // a multiple of 32
  for (long long i0 = (long long)blockIdx.x * kEncBlockThreads + threadIdx.x; i0 - lane < n16;
       i0 += S * kEncGroups) {  // the loop condition is warp-uniform
    float v[kEncGroups][16];
#pragma unroll
    for (int u = 0; u < kEncGroups; u++) {
      const long long i = i0 + u * S;
      const float4* src = reinterpret_cast<const float4*>(g) + 4 * (i < n16 ? i : 0);
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const float4 q = __ldcs(src + k);
        v[u][4 * k] = q.x;
        v[u][4 * k + 1] = q.y;
        v[u][4 * k + 2] = q.z;
        v[u][4 * k + 3] = q.w;
      }
    }
#pragma unroll
    for (int u = 0; u < kEncGroups; u++) {
      const long long i = i0 + u * S;
      float mn, mx;
#pragma unroll
      for (int j = 0; j < 16; j++) {
        v[u][j] = __fmul_rn(c, v[u][j]);
        mn = j ? fminf(mn, v[u][j]) : v[u][j];
        mx = j ? fmaxf(mx, v[u][j]) : v[u][j];
      }
#pragma unroll
      for (int o = 1; o < L; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      }
      const float D = __fsub_rn(mx, mn);
      const bool live = D >= cut;
      // lane 0 of the tile: Q / D; lane 1: D / Q (the scale)
      const float r = (sub & 1) ? __fdiv_rn(D, Qf) : __fdiv_rn(Qf, D);
      const float o = __shfl_xor_sync(kFull, r, 1);
      const float inv = live ? ((sub & 1) ? o : r) : 0.0f;
      const float scale = live ? ((sub & 1) ? r : o) : 0.0f;
      uint32_t w[B / 2];  // 16 codes of B bits
#pragma unroll
      for (int k = 0; k < B / 2; k++) w[k] = 0u;
#pragma unroll
      for (int j = 0; j < 16; j++) {
        uint32_t q = __float_as_uint(__fmaf_rn(__fsub_rn(v[u][j], mn), inv, 12582912.0f)) - 0x4B400000u;
        q = live ? min(q, Q) : 0u;
        w[(j * B) / 32] |= q << ((j * B) % 32);
      }
      if (i < n16) {
        uint8_t* dst = codes + i * (2 * B);
        if constexpr (B == 4) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
        } else {
#pragma unroll
          for (int k = 0; k < B / 2; k += 4)
            *reinterpret_cast<uint4*>(dst + 4 * k) = make_uint4(w[k], w[k + 1], w[k + 2], w[k + 3]);
        }
        if (sub == 0) {
          const long long t = i / L;
          scales[t] = scale;
          zeros[t] = __fadd_rn(mn, 0.0f);  // a zero minimum as +0
        }
      }
    }
  }
}

// Decode: thread i takes groups of 4 consecutive values (group i, i + S, ..., S the grid's
// threads; kDecGroups of them in flight), so that a warp's stores are 512 contiguous
// bytes and its code loads 32 consecutive words or so.  The 4 codes of group k start at
// bit 4 k b: one word at b = 8, else a 64-bit window of up to three words (b <= 16).
constexpr int kDecGroups = 4;
constexpr int kDecBlockThreads = 256;

template <int G>
__global__ void __launch_bounds__(kDecBlockThreads) k_naive_decode(const uint8_t* __restrict__ codes,
                                                                   const float* __restrict__ scales,
                                                                   const float* __restrict__ zeros,
                                                                   long long n_tiles, int b, float c,
                                                                   float* out) {
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes);
  const long long n4 = n_tiles * (G / 4);                    // groups of 4 values
  const long long n_words = (n_tiles * G * (long long)b + 31) / 32;
  const uint32_t mask = (1u << b) - 1u;
  const float inv_c = 1.0f / c;  // c is a power of two: RN(y / c) = y * (1 / c)
  const float2 ic2 = make_float2(inv_c, inv_c), m2 = make_float2(-8388608.0f, -8388608.0f);
  const long long S = (long long)gridDim.x * kDecBlockThreads;
  for (long long i0 = (long long)blockIdx.x * kDecBlockThreads + threadIdx.x; i0 < n4;
       i0 += S * kDecGroups) {
    unsigned long long v64[kDecGroups];
    float sc[kDecGroups], z[kDecGroups];
#pragma unroll
    for (int u = 0; u < kDecGroups; u++) {
      const long long i = i0 + u * S;
      v64[u] = 0ull;
      sc[u] = z[u] = 0.0f;
      if (i < n4) {
        const long long t = i / (G / 4);
        sc[u] = __ldg(scales + t);
        z[u] = __ldg(zeros + t);
        if (b == 8) {
          v64[u] = __ldg(cw + i);
        } else {
          const long long bit = i * 4 * (long long)b, w = bit >> 5;
          const int sh = (int)(bit & 31);
          const uint32_t w0 = __ldg(cw + w);
          const uint32_t w1 = w + 1 < n_words ? __ldg(cw + w + 1) : 0u;
          const uint32_t w2 = (sh + 4 * b > 64 && w + 2 < n_words) ? __ldg(cw + w + 2) : 0u;
          v64[u] = ((unsigned long long)__funnelshift_r(w1, w2, sh) << 32) | __funnelshift_r(w0, w1, sh);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kDecGroups; u++) {
      const long long i = i0 + u * S;
      if (i >= n4) break;
      const float2 s2 = make_float2(sc[u], sc[u]), z2 = make_float2(z[u], z[u]);
      float y[4];
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        const uint32_t c0 = (uint32_t)(v64[u] >> (j * b)) & mask;
        const uint32_t c1 = (uint32_t)(v64[u] >> ((j + 1) * b)) & mask;
        // (float)q exactly: the bits 0x4B000000 | q are 2^23 + q
        const float2 qf = add2(make_float2(__uint_as_float(0x4B000000u | c0),
                                           __uint_as_float(0x4B000000u | c1)), m2);
        const float2 r = fma2(qf, s2, z2);
        y[j] = __fmul_rn(r.x, ic2.x);
        y[j + 1] = __fmul_rn(r.y, ic2.y);
      }
      __stcs(reinterpret_cast<float4*>(out) + i, make_float4(y[0], y[1], y[2], y[3]));
    }
  }
}

int naive_blocks(long long n_tiles) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 0;
  const long long per = kNaiveWarps * kNaiveTiles;
  const long long want = (n_tiles + per - 1) / per;
  return (int)std::max<long long>(1, std::min<long long>(want, (long long)sms * 8));
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape and argument checks shared by the three entry points.
tahq_status naive_check(int64_t tokens, int64_t channels, int tile, int bits, float c) {
  if (tokens < 0 || channels <= 0 || tile <= 0 || bits < 1 || bits > 16) return TAHQ_ERR_ARG;
  if (channels % tile) return TAHQ_ERR_ARG;
  int e = 0;
  if (!(c > 0.0f) || !std::isfinite(c) || std::frexp(c, &e) != 0.5f) return TAHQ_ERR_ARG;
  if (tile != 32 && tile != 64 && tile != 128) return TAHQ_ERR_UNSUPPORTED;
  return TAHQ_OK;
}

}  // namespace
}  // namespace tahq

extern "C" size_t tahq_naive_codes_bytes(int64_t tokens, int64_t channels, int tile, int bits) {
  if (tahq::naive_check(tokens, channels, tile, bits, 1.0f) != TAHQ_OK) return 0;
  return (size_t)(tokens * (channels / tile)) * (size_t)(tile * bits / 8);
}

extern "C" tahq_status tahq_naive_encode(const float* grad, int64_t tokens, int64_t channels,
                                         int tile, int bits, float scale_c, uint8_t* codes,
                                         float* scales, float* zeros, void* stream) {
  using namespace tahq;
  const tahq_status st = naive_check(tokens, channels, tile, bits, scale_c);
  if (st != TAHQ_OK) return st;
  const long long n = tokens * (channels / tile);
  if (n == 0) return TAHQ_OK;
  if (!grad || !codes || !scales || !zeros) return TAHQ_ERR_ARG;
  if (!aligned_to(grad, 16) || !aligned_to(codes, 16) || !aligned_to(scales, 4) ||
      !aligned_to(zeros, 4))
    return TAHQ_ERR_ARG;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (bits == 4 || bits == 8 || bits == 16) {  // 16 codes a lane make whole vector stores
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return TAHQ_ERR_CUDA;
    const long long groups = n * (tile / 16), per = (long long)kEncBlockThreads * kEncGroups;
    const int blocks16 = (int)std::max<long long>(1, std::min<long long>((groups + per - 1) / per, 8ll * sms));
    using EncFn = void (*)(const float*, long long, float, uint8_t*, float*, float*);
    EncFn k = nullptr;
#define TAHQ_NAIVE16(GG)                                                                        \
    if (tile == GG) k = bits == 4 ? k_naive_encode16<GG, 4> : bits == 8 ? k_naive_encode16<GG, 8> \
                                                                        : k_naive_encode16<GG, 16>;
    TAHQ_NAIVE16(32)
    TAHQ_NAIVE16(64)
    TAHQ_NAIVE16(128)
#undef TAHQ_NAIVE16
    k<<<blocks16, kEncBlockThreads, 0, cs>>>(grad, n, scale_c, codes, scales, zeros);
    return cudaGetLastError() == cudaSuccess ? TAHQ_OK : TAHQ_ERR_CUDA;
  }
  const int blocks = naive_blocks(n);
  if (blocks <= 0) return TAHQ_ERR_CUDA;
  const dim3 grid(blocks), block(32 * kNaiveWarps);
  if (tile == 32) k_naive_encode<32><<<grid, block, 0, cs>>>(grad, n, bits, scale_c, codes, scales, zeros);
  if (tile == 64) k_naive_encode<64><<<grid, block, 0, cs>>>(grad, n, bits, scale_c, codes, scales, zeros);
  if (tile == 128) k_naive_encode<128><<<grid, block, 0, cs>>>(grad, n, bits, scale_c, codes, scales, zeros);
  return cudaGetLastError() == cudaSuccess ? TAHQ_OK : TAHQ_ERR_CUDA;
}

extern "C" tahq_status tahq_naive_decode(const uint8_t* codes, const float* scales,
                                         const float* zeros, int64_t tokens, int64_t channels,
                                         int tile, int bits, float scale_c, float* out,
                                         void* stream) {
  using namespace tahq;
  const tahq_status st = naive_check(tokens, channels, tile, bits, scale_c);
  if (st != TAHQ_OK) return st;
  const long long n = tokens * (channels / tile);
  if (n == 0) return TAHQ_OK;
  if (!codes || !scales || !zeros || !out) return TAHQ_ERR_ARG;
  if (!aligned_to(codes, 16) || !aligned_to(out, 16) || !aligned_to(scales, 4) ||
      !aligned_to(zeros, 4))
    return TAHQ_ERR_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return TAHQ_ERR_CUDA;
  const long long groups = n * (tile / 4), per = (long long)kDecBlockThreads * kDecGroups;
  const int blocks = (int)std::max<long long>(1, std::min<long long>((groups + per - 1) / per, 8ll * sms));
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const dim3 grid(blocks), block(kDecBlockThreads);
  if (tile == 32) k_naive_decode<32><<<grid, block, 0, cs>>>(codes, scales, zeros, n, bits, scale_c, out);
  if (tile == 64) k_naive_decode<64><<<grid, block, 0, cs>>>(codes, scales, zeros, n, bits, scale_c, out);
  if (tile == 128) k_naive_decode<128><<<grid, block, 0, cs>>>(codes, scales, zeros, n, bits, scale_c, out);
  return cudaGetLastError() == cudaSuccess ? TAHQ_OK : TAHQ_ERR_CUDA;
}
