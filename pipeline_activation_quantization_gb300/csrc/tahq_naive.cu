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
// A warp takes four consecutive tiles at a time (G = 32, 64 or 128: V = G / 32 values a
// lane, positions lane * V ...), every load of the four in flight first.  Encode stages a
// tile's codes in shared memory and writes each 32-bit word of the slot from the codes it
// covers; decode extracts each code from the one or two words it spans.  Both are streams
// bound by HBM (4 bytes read and b / 8 written an element, or the reverse).
#include <algorithm>
#include <cmath>

#include "../../include/tahq.h"
#include "tahq_device.cuh"

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

template <int G>
__global__ void __launch_bounds__(32 * kNaiveWarps) k_naive_decode(const uint8_t* __restrict__ codes,
                                                                   const float* __restrict__ scales,
                                                                   const float* __restrict__ zeros,
                                                                   long long n_tiles, int b, float c,
                                                                   float* out) {
  constexpr int V = G / 32;
  constexpr int kDecTiles = 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t mask = (1u << b) - 1u;
  const float inv_c = 1.0f / c;  // c is a power of two: RN(y / c) = y * (1 / c)
  const long long stride = (long long)gridDim.x * kNaiveWarps * kDecTiles;
  for (long long t0 = ((long long)blockIdx.x * kNaiveWarps + warp) * kDecTiles; t0 < n_tiles;
       t0 += stride) {
    const int nu = (int)min((long long)kDecTiles, n_tiles - t0);
    uint32_t qv[kDecTiles][V];
    float sc[kDecTiles], z[kDecTiles];
#pragma unroll
    for (int u = 0; u < kDecTiles; u++) {
      if (u >= nu) break;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(codes + (t0 + u) * (long long)(G * b / 8));
      sc[u] = __ldg(scales + t0 + u);
      z[u] = __ldg(zeros + t0 + u);
#pragma unroll
      for (int j = 0; j < V; j++) {
        const int bit = (lane * V + j) * b, w = bit >> 5, sh = bit & 31;
        uint32_t q = __ldg(src + w) >> sh;
        if (sh + b > 32) q |= __ldg(src + w + 1) << (32 - sh);
        qv[u][j] = q & mask;
      }
    }
#pragma unroll
    for (int u = 0; u < kDecTiles; u++) {
      if (u >= nu) break;
      float y[V];
#pragma unroll
      for (int j = 0; j < V; j++) y[j] = __fmul_rn(__fmaf_rn((float)qv[u][j], sc[u], z[u]), inv_c);
      float* dst = out + (t0 + u) * G + lane * V;
      if constexpr (V == 4) {
        __stcs(reinterpret_cast<float4*>(dst), make_float4(y[0], y[1], y[2], y[3]));
      } else if constexpr (V == 2) {
        __stcs(reinterpret_cast<float2*>(dst), make_float2(y[0], y[1]));
      } else {
        __stcs(dst, y[0]);
      }
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
  const int blocks = naive_blocks(n);
  if (blocks <= 0) return TAHQ_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
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
  const int blocks = naive_blocks(n);
  if (blocks <= 0) return TAHQ_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const dim3 grid(blocks), block(32 * kNaiveWarps);
  if (tile == 32) k_naive_decode<32><<<grid, block, 0, cs>>>(codes, scales, zeros, n, bits, scale_c, out);
  if (tile == 64) k_naive_decode<64><<<grid, block, 0, cs>>>(codes, scales, zeros, n, bits, scale_c, out);
  if (tile == 128) k_naive_decode<128><<<grid, block, 0, cs>>>(codes, scales, zeros, n, bits, scale_c, out);
  return cudaGetLastError() == cudaSuccess ? TAHQ_OK : TAHQ_ERR_CUDA;
}
