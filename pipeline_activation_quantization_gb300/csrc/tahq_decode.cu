// tahq_decode.cu -- decode kernel of the TAH-Quant activation codec for sm_103a.
//
// "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over Slow
// Network" (arXiv 2506.01352v2), §3.3 last paragraph ("apply H_G^T to the de-quantized
// values") and Algorithm 1 step 5 (stage b de-quantises what it received); the stream
// layout is §3.4's contiguous uint8 buffer with slots in tile order.
//
// One block decodes a chunk of consecutive tiles: slot offsets come from the running sum
// of tile*bits/8 (block scan + decoupled look-back over earlier chunks), the chunk's
// bytes are staged in shared memory with 16-byte loads, and each team of G/8 lanes
// unpacks, de-quantises (fma(q, scale, zero)), inverse-transforms flagged tiles
// (Hadamard, x 1/sqrt(h), swap positions 0 and d) and stores 8 floats per lane.
#include <algorithm>

#include "tahq_device.cuh"
#include "tahq_launch.h"

namespace tahq {

template <int kThreads>
__device__ __forceinline__ uint32_t block_exclusive_scan_dec(uint32_t v, uint32_t& total,
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

template <int G>
struct DecCfg {
  static constexpr int V = 8;
  using Gm = Geom<V, G>;
  static constexpr int kThreads = 256;
  static constexpr int kSteps = 8;
  static constexpr int CH = 8 * kSteps * Gm::TPW;             // tiles per chunk
  static constexpr int kPer = (CH + kThreads - 1) / kThreads;
  static constexpr int kStageBytes = CH * G + 48;              // b <= 8, plus pad
};

template <int G>
__global__ void __launch_bounds__(256) k_decode(DecodeArgs a, long long n_chunks) {
  using Cf = DecCfg<G>;
  constexpr int V = Cf::V, L = Cf::Gm::L, TPW = Cf::Gm::TPW, CH = Cf::CH;
  __shared__ __align__(16) uint32_t s_stage[Cf::kStageBytes / 4];
  __shared__ uint16_t s_off[CH];
  __shared__ uint8_t s_bits[CH];
  __shared__ uint32_t s_warp[9];
  __shared__ long long s_c;
  __shared__ unsigned long long s_base;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L;
  const unsigned long long limit = a.codes_bytes;
  const uint8_t* sb = reinterpret_cast<const uint8_t*>(s_stage);

  for (;;) {
    if (threadIdx.x == 0) s_c = (long long)atomicAdd(a.ticket, 1u);
    __syncthreads();
    const long long c = s_c;
    if (c >= n_chunks) break;
    const long long t0 = c * CH;
    const int nt = (int)min((long long)CH, a.n_tiles - t0);

    // 1. slot sizes of this chunk and their exclusive running sum
    uint32_t mine = 0u;
    uint8_t bl[Cf::kPer];
#pragma unroll
    for (int j = 0; j < Cf::kPer; j++) {
      const int k = threadIdx.x * Cf::kPer + j;
      bl[j] = 0;
      if (k < nt) {
        int b = a.bits[t0 + k];
        if (b < 1 || b > 8) {
          set_status(a.status, kStBadBits);
          b = 0;
        }
        bl[j] = (uint8_t)b;
        mine += (uint32_t)(G * b / 8);
      }
    }
    uint32_t chunk_bytes;
    uint32_t off = block_exclusive_scan_dec<256>(mine, chunk_bytes, s_warp);
#pragma unroll
    for (int j = 0; j < Cf::kPer; j++) {
      const int k = threadIdx.x * Cf::kPer + j;
      if (k < nt) {
        s_bits[k] = bl[j];
        s_off[k] = (uint16_t)off;
        off += (uint32_t)(G * bl[j] / 8);
      }
    }

    // 2. byte offset of the chunk: look-back over all earlier chunks
    if (threadIdx.x == 0) {
      unsigned long long prefix = 0ull;
      if (c == 0) {
        st_release_u64(&a.lookback[c], kLbPre | (unsigned long long)chunk_bytes);
      } else {
        st_release_u64(&a.lookback[c], kLbAgg | (unsigned long long)chunk_bytes);
        prefix = lookback_prefix(a.lookback, c, 0, a.status);
        st_release_u64(&a.lookback[c], kLbPre | (prefix + chunk_bytes));
      }
      if (prefix + chunk_bytes > limit) set_status(a.status, kStOverrun);
      s_base = prefix;
    }
    __syncthreads();
    const unsigned long long base = s_base;
    const int pad = (int)(base & 15ull);

    // 3. stage [base, base + chunk_bytes) in shared memory, never reading past codes_bytes
    const unsigned long long a0 = base - (unsigned long long)pad;
    const int n16 = (pad + (int)chunk_bytes + 15) / 16;
    for (int w16 = threadIdx.x; w16 < n16; w16 += Cf::kThreads) {
      const unsigned long long gb = a0 + 16ull * w16;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (gb + 16ull <= limit) {
        w = __ldg(reinterpret_cast<const uint4*>(a.codes + gb));
      } else {
        uint32_t tmp[4] = {0u, 0u, 0u, 0u};
        for (int k = 0; k < 16; k++)
          if (gb + k < limit) tmp[k >> 2] |= (uint32_t)a.codes[gb + k] << (8 * (k & 3));
        w = make_uint4(tmp[0], tmp[1], tmp[2], tmp[3]);
      }
      reinterpret_cast<uint4*>(s_stage)[w16] = w;
    }
    __syncthreads();

    // 4. per tile: unpack, de-quantise, inverse transform, store
#pragma unroll 1
    for (int s = 0; s < Cf::kSteps; s++) {
      const int kt = (s * 8 + warp) * TPW + team;
      const bool valid = kt < nt;
      const long long t = t0 + kt;
      int b = 0, piv = 0xFF;
      float sc = 0.0f, mn = 0.0f;
      bool ok = false;
      if (valid) {
        b = s_bits[kt];
        piv = a.pivots[t];
        sc = a.scales[t];
        mn = a.zeros[t];
        ok = b > 0 && base + s_off[kt] + (unsigned long long)(G * b / 8) <= limit;
        if (piv != 0xFF && piv >= G) {
          if (sub == 0) set_status(a.status, kStBadBits);
          ok = false;
        }
      }
      unsigned long long acc = 0ull;
      if (ok) {
        const int start = pad + (int)s_off[kt] + sub * b;  // V = 8 codes = b whole bytes
        for (int k = 0; k < b; k++) acc |= (unsigned long long)sb[start + k] << (8 * k);
      }
      const uint32_t qmask = (b >= 1) ? ((1u << b) - 1u) : 0u;
      float v[V];
#pragma unroll
      for (int j = 0; j < V; j++) {
        const uint32_t q = (uint32_t)(acc >> (j * b)) & qmask;
        v[j] = __fmaf_rn(__uint2float_rn(q), sc, mn);
      }
      const bool flag = ok && piv != 0xFF;
      if (__any_sync(kFull, flag)) {
        float w[V];
#pragma unroll
        for (int j = 0; j < V; j++) w[j] = v[j];
        team_fwht<V, L>(w, a.h, sub);
#pragma unroll
        for (int j = 0; j < V; j++) w[j] = __fmul_rn(w[j], a.c_h);
        team_swap0<V>(w, flag ? piv : 0, sub, lane - sub);
        if (flag) {
#pragma unroll
          for (int j = 0; j < V; j++) v[j] = w[j];
        }
      }
      if (!ok) {
#pragma unroll
        for (int j = 0; j < V; j++) v[j] = 0.0f;
      }
      if (valid) {
        float4* o = reinterpret_cast<float4*>(a.out + t * G + sub * V);
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
    __syncthreads();
  }
}

long long decode_chunks(int G, long long n_tiles) {
  const long long ch = 8ll * 8 * (32 / (G / 8));
  return (n_tiles + ch - 1) / ch;
}

template <int G>
static cudaError_t run_decode(const DecodeArgs& a, cudaStream_t st) {
  const long long n_chunks = decode_chunks(G, a.n_tiles);
  const int blocks = (int)std::max<long long>(1, std::min<long long>((long long)a.num_sms * 6, n_chunks));
  k_decode<G><<<blocks, 256, 0, st>>>(a, n_chunks);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  switch (a.G) {
    case 8: return run_decode<8>(a, st);
    case 16: return run_decode<16>(a, st);
    case 32: return run_decode<32>(a, st);
    case 64: return run_decode<64>(a, st);
    case 128: return run_decode<128>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tahq
