// tahq_decode.cu -- decode kernel of the TAH-Quant activation codec for sm_103a.
//
// "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over Slow
// Network" (arXiv 2506.01352v2), §3.3 last paragraph ("apply H_G^T to the de-quantized
// values") and Algorithm 1 step 5 (stage b de-quantises what it received); the stream
// layout is §3.4's contiguous uint8 buffer with slots in tile order.
//
// Two launches.  k_dec_totals: the slot bytes of every chunk of consecutive tiles (one
// warp per chunk, from the bit widths) and their running sum inside each block of 8
// chunks; the last of its blocks to finish turns the block totals into stream offsets.
// k_decode (a dependent launch): blocks take chunks in a grid-stride
// loop; a block scan gives each tile's offset inside its chunk, the chunk's bytes and
// metadata are staged in shared memory, and each team of G/8 lanes then
// unpacks 8 codes per lane, de-quantises (fma(q, scale, zero)) and stores 8 floats per
// lane.  Transformed tiles (pivot != 0xFF) are collected per warp and handled in a
// second, compacted pass: Hadamard per hblock, x 1/sqrt(h), swap positions 0 and d.
#include <algorithm>

#include "tahq_device.cuh"
#include "tahq_launch.h"

namespace tahq {

template <int kN>
__device__ __forceinline__ uint32_t block_exclusive_scan_dec(uint32_t v, uint32_t& total,
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

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;

template <int G>
struct DecCfg {
  static constexpr int V = 8;  // codes / output floats per lane
  using Gm = Geom<V, G>;
  static constexpr int L = Gm::L, TPW = Gm::TPW;
  static constexpr int kSteps = 8;
  static constexpr int CH = kDecWarps * kSteps * TPW;  // tiles per chunk
  static constexpr int NS = kSteps * TPW;              // tiles per warp
  static constexpr int kPer = (CH + kDecThreads - 1) / kDecThreads;
  static constexpr int kStage = CH * G + 64;           // b <= 8, plus pad and slack
  // blocks per SM the registers must allow (six fit the shared memory; the prefetched
  // metadata of 8 tiles a thread at G = 8 needs more registers than six leave)
  static constexpr int kMinBlocks = G >= 16 ? 6 : 4;
};

template <int G>
struct alignas(16) DecSmem {
  using C = DecCfg<G>;
  uint32_t stage[2][C::kStage / 4];  // this chunk's bytes and the next one's, in flight
  float scale[C::CH], zero[C::CH];
  uint16_t off[C::CH];
  uint16_t flagged[C::CH];
  uint8_t bits[C::CH], piv[C::CH];
  uint32_t scan[kDecWarps + 1];
};

// Bytes of all slots of chunk c (bit widths outside 1..8 count as 0, as in the scan).
template <int G>
__device__ __forceinline__ uint32_t warp_chunk_bytes(const uint8_t* bits, long long n_tiles,
                                                     long long c) {
  constexpr int CH = DecCfg<G>::CH;
  const long long t0 = c * CH;
  const int nt = (int)min((long long)CH, n_tiles - t0);
  const int lane = threadIdx.x & 31;
  uint32_t sum = 0;
  for (int k = lane; k < nt; k += 32) {
    const int b = bits[t0 + k];
    sum += (b >= 1 && b <= 8) ? (uint32_t)(G * b / 8) : 0u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  return sum;
}

// Packed ops on register pairs (mov.b64 {lo, hi}): (q0, q1) * s + z componentwise, each an
// fma rounded once (as fmaf); and the packed add.
__device__ __forceinline__ float2 fma2(float2 q, float2 s, float2 z) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(q.x), "f"(q.y), "f"(s.x), "f"(s.y), "f"(z.x), "f"(z.y));
  return d;
}
__device__ __forceinline__ float2 addp(float2 a, float2 b) {
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

// The lane's 8 codes of b bits (b whole bytes at stage byte `start`), de-quantised.  Up
// to 4 bits the 8 codes sit in one 32-bit word.
__device__ __forceinline__ void dequant8(const uint32_t* sw, int start, int b, float sc, float mn,
                                         float* v) {
  const int q = start >> 2, sh = (start & 3) * 8;
  const uint32_t w0 = sw[q], w1 = sw[q + 1];
  const uint32_t lo = __funnelshift_r(w0, w1, sh);
  const uint32_t mask = (1u << b) - 1u;
  const float2 s2 = make_float2(sc, sc), z2 = make_float2(mn, mn);
  const float2 m2 = make_float2(-8388608.0f, -8388608.0f);
  if (b <= 4) {
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const uint32_t c0 = (lo >> (j * b)) & mask;
      const uint32_t c1 = (lo >> ((j + 1) * b)) & mask;
      const float2 qf = addp(make_float2(__uint_as_float(0x4B000000u | c0),
                                         __uint_as_float(0x4B000000u | c1)), m2);
      const float2 r = fma2(qf, s2, z2);
      v[j] = r.x;
      v[j + 1] = r.y;
    }
    return;
  }
  const uint32_t hi = __funnelshift_r(w1, sw[q + 2], sh);
  const unsigned long long acc = ((unsigned long long)hi << 32) | lo;
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const uint32_t c0 = (uint32_t)(acc >> (j * b)) & mask;
    const uint32_t c1 = (uint32_t)(acc >> ((j + 1) * b)) & mask;
    // (float)q exactly: the bits 0x4B000000 | q are 2^23 + q
    const float2 qf = addp(make_float2(__uint_as_float(0x4B000000u | c0),
                                       __uint_as_float(0x4B000000u | c1)), m2);
    const float2 r = fma2(qf, s2, z2);
    v[j] = r.x;
    v[j + 1] = r.y;
  }
}

// dequant8 for b <= 4 (the 8 codes in one word), for warps whose tiles all have b <= 4.
__device__ __forceinline__ void dequant8_le4(const uint32_t* sw, int start, int b, float sc,
                                             float mn, float* v) {
  const int q = start >> 2, sh = (start & 3) * 8;
  const uint32_t lo = __funnelshift_r(sw[q], sw[q + 1], sh);
  const uint32_t mask = (1u << b) - 1u;
  const float2 s2 = make_float2(sc, sc), z2 = make_float2(mn, mn);
  const float2 m2 = make_float2(-8388608.0f, -8388608.0f);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const uint32_t c0 = (lo >> (j * b)) & mask;
    const uint32_t c1 = (lo >> ((j + 1) * b)) & mask;
    const float2 qf = addp(make_float2(__uint_as_float(0x4B000000u | c0),
                                       __uint_as_float(0x4B000000u | c1)), m2);
    const float2 r = fma2(qf, s2, z2);
    v[j] = r.x;
    v[j + 1] = r.y;
  }
}

// Slot bytes of every chunk (one warp per chunk, kDecChunksPerBlock chunks per block);
// bit widths outside 1..8 count as 0.  Each chunk gets its offset inside its block
// (ctot), each block its total (bsum, turned into stream offsets by the last block).
static_assert(kDecWarps == kDecChunksPerBlock, "one warp per chunk of a block");
template <int G>
__global__ void __launch_bounds__(kDecThreads) k_dec_totals(DecodeArgs a, long long n_chunks,
                                                           long long n_blocks) {
  __shared__ uint32_t s_t[kDecWarps];
  __shared__ unsigned long long s_w[kDecWarps + 1];
  __shared__ uint32_t s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long c = (long long)blockIdx.x * kDecWarps + warp;
  const uint32_t tot = c < n_chunks ? warp_chunk_bytes<G>(a.bits, a.n_tiles, c) : 0u;
  if (lane == 0) s_t[warp] = tot;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = lane < kDecWarps ? s_t[lane] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < kDecWarps; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    const long long cc = (long long)blockIdx.x * kDecWarps + lane;
    if (lane < kDecWarps && cc < n_chunks) a.ctot[cc] = incl - v;
    if (lane == kDecWarps - 1) a.bsum[blockIdx.x] = incl;
  }
  // the last block to finish turns the block totals into stream offsets
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1u ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  // the unpack kernel's blocks may now take the SMs (the other blocks have exited)
  dep_launch();
  __threadfence();
  constexpr int kPer = 4, kPass = kDecThreads * kPer;
  unsigned long long carry = 0;
  for (long long p0 = 0; p0 < n_blocks; p0 += kPass) {
    const long long i0 = p0 + (long long)threadIdx.x * kPer;
    unsigned long long v[kPer], mine = 0;
#pragma unroll
    for (int k = 0; k < kPer; k++) {
      v[k] = i0 + k < n_blocks ? __ldcg(&a.bsum[i0 + k]) : 0ull;
      mine += v[k];
    }
    unsigned long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const unsigned long long w = lane < kDecWarps ? s_w[lane] : 0ull;
      unsigned long long wi = w;
#pragma unroll
      for (int o = 1; o < kDecWarps; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(kFull, wi, o);
        if (lane >= o) wi += y;
      }
      __syncwarp();
      if (lane < kDecWarps) s_w[lane] = wi - w;
      if (lane == kDecWarps - 1) s_w[kDecWarps] = wi;
    }
    __syncthreads();
    unsigned long long acc = carry + s_w[warp] + incl - mine;
#pragma unroll
    for (int k = 0; k < kPer; k++) {
      if (i0 + k < n_blocks) a.bsum[i0 + k] = acc;
      acc += v[k];
    }
    carry += s_w[kDecWarps];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.bsum[n_blocks] = carry;  // the end of the last slot
    if (carry > a.codes_bytes) set_status(a.status, kStOverrun);
  }
}

// Exclusive prefix of the block totals, in place (one block of 1024 threads, coalesced
// passes of 4096 entries); flags a stream shorter than the sum of all slots.

// 16-byte asynchronous copy global -> shared (both 16-byte aligned), in the thread's
// current copy group.
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Start copying the bytes of chunk c (from the 16-byte boundary at or below its first
// byte) into `stage`; returns that first byte's offset in the stage.  Bytes past
// codes_bytes are never read (the last partial 16 bytes go by plain loads), and a chunk
// longer than its largest possible size is cut (the offsets were corrupted).
template <int G>
__device__ __forceinline__ int issue_chunk_bytes(const DecodeArgs& a, long long c, long long n_chunks,
                                                 long long n_blocks, uint32_t* stage) {
  using C = DecCfg<G>;
  auto start = [&](long long cc) {
    return cc < n_chunks ? a.bsum[cc / kDecChunksPerBlock] + a.ctot[cc] : a.bsum[n_blocks];
  };
  const unsigned long long base = start(c), end = max(base, start(c + 1));
  const int pad = (int)(base & 15ull);
  const unsigned long long a0 = base - (unsigned long long)pad;
  const unsigned long long bytes = min(end - base, (unsigned long long)(C::CH * G));
  const int n16 = (pad + (int)bytes + 15) / 16;
  const unsigned long long limit = a.codes_bytes;
  for (int w16 = threadIdx.x; w16 < n16; w16 += kDecThreads) {
    const unsigned long long gb = a0 + 16ull * w16;
    if (gb + 16ull <= limit) {
      cp_async16(stage + 4 * w16, a.codes + gb);
    } else {
      uint32_t tmp[4] = {0u, 0u, 0u, 0u};
      for (int k = 0; k < 16; k++)
        if (gb + k < limit) tmp[k >> 2] |= (uint32_t)a.codes[gb + k] << (8 * (k & 3));
      reinterpret_cast<uint4*>(stage)[w16] = make_uint4(tmp[0], tmp[1], tmp[2], tmp[3]);
    }
  }
  cp_async_commit();
  return pad;
}

// kS: every value stored as RN(value x a.inv_c) (the gradient codec's 1 / c).
template <int G, bool kS>
__global__ void __launch_bounds__(kDecThreads, DecCfg<G>::kMinBlocks) k_decode(DecodeArgs a, long long n_chunks,
                                                        long long n_blocks) {
  using C = DecCfg<G>;
  constexpr int V = C::V, L = C::L, TPW = C::TPW, CH = C::CH, NS = C::NS;
  extern __shared__ __align__(16) unsigned char dec_smem[];
  DecSmem<G>& s = *reinterpret_cast<DecSmem<G>*>(dec_smem);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = lane / L, sub = lane % L;
  const unsigned long long limit = a.codes_bytes;

  // the bytes of the block's first chunk; in each iteration the next chunk's bytes are
  // copied while this one is unpacked, and the next chunk's per-tile metadata (width |
  // pivot << 8, scale, zero of tile k = thread * kPer + j) and first byte are loaded into
  // registers
  dep_wait();  // the chunk offsets
  int slot = 0;
  int pad = blockIdx.x < n_chunks ? issue_chunk_bytes<G>(a, blockIdx.x, n_chunks, n_blocks, s.stage[0]) : 0;
  uint32_t nbp[C::kPer];
  float nsc[C::kPer], nze[C::kPer];
  unsigned long long nbase = 0ull;
  auto load_meta = [&](long long cc) {
    if (cc >= n_chunks) return;
    const long long tt = cc * CH;
    const int ntt = (int)min((long long)CH, a.n_tiles - tt);
#pragma unroll
    for (int j = 0; j < C::kPer; j++) {
      const int k = threadIdx.x * C::kPer + j;
      if (k < ntt) {
        nbp[j] = (uint32_t)a.bits[tt + k] | ((uint32_t)a.pivots[tt + k] << 8);
        nsc[j] = a.scales[tt + k];
        nze[j] = a.zeros[tt + k];
      }
    }
    nbase = a.bsum[cc / kDecChunksPerBlock] + a.ctot[cc];
  };
  load_meta(blockIdx.x);
  for (long long c = blockIdx.x; c < n_chunks; c += gridDim.x, slot ^= 1) {
    const long long cn = c + gridDim.x;
    int pad_next = 0;
    if (cn < n_chunks) {
      pad_next = issue_chunk_bytes<G>(a, cn, n_chunks, n_blocks, s.stage[slot ^ 1]);
    } else {
      cp_async_commit();  // an empty group keeps the wait below uniform
    }
    const uint32_t* stage = s.stage[slot];
    const long long t0 = c * CH;
    const int nt = (int)min((long long)CH, a.n_tiles - t0);
    uint32_t cbp[C::kPer];
#pragma unroll
    for (int j = 0; j < C::kPer; j++) {
      const int k = threadIdx.x * C::kPer + j;
      cbp[j] = nbp[j];
      if (k < nt) {
        s.scale[k] = nsc[j];
        s.zero[k] = nze[j];
      }
    }
    const unsigned long long base = nbase;
    load_meta(cn);

    // 1. slot sizes of this chunk and their exclusive running sum
    uint32_t mine = 0u;
    uint8_t bl[C::kPer];
#pragma unroll
    for (int j = 0; j < C::kPer; j++) {
      const int k = threadIdx.x * C::kPer + j;
      bl[j] = 0;
      if (k < nt) {
        int b = (int)(cbp[j] & 0xFFu);
        if (b < 1 || b > 8) {
          set_status(a.status, kStBadBits);
          b = 0;
        }
        bl[j] = (uint8_t)b;
        mine += (uint32_t)(G * b / 8);
      }
    }
    uint32_t chunk_bytes;
    uint32_t off = block_exclusive_scan_dec<kDecThreads>(mine, chunk_bytes, s.scan);
    (void)chunk_bytes;
    // each tile's slot (the chunk's first byte in the stream from k_dec_totals and
    // its last block), and, settled once here, whether it decodes (width 0: its slot runs past
    // the stream or its width or pivot is invalid, and it decodes to zeros) and is
    // transformed
#pragma unroll
    for (int j = 0; j < C::kPer; j++) {
      const int k = threadIdx.x * C::kPer + j;
      if (k < nt) {
        const int b = bl[j];
        const int piv = (int)(cbp[j] >> 8);
        const bool bad_piv = piv != 0xFF && piv >= G;
        if (bad_piv) set_status(a.status, kStBadBits);
        const bool ok = b > 0 && !bad_piv && base + off + (unsigned long long)(G * b / 8) <= limit;
        s.bits[k] = (uint8_t)(ok ? b : 0);
        s.piv[k] = (uint8_t)(ok ? piv : 0xFF);
        s.off[k] = (uint16_t)off;
        off += (uint32_t)(G * b / 8);
      }
    }
    cp_async_wait_prev();  // this chunk's bytes have landed
    __syncthreads();

    // 4. untransformed tiles; transformed ones are listed for the second pass
    uint16_t* fl = s.flagged + warp * NS;
    int nflag = 0;
    float* outc = a.out + t0 * G;  // the chunk's first value
#pragma unroll 1
    for (int st = 0; st < C::kSteps; st++) {
      const int kt = (st * kDecWarps + warp) * TPW + team;
      const bool valid = kt < nt;
      const int b = valid ? (int)s.bits[kt] : 0;  // 0: decodes to zeros (settled above)
      const bool ok = b > 0;
      const bool flag = valid && s.piv[kt] != 0xFF;
      const unsigned fm = __ballot_sync(kFull, flag && sub == 0);
      if (flag && sub == 0) fl[nflag + __popc(fm & ((1u << lane) - 1u))] = (uint16_t)kt;
      nflag += __popc(fm);
      const bool narrow = __all_sync(kFull, b <= 4);  // warp-uniform
      if (!valid || flag) continue;
      float v[V];
      const int start = pad + (int)s.off[kt] + sub * b;
      if (narrow) {  // b = 0 decodes to zeros: codes 0, scale and zero 0
        dequant8_le4(stage, start, b, ok ? s.scale[kt] : 0.0f, ok ? s.zero[kt] : 0.0f, v);
      } else if (ok) {
        dequant8(stage, start, b, s.scale[kt], s.zero[kt], v);
      } else {
#pragma unroll
        for (int j = 0; j < V; j++) v[j] = 0.0f;
      }
      if constexpr (kS) {
#pragma unroll
        for (int j = 0; j < V; j++) v[j] = __fmul_rn(v[j], a.inv_c);
      }
      float4* o = reinterpret_cast<float4*>(outc + kt * G + sub * V);
      o[0] = make_float4(v[0], v[1], v[2], v[3]);
      o[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncwarp();
    // 5. transformed tiles of this warp, TPW at a time
#pragma unroll 1
    for (int j0 = 0; j0 < nflag; j0 += TPW) {
      const int ci = j0 + team;
      const bool valid = ci < nflag;
      const int kt = valid ? (int)fl[ci] : 0;
      const int b = valid ? (int)s.bits[kt] : 1;
      const int piv = valid ? (int)s.piv[kt] : 0;
      float v[V];
      const int start = valid ? pad + (int)s.off[kt] + sub * b : 0;
      const float sc = valid ? s.scale[kt] : 0.0f, zr = valid ? s.zero[kt] : 0.0f;
      if (__all_sync(kFull, b <= 4)) {  // warp-uniform
        dequant8_le4(stage, start, b, sc, zr, v);
      } else {
        dequant8(stage, start, b, sc, zr, v);
      }
      team_fwht<V, L>(v, a.h, sub);
#pragma unroll
      for (int j = 0; j < V; j++) v[j] = __fmul_rn(v[j], a.c_h);
      team_swap0<V>(v, piv, sub, lane - sub);
      if constexpr (kS) {
#pragma unroll
        for (int j = 0; j < V; j++) v[j] = __fmul_rn(v[j], a.inv_c);
      }
      if (valid) {
        float4* o = reinterpret_cast<float4*>(a.out + (t0 + kt) * G + sub * V);
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
    __syncthreads();
    pad = pad_next;
  }
}

long long decode_chunks(int G, long long n_tiles) {
  const long long ch = (long long)kDecWarps * 8 * (32 / (G / 8));
  return (n_tiles + ch - 1) / ch;
}

template <int G>
static cudaError_t run_decode(const DecodeArgs& a, cudaStream_t st) {
  const long long n_chunks = decode_chunks(G, a.n_tiles);
  const long long n_blocks = decode_blocks(G, a.n_tiles);
  const size_t smem = sizeof(DecSmem<G>);
  static const cudaError_t e_attr = [smem] {
    const cudaError_t e0 = cudaFuncSetAttribute(k_decode<G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const cudaError_t e1 = cudaFuncSetAttribute(k_decode<G, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return e0 != cudaSuccess ? e0 : e1;
  }();
  if (e_attr != cudaSuccess) return e_attr;
  // one wave of the blocks an SM holds (registers and shared memory: 6 at tiles of 64 and
  // 128, 5 at 32, whose stages and per-tile arrays are larger), so that the blocks' load,
  // scan and unpack phases overlap and no block waits for a second wave
  static const int per_sm = [smem] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode<G, false>, kDecThreads, smem) != cudaSuccess || n < 1)
      n = 1;
    return n;
  }();
  const int blocks = (int)std::max<long long>(1, std::min<long long>((long long)a.num_sms * per_sm, n_chunks));
  k_dec_totals<G><<<(unsigned)n_blocks, kDecThreads, 0, st>>>(a, n_chunks, n_blocks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the unpack starts while the kernel before drains (dep_wait inside)
  return launch_dependent(a.inv_c != 1.0f ? k_decode<G, true> : k_decode<G, false>, (unsigned)blocks,
                          (unsigned)kDecThreads, smem, st, a, n_chunks, n_blocks);
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
