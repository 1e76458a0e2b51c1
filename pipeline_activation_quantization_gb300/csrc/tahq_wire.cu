// Wire format: the encoder's per-tile metadata packed next to its payload in one buffer,
// and back ("TAH-Quant" §3.2: the 1-bit per-tile width map travels with the payload as
// metadata; §3.4: one contiguous uint8 byte stream of fixed size per shape).
//
// Sections, each at a 16-byte boundary: a 128-byte header; the width map (bit t = tile t
// has bits_hi, LSB first); a (scale, zero) pair of fp16 per tile, the transform flag in
// the sign bit of the scale; the pivot fields (pb = log2 tile bits each, LSB first, 0
// for untransformed tiles); the payload (the packed slots of tahq_encode).  The encoder
// writes the payload in place and the fp16-exact scales and zeros to workspace arrays;
// k_wire_pack moves the metadata into the buffer, k_wire_unpack back out for the decoder.
#include <algorithm>

#include "tahq_device.cuh"
#include "tahq_launch.h"

namespace tahq {

namespace {

constexpr int kWireThreads = 256;

__device__ __forceinline__ void st_u32(uint8_t* base, long long byte_off, uint32_t v) {
  *reinterpret_cast<uint32_t*>(base + byte_off) = v;
}

// One thread per tile (the grid covers whole warps of tiles).
__global__ void __launch_bounds__(kWireThreads) k_wire_pack(const __grid_constant__ WirePackArgs a) {
  const long long t = (long long)blockIdx.x * kWireThreads + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool valid = t < a.n;
  const uint8_t b = valid ? a.bits[t] : (uint8_t)0;
  const uint8_t pv = valid ? a.pivots[t] : (uint8_t)0xFF;
  const bool flag = pv != 0xFFu;
  // width map: one word per 32 tiles
  const unsigned m = __ballot_sync(0xFFFFFFFFu, valid && b == (uint8_t)a.hi);
  const long long map_words = (a.n + 31) / 32;
  if (lane == 0 && (t >> 5) < map_words) st_u32(a.wire, a.off_map + 4 * (t >> 5), m);
  // (scale | flag << 15, zero): both are fp16 numbers already, converted exactly
  if (valid) {
    const uint32_t s16 = __half_as_ushort(__float2half_rn(a.scales[t])) | (flag ? 0x8000u : 0u);
    const uint32_t z16 = __half_as_ushort(__float2half_rn(a.zeros[t]));
    st_u32(a.wire, a.off_meta + 4 * t, s16 | (z16 << 16));
  }
  // pivot fields: the warp's 32 tiles fill pb whole words (its first bit is 32 pb (t / 32))
  const uint32_t p = flag ? (uint32_t)pv : 0u;
  const long long piv_words = (a.n * a.pb + 31) / 32;
  for (int w = 0; w < a.pb; w++) {
    const int bit = lane * a.pb - 32 * w;  // where the lane's field starts within word w
    uint32_t part = 0u;
    if (bit >= 0 && bit < 32) part = p << bit;
    else if (bit < 0 && bit + a.pb > 0) part = p >> (-bit);
    part = __reduce_or_sync(0xFFFFFFFFu, part);
    const long long W = ((t - lane) >> 5) * a.pb + w;
    if (lane == w && W < piv_words) st_u32(a.wire, a.off_piv + 4 * W, part);
  }
  if (blockIdx.x == 0) {
    if (threadIdx.x < 32) st_u32(a.wire, 4 * threadIdx.x, a.header[threadIdx.x]);
    // zero the padding after each section (the payload's slots end at off_pay + pay)
    const long long ends[4][2] = {{a.off_map + 4 * map_words, a.off_meta},
                                  {a.off_meta + 4 * a.n, a.off_piv},
                                  {a.off_piv + 4 * piv_words, a.off_pay},
                                  {a.off_pay + a.pay, a.total}};
    for (int r = 0; r < 4; r++)
      for (long long i = ends[r][0] + threadIdx.x; i < ends[r][1]; i += kWireThreads) a.wire[i] = 0;
  }
}

__global__ void __launch_bounds__(kWireThreads) k_wire_unpack(const __grid_constant__ WireUnpackArgs a) {
  const long long t = (long long)blockIdx.x * kWireThreads + threadIdx.x;
  if (blockIdx.x == 0 && threadIdx.x < 32 && threadIdx.x != 11) {  // word 11 is tau
    const uint32_t got = *reinterpret_cast<const uint32_t*>(a.wire + 4 * threadIdx.x);
    if (got != a.header[threadIdx.x]) set_status(a.status, kStBadWire);
  }
  if (t >= a.n) return;
  const uint32_t mw = *reinterpret_cast<const uint32_t*>(a.wire + a.off_map + 4 * (t >> 5));
  const uint32_t meta = *reinterpret_cast<const uint32_t*>(a.wire + a.off_meta + 4 * t);
  const long long bit = t * a.pb;
  const long long W = bit >> 5;
  const int sh = (int)(bit & 31);
  const uint32_t* pw = reinterpret_cast<const uint32_t*>(a.wire + a.off_piv);
  uint32_t f = pw[W] >> sh;
  if (sh + a.pb > 32) f |= pw[W + 1] << (32 - sh);
  f &= (1u << a.pb) - 1u;
  a.bits[t] = (uint8_t)(((mw >> (t & 31)) & 1u) ? a.hi : a.lo);
  a.scales[t] = __half2float(__ushort_as_half((uint16_t)(meta & 0x7FFFu)));
  a.zeros[t] = __half2float(__ushort_as_half((uint16_t)(meta >> 16)));
  a.pivots[t] = (meta & 0x8000u) ? (uint8_t)f : (uint8_t)0xFF;
}

}  // namespace

cudaError_t launch_wire_pack(const WirePackArgs& a, cudaStream_t st) {
  const long long blocks = std::max<long long>(1, (a.n + kWireThreads - 1) / kWireThreads);
  k_wire_pack<<<(unsigned)blocks, kWireThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_wire_unpack(const WireUnpackArgs& a, cudaStream_t st) {
  const long long blocks = std::max<long long>(1, (a.n + kWireThreads - 1) / kWireThreads);
  k_wire_unpack<<<(unsigned)blocks, kWireThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tahq
