// tahq_api.cu -- the C ABI of the codec (declared in include/tahq.h): argument checks,
// workspace layout, and the launch sequence on the caller's stream.  Allocates nothing.
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/tahq.h"
#include "tahq_launch.h"

namespace {

using tahq::LgTables;

constexpr int kVersion = 20200;  // 2.2.0: streaming encoder, scaled gradients, wait test
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
bool is_pow2(long long v) { return v > 0 && (v & (v - 1)) == 0; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Tables of the canonical base-2 logarithm (nearest floats of double-precision values).
const LgTables& lg_tables() {
  static LgTables tabs;
  static std::once_flag once;
  std::call_once(once, [] {
    const double ln2 = 0.69314718055994530942;
    for (int j = 0; j < 3; j++) tabs.k[j] = (float)(((j % 2) ? -1.0 : 1.0) / ((j + 1) * ln2));
    for (int i = 0; i < 128; i++) {
      const double c = 1.0 + i / 128.0;
      tabs.R[i] = (float)(1.0 / c);
      tabs.T[i] = (float)(-std::log2((double)tabs.R[i]));
      // fraction part of lg(c_i) by the general path (c_i is exact in float)
      const float r = std::fmaf((float)c, tabs.R[i], -1.0f);
      float p = std::fmaf(tabs.k[2], r, tabs.k[1]);
      p = std::fmaf(p, r, tabs.k[0]);
      tabs.TB[i] = std::fmaf(p, r, tabs.T[i]);
    }
  });
  return tabs;
}

int num_sms_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

struct Shape {
  long long T, C, n, n_g, n_groups, K, group_bytes, payload;
  int G, h, lo, hi;
  int mlog;  // allocation tile A = 2^mlog G; K counts allocation tiles (n_g >> mlog a group)
};

// Shape checks shared by every entry point.  hblock < 0 means "not given".
tahq_status check_shape(long long T, long long C, int G, int h, Shape& s) {
  if (T < 0 || C <= 0) return TAHQ_ERR_ARG;
  if (G < 8 || G > 128 || G % 8) return TAHQ_ERR_ARG;
  if (!is_pow2(G)) return TAHQ_ERR_UNSUPPORTED;
  if (C % G) return TAHQ_ERR_ARG;
  if (h >= 0 && (h < 2 || h > G || !is_pow2(h))) return TAHQ_ERR_ARG;
  if (T > 0 && C > (1ll << 40) / T) return TAHQ_ERR_ARG;
  s.T = T;
  s.C = C;
  s.G = G;
  s.h = h;
  s.n = T * (C / G);
  return TAHQ_OK;
}

// A = the allocation tile (0: A = G), a power-of-two multiple of G that divides C.
tahq_status check_codec(long long T, long long C, int G, int h, int lo, int hi, float budget,
                        long long S, Shape& s, long long A = 0) {
  tahq_status st = check_shape(T, C, G, h, s);
  if (st != TAHQ_OK) return st;
  if (A == 0) A = G;
  if (A < G || A % G || C % A || !is_pow2(A / G)) return TAHQ_ERR_ARG;
  s.mlog = 0;
  while ((1ll << s.mlog) < A / G) s.mlog++;
  if (lo < 1 || hi > 8 || lo >= hi) return TAHQ_ERR_ARG;
  if (!(std::isfinite(budget) && (double)budget >= lo && (double)budget <= hi)) return TAHQ_ERR_ARG;
  if (S < 0) return TAHQ_ERR_ARG;
  if (S == 0) S = T;
  if (T > 0 && T % S) return TAHQ_ERR_ARG;
  s.lo = lo;
  s.hi = hi;
  s.n_g = S * (C / G);
  if (s.n_g >= (1ll << 31)) return TAHQ_ERR_UNSUPPORTED;
  s.n_groups = (T > 0) ? T / S : 0;
  const long long n_ga = s.n_g >> s.mlog;
  s.K = (long long)std::floor(((double)budget - lo) * (double)n_ga / (double)(hi - lo));
  s.group_bytes = s.n_g * G * lo / 8 + (s.K << s.mlog) * G * (hi - lo) / 8;
  s.payload = s.n_groups * s.group_bytes;
  return TAHQ_OK;
}

struct EncLayout {
  size_t status, ticket, cand_cnt, doneA, doneB, doneB2, selready, sel, hist_coarse, hist_fine, lookback,
      ctrl_end, keys, cand, segmask, scratch_lo, scratch_hi, items, items_cap, total;
};

// Offset words are sized for the input type that needs the most compaction chunks.
EncLayout enc_layout(const Shape& s) {
  EncLayout L{};
  size_t off = 0;
  L.status = off;
  off = align_up(off + 16);
  L.ticket = off;
  off = align_up(off + 64);
  L.cand_cnt = off;
  off = align_up(off + 4 * (size_t)s.n_groups);
  L.doneA = off;
  off = align_up(off + 4 * (size_t)s.n_groups);
  L.doneB = off;
  off = align_up(off + 4 * (size_t)s.n_groups);
  L.doneB2 = off;
  off = align_up(off + 4 * (size_t)s.n_groups);
  L.selready = off;
  off = align_up(off + 4 * (size_t)s.n_groups);
  L.sel = off;
  off = align_up(off + sizeof(tahq::SelResult) * (size_t)s.n_groups);
  L.hist_coarse = off;
  off = align_up(off + 4ull * tahq::kCoarseBins * (size_t)s.n_groups);
  L.hist_fine = off;
  off = align_up(off + 4ull * tahq::kFineBins * (size_t)s.n_groups);
  L.lookback = off;
  const long long chunks = std::max(tahq::encode_chunks(0, s.G, s.hi, s.n_g, s.n_groups),
                                    tahq::encode_chunks(1, s.G, s.hi, s.n_g, s.n_groups));
  off = align_up(off + 8 * (size_t)chunks);
  L.ctrl_end = off;
  L.keys = off;
  off = align_up(off + 4 * (size_t)s.n);
  L.cand = off;
  off = align_up(off + 8 * (size_t)s.n);
  L.segmask = off;
  off = align_up(off + 4 * (size_t)s.n_groups * (size_t)((s.n_g + 31) / 32));
  // every tile quantised at both widths, fixed slots (read back by the compaction)
  L.scratch_lo = off;
  off = align_up(off + (size_t)s.n * (size_t)(s.G * s.lo / 8));
  L.scratch_hi = off;
  off = align_up(off + (size_t)s.n * (size_t)(s.G * s.hi / 8));
  // the decoded work queue, sized for the input type with the most items
  L.items = off;
  L.items_cap = (size_t)std::max(tahq::encode_queue_items(0, s.G, s.hi, s.n_g, s.n_groups),
                                 tahq::encode_queue_items(1, s.G, s.hi, s.n_g, s.n_groups));
  off = align_up(off + 8 * L.items_cap);
  L.total = off;
  return L;
}

struct DecLayout {
  size_t status, ticket, ctot, bsum, total;
};

DecLayout dec_layout(const Shape& s) {
  DecLayout L{};
  size_t off = 0;
  L.status = off;
  off = align_up(off + 16);
  L.ticket = off;
  off = align_up(off + 64);
  L.ctot = off;
  off = align_up(off + 4 * (size_t)tahq::decode_chunks(s.G, s.n));
  L.bsum = off;
  off = align_up(off + 8 * ((size_t)tahq::decode_blocks(s.G, s.n) + 1));
  L.total = off;
  return L;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

}  // namespace

extern "C" {

size_t tahq_payload_size(int64_t tokens, int64_t channels, int tile, int bits_lo, int bits_hi,
                         float budget, int64_t tokens_per_group) {
  Shape s;
  if (check_codec(tokens, channels, tile, -1, bits_lo, bits_hi, budget, tokens_per_group, s) !=
      TAHQ_OK)
    return 0;
  return (size_t)s.payload;
}

int64_t tahq_hi_count(int64_t tokens, int64_t channels, int tile, int bits_lo, int bits_hi,
                      float budget, int64_t tokens_per_group) {
  Shape s;
  if (check_codec(tokens, channels, tile, -1, bits_lo, bits_hi, budget, tokens_per_group, s) !=
      TAHQ_OK)
    return -1;
  return s.K;
}

size_t tahq_workspace_size(int64_t tokens, int64_t channels, int tile, int hblock, int bits_lo,
                           int bits_hi, float budget, int64_t tokens_per_group) {
  Shape s;
  if (check_codec(tokens, channels, tile, hblock, bits_lo, bits_hi, budget, tokens_per_group,
                  s) != TAHQ_OK)
    return 0;
  return enc_layout(s).total;
}

size_t tahq_decode_workspace_size(int64_t tokens, int64_t channels, int tile) {
  Shape s;
  if (check_shape(tokens, channels, tile, -1, s) != TAHQ_OK) return 0;
  return dec_layout(s).total;
}

namespace {

// tahq_encode_ex, and the wire format's encoder (wire: fp16 zero and scales).
tahq_status encode_impl(const void* x, tahq_dtype dtype, int64_t tokens, int64_t channels,
                        int tile, int hblock, int bits_lo, int bits_hi, float budget,
                        int64_t tokens_per_group, float tau, int alloc_tile, bool wire,
                        uint8_t* codes, float* scales, float* zeros, uint8_t* bits,
                        uint8_t* pivots, void* workspace, size_t workspace_bytes, void* stream,
                        float scale_c = 1.0f) {
  if (!(tau >= 0.0f)) return TAHQ_ERR_ARG;  // negative or NaN
  if (alloc_tile < 0) return TAHQ_ERR_ARG;
  Shape s;
  tahq_status st = check_codec(tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                               tokens_per_group, s, alloc_tile);
  if (st != TAHQ_OK) return st;
  // an allocation tile is never split between two of the encoder's 32 KB input chunks
  if (((long long)tile << s.mlog) * (dtype == TAHQ_BF16 ? 2 : 4) > 32768)
    return TAHQ_ERR_UNSUPPORTED;
  if (hblock < 0) return TAHQ_ERR_ARG;
  if (dtype != TAHQ_F32 && dtype != TAHQ_BF16) return TAHQ_ERR_ARG;
  if (s.n > 0) {
    if (!x || !codes || !scales || !zeros || !bits || !pivots) return TAHQ_ERR_ARG;
    if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4) || !aligned(zeros, 4))
      return TAHQ_ERR_ARG;
  }
  if (!workspace || !aligned(workspace, kAlign)) return TAHQ_ERR_WORKSPACE;
  const bool bf16 = dtype == TAHQ_BF16;
  const EncLayout L = enc_layout(s);
  if (workspace_bytes < L.total) return TAHQ_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // every tile at one width (K = 0 or K = all): only the status word and the ticket are
  // used, else the histograms, counters and offsets too
  const bool one_width = s.K == 0 || s.K == (s.n_g >> s.mlog);
  if (cudaMemsetAsync(workspace, 0, one_width ? L.cand_cnt : L.ctrl_end, cs) != cudaSuccess)
    return TAHQ_ERR_CUDA;
  if (s.n == 0) return TAHQ_OK;
  const int sms = num_sms_current();
  if (sms <= 0) return TAHQ_ERR_CUDA;

  tahq::EncodeArgs a{};
  a.x = x;
  a.bf16 = bf16;
  a.G = s.G;
  a.h = s.h;
  a.lo = s.lo;
  a.hi = s.hi;
  a.c_h = (float)(1.0 / std::sqrt((double)s.h));
  a.tau = tau;
  a.wire = wire;
  a.mlog = s.mlog;
  a.n_tiles = s.n;
  a.n_g = s.n_g;
  a.n_groups = s.n_groups;
  a.K = s.K;
  a.group_bytes = s.group_bytes;
  a.num_sms = sms;
  a.tabs = &lg_tables();
  a.codes = codes;
  a.scales = scales;
  a.zeros = zeros;
  a.bits = bits;
  a.pivots = pivots;
  a.status = at<uint32_t>(workspace, L.status);
  a.ticket = at<uint32_t>(workspace, L.ticket);
  a.cand_cnt = at<uint32_t>(workspace, L.cand_cnt);
  a.doneA = at<uint32_t>(workspace, L.doneA);
  a.doneB = at<uint32_t>(workspace, L.doneB);
  a.doneB2 = at<uint32_t>(workspace, L.doneB2);
  a.selready = at<uint32_t>(workspace, L.selready);
  a.sel = at<tahq::SelResult>(workspace, L.sel);
  a.hist_coarse = at<uint32_t>(workspace, L.hist_coarse);
  a.hist_fine = at<uint32_t>(workspace, L.hist_fine);
  a.lookback = at<unsigned long long>(workspace, L.lookback);
  a.keys = at<float>(workspace, L.keys);
  a.cand = at<unsigned long long>(workspace, L.cand);
  a.segmask = at<uint32_t>(workspace, L.segmask);
  a.scratch_lo = at<uint8_t>(workspace, L.scratch_lo);
  a.scratch_hi = at<uint8_t>(workspace, L.scratch_hi);
  a.items = at<unsigned long long>(workspace, L.items);
  a.items_cap = (long long)L.items_cap;
  a.scale_c = scale_c;
  const cudaError_t e = tahq::launch_encode(a, cs);
  if (e == cudaErrorNotYetImplemented) return TAHQ_ERR_UNSUPPORTED;  // scale_c off the streaming path
  return e == cudaSuccess ? TAHQ_OK : TAHQ_ERR_CUDA;
}

}  // namespace

tahq_status tahq_encode_ex(const void* x, tahq_dtype dtype, int64_t tokens, int64_t channels,
                           int tile, int hblock, int bits_lo, int bits_hi, float budget,
                           int64_t tokens_per_group, float tau, int alloc_tile, uint8_t* codes,
                           float* scales, float* zeros, uint8_t* bits, uint8_t* pivots,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return encode_impl(x, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                     tokens_per_group, tau, alloc_tile, false, codes, scales, zeros, bits, pivots,
                     workspace, workspace_bytes, stream);
}

size_t tahq_payload_size_ex(int64_t tokens, int64_t channels, int tile, int alloc_tile,
                            int bits_lo, int bits_hi, float budget, int64_t tokens_per_group) {
  Shape s;
  if (alloc_tile < 0 || check_codec(tokens, channels, tile, -1, bits_lo, bits_hi, budget,
                                    tokens_per_group, s, alloc_tile) != TAHQ_OK)
    return 0;
  return (size_t)s.payload;
}

tahq_status tahq_encode(const void* x, tahq_dtype dtype, int64_t tokens, int64_t channels,
                        int tile, int hblock, int bits_lo, int bits_hi, float budget,
                        int64_t tokens_per_group, uint8_t* codes, float* scales, float* zeros,
                        uint8_t* bits, uint8_t* pivots, void* workspace, size_t workspace_bytes,
                        void* stream) {
  return tahq_encode_ex(x, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                        tokens_per_group, 2.0f, 0, codes, scales, zeros, bits, pivots, workspace,
                        workspace_bytes, stream);
}

namespace {

// tahq_decode; clear = false when the caller has already cleared the status word (and
// may have set bits in it on the same stream).
tahq_status decode_impl(const uint8_t* codes, size_t codes_bytes, const float* scales,
                        const float* zeros, const uint8_t* bits, const uint8_t* pivots,
                        int64_t tokens, int64_t channels, int tile, int hblock, float* out,
                        void* workspace, size_t workspace_bytes, void* stream, bool clear,
                        float inv_c = 1.0f) {
  Shape s;
  tahq_status st = check_shape(tokens, channels, tile, hblock, s);
  if (st != TAHQ_OK) return st;
  if (hblock < 0) return TAHQ_ERR_ARG;
  if (s.n > 0) {
    if (!scales || !zeros || !bits || !pivots || !out) return TAHQ_ERR_ARG;
    if (codes_bytes > 0 && (!codes || !aligned(codes, 16))) return TAHQ_ERR_ARG;
    if (!aligned(out, 16) || !aligned(scales, 4) || !aligned(zeros, 4)) return TAHQ_ERR_ARG;
  }
  if (!workspace || !aligned(workspace, kAlign)) return TAHQ_ERR_WORKSPACE;
  const DecLayout L = dec_layout(s);
  if (workspace_bytes < L.total) return TAHQ_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // status and ticket; the offset arrays are written in full before they are read
  if (clear && cudaMemsetAsync(workspace, 0, L.ctot, cs) != cudaSuccess) return TAHQ_ERR_CUDA;
  if (s.n == 0) return TAHQ_OK;
  const int sms = num_sms_current();
  if (sms <= 0) return TAHQ_ERR_CUDA;
  tahq::DecodeArgs a{};
  a.codes = codes;
  a.codes_bytes = codes_bytes;
  a.scales = scales;
  a.zeros = zeros;
  a.bits = bits;
  a.pivots = pivots;
  a.G = s.G;
  a.h = s.h;
  a.c_h = (float)(1.0 / std::sqrt((double)s.h));
  a.n_tiles = s.n;
  a.num_sms = sms;
  a.out = out;
  a.status = at<uint32_t>(workspace, L.status);
  a.ticket = at<uint32_t>(workspace, L.ticket);
  a.ctot = at<uint32_t>(workspace, L.ctot);
  a.bsum = at<unsigned long long>(workspace, L.bsum);
  a.inv_c = inv_c;
  return tahq::launch_decode(a, cs) == cudaSuccess ? TAHQ_OK : TAHQ_ERR_CUDA;
}

}  // namespace

tahq_status tahq_decode(const uint8_t* codes, size_t codes_bytes, const float* scales,
                        const float* zeros, const uint8_t* bits, const uint8_t* pivots,
                        int64_t tokens, int64_t channels, int tile, int hblock, float* out,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(codes, codes_bytes, scales, zeros, bits, pivots, tokens, channels, tile,
                     hblock, out, workspace, workspace_bytes, stream, true);
}

// ------------------------------------------------------------------------ gradients

}  // extern "C"

namespace {

bool power_of_two(float c) {
  int e = 0;
  return c > 0.0f && std::isfinite(c) && std::frexp(c, &e) == 0.5f;
}

// y = RN(c x) elementwise (c a power of two: exact unless c x leaves the normal range),
// 16 bytes a thread and step; bf16 values stay bf16 (x 2^k is again a bf16 value).
template <bool kBf16>
__global__ void k_scale_input(const uint4* __restrict__ x, uint4* __restrict__ y, long long n16, float c) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x) {
    uint4 q = x[i];
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      if constexpr (kBf16) {
        const uint32_t lo = __float_as_uint(__fmul_rn(__uint_as_float(w[k] << 16), c));
        const uint32_t hi = __float_as_uint(__fmul_rn(__uint_as_float(w[k] & 0xFFFF0000u), c));
        // round to bf16, ties to even (exact here unless the range was left)
        const uint32_t rl = (lo + ((lo >> 16) & 1u) + 0x7FFFu) >> 16;
        const uint32_t rh = (hi + ((hi >> 16) & 1u) + 0x7FFFu) >> 16;
        w[k] = (rl & 0xFFFFu) | (rh << 16);
      } else {
        w[k] = __float_as_uint(__fmul_rn(__uint_as_float(w[k]), c));
      }
    }
    y[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

unsigned stream_blocks(long long n) {
  const int sms = num_sms_current();
  return (unsigned)std::max<long long>(1, std::min<long long>((n + 255) / 256, (long long)std::max(sms, 1) * 8));
}

}  // namespace

extern "C" {

size_t tahq_scaled_workspace_size(int64_t tokens, int64_t channels, int tile, int hblock,
                                  int bits_lo, int bits_hi, float budget,
                                  int64_t tokens_per_group, tahq_dtype dtype) {
  const size_t ws = tahq_workspace_size(tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                                        tokens_per_group);
  if (ws == 0 || (dtype != TAHQ_F32 && dtype != TAHQ_BF16)) return 0;
  return ws + align_up((size_t)(tokens * channels) * (dtype == TAHQ_BF16 ? 2 : 4));
}

tahq_status tahq_encode_scaled(const void* x, tahq_dtype dtype, int64_t tokens, int64_t channels,
                               int tile, int hblock, int bits_lo, int bits_hi, float budget,
                               int64_t tokens_per_group, float tau, float scale_c,
                               uint8_t* codes, float* scales, float* zeros, uint8_t* bits,
                               uint8_t* pivots, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (!power_of_two(scale_c)) return TAHQ_ERR_ARG;
  const size_t ws = tahq_workspace_size(tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                                        tokens_per_group);
  if (ws == 0 || (dtype != TAHQ_F32 && dtype != TAHQ_BF16)) return TAHQ_ERR_ARG;
  const size_t esz = dtype == TAHQ_BF16 ? 2 : 4;
  const size_t nbytes = (size_t)(tokens * channels) * esz;
  if (!workspace || !aligned(workspace, kAlign)) return TAHQ_ERR_WORKSPACE;
  if (workspace_bytes < ws + align_up(nbytes)) return TAHQ_ERR_WORKSPACE;
  if (nbytes && (!x || !aligned(x, 16))) return TAHQ_ERR_ARG;
  // the streaming encoder reads RN(c x) itself; the other encoders read a scaled copy
  const tahq_status direct = encode_impl(x, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi,
                                         budget, tokens_per_group, tau, 0, false, codes, scales,
                                         zeros, bits, pivots, workspace, ws, stream, scale_c);
  if (direct != TAHQ_ERR_UNSUPPORTED) return direct;
  void* xs = static_cast<unsigned char*>(workspace) + ws;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (nbytes) {  // channels are a multiple of 8, so the tensor is whole 16-byte units
    const long long n16 = (long long)(nbytes / 16);
    if (dtype == TAHQ_BF16)
      k_scale_input<true><<<stream_blocks(n16), 256, 0, cs>>>(static_cast<const uint4*>(x),
                                                              static_cast<uint4*>(xs), n16, scale_c);
    else
      k_scale_input<false><<<stream_blocks(n16), 256, 0, cs>>>(static_cast<const uint4*>(x),
                                                               static_cast<uint4*>(xs), n16, scale_c);
    if (cudaGetLastError() != cudaSuccess) return TAHQ_ERR_CUDA;
  }
  return encode_impl(xs, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                     tokens_per_group, tau, 0, false, codes, scales, zeros, bits, pivots,
                     workspace, ws, stream);
}

tahq_status tahq_decode_scaled(const uint8_t* codes, size_t codes_bytes, const float* scales,
                               const float* zeros, const uint8_t* bits, const uint8_t* pivots,
                               int64_t tokens, int64_t channels, int tile, int hblock,
                               float scale_c, float* out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!power_of_two(scale_c)) return TAHQ_ERR_ARG;
  // RN(decode / c) = decode x (1 / c), applied by the decoder to every value it stores
  return decode_impl(codes, codes_bytes, scales, zeros, bits, pivots, tokens, channels, tile,
                     hblock, out, workspace, workspace_bytes, stream, true, 1.0f / scale_c);
}

// ------------------------------------------------------------------------ wire format

namespace {

struct WireLayout {
  long long off_map, off_meta, off_piv, off_pay, pay, total;
  int pb;
};

long long up16(long long v) { return (v + 15) / 16 * 16; }

// Sections at 16-byte boundaries: 128-byte header, width map (1 bit a tile), (scale, zero)
// fp16 pairs (4 bytes a tile), pivot fields (log2 tile bits a tile), payload.
WireLayout wire_layout(const Shape& s) {
  WireLayout W{};
  W.pb = 0;
  while ((1 << W.pb) < s.G) W.pb++;
  W.off_map = 128;
  W.off_meta = W.off_map + up16((s.n + 7) / 8);
  W.off_piv = W.off_meta + up16(4 * s.n);
  W.off_pay = W.off_piv + up16((s.n * W.pb + 7) / 8);
  W.pay = s.payload;
  W.total = W.off_pay + up16(s.payload);
  return W;
}

// The 128-byte header (little-endian fields; the host is little-endian like the device).
void wire_header(const Shape& s, float budget, float tau, const WireLayout& W, uint32_t* words) {
  unsigned char b[128];
  std::memset(b, 0, sizeof(b));
  auto put = [&](int off, const void* v, size_t n) { std::memcpy(b + off, v, n); };
  const uint32_t magic = 0x51484154u;  // bytes 'T' 'A' 'H' 'Q'
  const uint16_t version = 1, header_bytes = 128, G = (uint16_t)s.G, h = (uint16_t)s.h;
  const int64_t T = s.T, C = s.C, S = s.n_g / (s.C / s.G);
  const uint8_t lo = (uint8_t)s.lo, hi = (uint8_t)s.hi, pb = (uint8_t)W.pb;
  const uint64_t n = (uint64_t)s.n;
  const uint64_t offs[6] = {(uint64_t)W.off_map, (uint64_t)W.off_meta, (uint64_t)W.off_piv,
                            (uint64_t)W.off_pay, (uint64_t)W.pay, (uint64_t)W.total};
  put(0, &magic, 4);
  put(4, &version, 2);
  put(6, &header_bytes, 2);
  put(8, &T, 8);
  put(16, &C, 8);
  put(24, &S, 8);
  put(32, &G, 2);
  put(34, &h, 2);
  put(36, &lo, 1);
  put(37, &hi, 1);
  put(38, &pb, 1);
  put(40, &budget, 4);
  put(44, &tau, 4);
  put(48, &n, 8);
  put(56, offs, sizeof(offs));
  std::memcpy(words, b, sizeof(b));
}

// Per-tile arrays after a codec workspace of `base` bytes: scales, zeros, bits, pivots.
struct WireArrays {
  size_t scales, zeros, bits, pivots, total;
};
WireArrays wire_arrays(size_t base, long long n) {
  WireArrays A{};
  A.scales = align_up(base);
  A.zeros = align_up(A.scales + 4 * (size_t)n);
  A.bits = align_up(A.zeros + 4 * (size_t)n);
  A.pivots = align_up(A.bits + (size_t)n);
  A.total = align_up(A.pivots + (size_t)n);
  return A;
}

}  // namespace

size_t tahq_wire_size(int64_t tokens, int64_t channels, int tile, int bits_lo, int bits_hi,
                      float budget, int64_t tokens_per_group) {
  Shape s;
  if (check_codec(tokens, channels, tile, -1, bits_lo, bits_hi, budget, tokens_per_group, s) !=
      TAHQ_OK)
    return 0;
  return (size_t)wire_layout(s).total;
}

size_t tahq_wire_workspace_size(int64_t tokens, int64_t channels, int tile, int hblock,
                                int bits_lo, int bits_hi, float budget,
                                int64_t tokens_per_group) {
  Shape s;
  if (check_codec(tokens, channels, tile, hblock, bits_lo, bits_hi, budget, tokens_per_group,
                  s) != TAHQ_OK)
    return 0;
  return wire_arrays(enc_layout(s).total, s.n).total;
}

size_t tahq_wire_decode_workspace_size(int64_t tokens, int64_t channels, int tile) {
  Shape s;
  if (check_shape(tokens, channels, tile, -1, s) != TAHQ_OK) return 0;
  return wire_arrays(dec_layout(s).total, s.n).total;
}

tahq_status tahq_encode_wire(const void* x, tahq_dtype dtype, int64_t tokens, int64_t channels,
                             int tile, int hblock, int bits_lo, int bits_hi, float budget,
                             int64_t tokens_per_group, float tau, uint8_t* wire, size_t wire_bytes,
                             void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  tahq_status st = check_codec(tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                               tokens_per_group, s);
  if (st != TAHQ_OK) return st;
  if (hblock < 0 || !(tau >= 0.0f)) return TAHQ_ERR_ARG;
  const WireLayout W = wire_layout(s);
  if (!wire || !aligned(wire, 16) || wire_bytes < (size_t)W.total) return TAHQ_ERR_ARG;
  if (!workspace || !aligned(workspace, kAlign)) return TAHQ_ERR_WORKSPACE;
  const EncLayout L = enc_layout(s);
  const WireArrays A = wire_arrays(L.total, s.n);
  if (workspace_bytes < A.total) return TAHQ_ERR_WORKSPACE;
  float* scales = at<float>(workspace, A.scales);
  float* zeros = at<float>(workspace, A.zeros);
  uint8_t* bits = at<uint8_t>(workspace, A.bits);
  uint8_t* pivots = at<uint8_t>(workspace, A.pivots);
  st = encode_impl(x, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                   tokens_per_group, tau, 0, true, wire + W.off_pay, scales, zeros, bits, pivots,
                   workspace, L.total, stream);
  if (st != TAHQ_OK) return st;
  tahq::WirePackArgs a{};
  a.scales = scales;
  a.zeros = zeros;
  a.bits = bits;
  a.pivots = pivots;
  a.wire = wire;
  a.n = s.n;
  a.off_map = W.off_map;
  a.off_meta = W.off_meta;
  a.off_piv = W.off_piv;
  a.off_pay = W.off_pay;
  a.pay = W.pay;
  a.total = W.total;
  a.hi = s.hi;
  a.pb = W.pb;
  wire_header(s, budget, tau, W, a.header);
  return tahq::launch_wire_pack(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? TAHQ_OK
             : TAHQ_ERR_CUDA;
}

tahq_status tahq_decode_wire(const uint8_t* wire, size_t wire_bytes, int64_t tokens,
                             int64_t channels, int tile, int hblock, int bits_lo, int bits_hi,
                             float budget, int64_t tokens_per_group, float* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  Shape s;
  tahq_status st = check_codec(tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                               tokens_per_group, s);
  if (st != TAHQ_OK) return st;
  if (hblock < 0) return TAHQ_ERR_ARG;
  const WireLayout W = wire_layout(s);
  if (!wire || !aligned(wire, 16) || wire_bytes < (size_t)W.total) return TAHQ_ERR_ARG;
  if (s.n > 0 && (!out || !aligned(out, 16))) return TAHQ_ERR_ARG;
  if (!workspace || !aligned(workspace, kAlign)) return TAHQ_ERR_WORKSPACE;
  const DecLayout L = dec_layout(s);
  const WireArrays A = wire_arrays(L.total, s.n);
  if (workspace_bytes < A.total) return TAHQ_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, L.ctot, cs) != cudaSuccess) return TAHQ_ERR_CUDA;
  tahq::WireUnpackArgs a{};
  a.wire = wire;
  a.scales = at<float>(workspace, A.scales);
  a.zeros = at<float>(workspace, A.zeros);
  a.bits = at<uint8_t>(workspace, A.bits);
  a.pivots = at<uint8_t>(workspace, A.pivots);
  a.status = at<uint32_t>(workspace, L.status);
  a.n = s.n;
  a.off_map = W.off_map;
  a.off_meta = W.off_meta;
  a.off_piv = W.off_piv;
  a.lo = s.lo;
  a.hi = s.hi;
  a.pb = W.pb;
  wire_header(s, budget, 0.0f, W, a.header);  // tau (word 11) is not compared
  if (tahq::launch_wire_unpack(a, cs) != cudaSuccess) return TAHQ_ERR_CUDA;
  return decode_impl(wire + W.off_pay, (size_t)W.pay, a.scales, a.zeros, a.bits, a.pivots,
                     tokens, channels, tile, hblock, out, workspace, L.total, stream, false);
}

}  // extern "C"

namespace {

// One thread waits in turn on eight counters that nothing advances.
__global__ void k_wait_probe(const uint32_t* counters, uint32_t* status,
                             unsigned long long limit_ns, unsigned long long* elapsed) {
  if (threadIdx.x != 0) return;
  const unsigned long long t0 = tahq::global_ns();
  unsigned long long gave_up = 0;
  for (int i = 0; i < 8; i++) gave_up += tahq::wait_counter(counters + i, 1u, status, limit_ns) ? 0 : 1;
  if (elapsed) {
    elapsed[0] = tahq::global_ns() - t0;
    elapsed[1] = gave_up;
  }
}

}  // namespace

extern "C" {

tahq_status tahq_test_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t limit_ns,
                                   uint64_t* elapsed_ns, void* stream) {
  if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < 1024) return TAHQ_ERR_WORKSPACE;
  if (limit_ns < 1 || limit_ns > 10000000000ull) return TAHQ_ERR_ARG;
  if (elapsed_ns && !aligned(elapsed_ns, 8)) return TAHQ_ERR_ARG;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, 1024, cs) != cudaSuccess) return TAHQ_ERR_CUDA;
  uint32_t* status = static_cast<uint32_t*>(workspace);
  const uint32_t* counters = at<uint32_t>(workspace, 512);
  k_wait_probe<<<1, 32, 0, cs>>>(counters, status, (unsigned long long)limit_ns,
                                 reinterpret_cast<unsigned long long*>(elapsed_ns));
  return cudaGetLastError() == cudaSuccess ? TAHQ_OK : TAHQ_ERR_CUDA;
}

tahq_status tahq_get_device_status(const void* workspace, uint32_t* status_out, void* stream) {
  if (!workspace) return TAHQ_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
    return TAHQ_ERR_CUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return TAHQ_ERR_CUDA;
  if (status_out) *status_out = word;
  return word ? TAHQ_ERR_DEVICE_STATUS : TAHQ_OK;
}

const char* tahq_status_string(int status) {
  switch (status) {
    case TAHQ_OK: return "TAHQ_OK";
    case TAHQ_ERR_ARG: return "TAHQ_ERR_ARG: an argument is outside the supported limits";
    case TAHQ_ERR_UNSUPPORTED: return "TAHQ_ERR_UNSUPPORTED: valid parameters not built here";
    case TAHQ_ERR_WORKSPACE: return "TAHQ_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case TAHQ_ERR_CUDA: return "TAHQ_ERR_CUDA: a CUDA call or kernel launch failed";
    case TAHQ_ERR_DEVICE_STATUS: return "TAHQ_ERR_DEVICE_STATUS: the device reported an error";
  }
  return "unknown tahq_status";
}

int tahq_version(void) { return kVersion; }

void tahq_log2_tables(float* T, float* R, float* k) {
  const LgTables& t = lg_tables();
  if (T) std::memcpy(T, t.T, sizeof t.T);
  if (R) std::memcpy(R, t.R, sizeof t.R);
  if (k) std::memcpy(k, t.k, sizeof t.k);
}

}  // extern "C"
