// tahq_launch.h -- host-side launch interface between the C ABI (tahq_api.cu) and the
// kernel translation units (tahq_encode.cu, tahq_decode.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tahq_device.cuh"

namespace tahq {

// Everything one encode launch sequence needs; pointers are device pointers carved out
// of the caller's output buffers and workspace.
struct EncodeArgs {
  const void* x;
  bool bf16;
  int G, h, lo, hi;
  float c_h;                 // RN(1/sqrt(h))
  float tau;                 // outlier threshold: transform where r > tau (>= 0, +inf: never)
  bool wire;                 // fp16 zero and scales of the wire format (else the fp32 quantiser)
  float scale_c = 1.0f;      // streaming encoder only: the codec sees RN(c x) (c a power of two)
  int mlog;                  // allocation tiles of 2^mlog tiles (one key each); K counts them
  long long n_tiles, n_g, n_groups, K, group_bytes;
  int num_sms;
  const LgTables* tabs;
  uint8_t* codes;
  float* scales;
  float* zeros;
  uint8_t* bits;
  uint8_t* pivots;
  // workspace
  uint32_t* status;
  uint32_t* ticket;
  uint32_t* cand_cnt;        // [n_groups]
  uint32_t* doneA;           // [n_groups] finished stats items
  uint32_t* doneB;           // [n_groups] finished select items
  uint32_t* doneB2;          // [n_groups] finished offsets items
  uint32_t* selready;        // [n_groups] 1 once sel[g] is published
  SelResult* sel;            // [n_groups]
  uint32_t* hist_coarse;     // [n_groups * kCoarseBins]
  uint32_t* hist_fine;       // [n_groups * kFineBins]
  unsigned long long* lookback;  // [encode_chunks] compaction chunk counts, then offsets
  float* keys;               // [n_tiles]
  unsigned long long* cand;  // [n_tiles]
  uint32_t* segmask;         // [n_groups * ceil(n_g / 32)] hi tiles of each 32-tile segment
  uint8_t* scratch_lo;       // [n_tiles * G * lo / 8] every tile quantised at bits_lo
  uint8_t* scratch_hi;       // [n_tiles * G * hi / 8] every tile quantised at bits_hi
  unsigned long long* items; // [items_cap] the decoded work queue
  long long items_cap;
  unsigned long long wait_ns;  // bound of every wait in the kernels (0: kWaitNs)
};

struct DecodeArgs {
  const uint8_t* codes;
  unsigned long long codes_bytes;
  const float* scales;
  const float* zeros;
  const uint8_t* bits;
  const uint8_t* pivots;
  int G, h;
  float c_h;
  long long n_tiles;
  int num_sms;
  float* out;
  uint32_t* status;
  uint32_t* ticket;
  uint32_t* ctot;                // [decode_chunks] chunk offset inside its block of 8 chunks
  unsigned long long* bsum;      // [decode_blocks + 1] stream offset of each block of 8
                                 // chunks, then the end of the last slot
  float inv_c = 1.0f;            // every output value is RN(value x inv_c) (a power of two)
};

// Encode geometry: bytes of input per tiles item; tiles per compaction chunk, at most.
constexpr int kEncChunkBytes = 32768;
constexpr int kEncMaxCC = 2048;

// Tiles per compaction chunk of the encode kernel, and the number of compaction chunks
// (one offset word each) for these shapes.
long long encode_cchunk_tiles(int bf16, int G, int hi);
long long encode_chunks(int bf16, int G, int hi, long long n_g, long long n_groups);
// Select (and offsets) items per group; work-queue items of a whole encode.
long long encode_sel_items(long long nA, long long nC);
long long encode_queue_items(int bf16, int G, int hi, long long n_g, long long n_groups);
// Number of decode chunks, and of blocks of kDecChunksPerBlock chunks, for these shapes.
constexpr int kDecChunksPerBlock = 8;
long long decode_chunks(int G, long long n_tiles);
inline long long decode_blocks(int G, long long n_tiles) {
  return (decode_chunks(G, n_tiles) + kDecChunksPerBlock - 1) / kDecChunksPerBlock;
}

// Wire format (tahq_wire.cu): per-tile metadata into / out of one buffer.  Offsets are
// byte offsets of the sections in `wire` (16-byte aligned); header = its 128 bytes.
struct WirePackArgs {
  const float* scales;   // [n] fp16-exact scales
  const float* zeros;    // [n] fp16-exact zeros
  const uint8_t* bits;   // [n]
  const uint8_t* pivots; // [n] 0xFF = untransformed
  uint8_t* wire;
  long long n, off_map, off_meta, off_piv, off_pay, pay, total;
  int hi, pb;
  uint32_t header[32];
};
struct WireUnpackArgs {
  const uint8_t* wire;
  float* scales;
  float* zeros;
  uint8_t* bits;
  uint8_t* pivots;
  uint32_t* status;      // kStBadWire when the header differs from `header` (tau aside)
  long long n, off_map, off_meta, off_piv;
  int lo, hi, pb;
  uint32_t header[32];
};

cudaError_t launch_encode(const EncodeArgs& a, cudaStream_t st);
cudaError_t launch_wire_pack(const WirePackArgs& a, cudaStream_t st);
cudaError_t launch_wire_unpack(const WireUnpackArgs& a, cudaStream_t st);
cudaError_t launch_encode_f32(const EncodeArgs& a, cudaStream_t st);
cudaError_t launch_encode_bf16(const EncodeArgs& a, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);

}  // namespace tahq
