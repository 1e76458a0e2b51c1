// tahq_encode.cu -- host side of the encode launch: geometry of the compaction chunks
// and the dispatch to the per-input-type instantiations (tahq_encode_f32.cu,
// tahq_encode_bf16.cu).
#include <algorithm>

#include "tahq_launch.h"

namespace tahq {

long long encode_cchunk_tiles(int bf16, int G, int hi) {
  const long long ch = kEncChunkBytes / (G * (bf16 ? 2 : 4));
  long long m = 1;
  while (m < 8 && 2 * m * ch * G * hi / 8 <= kEncChunkBytes - 64 && 2 * m * ch <= kEncMaxCC) m *= 2;
  return m * ch;
}

long long encode_chunks(int bf16, int G, int hi, long long n_g, long long n_groups) {
  const long long chc = encode_cchunk_tiles(bf16, G, hi);
  return n_groups * ((n_g + chc - 1) / chc);
}

// An offsets item covers at most 256 compaction chunks (their counts collect in shared
// memory); otherwise one select / offsets item per 32 tiles items, at most 256 (fewer,
// larger items spend less of their time waiting and synchronising; measured on 64 MiB
// groups: 1/8 -> 0.79 ms, 1/32 -> 0.72 ms, 1/64 -> 0.83 ms per encode).
long long encode_sel_items(long long nA, long long nC) {
  return std::max<long long>({1ll, std::min<long long>(256, nA / 32), (nC + 255) / 256});
}

long long encode_queue_items(int bf16, int G, int hi, long long n_g, long long n_groups) {
  const long long ch = kEncChunkBytes / (G * (bf16 ? 2 : 4));
  const long long nA = (n_g + ch - 1) / ch;
  const long long chc = encode_cchunk_tiles(bf16, G, hi);
  const long long nC = (n_g + chc - 1) / chc;
  return n_groups * (nA + 2 * encode_sel_items(nA, nC) + nC);
}

cudaError_t launch_encode(const EncodeArgs& a, cudaStream_t st) {
  return a.bf16 ? launch_encode_bf16(a, st) : launch_encode_f32(a, st);
}

}  // namespace tahq
