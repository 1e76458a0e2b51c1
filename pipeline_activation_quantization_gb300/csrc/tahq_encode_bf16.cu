// tahq_encode_bf16.cu -- encode kernels for bf16 input (one translation unit per
// input type, so that the two compile in parallel).
#include "tahq_encode.cuh"

namespace tahq {

cudaError_t launch_encode_bf16(const EncodeArgs& a, cudaStream_t st) {
  switch (a.G) {
    case 8: return run_encode<uint16_t, 8>(a, st);
    case 16: return run_encode<uint16_t, 16>(a, st);
    case 32: return run_encode<uint16_t, 32>(a, st);
    case 64: return run_encode<uint16_t, 64>(a, st);
    case 128: return run_encode<uint16_t, 128>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tahq
