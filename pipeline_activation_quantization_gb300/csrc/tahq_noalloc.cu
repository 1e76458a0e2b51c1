// tahq_noalloc.cu -- decode for callers that cannot allocate device memory.
//
// tahq_decode needs a small device workspace (a status word, a block ticket, each decode
// chunk's offset inside its block of chunks and each block's stream offset).  Some
// callers have no way to provide it: a
// receiving pipeline stage driven by a runtime that plans all device memory ahead of
// time and hands the codec only its inputs and outputs, or a C caller without a
// device allocator of its own, for which a cudaMalloc in the receive loop would also
// synchronise the whole device.  tahq_decode_noalloc serves them from a fixed scratch
// array compiled into the library instead.
//
// The array lives in device memory of every GPU that loads the library, until the
// process exits.  In host code its name is only a host-side stand-in, so the device
// address is looked up once per device with cudaGetSymbolAddress and cached.
#include <mutex>

#include "../../include/tahq.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[TAHQ_NOALLOC_SCRATCH_BYTES];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device; looked up on the first call
// on each device (with that device current), nullptr if the lookup failed.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" tahq_status tahq_decode_noalloc(const uint8_t* codes, size_t codes_bytes,
                                           const float* scales, const float* zeros,
                                           const uint8_t* bits, const uint8_t* pivots,
                                           int64_t tokens, int64_t channels, int tile,
                                           int hblock, float* out, uint32_t* device_status,
                                           void* stream) {
  const size_t need = tahq_decode_workspace_size(tokens, channels, tile);
  if (need == 0) return TAHQ_ERR_ARG;
  if (need > (size_t)TAHQ_NOALLOC_SCRATCH_BYTES) return TAHQ_ERR_WORKSPACE;
  void* scratch = scratch_address();
  if (!scratch) return TAHQ_ERR_CUDA;
  // tahq_decode clears the part of the scratch it uses before launching its kernel.
  const tahq_status st = tahq_decode(codes, codes_bytes, scales, zeros, bits, pivots, tokens,
                                     channels, tile, hblock, out, scratch,
                                     (size_t)TAHQ_NOALLOC_SCRATCH_BYTES, stream);
  if (st != TAHQ_OK || !device_status) return st;
  // the status word sits at the head of the scratch
  if (cudaMemcpyAsync(device_status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TAHQ_ERR_CUDA;
  return TAHQ_OK;
}
