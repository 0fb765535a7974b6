// The device status word shared by every kernel of the library, one per
// device (a file-scope __device__ variable, so no allocation is needed).
#include <cuda_runtime.h>

#include "internal.h"

namespace fmsa {

static __device__ unsigned g_status_word;

unsigned* status_word_ptr() {
  constexpr int kMaxDevices = 64;
  static unsigned* cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned*>(ptr);
  }
  return cache[dev];
}

}  // namespace fmsa
