// The device status word shared by every kernel of the library, one per
// device, and the pool of work counters of the persistent kernels (both
// file-scope __device__ variables, so no allocation is needed).
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
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

// Work counters of persistent launches.  Each launch takes the next slot
// round-robin and zeroes it on its own stream before the kernel runs, so
// launches that overlap on the GPU (different streams) use different slots
// unless more than kSchedSlots of them are in flight at once.
static __device__ int g_sched[kSchedSlots];

int* sched_counter() {
  constexpr int kMaxDevices = 64;
  static int* cache[kMaxDevices] = {};
  static std::atomic<unsigned> next{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_sched) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int*>(ptr);
  }
  return cache[dev] + (next.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
}

int sm_count() {
  constexpr int kMaxDevices = 64;
  static int cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// Failure-detection probe: one thread waits, through the same bounded wait
// every kernel of the library uses, on an mbarrier that nothing arrives on.
// The wait gives up after kWaitLimitNs and records FLASH_MSA_ERR_TIMEOUT
// (site kTimeoutProbeSite) in the status word; the kernel then returns, so
// the context stays usable.
constexpr unsigned kTimeoutProbeSite = 0xEE;

__global__ void wait_timeout_probe_kernel(unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  wait_bar(smem_u32(&bar), 0, &abort_flag, status, kTimeoutProbeSite);
}

flash_msa_status launch_wait_timeout_probe(cudaStream_t stream) {
  unsigned* status = status_word_ptr();
  if (!status) return set_cuda_error("selftest: status word");
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status);
  if (cudaGetLastError() != cudaSuccess) return set_cuda_error("selftest: launch");
  return FLASH_MSA_OK;
}

}  // namespace fmsa
