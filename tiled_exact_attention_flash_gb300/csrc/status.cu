// Per-device state of the library: the device status word shared by every
// kernel, the pool of work counters of the persistent kernels (both
// file-scope __device__ variables, so no allocation is needed), cached device
// attributes, the once-per-device kernel attribute setting and the limit of
// the kernels' bounded waits.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace fmsa {

constexpr int kMaxDevices = 64;

static __device__ unsigned g_status_word;

// Device ordinal of the calling thread's current device, or -1.
static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Address of a __device__ symbol on the current device, looked up once per
// device.  Concurrent first calls may both look it up; both store the same
// value into the atomic slot.
static void* symbol_address(std::atomic<void*> (&cache)[kMaxDevices], const void* symbol) {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  void* ptr = cache[dev].load(std::memory_order_acquire);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, symbol) != cudaSuccess) return nullptr;
    cache[dev].store(ptr, std::memory_order_release);
  }
  return ptr;
}

unsigned* status_word_ptr() {
  static std::atomic<void*> cache[kMaxDevices];
  return static_cast<unsigned*>(symbol_address(cache, reinterpret_cast<const void*>(&g_status_word)));
}

// Work counters of persistent launches.  Each launch takes the next slot
// round-robin and a fresh ticket, and sets both 32-bit halves of the slot to
// the ticket on its own stream before the kernel runs (see claim_unit in
// common.cuh).  Launches that overlap on the GPU (different streams) use
// different slots unless more than kSchedSlots of them are in flight at once;
// if they do share one, the kernels see a foreign ticket and report
// FLASH_MSA_ERR_SCHEDULE.
static __device__ unsigned long long g_sched[kSchedSlots];

static PFN_cuMemsetD32Async_v3020 memset_d32_fn() {
  static std::atomic<PFN_cuMemsetD32Async_v3020> fn{nullptr};
  PFN_cuMemsetD32Async_v3020 f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemsetD32Async", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<PFN_cuMemsetD32Async_v3020>(ptr);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

flash_msa_status claim_sched_counter(cudaStream_t stream, SchedCounter* out) {
  static std::atomic<void*> cache[kMaxDevices];
  static std::atomic<unsigned> next_slot{0};
  static std::atomic<unsigned> next_ticket{0};
  auto* base = static_cast<unsigned long long*>(
      symbol_address(cache, reinterpret_cast<const void*>(&g_sched)));
  if (!base) return set_cuda_error("work counter: symbol address");
  PFN_cuMemsetD32Async_v3020 memset32 = memset_d32_fn();
  if (!memset32) return set_error(FLASH_MSA_ERR_CUDA, "cuMemsetD32Async is not available");
  out->counter = base + (next_slot.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
  // tickets 1 .. 2^31 - 1: the low half (ticket + claims) stays below 2^32
  out->ticket = next_ticket.fetch_add(1, std::memory_order_relaxed) % 0x7FFFFFFFu + 1u;
  const CUresult r = memset32(reinterpret_cast<CUdeviceptr>(out->counter), out->ticket, 2,
                              reinterpret_cast<CUstream>(stream));
  if (r != CUDA_SUCCESS)
    return set_error(FLASH_MSA_ERR_CUDA, "work counter reset failed (CUresult %d)", int(r));
  return FLASH_MSA_OK;
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Large dynamic shared memory must be enabled per kernel and per device; the
// bit `which` of the current device's mask records that it was.
flash_msa_status enable_smem(const void* kernel, int bytes, unsigned which, const char* what) {
  static std::atomic<unsigned> done[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return set_cuda_error("cudaGetDevice");
  const unsigned bit = 1u << which;
  if (done[dev].load(std::memory_order_acquire) & bit) return FLASH_MSA_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return set_cuda_error(what);
  done[dev].fetch_or(bit, std::memory_order_acq_rel);
  return FLASH_MSA_OK;
}

// Limit of any single bounded wait inside the kernels (process-wide).
static std::atomic<unsigned> g_wait_limit_ms{kDefaultWaitLimitMs};

unsigned wait_limit_ms() { return g_wait_limit_ms.load(std::memory_order_relaxed); }

void set_wait_limit_ms(unsigned ms) { g_wait_limit_ms.store(ms, std::memory_order_relaxed); }

// Failure-detection probe: one thread waits, through the same bounded wait
// every kernel of the library uses, on an mbarrier that nothing arrives on.
// The wait gives up after kProbeWaitMs and records FLASH_MSA_ERR_TIMEOUT
// (site kTimeoutProbeSite) in the status word; the kernel then returns, so
// the context stays usable.
constexpr unsigned kTimeoutProbeSite = 0xEE;
constexpr int kProbeWaitMs = 200;

__global__ void wait_timeout_probe_kernel(unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int ctl[2];  // abort flag, wait limit (ms)
  if (threadIdx.x != 0) return;
  ctl[0] = 0;
  ctl[1] = kProbeWaitMs;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  wait_bar(smem_u32(&bar), 0, ctl, status, kTimeoutProbeSite);
}

flash_msa_status launch_wait_timeout_probe(cudaStream_t stream) {
  unsigned* status = status_word_ptr();
  if (!status) return set_cuda_error("selftest: status word");
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status);
  if (cudaGetLastError() != cudaSuccess) return set_cuda_error("selftest: launch");
  return FLASH_MSA_OK;
}

}  // namespace fmsa
