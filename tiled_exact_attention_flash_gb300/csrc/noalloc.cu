// flash_msa_bwd_noalloc: the backward pass for callers that are not allowed
// to allocate device memory at call time -- e.g. a host program whose
// framework owns the whole device memory pool and hands out no extra
// buffers, or a latency-critical loop in which cudaMalloc / cudaFree are
// banned because they can synchronise the whole device.  Such a caller cannot
// provide the workspace flash_msa_bwd() asks for, so this entry point uses a
// fixed scratch array that is part of the library image instead.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  All calls
// on a device share it and it keeps whatever the previous call left there;
// the backward's first launch rewrites every element it later reads, so
// nothing needs clearing between calls.  Calls whose kernels overlap on the
// GPU (different streams, no ordering between them) race on the array.
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"

namespace fmsa {

// 16 MiB: two fp32 vectors of B * H * ceil(N/128) * 128 entries, i.e.
// B * H * ceil(N/128) * 128 <= 2^21 (for example B*H = 32 heads at N = 65536).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

// Device address of the scratch array for the current device.  Host code may
// not pass g_bwd_scratch itself to a kernel: in host code that name is a
// host-side stand-in, not a device address.  Looked up once per device
// (threads making their first calls at the same time may both look it up and
// store the same value).
static flash_msa_status scratch_address(void** out) {
  constexpr int kMaxDevices = 64;
  static std::atomic<void*> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_cuda_error("bwd_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(FLASH_MSA_ERR_CUDA, "bwd_noalloc: device ordinal %d out of range", dev);
  void* ptr = cache[dev].load(std::memory_order_acquire);
  if (!ptr) {
    const cudaError_t rc = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (rc != cudaSuccess || !ptr)
      return set_error(FLASH_MSA_ERR_CUDA, "bwd_noalloc: cudaGetSymbolAddress failed: %s",
                       cudaGetErrorString(rc));
    cache[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return FLASH_MSA_OK;
}

}  // namespace fmsa

using namespace fmsa;

extern "C" flash_msa_status flash_msa_bwd_noalloc(const void* q, const void* k, const void* v,
                                                  const void* o, const float* lse, const void* dO,
                                                  void* dq, void* dk, void* dv, int B, int H,
                                                  int64_t N, int d, float scale,
                                                  const flash_msa_mask_desc* mask, void* stream) {
  const size_t need = flash_msa_bwd_workspace_bytes(B, H, N, d);
  if (need > kNoAllocScratchBytes)
    return set_error(FLASH_MSA_ERR_WORKSPACE,
                     "bwd_noalloc: B=%d H=%d N=%lld needs %zu bytes of scratch, more than the "
                     "fixed %zu bytes; use flash_msa_bwd() with a caller-provided workspace",
                     B, H, static_cast<long long>(N), need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  const flash_msa_status st = scratch_address(&scratch);
  if (st != FLASH_MSA_OK) return st;
  // Same kernels and launches as flash_msa_bwd(); only the workspace differs.
  // need == 0 means invalid sizes, which flash_msa_bwd() reports.
  return flash_msa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, mask, scratch,
                       kNoAllocScratchBytes, stream);
}
