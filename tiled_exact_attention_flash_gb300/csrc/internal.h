// Host-side declarations shared by the library's translation units (not part
// of the public C ABI, which is include/flashmsa.h).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "flashmsa.h"

namespace fmsa {

// error reporting (api.cpp): store a message for flash_msa_last_error_string
flash_msa_status set_error(flash_msa_status code, const char* fmt, ...);
flash_msa_status set_cuda_error(const char* what);

// 4-D TMA map over a bf16 (B, N, H, d) tensor: dims (d, N, H, B), box
// (64, 128, 1, 1), 128-byte swizzle, zero fill past N.  Encoded on the host.
flash_msa_status make_tile_map(CUtensorMap* m, const void* base, int B, int64_t N, int H, int d);
// 4-D TMA map over an fp32 (B, H, NP, d) accumulator: dims (d, NP, H, B), box
// (32, 128, 1, 1), 128-byte swizzle (the target of bulk tensor reductions).
flash_msa_status make_acc_map(CUtensorMap* m, float* base, int B, int H, int64_t NP, int d);

// per-device state (status.cu)
unsigned* status_word_ptr();  // device address for the current device, or null on error
constexpr int kSchedSlots = 256;
struct SchedCounter {
  unsigned long long* counter;  // device address of the launch's work counter
  unsigned ticket;              // the launch's ticket (see claim_unit)
};
// A work counter of the current device for one launch, initialised on
// `stream` with a fresh ticket.
flash_msa_status claim_sched_counter(cudaStream_t stream, SchedCounter* out);
int sm_count();  // multiprocessors of the current device, 0 on error
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel (bit
// `which`, one per kernel instantiation) and device
flash_msa_status enable_smem(const void* kernel, int bytes, unsigned which, const char* what);
constexpr unsigned kDefaultWaitLimitMs = 4000;
unsigned wait_limit_ms();  // limit of any single bounded wait in the kernels
void set_wait_limit_ms(unsigned ms);
flash_msa_status launch_wait_timeout_probe(cudaStream_t stream);

struct FwdLaunch {
  const void *q, *k, *v;
  void* o;
  float* lse;
  int B, H, d;
  int Hkv;          // key/value heads (H % Hkv == 0; query head h reads kv head h / (H / Hkv))
  int64_t N;
  float scale;
  MaskParams mask;
  ListParams list;     // CSR by query block (or arithmetic)
  float pair_overlap;  // the index's pair_overlap (0 without an index)
  unsigned* status;
};
flash_msa_status launch_fwd(const FwdLaunch& a, cudaStream_t stream);

struct BwdLaunch {
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float* dsum;   // workspace: [-LSE * log2(e) | D], fp32 (B, H, padded N) each
  float* dqacc;  // workspace: fp32 dQ accumulator (B, H, padded N, d), or null
  int B, H, d;
  int Hkv;      // key/value heads
  int64_t N;
  float scale;
  MaskParams mask;
  ListParams rows;  // CSR by query block (dQ pass)
  ListParams cols;  // CSC by key block (dK/dV pass)
  unsigned* status;
  unsigned stages;  // FLASH_MSA_BWD_* bits
};
flash_msa_status launch_bwd(const BwdLaunch& a, cudaStream_t stream);

}  // namespace fmsa
