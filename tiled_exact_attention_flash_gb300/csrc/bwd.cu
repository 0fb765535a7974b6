// Backward attention kernels for sm_103a.  Recompute backward ("Flash MSA
// Attention Kernel Implementation", section "The Backward Pass: The Real
// Beast"): with P = exp(scale S - LSE) recomputed from Q, K and the stored
// LSE,
//     dV = P^T dO,  dP = dO V^T,  D = rowsum(dO o O),  dS = P o (dP - D),
//     dQ = scale dS K,  dK = scale dS^T Q.
// (rowsum(P o dP) = rowsum(dO o O) because O = P V.)
//
// Three launches:
//   bwd_pre   D_i = sum_c dO_ic O_ic and LSE_i * log2(e), padded to whole
//             128-row tiles (padding rows get LSE = +inf, so P = 0 there)
//   bwd_dkdv  key-stationary: per (b, h, key tile) loop over the live query
//             tiles; S^T = K Q^T and dP^T = V dO^T in TMEM, P^T and dS^T
//             written back to TMEM as bf16, dV += P^T dO and dK += dS^T Q
//             accumulated in TMEM
//   bwd_dq    query-stationary: per (b, h, query tile) loop over the live key
//             tiles; S = Q K^T, dP = dO V^T, dS to TMEM, dQ += dS K in TMEM
// Each tile pair costs 4 + 3 tensor-core products; no atomics, so all three
// outputs are deterministic.
//
// CTA layout of the two main kernels (256 threads, one CTA per SM):
//   warp 0 TMA producer (one lane), warp 1 MMA issuer (one lane), warp 2
//   TMEM allocator, warps 4-7 elementwise work, thread = row of the
//   stationary tile (key row in bwd_dkdv, query row in bwd_dq).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fmsa {

constexpr int kBwdThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// bwd_pre
// ---------------------------------------------------------------------------
struct PreParams {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  float* lse2;  // (B, H, NP)
  float* dsum;  // (B, H, NP)
  int B, H, N, NP;
};

template <int HD>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreParams p) {
  constexpr int kTpr = HD / 8;            // threads per row, 8 bf16 (16 bytes) each
  constexpr int kRows = 256 / kTpr;       // rows per block
  const int h = blockIdx.y, b = blockIdx.z;
  const int r = threadIdx.x / kTpr, c = threadIdx.x % kTpr;
  const int64_t i = int64_t(blockIdx.x) * kRows + r;  // grid covers NP exactly
  float acc = 0.f;
  if (i < p.N) {
    const int64_t off = ((int64_t(b) * p.N + i) * p.H + h) * HD + c * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(p.o + off);
    const uint4 gv = *reinterpret_cast<const uint4*>(p.dout + off);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 of = __bfloat1622float2(o2[e]);
      const float2 gf = __bfloat1622float2(g2[e]);
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
  }
#pragma unroll
  for (int s = kTpr / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, s, kTpr);
  if (c == 0 && i < p.NP) {
    const int64_t at = (int64_t(b) * p.H + h) * p.NP + i;
    float l2 = INFINITY;
    if (i < p.N) {
      const float l = p.lse[(int64_t(b) * p.H + h) * p.N + i];
      l2 = (l == -INFINITY) ? INFINITY : l * kLog2e;
    }
    p.lse2[at] = l2;
    p.dsum[at] = acc;
  }
}

// ---------------------------------------------------------------------------
// shared layout pieces for the two main kernels
// ---------------------------------------------------------------------------
struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  __nv_bfloat16* out_a;  // dkdv: dK, dq: dQ
  __nv_bfloat16* out_b;  // dkdv: dV
  const float* lse2;
  const float* dsum;
  int B, H, N, NP;
  int n_units;
  float scale, scale_log2;
  MaskParams mask;
  ListParams list;
  unsigned* status;
};

template <int HD>
struct BwdLayout {
  static constexpr int kTileBytes = kTile * HD * 2;
  static constexpr int kStages = HD == 128 ? 4 : 8;  // even: tiles come in pairs
  static constexpr int kFixOff = 0;                  // two stationary tiles
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kVecOff = kRingOff + kStages * kTileBytes;  // (stages/2) x 1 KB
  static constexpr int kBarOff = kVecOff + (kStages / 2) * 1024;
  static constexpr int kFixFull = 0, kFixEmpty = 1, kSFull = 2, kPFull = 3, kAccFull = 4,
                       kAccEmpty = 5, kMmaDone = 6, kRingFull = 7, kRingEmpty = 7 + kStages;
  static constexpr int kNumBars = 7 + 2 * kStages;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
};

template <int HD>
__device__ __forceinline__ void load_tile_2d(const CUtensorMap* m, uint32_t dst, uint32_t bar,
                                             int row, int h, int b) {
#pragma unroll
  for (int c = 0; c < HD / 64; ++c) tma_load_4d(dst + c * (kTile * 128), m, bar, c * 64, row, h, b);
}

__device__ __forceinline__ bool next_unit(int& k, Unit& un, const BwdParams& p) {
  while (true) {
    const int u = int(blockIdx.x) + k * int(gridDim.x);
    if (u >= p.n_units) return false;
    ++k;
    un = decode_unit(u, p.H, p.list, p.status);
    if (un.n > 0) return true;
  }
}

template <int HD>
__device__ __forceinline__ void init_bwd_barriers(uint64_t* bars) {
  using L = BwdLayout<HD>;
  mbar_init(smem_u32(bars + L::kFixFull), 1);
  mbar_init(smem_u32(bars + L::kFixEmpty), 1);
  mbar_init(smem_u32(bars + L::kSFull), 1);
  mbar_init(smem_u32(bars + L::kPFull), 128);
  mbar_init(smem_u32(bars + L::kAccFull), 1);
  mbar_init(smem_u32(bars + L::kAccEmpty), 128);
  mbar_init(smem_u32(bars + L::kMmaDone), 1);
  for (int i = 0; i < L::kStages; ++i) {
    mbar_init(smem_u32(bars + L::kRingFull + i), 1);
    mbar_init(smem_u32(bars + L::kRingEmpty + i), 1);
  }
  fence_mbar_init();
}

// Producer shared by both kernels.  Per unit: the two stationary tiles
// (dkdv: K, V of the key block; dq: Q, dO of the query block), then per inner
// tile two ring stages (dkdv: Q_t + its LSE2/D vectors, dO_t; dq: K_t, V_t).
template <int HD, bool kKeyStationary>
__device__ __forceinline__ void bwd_producer(const BwdParams& p, uint8_t* smem, uint64_t* bars,
                                             volatile int* abort_flag) {
  using L = BwdLayout<HD>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const CUtensorMap* fix_a = kKeyStationary ? &p.tm_k : &p.tm_q;
  const CUtensorMap* fix_b = kKeyStationary ? &p.tm_v : &p.tm_do;
  const CUtensorMap* ring_a = kKeyStationary ? &p.tm_q : &p.tm_k;
  const CUtensorMap* ring_b = kKeyStationary ? &p.tm_do : &p.tm_v;
  uint32_t cnt = 0, fe_cnt = 0;
  int last[L::kStages];
  for (int i = 0; i < L::kStages; ++i) last[i] = -1;
  int last_fix = -1;
  bool ok = true;
  int k = 0;
  Unit un;
  while (ok && next_unit(k, un, p)) {
    if (!wait_bar(bar(L::kFixEmpty), (fe_cnt & 1) ^ 1, abort_flag, p.status, 1)) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(bar(L::kFixFull), 2 * L::kTileBytes);
    load_tile_2d<HD>(fix_a, smem_u32(smem + L::kFixOff), bar(L::kFixFull), un.ob * kTile, un.h,
                     un.b);
    load_tile_2d<HD>(fix_b, smem_u32(smem + L::kFixOff + L::kTileBytes), bar(L::kFixFull),
                     un.ob * kTile, un.h, un.b);
    last_fix = int(fe_cnt);
    ++fe_cnt;
    for (int t = 0; t < un.n && ok; ++t) {
      const InnerTile it = inner_tile(un, t, p.list, p.status);
      for (int half = 0; half < 2; ++half) {
        const int stage = cnt % L::kStages;
        if (!wait_bar(bar(L::kRingEmpty + stage), ((cnt / L::kStages) & 1) ^ 1, abort_flag,
                      p.status, 2)) {
          ok = false;
          break;
        }
        const uint32_t dst = smem_u32(smem + L::kRingOff + stage * L::kTileBytes);
        if (half == 0) {
          const bool vec = kKeyStationary;
          mbar_arrive_expect_tx(bar(L::kRingFull + stage), L::kTileBytes + (vec ? 1024 : 0));
          load_tile_2d<HD>(ring_a, dst, bar(L::kRingFull + stage), it.blk * kTile, un.h, un.b);
          if (vec) {
            const int64_t row0 = (int64_t(un.b) * p.H + un.h) * p.NP + int64_t(it.blk) * kTile;
            const uint32_t vdst = smem_u32(smem + L::kVecOff + (stage / 2) * 1024);
            bulk_load(vdst, p.lse2 + row0, 512, bar(L::kRingFull + stage));
            bulk_load(vdst + 512, p.dsum + row0, 512, bar(L::kRingFull + stage));
          }
        } else {
          mbar_arrive_expect_tx(bar(L::kRingFull + stage), L::kTileBytes);
          load_tile_2d<HD>(ring_b, dst, bar(L::kRingFull + stage), it.blk * kTile, un.h, un.b);
        }
        last[stage] = int(cnt);
        ++cnt;
      }
    }
  }
  if (!ok) {
    for (int i = 0; i < L::kStages; ++i)
      if (last[i] >= 0) drain_bar(bar(L::kRingFull + i), (last[i] / L::kStages) & 1);
    if (last_fix >= 0) drain_bar(bar(L::kFixFull), last_fix & 1);
  }
}

// MMA issuer shared by both kernels.
//  dkdv: tS = K Q_t^T, tD = V dO_t^T; then dV (+)= P^T dO_t, dK (+)= dS^T Q_t
//  dq:   tS = Q K_t^T, tD = dO V_t^T; then dQ (+)= dS K_t
// TMEM columns: tS [0,128), tD [128,256), acc0 [256, 256+d), acc1 [384, 384+d).
template <int HD, bool kKeyStationary>
__device__ __forceinline__ void bwd_mma(const BwdParams& p, uint8_t* smem, uint64_t* bars,
                                        uint32_t tmem, volatile int* abort_flag) {
  using L = BwdLayout<HD>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdAcc = idesc_bf16_f32(128, HD, false, true);
  const uint32_t tS = tmem, tD = tmem + 128, tA0 = tmem + 256, tA1 = tmem + 384;
  const uint32_t fa = smem_u32(smem + L::kFixOff);
  const uint32_t fb = fa + L::kTileBytes;
  uint32_t cnt = 0, ff_cnt = 0, sp_cnt = 0, ae_cnt = 0;
  bool ok = true;
  int k = 0;
  Unit un;
  while (ok && next_unit(k, un, p)) {
    if (!wait_bar(bar(L::kFixFull), ff_cnt & 1, abort_flag, p.status, 10)) {
      ok = false;
      break;
    }
    ++ff_cnt;
    for (int t = 0; t < un.n; ++t) {
      const int sa = cnt % L::kStages, sb = (cnt + 1) % L::kStages;
      if (!wait_bar(bar(L::kRingFull + sa), (cnt / L::kStages) & 1, abort_flag, p.status, 11) ||
          !wait_bar(bar(L::kRingFull + sb), ((cnt + 1) / L::kStages) & 1, abort_flag, p.status,
                    12)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t ra = smem_u32(smem + L::kRingOff + sa * L::kTileBytes);
      const uint32_t rb = smem_u32(smem + L::kRingOff + sb * L::kTileBytes);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk / 4) * (kTile * 128) + (kk % 4) * 32;
        mma_ss(tS, sdesc_sw128(fa + off, 16, 1024), sdesc_sw128(ra + off, 16, 1024), kIdS,
               kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk / 4) * (kTile * 128) + (kk % 4) * 32;
        mma_ss(tD, sdesc_sw128(fb + off, 16, 1024), sdesc_sw128(rb + off, 16, 1024), kIdS,
               kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kSFull));
      if (t == 0) {
        if (!wait_bar(bar(L::kAccEmpty), (ae_cnt & 1) ^ 1, abort_flag, p.status, 13)) {
          ok = false;
          break;
        }
        ++ae_cnt;
      }
      if (!wait_bar(bar(L::kPFull), sp_cnt & 1, abort_flag, p.status, 14)) {
        ok = false;
        break;
      }
      ++sp_cnt;
      tc_fence_after();
      if (kKeyStationary) {
        // dV += P^T dO_t (P^T bf16 in tS), dK += dS^T Q_t (dS^T bf16 in tD)
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t bo = sdesc_sw128(rb + kk * 2048, kTile * 128, 1024);
          mma_ts(tA0, tS + kk * 8, bo, kIdAcc, (t > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t bq = sdesc_sw128(ra + kk * 2048, kTile * 128, 1024);
          mma_ts(tA1, tD + kk * 8, bq, kIdAcc, (t > 0 || kk > 0) ? 1u : 0u);
        }
      } else {
        // dQ += dS K_t (dS bf16 in tS)
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t bk = sdesc_sw128(ra + kk * 2048, kTile * 128, 1024);
          mma_ts(tA0, tS + kk * 8, bk, kIdAcc, (t > 0 || kk > 0) ? 1u : 0u);
        }
      }
      mma_commit(bar(L::kRingEmpty + sa));
      mma_commit(bar(L::kRingEmpty + sb));
      cnt += 2;
    }
    if (!ok) break;
    mma_commit(bar(L::kFixEmpty));
    mma_commit(bar(L::kAccFull));
  }
  mma_commit(bar(L::kMmaDone));
  drain_bar(bar(L::kMmaDone), 0);
}

// Write 32 fp32 TMEM columns of one row, times `mul`, as bf16 to global.
__device__ __forceinline__ void store_row_chunk(uint32_t taddr, float mul, __nv_bfloat16* dst,
                                                bool valid) {
  uint32_t v[32];
  tmem_ld_x32(taddr, v);
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 16; ++j)
    w[j] = pack_bf16x2(__uint_as_float(v[2 * j]) * mul, __uint_as_float(v[2 * j + 1]) * mul);
  if (valid) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int j = 0; j < 4; ++j) d4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

__device__ __forceinline__ void zero_row(__nv_bfloat16* dst, int hd, bool valid) {
  if (!valid) return;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int j = 0; j < hd / 8; ++j) d4[j] = make_uint4(0, 0, 0, 0);
}

// Elementwise warpgroup of bwd_dkdv: thread = key row j of the key tile.
template <int HD>
__device__ __forceinline__ void dkdv_elementwise(const BwdParams& p, uint8_t* smem,
                                                 uint64_t* bars, uint32_t tmem,
                                                 volatile int* abort_flag) {
  using L = BwdLayout<HD>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int wq = int(warp_id()) & 3;
  const int row = wq * 32 + int(lane_id());
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t tS = tmem + lane_off, tD = tS + 128, tDV = tS + 256, tDK = tS + 384;
  const float sl2 = p.scale_log2;
  uint32_t sp_cnt = 0, af_cnt = 0, cnt = 0;
  for (int k = 0;; ++k) {
    const int u = int(blockIdx.x) + k * int(gridDim.x);
    if (u >= p.n_units) break;
    const Unit un = decode_unit(u, p.H, p.list, p.status);
    const int64_t j = int64_t(un.ob) * kTile + row;  // key token
    const bool valid = j < p.N;
    __nv_bfloat16* dk_row = p.out_a + ((int64_t(un.b) * p.N + j) * p.H + un.h) * HD;
    __nv_bfloat16* dv_row = p.out_b + ((int64_t(un.b) * p.N + j) * p.H + un.h) * HD;
    if (un.n == 0) {
      zero_row(dk_row, HD, valid);
      zero_row(dv_row, HD, valid);
      continue;
    }
    for (int t = 0; t < un.n; ++t) {
      const InnerTile it = inner_tile(un, t, p.list, p.status);
      int lo = 0, hi = kTile - 1;
      if (it.dead) hi = -1;
      else if (it.partial) col_live_range(j, it.blk, un.ob, p.N, p.mask, lo, hi);
      const float* vec =
          reinterpret_cast<const float*>(smem + L::kVecOff + ((cnt % L::kStages) / 2) * 1024);
      cnt += 2;
      bool ok = wait_bar(bar(L::kSFull), sp_cnt & 1, abort_flag, p.status, 20);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      ++sp_cnt;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t s[32], dp[32], pp[16], dd[16];
        tmem_ld_x32(tS + ch * 32, s);
        tmem_ld_x32(tD + ch * 32, dp);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int c = ch * 32 + e;
          const float4 ld = *reinterpret_cast<const float4*>(vec + (c & ~3));
          const float2 dv2 = *reinterpret_cast<const float2*>(vec + 128 + c);
          const float l0 = (c & 2) ? ld.z : ld.x;
          const float l1 = (c & 2) ? ld.w : ld.y;
          float p0 = ex2_approx(fmaf(__uint_as_float(s[e]), sl2, -l0));
          float p1 = ex2_approx(fmaf(__uint_as_float(s[e + 1]), sl2, -l1));
          if (c < lo || c > hi) p0 = 0.f;
          if (c + 1 < lo || c + 1 > hi) p1 = 0.f;
          const float d0 = p0 * (__uint_as_float(dp[e]) - dv2.x);
          const float d1 = p1 * (__uint_as_float(dp[e + 1]) - dv2.y);
          pp[e / 2] = pack_bf16x2(p0, p1);
          dd[e / 2] = pack_bf16x2(d0, d1);
        }
        tmem_st_x16(tS + ch * 16, pp);
        tmem_st_x16(tD + ch * 16, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::kPFull));
    }
    bool ok = wait_bar(bar(L::kAccFull), af_cnt & 1, abort_flag, p.status, 21);
    if (!__all_sync(0xFFFFFFFFu, ok)) return;
    ++af_cnt;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      store_row_chunk(tDV + c * 32, 1.f, dv_row + c * 32, valid);
      store_row_chunk(tDK + c * 32, p.scale, dk_row + c * 32, valid);
    }
    tc_fence_before();
    mbar_arrive(bar(L::kAccEmpty));
  }
}

// Elementwise warpgroup of bwd_dq: thread = query row i of the query tile.
template <int HD>
__device__ __forceinline__ void dq_elementwise(const BwdParams& p, uint64_t* bars, uint32_t tmem,
                                               volatile int* abort_flag) {
  using L = BwdLayout<HD>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int wq = int(warp_id()) & 3;
  const int row = wq * 32 + int(lane_id());
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t tS = tmem + lane_off, tD = tS + 128, tDQ = tS + 256;
  const float sl2 = p.scale_log2;
  uint32_t sp_cnt = 0, af_cnt = 0;
  for (int k = 0;; ++k) {
    const int u = int(blockIdx.x) + k * int(gridDim.x);
    if (u >= p.n_units) break;
    const Unit un = decode_unit(u, p.H, p.list, p.status);
    const int64_t i = int64_t(un.ob) * kTile + row;
    const bool valid = i < p.N;
    __nv_bfloat16* dq_row = p.out_a + ((int64_t(un.b) * p.N + i) * p.H + un.h) * HD;
    if (un.n == 0) {
      zero_row(dq_row, HD, valid);
      continue;
    }
    const int64_t vrow = (int64_t(un.b) * p.H + un.h) * p.NP + i;
    const float l2 = p.lse2[vrow];
    const float di = p.dsum[vrow];
    for (int t = 0; t < un.n; ++t) {
      const InnerTile it = inner_tile(un, t, p.list, p.status);
      int lo = 0, hi = kTile - 1;
      if (it.dead) hi = -1;
      else if (it.partial) row_live_range(i, un.ob, it.blk, p.N, p.mask, lo, hi);
      bool ok = wait_bar(bar(L::kSFull), sp_cnt & 1, abort_flag, p.status, 20);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      ++sp_cnt;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t s[32], dp[32], dd[16];
        tmem_ld_x32(tS + ch * 32, s);
        tmem_ld_x32(tD + ch * 32, dp);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int c = ch * 32 + e;
          float p0 = ex2_approx(fmaf(__uint_as_float(s[e]), sl2, -l2));
          float p1 = ex2_approx(fmaf(__uint_as_float(s[e + 1]), sl2, -l2));
          if (c < lo || c > hi) p0 = 0.f;
          if (c + 1 < lo || c + 1 > hi) p1 = 0.f;
          dd[e / 2] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - di),
                                  p1 * (__uint_as_float(dp[e + 1]) - di));
        }
        tmem_st_x16(tS + ch * 16, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::kPFull));
    }
    bool ok = wait_bar(bar(L::kAccFull), af_cnt & 1, abort_flag, p.status, 21);
    if (!__all_sync(0xFFFFFFFFu, ok)) return;
    ++af_cnt;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) store_row_chunk(tDQ + c * 32, p.scale, dq_row + c * 32, valid);
    tc_fence_before();
    mbar_arrive(bar(L::kAccEmpty));
  }
}

template <int HD, bool kKeyStationary>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const int warp = int(warp_id());
  const int lane = int(lane_id());
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    init_bwd_barriers<HD>(bars);
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0) {
    if (lane == 0) bwd_producer<HD, kKeyStationary>(p, smem, bars, abort_flag);
  } else if (warp == 1) {
    if (lane == 0) bwd_mma<HD, kKeyStationary>(p, smem, bars, tmem, abort_flag);
  } else if (warp >= 4) {
    if (kKeyStationary) dkdv_elementwise<HD>(p, smem, bars, tmem, abort_flag);
    else dq_elementwise<HD>(p, bars, tmem, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
template <int HD>
static flash_msa_status launch_bwd_hd(const BwdLaunch& a, cudaStream_t stream) {
  using L = BwdLayout<HD>;
  const int nb = a.rows.n_blocks;
  const int NP = nb * kTile;
  float* lse2 = a.dsum;                        // workspace: [lse2 | dsum]
  float* dsum = a.dsum + int64_t(a.B) * a.H * NP;
  if (a.stages & FLASH_MSA_BWD_PREPROCESS) {
    PreParams pp{reinterpret_cast<const __nv_bfloat16*>(a.o),
                 reinterpret_cast<const __nv_bfloat16*>(a.dout), a.lse, lse2, dsum,
                 a.B, a.H, int(a.N), NP};
    constexpr int kRows = 256 / (HD / 8);
    dim3 grid((NP + kRows - 1) / kRows, a.H, a.B);
    bwd_pre_kernel<HD><<<grid, 256, 0, stream>>>(pp);
    if (cudaGetLastError() != cudaSuccess) return set_cuda_error("bwd_pre launch");
  }
  BwdParams p;
  memset(&p, 0, sizeof(p));
  flash_msa_status st;
  if ((st = make_tile_map(&p.tm_q, a.q, a.B, a.N, a.H, HD)) != FLASH_MSA_OK) return st;
  if ((st = make_tile_map(&p.tm_k, a.k, a.B, a.N, a.H, HD)) != FLASH_MSA_OK) return st;
  if ((st = make_tile_map(&p.tm_v, a.v, a.B, a.N, a.H, HD)) != FLASH_MSA_OK) return st;
  if ((st = make_tile_map(&p.tm_do, a.dout, a.B, a.N, a.H, HD)) != FLASH_MSA_OK) return st;
  p.lse2 = lse2;
  p.dsum = dsum;
  p.B = a.B;
  p.H = a.H;
  p.N = int(a.N);
  p.NP = NP;
  p.n_units = a.B * a.H * nb;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.mask = a.mask;
  p.status = a.status;
  static bool attr_set[2][2] = {{false, false}, {false, false}};
  auto prep = [&](auto kern, int which) -> flash_msa_status {
    if (!attr_set[HD == 128][which]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes) !=
          cudaSuccess)
        return set_cuda_error("cudaFuncSetAttribute(bwd)");
      attr_set[HD == 128][which] = true;
    }
    return FLASH_MSA_OK;
  };
  if (a.stages & FLASH_MSA_BWD_DKDV) {
    if ((st = prep(bwd_main_kernel<HD, true>, 0)) != FLASH_MSA_OK) return st;
    p.list = a.cols;
    p.out_a = reinterpret_cast<__nv_bfloat16*>(a.dk);
    p.out_b = reinterpret_cast<__nv_bfloat16*>(a.dv);
    bwd_main_kernel<HD, true><<<p.n_units, kBwdThreads, L::kSmemBytes, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return set_cuda_error("bwd_dkdv launch");
  }
  if (a.stages & FLASH_MSA_BWD_DQ) {
    if ((st = prep(bwd_main_kernel<HD, false>, 1)) != FLASH_MSA_OK) return st;
    p.list = a.rows;
    p.out_a = reinterpret_cast<__nv_bfloat16*>(a.dq);
    p.out_b = nullptr;
    bwd_main_kernel<HD, false><<<p.n_units, kBwdThreads, L::kSmemBytes, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return set_cuda_error("bwd_dq launch");
  }
  return FLASH_MSA_OK;
}

flash_msa_status launch_bwd(const BwdLaunch& a, cudaStream_t stream) {
  if (a.d == 128) return launch_bwd_hd<128>(a, stream);
  return launch_bwd_hd<64>(a, stream);
}

}  // namespace fmsa
