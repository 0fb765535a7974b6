// Backward attention kernels for sm_103a.  Recompute backward ("Flash MSA
// Attention Kernel Implementation", section "The Backward Pass: The Real
// Beast"): with P = exp(scale S - LSE) recomputed from Q, K and the stored
// LSE,
//     dV = P^T dO,  dP = dO V^T,  D = rowsum(dO o O),  dS = P o (dP - D),
//     dQ = scale dS K,  dK = scale dS^T Q.
// (rowsum(P o dP) = rowsum(dO o O) because O = P V.)
//
// Three launches:
//   bwd_pre   D_i = sum_c dO_ic O_ic and -LSE_i * log2(e), padded to whole
//             128-row tiles (padding rows get -LSE = -inf, so P = 0 there)
//   bwd_dkdv  key-stationary: per (b, h, key tile) loop over the live query
//             tiles; S^T = K Q^T and dP^T = V dO^T in TMEM, P^T and dS^T
//             written back to TMEM as bf16, dV += P^T dO and dK += dS^T Q
//             accumulated in TMEM
//   bwd_dq    query-stationary: per (b, h, query tile) loop over the live key
//             tiles; S = Q K^T, dP = dO V^T, dS to TMEM, dQ += dS K in TMEM
// Each tile pair costs 4 + 3 tensor-core products; no atomics, so all three
// outputs are deterministic.
//
// CTA layout of the two main kernels (384 threads, one CTA per SM):
//   warp 0 TMA producer (one lane), warp 1 MMA issuer (the whole warp runs
//   the loop, one elected lane issues), warp 2
//   TMEM allocator, warps 4-11 elementwise work in two warpgroups: thread =
//   row of the stationary tile (key row in bwd_dkdv, query row in bwd_dq),
//   warpgroup g = columns [64 g, 64 g + 64) of the moving tile.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fmsa {

constexpr int kBwdThreads = 384;
constexpr int kEwWarps = 8;  // elementwise warps: two warpgroups, 64 columns each
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// bwd_pre
// ---------------------------------------------------------------------------
struct PreParams {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  float* nlse2;  // (B, H, NP)
  float* dsum;  // (B, H, NP)
  float* dqacc;  // (B, H, NP, d) fp32 dQ accumulator to zero, or null
  int B, H, N, NP;
  ListParams geo;  // tiles of the rows: row i of the vectors is entry i % 128 of tile i / 128
};

template <int HD>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreParams p) {
  constexpr int kTpr = HD / 8;            // threads per row, 8 bf16 (16 bytes) each
  constexpr int kRows = 256 / kTpr;       // rows per block
  const int h = blockIdx.y, b = blockIdx.z;
  const int r = threadIdx.x / kTpr, c = threadIdx.x % kTpr;
  const int64_t i = int64_t(blockIdx.x) * kRows + r;  // grid covers NP exactly
  if (p.dqacc && i < p.NP) {  // zero this thread's 8 accumulator entries of row i
    float4* z = reinterpret_cast<float4*>(p.dqacc + ((int64_t(b) * p.H + h) * p.NP + i) * HD + c * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // the token of vector row i: entry i % 128 of tile i / 128
  const TileGeo tg = tile_geo(p.geo, int(i / kTile), p.N);
  const int64_t loc = int64_t(tg.lb) * kTile + i % kTile;  // token within its sequence
  const int64_t tok = tg.row0 + i % kTile;                 // token on the sequence axis
  const bool live_row = i < p.NP && loc < tg.n;
  float acc = 0.f;
  if (live_row) {
    const int64_t off = ((int64_t(b) * p.N + tok) * p.H + h) * HD + c * 8;
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
    float nl2 = -INFINITY;  // a row without live keys has P = 0, like padding
    if (live_row) {
      const float l = p.lse[(int64_t(b) * p.H + h) * p.N + tok];
      nl2 = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
    }
    p.nlse2[at] = nl2;
    p.dsum[at] = acc;
  }
}

// ---------------------------------------------------------------------------
// shared layout pieces for the two main kernels
// ---------------------------------------------------------------------------
struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  CUtensorMap tm_dqacc;  // fused: the fp32 dQ accumulator (target of bulk reductions)
  __nv_bfloat16* out_a;  // dkdv: dK, dq: dQ
  __nv_bfloat16* out_b;  // dkdv: dV
  const float* nlse2;
  const float* dsum;
  const __nv_bfloat16* dout;  // dQ pass: rows staged into TMEM by the elementwise side
  int B, H, N, NP;  // H: query heads
  int Hkv, G;       // key/value heads, query heads per key/value head
  int n_units;
  int head_group;             // units are handed out in groups of this many heads
  float* dqacc;               // fused: fp32 dQ accumulator (B, H, NP, d)
  unsigned long long* sched;  // work counter of this launch (see claim_unit)
  unsigned ticket;
  int wait_limit_ms;          // limit of any single bounded wait
  float scale, scale_log2;
  MaskParams mask;
  ListParams list;
  unsigned* status;
};

// Streamed tiles (dK/dV pass: Q and dO; dQ pass: K and V) are prefetched into
// L2 this many tiles ahead of their shared-memory load.  Measured +6% on the
// backward at N = 16384 when units ran (b, h)-major; with the rank-major
// order 0 to 6 tiles all measure within 1% (3 kept).
constexpr int kL2PrefetchTiles = 3;

// Modes of bwd_main_kernel.
constexpr int kModeDq = 0;     // query-stationary dQ pass (deterministic backward)
constexpr int kModeDkdv = 1;   // key-stationary dK/dV pass (deterministic backward)
constexpr int kModeFused = 2;  // key-stationary dK/dV plus dQ partial products added
                               // into the fp32 accumulator (default backward)

template <int HD, int kMode>
struct BwdLayout {
  static constexpr bool KS = kMode != kModeDq;  // key-stationary
  static constexpr int kTileBytes = kTile * HD * 2;
  // key-stationary: even (Q and dO of a tile in consecutive stages share a
  // vector slot); dQ: one more stage of prefetch (no vectors to stage)
  static constexpr int kStages = KS ? (HD == 128 ? 4 : 8) : (HD == 128 ? 6 : 12);
  static constexpr int kFixOff = 0;  // dK/dV: K and V tiles; dQ: the Q tile (dO lives in TMEM)
  static constexpr int kRingOff = (KS ? 2 : 1) * kTileBytes;
  static constexpr int kVecOff = kRingOff + kStages * kTileBytes;  // (stages/2) x 1 KB
  // fused: the dS tile of the current query tile, 128 keys x 128 queries
  // bf16, the MN-major A operand of dQ = dS K (two 16 KB chunks of 64
  // queries, one 128-byte swizzled row per key)
  static constexpr int kDsOff = kVecOff + (KS ? (kStages / 2) * 1024 : 0);  // vectors: KS only
  static constexpr int kDsBytes = kMode == kModeFused ? kTile * kTile * 2 : 0;
  static constexpr int kBarOff = kDsOff + kDsBytes;
  // kSFull / kPFull: two slots each.  dK/dV and fused: kSFull (S^T
  // computed), kSFull + 1 (dP^T computed), kPFull (P^T written), kPFull + 1
  // (dS^T written); dQ: kSFull, kPFull, kDpFree and kDsEmpty (= kSFull + 1,
  // the dS columns of TMEM may be overwritten).  Fused: kDqFull (the tile's
  // dQ partial product computed), kDqFree (read out of TMEM).
  static constexpr int kFixFull = 0, kFixEmpty = 1, kSFull = 2, kDsEmpty = 3, kPFull = 4,
                       kDpFree = 6, kAccFull = 7, kAccEmpty = 8, kMmaDone = 9, kDqFull = 10,
                       kDqFree = 11, kWgSync = 12, kRingFull = 14, kRingEmpty = 14 + kStages,
                       kUnitFull = 14 + 2 * kStages, kUnitEmpty = kUnitFull + 2;
  static constexpr int kNumBars = kUnitEmpty + 2;
  // misc: TMEM base address, abort flag, wait limit, (pad), the two
  // unit-queue slots
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // The fused layout fills the 227 KB a CTA may have, so it takes no
  // alignment slack: the kernel checks that the dynamic shared memory starts
  // on a 1024-byte boundary (as the 128-byte swizzle needs) and reports
  // FLASH_MSA_ERR_UNSUPPORTED otherwise.
  static constexpr int kSmemBytes = kMiscOff + 24 + (kMode == kModeFused ? 0 : 1024);
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

template <int HD>
__device__ __forceinline__ void load_tile_2d(const CUtensorMap* m, uint32_t dst, uint32_t bar,
                                             int row, int h, int b) {
#pragma unroll
  for (int c = 0; c < HD / 64; ++c) tma_load_4d(dst + c * (kTile * 128), m, bar, c * 64, row, h, b);
}

// Units: dK/dV pass (b, key/value head, key block), whose inner tiles are the
// key block's query-block list repeated for each of the G query heads that
// share the key/value head; dQ pass (b, query head, query block).
template <bool kKeyStationary>
__device__ __forceinline__ Unit bwd_decode(int u, const BwdParams& p) {
  const int H = kKeyStationary ? p.Hkv : p.H;
  int bh, rank;
  unit_order_grouped(u, p.B * H, p.list.n_blocks, p.head_group, bh, rank);
  Unit un = decode_unit_at(bh, rank, H, p.list, p.status);
  if (kKeyStationary) un.n = un.n0 * p.G;
  return un;
}

// Inner tile t of a unit and the query head it belongs to.
template <bool kKeyStationary>
__device__ __forceinline__ InnerTile bwd_inner(const Unit& un, int t, const BwdParams& p,
                                               int& hq) {
  if (!kKeyStationary) {
    hq = un.h;
    return inner_tile(un, t, p.list, p.status);
  }
  const int g = p.G == 1 ? 0 : t / un.n0;
  hq = un.h * p.G + g;
  return inner_tile(un, t - g * un.n0, p.list, p.status);
}

template <int HD, int kMode>
__device__ __forceinline__ void init_bwd_barriers(uint64_t* bars) {
  using L = BwdLayout<HD, kMode>;
  constexpr bool KS = L::KS;
  // dQ: the producer's Q tile plus every elementwise warp's rows of dO
  mbar_init(smem_u32(bars + L::kFixFull), KS ? 1 : 1 + kEwWarps);
  mbar_init(smem_u32(bars + L::kFixEmpty), 1);
  for (int i = 0; i < 2; ++i) {
    mbar_init(smem_u32(bars + L::kSFull + i), 1);
    mbar_init(smem_u32(bars + L::kPFull + i), kEwWarps);
  }
  mbar_init(smem_u32(bars + L::kDpFree), kEwWarps);
  mbar_init(smem_u32(bars + L::kAccFull), 1);
  mbar_init(smem_u32(bars + L::kAccEmpty), kEwWarps);
  mbar_init(smem_u32(bars + L::kMmaDone), 1);
  mbar_init(smem_u32(bars + L::kDqFull), 1);
  mbar_init(smem_u32(bars + L::kDqFree), kEwWarps);
  for (int i = 0; i < 2; ++i) mbar_init(smem_u32(bars + L::kWgSync + i), 4);
  // The ring holds pairs loaded together: (K_t, V_t) in the dQ pass, (Q_t,
  // dO_t) in the key-stationary kernels, in stages 2i and 2i + 1.  Both
  // copies of a pair arrive on the full barrier of stage 2i (count 2; the
  // odd stages' full barriers are unused), so the MMA warp waits once per
  // inner tile; the empty barriers stay per stage (the halves are released
  // apart).
  static_assert(L::kStages % 2 == 0, "ring stages come in pairs");
  for (int i = 0; i < L::kStages; ++i) {
    mbar_init(smem_u32(bars + L::kRingFull + i), (i % 2 == 0) ? 2 : 1);
    mbar_init(smem_u32(bars + L::kRingEmpty + i), 1);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(smem_u32(bars + L::kUnitFull + i), 1);               // the producer
    mbar_init(smem_u32(bars + L::kUnitEmpty + i), 1 + kEwWarps);  // MMA warp, EW warps
  }
  fence_mbar_init();
}

template <int HD, int kMode>
__device__ __forceinline__ UnitQueue unit_queue(uint8_t* smem, uint64_t* bars) {
  using L = BwdLayout<HD, kMode>;
  return UnitQueue{smem_u32(bars + L::kUnitFull), smem_u32(bars + L::kUnitEmpty),
                   reinterpret_cast<volatile int*>(smem + L::kMiscOff + 16), 0u};
}

// Producer shared by both kernels.  Per unit: the stationary tiles (dkdv: K,
// V of the key block; dq: Q of the query block), then per inner tile two ring
// stages (dkdv: Q_t + its LSE2/D vectors, dO_t; dq: K_t, V_t).
template <int HD, int kMode>
__device__ __forceinline__ void bwd_producer(const BwdParams& p, uint8_t* smem, uint64_t* bars,
                                             volatile int* abort_flag) {
  using L = BwdLayout<HD, kMode>;
  constexpr bool kKeyStationary = L::KS;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const CUtensorMap* fix_a = kKeyStationary ? &p.tm_k : &p.tm_q;
  const CUtensorMap* fix_b = kKeyStationary ? &p.tm_v : &p.tm_do;
  const CUtensorMap* ring_a = kKeyStationary ? &p.tm_q : &p.tm_k;
  const CUtensorMap* ring_b = kKeyStationary ? &p.tm_do : &p.tm_v;
  // ring position (stage, phase) advanced by one per load; no divisions
  // (the dQ ring has 6 or 12 stages)
  int stage = 0;
  uint32_t phase = 0, fe_cnt = 0;
  int last[L::kStages];  // phase of the last load into each stage, -1 if none
  for (int i = 0; i < L::kStages; ++i) last[i] = -1;
  int last_fix = -1;
  bool ok = true;
  UnitQueue queue = unit_queue<HD, kMode>(smem, bars);
  // units are claimed one ahead (the dQ pass prefetches the next unit's dO)
  int u = queue_push(queue, p.sched, p.ticket, p.n_units, abort_flag, p.status);
  while (ok && u >= 0) {
    const int u_next = queue_push(queue, p.sched, p.ticket, p.n_units, abort_flag, p.status);
    if (u_next == -2) {
      ok = false;
      break;
    }
    const Unit un = bwd_decode<kKeyStationary>(u, p);
    u = u_next;
    if (un.n == 0) continue;
    if (!wait_bar(bar(L::kFixEmpty), (fe_cnt & 1) ^ 1, abort_flag, p.status, 1)) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(bar(L::kFixFull), (kKeyStationary ? 2 : 1) * L::kTileBytes);
    const int fix_row = int(tile_geo(p.list, un.ob, p.N).row0);
    load_tile_2d<HD>(fix_a, smem_u32(smem + L::kFixOff), bar(L::kFixFull), fix_row, un.h, un.b);
    if (kKeyStationary) {
      load_tile_2d<HD>(fix_b, smem_u32(smem + L::kFixOff + L::kTileBytes), bar(L::kFixFull),
                       fix_row, un.h, un.b);
    } else {
      // the elementwise warps read the next unit's dO rows with plain loads:
      // start pulling them into L2 now
      if (u_next >= 0) {
        const Unit nx = bwd_decode<false>(u_next, p);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c)
          tma_prefetch_l2_4d(fix_b, c * 64, int(tile_geo(p.list, nx.ob, p.N).row0), nx.h, nx.b);
      }
    }
    last_fix = int(fe_cnt);
    ++fe_cnt;
    const int hkv = kKeyStationary ? 0 : un.h / p.G;  // dQ pass: head of the K / V tiles
    for (int t = 0; t < un.n && ok; ++t) {
      int hq;
      const InnerTile it = bwd_inner<kKeyStationary>(un, t, p, hq);
      const int hr = kKeyStationary ? hq : hkv;  // head of the streamed tiles
      const int ring_row = int(tile_geo(p.list, it.blk, p.N).row0);
      // the pair: ring_a's tile (Q or K) into stage `stage` (even), ring_b's
      // (dO or V) into stage + 1, both completing the full barrier of
      // `stage`.  The key-stationary kernels copy dO first: its stage is
      // released earlier (after dV) than Q's (after dK), so Q, which the
      // pair's first product S^T needs, is the later copy and waiting for
      // the whole pair costs nothing
      const uint32_t full = bar(L::kRingFull + stage);
      for (int half = 0; half < 2; ++half) {
        const bool is_a = kKeyStationary ? (half == 1) : (half == 0);
        const int st = stage + (is_a ? 0 : 1);
        if (!wait_bar(bar(L::kRingEmpty + st), phase ^ 1, abort_flag, p.status, 2)) {
          ok = false;
          break;
        }
        const uint32_t dst = smem_u32(smem + L::kRingOff + st * L::kTileBytes);
        if (is_a) {
          const bool vec = kKeyStationary;
          mbar_arrive_expect_tx(full, L::kTileBytes + (vec ? 1024 : 0));
          load_tile_2d<HD>(ring_a, dst, full, ring_row, hr, un.b);
          if (vec) {
            const int64_t row0 = (int64_t(un.b) * p.H + hq) * p.NP + int64_t(it.blk) * kTile;
            const uint32_t vdst = smem_u32(smem + L::kVecOff + (stage / 2) * 1024);
            bulk_load(vdst, p.nlse2 + row0, 512, full);
            bulk_load(vdst + 512, p.dsum + row0, 512, full);
          }
        } else {
          mbar_arrive_expect_tx(full, L::kTileBytes);
          load_tile_2d<HD>(ring_b, dst, full, ring_row, hr, un.b);
        }
        last[st] = int(phase);
      }
      if (!ok) break;
      stage += 2;
      if (stage == L::kStages) {
        stage = 0;
        phase ^= 1;
      }
      if (t + kL2PrefetchTiles < un.n) {
        int fq;
        const InnerTile ft = bwd_inner<kKeyStationary>(un, t + kL2PrefetchTiles, p, fq);
        const int fr = kKeyStationary ? fq : hkv;
#pragma unroll
        const int pf_row = int(tile_geo(p.list, ft.blk, p.N).row0);
        for (int c = 0; c < HD / 64; ++c) {
          tma_prefetch_l2_4d(ring_a, c * 64, pf_row, fr, un.b);
          tma_prefetch_l2_4d(ring_b, c * 64, pf_row, fr, un.b);
        }
      }
    }
  }
  if (!ok) {  // (a pair whose second copy was never issued waits out the drain limit)
    for (int i = 0; i < L::kStages; ++i)
      if (last[i] >= 0) drain_bar(bar(L::kRingFull + (i & ~1)), uint32_t(last[i]));
    if (last_fix >= 0) drain_bar(bar(L::kFixFull), last_fix & 1);
  }
}

// One arrival per warp, after every lane's TMEM traffic is ordered before it.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  tc_fence_before();
  __syncwarp();
  if (lane_id() == 0) mbar_arrive(bar);
}

// Common MMA pieces.  K-major operands: 16-element k-steps are 32 bytes
// apart inside a 128-byte swizzle row, 64-element chunks 16 KB apart.
// MN-major B operands (rows = the reduction index): 16 rows = 2 KB per
// k-step, 64-column chunks 16 KB apart.
template <int HD>
__device__ __forceinline__ void mma_kmajor(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc) {
  const uint32_t ad = sdesc_lo(a, 16), bd = sdesc_lo(b, 16);
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
    mma_ss(d, ad + off, bd + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// D (+)= A[tmem] * B[smem], reduction over 128 rows of B in 8 k-steps of 16.
// A is the bf16 output of the two elementwise warpgroups: warpgroup g packed
// its 64 reduction indices (two per column) into columns [64 g, 64 g + 32)
// of the region at a_tmem, so k-step kk reads 8 columns at
// a_tmem + 64 (kk / 4) + 8 (kk % 4).
__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a_tmem, uint32_t b,
                                           uint32_t idesc, bool accumulate) {
  const uint32_t bd = sdesc_lo(b, kTile * 128);
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    mma_ts(d, a_tmem + (kk / 4) * 64 + (kk % 4) * 8, bd + kk * (2048 >> 4), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
}

// MMA issuer of bwd_dq (query-stationary; Q of the query block in shared
// memory, its dO in TMEM written by the elementwise warpgroups; ring K_t, V_t).
// TMEM: S at [0,128), dP at [128,256), dQ at [256, 256+d), dS (bf16 pairs)
// at [384,448), dO (bf16 pairs) at [448, 448+d/2).  The elementwise side
// pulls S(t) and dP(t) into registers first (sdp_free), so the next tile's
// products run while it computes dS(t).  Order per key tile t:
//   [sdp_free(t)] S(t+1), dP(t+1) -> s_full(t+1), release V_(t+1);
//   [P full(t)] dQ += dS(t) K_t -> ds_empty, release K_t.
template <int HD>
__device__ __forceinline__ void dq_mma(const BwdParams& p, uint8_t* smem, uint64_t* bars,
                                       uint32_t tmem, volatile int* abort_flag) {
  using L = BwdLayout<HD, kModeDq>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdAcc = idesc_bf16_f32(128, HD, false, true);
  const uint32_t tS = tmem, tDP = tmem + 128, tDQ = tmem + 256;
  const uint32_t tDS = tmem + 384, tDO = tmem + 448;
  const uint32_t fq = smem_u32(smem + L::kFixOff);
  const uint32_t ring = smem_u32(smem + L::kRingOff);
  // ring position of a key tile: K_t in stage s (even), V_t in s + 1, both
  // filled in phase ph (the ring has an even number of stages)
  struct Pos {
    int s;
    uint32_t ph;
  };
  auto advance = [](Pos r) {
    r.s += 2;
    if (r.s == L::kStages) {
      r.s = 0;
      r.ph ^= 1;
    }
    return r;
  };
  auto stage_addr = [&](int s) { return ring + uint32_t(s) * L::kTileBytes; };
  auto ring_wait = [&](int s, uint32_t ph, unsigned where) {
    return wait_bar_warp(bar(L::kRingFull + s), ph, abort_flag, p.status, where);
  };
  // S = Q K^T (both operands in shared memory), dP = dO[tmem] V^T, for the
  // tile at ring position r
  auto issue_sdp = [&](Pos r) {
    mma_kmajor<HD>(tS, fq, stage_addr(r.s), kIdS);
    const uint32_t vd = sdesc_lo(stage_addr(r.s + 1), 16);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
      mma_ts(tDP, tDO + kk * 8, vd + off, kIdS, kk > 0 ? 1u : 0u);
    }
    mma_commit(bar(L::kSFull));
    mma_commit(bar(L::kRingEmpty + r.s + 1));  // V_t is not read again
  };
  Pos pos{0, 0};  // ring position of the current unit's first tile
  uint32_t ff_cnt = 0, pf_cnt = 0, sdp_cnt = 0, ae_cnt = 0;
  bool ok = true, pending_sdp = false;
  UnitQueue queue = unit_queue<HD, kModeDq>(smem, bars);
  int u;
  while (ok && (u = queue_pop<true>(queue, abort_flag, p.status)) >= 0) {
    const Unit un = bwd_decode<false>(u, p);
    if (un.n == 0) continue;
    if (!wait_bar_warp(bar(L::kFixFull), ff_cnt & 1, abort_flag, p.status, 10)) break;
    ++ff_cnt;
    if (!ring_wait(pos.s, pos.ph, 11)) break;  // K_t and V_t: one barrier per pair
    // the previous unit's last S / dP must be in registers before S(0) and
    // dP(0) overwrite them
    if (pending_sdp) {
      if (!wait_bar_warp(bar(L::kDpFree), sdp_cnt & 1, abort_flag, p.status, 15)) break;
      ++sdp_cnt;
    }
    tc_fence_after();
    issue_sdp(pos);
    if (un.n == 1) mma_commit(bar(L::kFixEmpty));  // Q and dO are not read again
    for (int t = 0; t < un.n && ok; ++t) {
      const Pos nxt = advance(pos);  // pos: tile t, nxt: tile t + 1
      if (t + 1 < un.n) {
        if (!ring_wait(nxt.s, nxt.ph, 11)) { ok = false; break; }
        if (!wait_bar_warp(bar(L::kDpFree), sdp_cnt & 1, abort_flag, p.status, 15)) { ok = false; break; }
        ++sdp_cnt;
        tc_fence_after();
        issue_sdp(nxt);
        if (t + 2 == un.n) mma_commit(bar(L::kFixEmpty));
      }
      if (t == 0) {
        if (!wait_bar_warp(bar(L::kAccEmpty), (ae_cnt & 1) ^ 1, abort_flag, p.status, 13)) { ok = false; break; }
        ++ae_cnt;
      }
      if (!wait_bar_warp(bar(L::kPFull), pf_cnt & 1, abort_flag, p.status, 14)) { ok = false; break; }
      ++pf_cnt;
      tc_fence_after();
      // dQ (+)= dS K_t: dS from TMEM (k-step kk = keys [16 kk, 16 kk + 16) =
      // columns tDS + 8 kk), K_t as an MN-major B operand
      const uint32_t kd = sdesc_lo(stage_addr(pos.s), kTile * 128);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_ts(tDQ, tDS + kk * 8, kd + kk * (2048 >> 4), kIdAcc, (t > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar(L::kDsEmpty));
      mma_commit(bar(L::kRingEmpty + pos.s));
      pos = nxt;
    }
    if (!ok) break;
    mma_commit(bar(L::kAccFull));
    pending_sdp = true;
  }
  mma_commit(bar(L::kMmaDone));
  drain_bar(bar(L::kMmaDone), 0);
}

// MMA issuer of bwd_dkdv (key-stationary; fixed tiles K, V; ring Q_t, dO_t).
// TMEM: S^T at A = [0,128), dP^T at B = [128,256), dV at [256, 256+d), dK at
// [384, 384+d).  The elementwise side reads S^T, writes P^T (bf16) over it
// and signals p_full; then reads dP^T, writes dS^T (bf16) over it and
// signals ds_full.  Each region is refilled for the next tile as soon as
// the product reading it has been issued, so the next tile's S^T is ready
// while dS^T is still being computed.  Order per tile t:
//   [p_full(t)] dV += P^T dO_t, release dO_t, S^T(t+1) -> s_full;
//   [ds_full(t)] dK += dS^T Q_t, release Q_t, dP^T(t+1) -> dp_full.
template <int HD>
__device__ __forceinline__ void dkdv_mma(const BwdParams& p, uint8_t* smem, uint64_t* bars,
                                         uint32_t tmem, volatile int* abort_flag) {
  using L = BwdLayout<HD, kModeDkdv>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdAcc = idesc_bf16_f32(128, HD, false, true);
  const uint32_t tA = tmem, tB = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;
  const uint32_t fk = smem_u32(smem + L::kFixOff);
  const uint32_t fv = fk + L::kTileBytes;
  auto stage_addr = [&](uint32_t c) {
    return smem_u32(smem + L::kRingOff + (c % L::kStages) * L::kTileBytes);
  };
  auto ring_wait = [&](uint32_t c, unsigned where) {
    return wait_bar_warp(bar(L::kRingFull + c % L::kStages), (c / L::kStages) & 1, abort_flag,
                    p.status, where);
  };
  uint32_t cnt = 0, ff_cnt = 0, pf_cnt = 0, ae_cnt = 0;
  bool ok = true;
  UnitQueue queue = unit_queue<HD, kModeDkdv>(smem, bars);
  int u;
  while (ok && (u = queue_pop<true>(queue, abort_flag, p.status)) >= 0) {
    const Unit un = bwd_decode<true>(u, p);
    if (un.n == 0) continue;
    if (!wait_bar_warp(bar(L::kFixFull), ff_cnt & 1, abort_flag, p.status, 10)) break;
    ++ff_cnt;
    if (!ring_wait(cnt, 11)) break;  // Q_0 and dO_0 (one barrier per ring pair)
    tc_fence_after();
    mma_kmajor<HD>(tA, fk, stage_addr(cnt), kIdS);  // S^T(0) = K Q_0^T
    mma_commit(bar(L::kSFull));
    mma_kmajor<HD>(tB, fv, stage_addr(cnt + 1), kIdS);  // dP^T(0) = V dO_0^T
    mma_commit(bar(L::kSFull + 1));
    if (un.n == 1) mma_commit(bar(L::kFixEmpty));  // K and V are not read again
    for (int t = 0; t < un.n && ok; ++t) {
      const uint32_t c = cnt + 2 * t;  // Q_t at c, dO_t at c + 1
      const bool more = t + 1 < un.n;
      if (t == 0) {
        if (!wait_bar_warp(bar(L::kAccEmpty), (ae_cnt & 1) ^ 1, abort_flag, p.status, 13)) { ok = false; break; }
        ++ae_cnt;
      }
      if (!wait_bar_warp(bar(L::kPFull), pf_cnt & 1, abort_flag, p.status, 14)) { ok = false; break; }
      tc_fence_after();
      mma_tmem_a(tDV, tA, stage_addr(c + 1), kIdAcc, t > 0);  // dV += P^T dO_t
      mma_commit(bar(L::kRingEmpty + (c + 1) % L::kStages));
      if (more) {
        if (!ring_wait(c + 2, 11)) { ok = false; break; }
        tc_fence_after();
        mma_kmajor<HD>(tA, fk, stage_addr(c + 2), kIdS);  // S^T(t+1) over P^T(t)
        mma_commit(bar(L::kSFull));
      }
      if (!wait_bar_warp(bar(L::kPFull + 1), pf_cnt & 1, abort_flag, p.status, 16)) { ok = false; break; }
      ++pf_cnt;
      tc_fence_after();
      mma_tmem_a(tDK, tB, stage_addr(c), kIdAcc, t > 0);  // dK += dS^T Q_t
      mma_commit(bar(L::kRingEmpty + c % L::kStages));
      if (more) {  // dO_t+1 arrived with Q_t+1 (waited for before S^T(t+1))
        mma_kmajor<HD>(tB, fv, stage_addr(c + 3), kIdS);  // dP^T(t+1) over dS^T(t)
        mma_commit(bar(L::kSFull + 1));
        if (t + 2 == un.n) mma_commit(bar(L::kFixEmpty));
      }
    }
    if (!ok) break;
    cnt += 2 * un.n;
    mma_commit(bar(L::kAccFull));
  }
  mma_commit(bar(L::kMmaDone));
  drain_bar(bar(L::kMmaDone), 0);
}

// MMA issuer of the fused kernel (key-stationary, like dkdv_mma, plus the dQ
// partial product of every tile).  TMEM: S^T at A = [0,128), dP^T at
// B = [128,256), dV at [256, 256+d), dK at [384, 384+d); dQ(t) = dS(t) K
// (fp32, query rows in the lanes) is written over B once dK(t) has read
// dS^T(t) from it, and the elementwise side reads it out (dq_free) before
// dP^T(t+1) overwrites it.  dS(t) reaches the tensor core through shared
// memory (MN-major A operand), written by the elementwise side next to dS^T.
// Order per tile t:
//   [p_full(t)] dV += P^T dO_t, release dO_t, S^T(t+1) -> s_full;
//   [ds_full(t)] dK += dS^T Q_t, dQ(t) = dS K -> dq_full, release Q_t;
//   [dq_free(t)] dP^T(t+1) -> dp_full.
// K is read by the unit's last dQ product, so K and V are released after it.
template <int HD>
__device__ __forceinline__ void fused_mma(const BwdParams& p, uint8_t* smem, uint64_t* bars,
                                          uint32_t tmem, volatile int* abort_flag) {
  using L = BwdLayout<HD, kModeFused>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdAcc = idesc_bf16_f32(128, HD, false, true);
  constexpr uint32_t kIdDq = idesc_bf16_f32(128, HD, true, true);
  const uint32_t tA = tmem, tB = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;
  const uint32_t fk = smem_u32(smem + L::kFixOff);
  const uint32_t fv = fk + L::kTileBytes;
  // dQ = dS K: A = dS (MN-major: 64-query chunks 16 KB apart, 16 keys = 2 KB
  // per k-step), B = K (MN-major, like V in the forward's P V)
  const uint32_t dq_a = sdesc_lo(smem_u32(smem + L::kDsOff), kTile * 128);
  const uint32_t dq_b = sdesc_lo(fk, kTile * 128);
  auto stage_addr = [&](uint32_t c) {
    return smem_u32(smem + L::kRingOff + (c % L::kStages) * L::kTileBytes);
  };
  auto ring_wait = [&](uint32_t c, unsigned where) {
    return wait_bar_warp(bar(L::kRingFull + c % L::kStages), (c / L::kStages) & 1, abort_flag,
                    p.status, where);
  };
  uint32_t cnt = 0, ff_cnt = 0, pf_cnt = 0, ae_cnt = 0, dq_cnt = 0;
  bool ok = true, pending_drain = false;
  UnitQueue queue = unit_queue<HD, kModeFused>(smem, bars);
  int u;
  while (ok && (u = queue_pop<true>(queue, abort_flag, p.status)) >= 0) {
    const Unit un = bwd_decode<true>(u, p);
    if (un.n == 0) continue;
    if (!wait_bar_warp(bar(L::kFixFull), ff_cnt & 1, abort_flag, p.status, 10)) break;
    ++ff_cnt;
    if (!ring_wait(cnt, 11)) break;  // Q_0 and dO_0 (one barrier per ring pair)
    tc_fence_after();
    mma_kmajor<HD>(tA, fk, stage_addr(cnt), kIdS);  // S^T(0) = K Q_0^T
    mma_commit(bar(L::kSFull));
    // the previous unit's last dQ product must be out of B
    if (pending_drain && !wait_bar_warp(bar(L::kDqFree), dq_cnt++ & 1, abort_flag, p.status, 17)) break;
    tc_fence_after();
    mma_kmajor<HD>(tB, fv, stage_addr(cnt + 1), kIdS);  // dP^T(0) = V dO_0^T
    mma_commit(bar(L::kSFull + 1));
    for (int t = 0; t < un.n && ok; ++t) {
      const uint32_t c = cnt + 2 * t;  // Q_t at c, dO_t at c + 1
      const bool more = t + 1 < un.n;
      if (t == 0) {
        if (!wait_bar_warp(bar(L::kAccEmpty), (ae_cnt & 1) ^ 1, abort_flag, p.status, 13)) { ok = false; break; }
        ++ae_cnt;
      }
      if (!wait_bar_warp(bar(L::kPFull), pf_cnt & 1, abort_flag, p.status, 14)) { ok = false; break; }
      tc_fence_after();
      mma_tmem_a(tDV, tA, stage_addr(c + 1), kIdAcc, t > 0);  // dV += P^T dO_t
      mma_commit(bar(L::kRingEmpty + (c + 1) % L::kStages));
      if (more) {
        if (!ring_wait(c + 2, 11)) { ok = false; break; }
        tc_fence_after();
        mma_kmajor<HD>(tA, fk, stage_addr(c + 2), kIdS);  // S^T(t+1) over P^T(t)
        mma_commit(bar(L::kSFull));
      }
      if (!wait_bar_warp(bar(L::kPFull + 1), pf_cnt & 1, abort_flag, p.status, 16)) { ok = false; break; }
      ++pf_cnt;
      tc_fence_after();
      mma_tmem_a(tDK, tB, stage_addr(c), kIdAcc, t > 0);  // dK += dS^T Q_t
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)  // dQ(t) = dS K over dS^T(t)
        mma_ss(tB, dq_a + kk * (2048 >> 4), dq_b + kk * (2048 >> 4), kIdDq, kk > 0 ? 1u : 0u);
      mma_commit(bar(L::kDqFull));
      mma_commit(bar(L::kRingEmpty + c % L::kStages));
      if (!more) mma_commit(bar(L::kFixEmpty));  // K and V are not read again
      if (more) {
        if (!wait_bar_warp(bar(L::kDqFree), dq_cnt++ & 1, abort_flag, p.status, 17)) { ok = false; break; }
        tc_fence_after();
        mma_kmajor<HD>(tB, fv, stage_addr(c + 3), kIdS);  // dP^T(t+1) over dQ(t)
        mma_commit(bar(L::kSFull + 1));
      }
    }
    if (!ok) break;
    cnt += 2 * un.n;
    mma_commit(bar(L::kAccFull));
    pending_drain = true;
  }
  mma_commit(bar(L::kMmaDone));
  drain_bar(bar(L::kMmaDone), 0);
}

// Write the warpgroup's HD/2 fp32 accumulator columns of this thread's row
// (TMEM address taddr), times `mul`, as bf16 to dst (the row's first element
// of the piece); rows of consecutive lanes are `stride` bytes apart.
template <int HD>
__device__ __forceinline__ void store_acc_piece(uint32_t taddr, float mul, __nv_bfloat16* dst,
                                                int64_t stride, bool valid) {
  constexpr int kC = HD / 16;  // 16-byte chunks: HD/2 bf16 = HD bytes
  uint4 c[kC];
#pragma unroll
  for (int q = 0; q < HD / 64; ++q) {
    uint32_t v[32];
    tmem_ld_x32(taddr + q * 32, v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* f = reinterpret_cast<const float*>(v + 8 * j);
      c[4 * q + j] = make_uint4(pack_bf16x2(f[0] * mul, f[1] * mul), pack_bf16x2(f[2] * mul, f[3] * mul),
                                pack_bf16x2(f[4] * mul, f[5] * mul), pack_bf16x2(f[6] * mul, f[7] * mul));
    }
  }
  // lane groups of 4: each store writes 64 contiguous bytes of 8 rows (fewer
  // shuffles than a full 8-lane transpose, still whole 32-byte sectors)
  store_rows_transposed<kC, 4>(c, reinterpret_cast<char*>(dst), stride, valid);
}

__device__ __forceinline__ void zero_row(__nv_bfloat16* dst, int hd, bool valid) {
  if (!valid) return;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int j = 0; j < hd / 8; ++j) d4[j] = make_uint4(0, 0, 0, 0);
}

// Elementwise warpgroups of bwd_dkdv: thread = key row j of the key tile,
// warpgroup g = query columns [64 g, 64 g + 64) of each query tile.
// Pass 1: P^T = exp2(scale*log2e * S^T - LSE*log2e) on live entries, bf16
// to the start of the warpgroup's S^T columns, p_full.  Pass 2 (once dP^T is
// in TMEM): dS^T = P^T o (dP^T - D), bf16 to the start of its dP^T columns,
// ds_full.  dV of the tile runs on the tensor cores during pass 2, and the
// next tile's S^T during dK.
template <int HD>
__device__ __forceinline__ void dkdv_elementwise(const BwdParams& p, uint8_t* smem,
                                                 uint64_t* bars, uint32_t tmem, int g,
                                                 volatile int* abort_flag) {
  using L = BwdLayout<HD, kModeDkdv>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int wq = int(warp_id()) & 3;
  const int row = wq * 32 + int(lane_id());
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t tA = tmem + lane_off + 64 * g, tB = tA + 128;
  const uint32_t tDV = tmem + lane_off + 256, tDK = tmem + lane_off + 384;
  const float sl2 = p.scale_log2;
  uint32_t sp_cnt = 0, af_cnt = 0, cnt = 0;
  UnitQueue queue = unit_queue<HD, kModeDkdv>(smem, bars);
  while (true) {
    const int u = queue_pop<true>(queue, abort_flag, p.status);
    if (u < 0) return;
    const Unit un = bwd_decode<true>(u, p);
    // this key row: token j of its sequence (kg.n tokens), token kg.row0 + row of the axis
    const TileGeo kg = tile_geo(p.list, un.ob, p.N);
    const int64_t j = int64_t(kg.lb) * kTile + row;
    const bool valid = j < kg.n;
    const int64_t ktok = kg.row0 + row;
    __nv_bfloat16* dk_row = p.out_a + ((int64_t(un.b) * p.N + ktok) * p.Hkv + un.h) * HD;
    __nv_bfloat16* dv_row = p.out_b + ((int64_t(un.b) * p.N + ktok) * p.Hkv + un.h) * HD;
    if (un.n == 0) {
      if (g == 0) {
        zero_row(dk_row, HD, valid);
        zero_row(dv_row, HD, valid);
      }
      continue;
    }
    for (int t = 0; t < un.n; ++t) {
      int hq;
      const InnerTile it = bwd_inner<true>(un, t, p, hq);
      int lo = 0, hi = kTile - 1;
      if (it.dead) hi = -1;
      else if (it.partial)
        col_live_range(j, tile_geo(p.list, it.blk, p.N).lb, kg.lb, kg.n, p.mask, lo, hi);
      prefetch_tile_bits(p.list, it.slot, row);
      const float* vec =
          reinterpret_cast<const float*>(smem + L::kVecOff + ((cnt % L::kStages) / 2) * 1024);
      cnt += 2;
      bool ok = wait_bar(bar(L::kSFull), sp_cnt & 1, abort_flag, p.status, 20);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_x64(tA, sv);
      if (it.partial || it.dead) {  // dead entries: S^T = -inf, so P^T = 0 below (scale > 0)
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (64 * g + e < lo || 64 * g + e > hi) sv[e] = kNegInfBits;
        if (it.slot >= 0) {  // bit-packed mask tile: this key row's bits over 64 queries
          uint32_t bw[2];
          load_tile_bits<2>(p.list, it.slot, row, 2 * g, bw);
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (!((bw[e >> 5] >> (e & 31)) & 1u)) sv[e] = kNegInfBits;
        }
      }
      // pass 1: P^T (kept in sv as fp32), bf16 to columns [64 g, 64 g + 32)
      {
        uint32_t pp[32];
        float4 l4n = *reinterpret_cast<const float4*>(vec + 64 * g);
#pragma unroll
        for (int x = 0; x < 64; x += 4) {
          const float4 l4 = l4n;
          if (x + 4 < 64)  // next group's -LSE, loaded one group ahead
            l4n = *reinterpret_cast<const float4*>(vec + 64 * g + x + 4);
          const float nl[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            float x0, x1;
            fma2(x0, x1, __uint_as_float(sv[x + e]), __uint_as_float(sv[x + e + 1]), sl2, sl2,
                 nl[e], nl[e + 1]);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            sv[x + e] = __float_as_uint(p0);
            sv[x + e + 1] = __float_as_uint(p1);
            pp[(x + e) / 2] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st_x32(tA, pp);
        tmem_wait_st();
        warp_arrive(bar(L::kPFull));
      }
      // pass 2: dS^T = P^T o (dP^T - D), bf16 to columns [64 g, 64 g + 32) of B
      ok = wait_bar(bar(L::kSFull + 1), sp_cnt & 1, abort_flag, p.status, 24);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      ++sp_cnt;
      tc_fence_after();
      uint32_t dpv[64];
      tmem_ld_x64(tB, dpv);
      uint32_t dd[32];
      float4 d4n = *reinterpret_cast<const float4*>(vec + 128 + 64 * g);
#pragma unroll
      for (int x = 0; x < 64; x += 4) {
        const float4 d4 = d4n;
        if (x + 4 < 64) d4n = *reinterpret_cast<const float4*>(vec + 128 + 64 * g + x + 4);
        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          float u0, u1, d0, d1;
          sub2(u0, u1, __uint_as_float(dpv[x + e]), __uint_as_float(dpv[x + e + 1]), dv[e],
               dv[e + 1]);
          mul2(d0, d1, __uint_as_float(sv[x + e]), __uint_as_float(sv[x + e + 1]), u0, u1);
          dd[(x + e) / 2] = pack_bf16x2(d0, d1);
        }
      }
      tmem_st_x32(tB, dd);
      tmem_wait_st();
      warp_arrive(bar(L::kPFull + 1));
    }
    const bool ok = wait_bar(bar(L::kAccFull), af_cnt & 1, abort_flag, p.status, 21);
    if (!__all_sync(0xFFFFFFFFu, ok)) return;
    ++af_cnt;
    tc_fence_after();
    // warpgroup g writes dV and dK columns [d/2 g, d/2 (g + 1))
    const int64_t stride = int64_t(p.Hkv) * HD * 2;  // bytes between consecutive key rows
    store_acc_piece<HD>(tDV + g * (HD / 2), 1.f, dv_row + g * (HD / 2), stride, valid);
    store_acc_piece<HD>(tDK + g * (HD / 2), p.scale, dk_row + g * (HD / 2), stride, valid);
    warp_arrive(bar(L::kAccEmpty));
  }
}

// Elementwise warpgroups of the fused kernel.  As in dkdv_elementwise, a
// thread owns key row j of the key tile and warpgroup g the query columns
// [64 g, 64 g + 64) of each query tile, in two passes per tile: P^T, then
// dS^T.  Pass 2 also writes the thread's dS values (its key row, 64 queries,
// bf16) into the dS tile in shared memory, the A operand of dQ = dS K.  After
// the next tile's pass 1 (or at the end of the unit) the warpgroup reads its
// half of the tile's dQ partial product out of TMEM -- query row
// 32 (warp % 4) + lane, columns [d/2 g, d/2 g + d/2) -- releases the columns,
// stages it in shared memory and adds it into the fp32 accumulator with TMA
// bulk tensor reductions.  Order per tile t: pass 2 (t), pass 1 (t + 1),
// drain (t).
template <int HD>
__device__ __forceinline__ void fused_elementwise(const BwdParams& p, uint8_t* smem,
                                                  uint64_t* bars, uint32_t tmem, int g,
                                                  volatile int* abort_flag) {
  using L = BwdLayout<HD, kModeFused>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int wq = int(warp_id()) & 3;
  const int row = wq * 32 + int(lane_id());
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t tA = tmem + lane_off + 64 * g, tB = tA + 128;
  const uint32_t tDV = tmem + lane_off + 256, tDK = tmem + lane_off + 384;
  const uint32_t tDQ = tmem + lane_off + 128 + g * (HD / 2);
  // this key row of the dS tile: chunk g, 128 bytes, 16-byte unit u stored at
  // unit position u ^ (row % 8) (the 128-byte swizzle the descriptor names)
  uint8_t* ds_row = smem + L::kDsOff + g * (kTile * 128) + row * 128;
  // the same 16 KB half of the dS tile stages the warpgroup's dQ rows
  const uint32_t stage = smem_u32(smem + L::kDsOff + g * (kTile * 128));
  const bool wg_leader = (threadIdx.x & 127) == 0;  // issues the warpgroup's bulk reductions
  const float sl2 = p.scale_log2;
  uint32_t s1_cnt = 0, s2_cnt = 0, af_cnt = 0, dq_cnt = 0, cnt = 0, ws_cnt = 0;
  // the four warps of this warpgroup meet (a bounded wait, like every other)
  auto wg_sync = [&]() -> bool {
    warp_arrive(bar(L::kWgSync + g));
    const bool ok = wait_bar(bar(L::kWgSync + g), ws_cnt & 1, abort_flag, p.status, 26);
    ++ws_cnt;
    return __all_sync(0xFFFFFFFFu, ok);
  };
  UnitQueue queue = unit_queue<HD, kModeFused>(smem, bars);
  auto vec_at = [&](uint32_t c) {  // -LSE log2(e) | D of the query tile at ring position c
    return reinterpret_cast<const float*>(smem + L::kVecOff + ((c % L::kStages) / 2) * 1024);
  };
  uint32_t sv[64];  // P^T of the current tile (fp32), from pass 1 to pass 2
  // pass 1: P^T = exp2(scale*log2e * S^T - LSE*log2e) on live entries, bf16
  // to columns [64 g, 64 g + 32) of A, p_full
  auto pass1 = [&](const Unit& un, int t, int64_t j, const TileGeo& kg, const float* vec) -> bool {
    int hq;
    const InnerTile it = bwd_inner<true>(un, t, p, hq);
    int lo = 0, hi = kTile - 1;
    if (it.dead) hi = -1;
    else if (it.partial)
      col_live_range(j, tile_geo(p.list, it.blk, p.N).lb, kg.lb, kg.n, p.mask, lo, hi);
    prefetch_tile_bits(p.list, it.slot, row);
    const bool ok = wait_bar(bar(L::kSFull), s1_cnt & 1, abort_flag, p.status, 20);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    ++s1_cnt;
    tc_fence_after();
    tmem_ld_x64(tA, sv);
    if (it.partial || it.dead) {  // dead entries: S^T = -inf, so P^T = 0 below (scale > 0)
#pragma unroll
      for (int e = 0; e < 64; ++e)
        if (64 * g + e < lo || 64 * g + e > hi) sv[e] = kNegInfBits;
      if (it.slot >= 0) {  // bit-packed mask tile: this key row's bits over 64 queries
        uint32_t bw[2];
        load_tile_bits<2>(p.list, it.slot, row, 2 * g, bw);
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (!((bw[e >> 5] >> (e & 31)) & 1u)) sv[e] = kNegInfBits;
      }
    }
    uint32_t pp[32];
    float4 l4n = *reinterpret_cast<const float4*>(vec + 64 * g);
#pragma unroll
    for (int x = 0; x < 64; x += 4) {
      const float4 l4 = l4n;
      if (x + 4 < 64)  // next group's -LSE, loaded one group ahead
        l4n = *reinterpret_cast<const float4*>(vec + 64 * g + x + 4);
      const float nl[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        float x0, x1;
        fma2(x0, x1, __uint_as_float(sv[x + e]), __uint_as_float(sv[x + e + 1]), sl2, sl2,
             nl[e], nl[e + 1]);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        sv[x + e] = __float_as_uint(p0);
        sv[x + e + 1] = __float_as_uint(p1);
        pp[(x + e) / 2] = pack_bf16x2(p0, p1);
      }
    }
    tmem_st_x32(tA, pp);
    tmem_wait_st();
    warp_arrive(bar(L::kPFull));
    return true;
  };
  // pass 2: dS^T = P^T o (dP^T - D), bf16 to columns [64 g, 64 g + 32) of B
  // and to this key row of the dS tile, ds_full
  auto pass2 = [&](const float* vec) -> bool {
    const bool ok = wait_bar(bar(L::kSFull + 1), s2_cnt & 1, abort_flag, p.status, 24);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    ++s2_cnt;
    tc_fence_after();
    uint32_t dpv[64];
    tmem_ld_x64(tB, dpv);
    uint32_t dd[32];
    float4 d4n = *reinterpret_cast<const float4*>(vec + 128 + 64 * g);
#pragma unroll
    for (int x = 0; x < 64; x += 4) {
      const float4 d4 = d4n;
      if (x + 4 < 64) d4n = *reinterpret_cast<const float4*>(vec + 128 + 64 * g + x + 4);
      const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        float u0, u1, d0, d1;
        sub2(u0, u1, __uint_as_float(dpv[x + e]), __uint_as_float(dpv[x + e + 1]), dv[e],
             dv[e + 1]);
        mul2(d0, d1, __uint_as_float(sv[x + e]), __uint_as_float(sv[x + e + 1]), u0, u1);
        dd[(x + e) / 2] = pack_bf16x2(d0, d1);
      }
    }
    tmem_st_x32(tB, dd);
    // the previous drain's bulk reductions must have read the buffer
    if (wg_leader) bulk_wait_read_all();
    if (!wg_sync()) return false;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<uint4*>(ds_row + ((q ^ (row & 7)) << 4)) =
          make_uint4(dd[4 * q], dd[4 * q + 1], dd[4 * q + 2], dd[4 * q + 3]);
    fence_proxy_async_smem();  // the tensor core reads the dS tile through the async proxy
    tmem_wait_st();
    warp_arrive(bar(L::kPFull + 1));
    return true;
  };
  // drain: the warpgroup's half of dQ(t) into the fp32 accumulator
  // (unscaled), in rounds of 32 columns staged through the warpgroup's 16 KB
  // half of the dS tile (free once dQ(t) has read it): each thread writes its
  // query row (128 bytes, 128-byte swizzled), and the warpgroup's first
  // thread has the TMA engine add the 128 x 32 tile into the accumulator
  auto drain = [&](const Unit& un, int t) -> bool {
    int hq;
    const InnerTile it = bwd_inner<true>(un, t, p, hq);
    const bool ok = wait_bar(bar(L::kDqFull), dq_cnt & 1, abort_flag, p.status, 25);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    ++dq_cnt;
    tc_fence_after();
    constexpr int kRounds = HD / 64;
#pragma unroll
    for (int q = 0; q < kRounds; ++q) {
      uint32_t v[32];
      tmem_ld_x32(tDQ + 32 * q, v);
      if (q == kRounds - 1) warp_arrive(bar(L::kDqFree));
      if (q > 0) {  // the previous round's copy must have left the staging buffer
        if (wg_leader) bulk_wait_read_all();
        if (!wg_sync()) return false;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(ds_row + ((k ^ (row & 7)) << 4)) =
            make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
      fence_proxy_async_smem();  // the TMA engine reads the tile through the async proxy
      if (!wg_sync()) return false;
      if (wg_leader && !it.dead) {
        tma_reduce_add_4d(&p.tm_dqacc, stage, g * (HD / 2) + 32 * q, it.blk * kTile, hq, un.b);
        bulk_commit_group();
      }
    }
    return true;
  };
  while (true) {
    const int u = queue_pop<true>(queue, abort_flag, p.status);
    if (u < 0) return;
    const Unit un = bwd_decode<true>(u, p);
    // this key row: token j of its sequence (kg.n tokens), token kg.row0 + row of the axis
    const TileGeo kg = tile_geo(p.list, un.ob, p.N);
    const int64_t j = int64_t(kg.lb) * kTile + row;
    const bool valid = j < kg.n;
    const int64_t ktok = kg.row0 + row;
    __nv_bfloat16* dk_row = p.out_a + ((int64_t(un.b) * p.N + ktok) * p.Hkv + un.h) * HD;
    __nv_bfloat16* dv_row = p.out_b + ((int64_t(un.b) * p.N + ktok) * p.Hkv + un.h) * HD;
    if (un.n == 0) {
      if (g == 0) {
        zero_row(dk_row, HD, valid);
        zero_row(dv_row, HD, valid);
      }
      continue;
    }
    if (!pass1(un, 0, j, kg, vec_at(cnt))) return;
    for (int t = 0; t < un.n; ++t) {
      const uint32_t c = cnt + 2 * t;
      if (!pass2(vec_at(c))) return;
      if (t + 1 < un.n && !pass1(un, t + 1, j, kg, vec_at(c + 2))) return;
      if (!drain(un, t)) return;
    }
    cnt += 2 * un.n;
    const bool ok = wait_bar(bar(L::kAccFull), af_cnt & 1, abort_flag, p.status, 21);
    if (!__all_sync(0xFFFFFFFFu, ok)) return;
    ++af_cnt;
    tc_fence_after();
    // warpgroup g writes dV and dK columns [d/2 g, d/2 (g + 1))
    const int64_t stride = int64_t(p.Hkv) * HD * 2;  // bytes between consecutive key rows
    store_acc_piece<HD>(tDV + g * (HD / 2), 1.f, dv_row + g * (HD / 2), stride, valid);
    store_acc_piece<HD>(tDK + g * (HD / 2), p.scale, dk_row + g * (HD / 2), stride, valid);
    warp_arrive(bar(L::kAccEmpty));
  }
}

// Elementwise warpgroups of bwd_dq: thread = query row i of the query tile,
// warpgroup g = key columns [64 g, 64 g + 64).  Per unit the warpgroups first
// write the row's dO into TMEM (warpgroup g: head-dimension half g).  Per key
// tile, S and dP are pulled into registers at once (releasing both regions
// for the next tile's products), dS is computed there and written as bf16
// to the dS columns.  The next unit's dO is staged before this unit's dQ is
// stored, so the next unit's first products overlap the store.
template <int HD>
__device__ __forceinline__ void dq_elementwise(const BwdParams& p, uint8_t* smem, uint64_t* bars,
                                               uint32_t tmem, int g, volatile int* abort_flag) {
  using L = BwdLayout<HD, kModeDq>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int wq = int(warp_id()) & 3;
  const int row = wq * 32 + int(lane_id());
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t tS = tmem + lane_off + 64 * g, tDP = tS + 128, tDQ = tmem + lane_off + 256;
  const uint32_t tDS = tmem + lane_off + 384 + 32 * g;  // keys [64 g, 64 g + 64) as pairs
  const uint32_t tDO = tmem + lane_off + 448 + (HD / 4) * g;
  const float sl2 = p.scale_log2;
  uint32_t sp_cnt = 0, af_cnt = 0, fe_cnt = 0, ds_cnt = 0;
  UnitQueue queue = unit_queue<HD, kModeDq>(smem, bars);
  // next unit with live key tiles; units without any get zero dQ rows here
  auto next = [&](Unit& un) -> bool {
    while (true) {
      const int u = queue_pop<true>(queue, abort_flag, p.status);
      if (u < 0) return false;
      un = bwd_decode<false>(u, p);
      if (un.n > 0) return true;
      const TileGeo qg = tile_geo(p.list, un.ob, p.N);
      if (g == 0)
        zero_row(p.out_a + ((int64_t(un.b) * p.N + qg.row0 + row) * p.H + un.h) * HD, HD,
                 int64_t(qg.lb) * kTile + row < qg.n);
    }
  };
  // this row's dO half into TMEM (after the previous unit's last dP has
  // been computed), its -LSE * log2(e) and D into nl2 / di
  auto stage_unit = [&](const Unit& un, float& nl2, float& di) -> bool {
    const TileGeo qg = tile_geo(p.list, un.ob, p.N);
    const bool valid = int64_t(qg.lb) * kTile + row < qg.n;
    const int64_t i = int64_t(un.ob) * kTile + row;  // row of the (tile-layout) vectors
    const uint4* src = reinterpret_cast<const uint4*>(
        p.dout + ((int64_t(un.b) * p.N + qg.row0 + row) * p.H + un.h) * HD + (HD / 2) * g);
    uint32_t rw[HD / 4];
#pragma unroll
    for (int j = 0; j < HD / 16; ++j) {
      const uint4 v = valid ? src[j] : make_uint4(0, 0, 0, 0);
      rw[4 * j] = v.x;
      rw[4 * j + 1] = v.y;
      rw[4 * j + 2] = v.z;
      rw[4 * j + 3] = v.w;
    }
    const int64_t vrow = (int64_t(un.b) * p.H + un.h) * p.NP + i;  // i < NP always
    nl2 = p.nlse2[vrow];
    di = p.dsum[vrow];
    const bool ok = wait_bar(bar(L::kFixEmpty), (fe_cnt & 1) ^ 1, abort_flag, p.status, 22);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    ++fe_cnt;
    tc_fence_after();
    if constexpr (HD == 128) tmem_st_x32(tDO, rw);
    else tmem_st_x16(tDO, rw);
    tmem_wait_st();
    warp_arrive(bar(L::kFixFull));
    return true;
  };
  Unit cur;
  bool has = next(cur);
  float nl2 = 0.f, di = 0.f;
  if (has && !stage_unit(cur, nl2, di)) return;
  while (has) {
    // this query row: token i of its sequence (qg.n tokens), token qg.row0 + row of the axis
    const TileGeo qg = tile_geo(p.list, cur.ob, p.N);
    const int64_t i = int64_t(qg.lb) * kTile + row;
    for (int t = 0; t < cur.n; ++t) {
      const InnerTile it = inner_tile(cur, t, p.list, p.status);
      int lo = 0, hi = kTile - 1;
      if (it.dead) hi = -1;
      else if (it.partial)
        row_live_range(i, qg.lb, tile_geo(p.list, it.blk, p.N).lb, qg.n, p.mask, lo, hi);
      prefetch_tile_bits(p.list, it.slot, row);
      bool ok = wait_bar(bar(L::kSFull), sp_cnt & 1, abort_flag, p.status, 20);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      ++sp_cnt;
      tc_fence_after();
      uint32_t sv[64], dpv[64];
      tmem_ld_x64x2(tS, tDP, sv, dpv);
      warp_arrive(bar(L::kDpFree));  // S and dP of this tile are in registers
      if (it.partial || it.dead) {  // dead entries: S = -inf, so P = 0 below (scale > 0)
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (64 * g + e < lo || 64 * g + e > hi) sv[e] = kNegInfBits;
        if (it.slot >= 0) {  // bit-packed mask tile: this query row's bits over 64 keys
          uint32_t bw[2];
          load_tile_bits<2>(p.list, it.slot, row, 2 * g, bw);
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (!((bw[e >> 5] >> (e & 31)) & 1u)) sv[e] = kNegInfBits;
        }
      }
      uint32_t dd[32];
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        float x0, x1, p0, p1, u0, u1, d0, d1;
        fma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), sl2, sl2, nl2, nl2);
        p0 = ex2_approx(x0);
        p1 = ex2_approx(x1);
        sub2(u0, u1, __uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1]), di, di);
        mul2(d0, d1, p0, p1, u0, u1);
        dd[e / 2] = pack_bf16x2(d0, d1);
      }
      ok = wait_bar(bar(L::kDsEmpty), (ds_cnt & 1) ^ 1, abort_flag, p.status, 23);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      ++ds_cnt;
      tc_fence_after();
      tmem_st_x32(tDS, dd);
      tmem_wait_st();
      warp_arrive(bar(L::kPFull));
    }
    Unit nxt;
    float nnl2 = 0.f, ndi = 0.f;
    const bool has_next = next(nxt);
    if (has_next && !stage_unit(nxt, nnl2, ndi)) return;
    const bool ok = wait_bar(bar(L::kAccFull), af_cnt & 1, abort_flag, p.status, 21);
    if (!__all_sync(0xFFFFFFFFu, ok)) return;
    ++af_cnt;
    tc_fence_after();
    __nv_bfloat16* dq_row =
        p.out_a + ((int64_t(cur.b) * p.N + qg.row0 + row) * p.H + cur.h) * HD;
    store_acc_piece<HD>(tDQ + g * (HD / 2), p.scale, dq_row + g * (HD / 2),
                        int64_t(p.H) * HD * 2, i < qg.n);
    warp_arrive(bar(L::kAccEmpty));
    cur = nxt;
    has = has_next;
    nl2 = nnl2;
    di = ndi;
  }
}

template <int HD, int kMode>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdLayout<HD, kMode>;
  extern __shared__ uint8_t smem_raw[];
  if (kMode == kModeFused && (smem_u32(smem_raw) & 1023u) != 0) {
    // no room for alignment slack (see BwdLayout): refuse, uniformly, before
    // any barrier or TMEM allocation
    if (threadIdx.x == 0) record_status(p.status, FLASH_MSA_ERR_UNSUPPORTED, 0xF5);
    return;
  }
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
    abort_flag[0] = 0;
    abort_flag[1] = p.wait_limit_ms;
    init_bwd_barriers<HD, kMode>(bars);
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_do);
    if (kMode == kModeFused) tma_prefetch_desc(&p.tm_dqacc);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp < 4) regs_shrink<80>();  // 384 x 168 at launch: 128 x 80 + 256 x 208
  if (warp == 0) {
    if (lane == 0) bwd_producer<HD, kMode>(p, smem, bars, abort_flag);
  } else if (warp == 1) {  // the whole warp: the MMA wrappers elect one lane
    if (kMode == kModeFused) fused_mma<HD>(p, smem, bars, tmem, abort_flag);
    else if (kMode == kModeDkdv) dkdv_mma<HD>(p, smem, bars, tmem, abort_flag);
    else dq_mma<HD>(p, smem, bars, tmem, abort_flag);
  } else if (warp >= 4) {
    const int g = (warp - 4) >> 2;  // elementwise warpgroup: columns [64 g, 64 g + 64)
    regs_grow<208>();
    if (kMode == kModeFused) {
      fused_elementwise<HD>(p, smem, bars, tmem, g, abort_flag);
      // bulk reductions still in flight read shared memory: finish them
      // before the CTA releases it
      if ((threadIdx.x & 127) == 0) bulk_wait_all();
    } else if (kMode == kModeDkdv) {
      dkdv_elementwise<HD>(p, smem, bars, tmem, g, abort_flag);
    } else {
      dq_elementwise<HD>(p, smem, bars, tmem, g, abort_flag);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dQ = scale * accumulator, fp32 (B, H, NP, d) -> bf16 (B, N, H, d); one
// thread per 8 elements, consecutive threads along the output.
template <int HD>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         __nv_bfloat16* __restrict__ dq, int B,
                                                         int H, int N, int NP, float scale) {
  constexpr int kChunks = HD / 8;
  const int64_t total = int64_t(B) * N * H * kChunks;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int c = int(e % kChunks);
    const int64_t r = e / kChunks;  // output row (b, i, h)
    const int h = int(r % H);
    const int64_t bi = r / H;
    const int i = int(bi % N);
    const int b = int(bi / N);
    const float4* src =
        reinterpret_cast<const float4*>(acc + ((int64_t(b) * H + h) * NP + i) * HD + c * 8);
    const float4 x = __ldg(src), y = __ldg(src + 1);
    uint4 w;
    w.x = pack_bf16x2(x.x * scale, x.y * scale);
    w.y = pack_bf16x2(x.z * scale, x.w * scale);
    w.z = pack_bf16x2(y.x * scale, y.y * scale);
    w.w = pack_bf16x2(y.z * scale, y.w * scale);
    *reinterpret_cast<uint4*>(dq + r * HD + c * 8) = w;
  }
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
// Heads per group of the fused kernel's unit order: the CTAs running at any
// time then add into the accumulators of about this many bytes of heads
// (plus their streamed Q and dO tiles), which stay resident in the 129 MB L2.
constexpr int64_t kFusedGroupBytes = int64_t(48) << 20;

// Units of the two-kernel backward are numbered rank-major within groups of
// heads whose streamed tiles (per_head_bytes each) fit kBwdGroupBytes, so
// the CTAs working at the same time re-read the same heads' tiles from L2
// (129 MB) instead of DRAM.  When fewer than two heads fit, one group of all
// heads keeps plain rank-major order (longest units first over the launch).
constexpr int64_t kBwdGroupBytes = int64_t(64) << 20;
static int bwd_head_group(int64_t per_head_bytes, int heads) {
  const int64_t g = kBwdGroupBytes / (per_head_bytes > 0 ? per_head_bytes : 1);
  return (g < 2 || g >= heads) ? heads : int(g);
}

template <int HD>
static flash_msa_status launch_bwd_hd(const BwdLaunch& a, cudaStream_t stream) {
  using LK = BwdLayout<HD, kModeDkdv>;
  using LQ = BwdLayout<HD, kModeDq>;
  using LF = BwdLayout<HD, kModeFused>;
  const int nb = a.rows.n_blocks;
  const int NP = nb * kTile;
  float* nlse2 = a.dsum;                        // workspace: [nlse2 | dsum | dQ accumulator]
  float* dsum = a.dsum + int64_t(a.B) * a.H * NP;
  if (a.stages & FLASH_MSA_BWD_PREPROCESS) {
    PreParams pp{reinterpret_cast<const __nv_bfloat16*>(a.o),
                 reinterpret_cast<const __nv_bfloat16*>(a.dout), a.lse, nlse2, dsum, a.dqacc,
                 a.B, a.H, int(a.N), NP, a.rows};
    constexpr int kRows = 256 / (HD / 8);
    dim3 grid((NP + kRows - 1) / kRows, a.H, a.B);
    bwd_pre_kernel<HD><<<grid, 256, 0, stream>>>(pp);
    if (cudaGetLastError() != cudaSuccess) return set_cuda_error("bwd_pre launch");
  }
  BwdParams p;
  memset(&p, 0, sizeof(p));
  flash_msa_status st;
  if (a.stages & (FLASH_MSA_BWD_DKDV | FLASH_MSA_BWD_DQ | FLASH_MSA_BWD_FUSED)) {
    if ((st = make_tile_map(&p.tm_q, a.q, a.B, a.N, a.H, HD)) != FLASH_MSA_OK) return st;
    if ((st = make_tile_map(&p.tm_k, a.k, a.B, a.N, a.Hkv, HD)) != FLASH_MSA_OK) return st;
    if ((st = make_tile_map(&p.tm_v, a.v, a.B, a.N, a.Hkv, HD)) != FLASH_MSA_OK) return st;
    if ((st = make_tile_map(&p.tm_do, a.dout, a.B, a.N, a.H, HD)) != FLASH_MSA_OK) return st;
  }
  p.nlse2 = nlse2;
  p.dsum = dsum;
  p.dqacc = a.dqacc;
  p.dout = reinterpret_cast<const __nv_bfloat16*>(a.dout);
  p.B = a.B;
  p.H = a.H;
  p.N = int(a.N);
  p.NP = NP;
  p.Hkv = a.Hkv;
  p.G = a.H / a.Hkv;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.mask = a.mask;
  p.status = a.status;
  p.wait_limit_ms = int(wait_limit_ms());
  // persistent launches: one CTA per SM (fewer for small problems), units
  // handed out in order by a counter set up just before each kernel
  const int sms = sm_count();
  if (sms <= 0) return set_cuda_error("bwd: multiprocessor count");
  auto claim_counter = [&]() -> flash_msa_status {
    SchedCounter c;
    const flash_msa_status r = claim_sched_counter(stream, &c);
    p.sched = c.counter;
    p.ticket = c.ticket;
    return r;
  };
  // which: bit of enable_smem for this kernel instantiation
  auto launch = [&](const void* kern, int smem_bytes, unsigned which, auto kernel_fn,
                    const char* what) -> flash_msa_status {
    flash_msa_status r = enable_smem(kern, smem_bytes, which, "cudaFuncSetAttribute(bwd)");
    if (r != FLASH_MSA_OK) return r;
    if ((r = claim_counter()) != FLASH_MSA_OK) return r;
    const int grid = p.n_units < sms ? p.n_units : sms;
    kernel_fn<<<grid, kBwdThreads, smem_bytes, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return set_cuda_error(what);
    return FLASH_MSA_OK;
  };
  const unsigned hd_bit = HD == 128 ? 1u : 0u;
  if (a.stages & FLASH_MSA_BWD_DKDV) {
    p.list = a.cols;
    p.n_units = a.B * a.Hkv * nb;
    // a key/value head's units stream the Q and dO tiles of its H / Hkv query heads
    p.head_group = bwd_head_group(int64_t(a.H / a.Hkv) * 2 * a.N * a.d * 2, a.B * a.Hkv);
    p.out_a = reinterpret_cast<__nv_bfloat16*>(a.dk);
    p.out_b = reinterpret_cast<__nv_bfloat16*>(a.dv);
    if ((st = launch(reinterpret_cast<const void*>(&bwd_main_kernel<HD, kModeDkdv>),
                     LK::kSmemBytes, 2 + hd_bit, bwd_main_kernel<HD, kModeDkdv>,
                     "bwd_dkdv launch")) != FLASH_MSA_OK)
      return st;
  }
  if (a.stages & FLASH_MSA_BWD_DQ) {
    p.list = a.rows;
    p.n_units = a.B * a.H * nb;
    p.head_group = bwd_head_group(int64_t(2) * a.N * a.d * 2, a.B * a.H);  // K and V tiles
    p.out_a = reinterpret_cast<__nv_bfloat16*>(a.dq);
    p.out_b = nullptr;
    if ((st = launch(reinterpret_cast<const void*>(&bwd_main_kernel<HD, kModeDq>),
                     LQ::kSmemBytes, 4 + hd_bit, bwd_main_kernel<HD, kModeDq>,
                     "bwd_dq launch")) != FLASH_MSA_OK)
      return st;
  }
  if (a.stages & FLASH_MSA_BWD_FUSED) {
    if (!a.dqacc) return set_error(FLASH_MSA_ERR_WORKSPACE, "bwd: no dQ accumulator");
    if ((st = make_acc_map(&p.tm_dqacc, a.dqacc, a.B, a.H, NP, HD)) != FLASH_MSA_OK) return st;
    p.list = a.cols;
    p.n_units = a.B * a.Hkv * nb;
    // key/value heads per group: accumulator (G query heads) plus Q and dO
    const int64_t per_head = int64_t(NP) * HD * (4 + 2 + 2) * p.G;
    int grp = int(kFusedGroupBytes / (per_head > 0 ? per_head : 1));
    if (grp < 1) grp = 1;
    if (grp > a.B * a.Hkv) grp = a.B * a.Hkv;
    p.head_group = grp;
    p.out_a = reinterpret_cast<__nv_bfloat16*>(a.dk);
    p.out_b = reinterpret_cast<__nv_bfloat16*>(a.dv);
    if ((st = launch(reinterpret_cast<const void*>(&bwd_main_kernel<HD, kModeFused>),
                     LF::kSmemBytes, 6 + hd_bit, bwd_main_kernel<HD, kModeFused>,
                     "bwd_fused launch")) != FLASH_MSA_OK)
      return st;
  }
  if (a.stages & FLASH_MSA_BWD_DQ_CONVERT) {
    const int64_t chunks = int64_t(a.B) * a.N * a.H * (HD / 8);
    int64_t blocks = (chunks + 255) / 256;
    if (blocks > int64_t(sms) * 16) blocks = int64_t(sms) * 16;
    dq_convert_kernel<HD><<<int(blocks), 256, 0, stream>>>(
        a.dqacc, reinterpret_cast<__nv_bfloat16*>(a.dq), a.B, a.H, int(a.N), NP, a.scale);
    if (cudaGetLastError() != cudaSuccess) return set_cuda_error("dq_convert launch");
  }
  return FLASH_MSA_OK;
}

flash_msa_status launch_bwd(const BwdLaunch& a, cudaStream_t stream) {
  if (a.d == 128) return launch_bwd_hd<128>(a, stream);
  return launch_bwd_hd<64>(a, stream);
}

}  // namespace fmsa
