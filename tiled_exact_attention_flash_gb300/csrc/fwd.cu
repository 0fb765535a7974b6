// Forward attention kernel for sm_103a: O = softmax(mask(Q K^T * scale)) V
// and LSE, two neighbouring 128-row query tiles per CTA, tile by tile over
// their live key tiles with an online softmax ("Flash MSA Attention Kernel
// Implementation", sections "The Flash Core: Tiling Over the Memory
// Hierarchy" and "Optimization Tricks That Actually Matter"; sparse lists
// from "How Does Flash-MSA Sparse Attention Work", section "How Flash-MSA
// Sparse Attention Works").
//
// CTA layout (384 threads, one CTA per SM, each working through pair units):
//   warp 0      TMA producer: Q tiles and the K/V ring, one elected lane
//   warp 1      MMA issuer: tcgen05.mma for S = Q K^T and O += P V (the
//               whole warp runs the loop, one elected lane issues; for
//               index lists whose pairs mostly differ: slot 0 only, warp 3
//               issuing for slot 1)
//   warp 2      TMEM allocator
//   warps 4-7   softmax + epilogue for query slot 0 (thread = query row)
//   warps 8-11  softmax + epilogue for query slot 1
// The two query slots hold two neighbouring query blocks of one head and
// share every key/value tile load; the tensor core works on one slot's
// products while the other slot's softmax runs.  TMEM (512 columns):
//   slot s: S at columns [256 s, 256 s + 128), P (bf16, two per column)
//   aliased onto the first 64 of them, O at [256 s + 128, 256 s + 128 + d).
// Shared memory: one Q tile per slot, a ring of K/V tile pairs, all 128-byte
// swizzled by TMA and read by the tensor core through matrix descriptors.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fmsa {

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;
  __nv_bfloat16* o;
  float* lse;
  int B, H, N;
  int G;  // query heads per key/value head
  int n_units;
  UnitOrder order;   // pair units: rank-major over all heads
  int slot_issuers;  // one MMA-issuing warp per query slot (else one for both)
  float scale_log2;  // scale * log2(e)
  int wait_limit_ms;  // limit of any single bounded wait
  MaskParams mask;
  ListParams list;
  unsigned* status;
};

template <int HD>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * HD * 2;
  // K/V ring: kSlots slots of two tile buffers; a slot holds what one step
  // of the MMA loop consumes and releases together: V of tile t in its first
  // buffer and K of the next tile in its second (a unit's first slot holds
  // only K of its first tile, its last only V of its last tile)
  static constexpr int kSlots = HD == 128 ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + 2 * kSlots * kTileBytes;
  // barrier slots
  static constexpr int kQFull = 0, kQEmpty = 2, kSFull = 4, kPFull = 6, kOFull = 8, kOEmpty = 10,
                       kMmaDone = 12, kKvFull = 13, kKvEmpty = 13 + kSlots;
  static constexpr int kNumBars = 13 + 2 * kSlots;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // misc: TMEM base address, abort flag, wait limit
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack for 1024-byte alignment
};

constexpr int kFwdThreads = 384;

// Work unit = a pair of query blocks of one (b, h): ranks 2r and 2r + 1 of
// the longest-first order (for causal and window masks, two neighbouring
// blocks whose key-tile lists nearly coincide).  Slot 0 takes rank 2r, slot
// 1 rank 2r + 1.  The producer loads each key/value tile of the UNION of the
// two lists once; the MMA issuer runs Q K^T and P V for whichever slots the
// tile belongs to.  Pair units are numbered rank-major (unit_order_grouped
// with one group of all heads: pair r
// of every (b, h) before pair r + 1), so the launch runs its longest units
// first; each CTA takes its units in the order of fwd_unit.
struct PairUnit {
  int b, h;
  int q[2];       // query block per slot (q[1] < 0: no second block)
  int beg[2], n[2];
};

// Unit k of this CTA.  One CTA per SM; units are dealt serpentine-wise (CTA c
// takes c, then 2G - 1 - c, then 2G + c, ...), which evens out the CTAs'
// shares of the rank-major (longest first) unit lengths.
__device__ __forceinline__ int fwd_unit(int k) {
  const int c = int(blockIdx.x), g = int(gridDim.x);
  return k * g + ((k & 1) ? g - 1 - c : c);
}

__device__ __forceinline__ PairUnit decode_pair(int u, const FwdParams& p) {
  const ListParams& L = p.list;
  PairUnit pu;
  int r;
  unit_order_grouped(u, (L.n_blocks + 1) / 2, p.order, pu.b, pu.h, r);
  for (int s = 0; s < 2; ++s) {
    const int rank = 2 * r + s;
    pu.q[s] = -1;
    pu.beg[s] = 0;
    pu.n[s] = 0;
    if (rank >= L.n_blocks) continue;
    // the single-unit decoder gives the block id and its list bounds
    Unit un;
    decode_block_at(un, rank, L, p.status);
    pu.q[s] = un.ob;
    pu.beg[s] = un.begin;
    pu.n[s] = un.n;
  }
  return pu;
}

// Merged walk over the two slots' key-tile lists (ascending key block).
struct PairWalk {
  int pos[2];  // next position in each list (index mode) or next key block (arithmetic)
  int end[2];
};

struct PairTile {
  int kb;
  bool in[2];
};

__device__ __forceinline__ void walk_init(PairWalk& w, const PairUnit& pu, const ListParams& L) {
  for (int s = 0; s < 2; ++s) {
    if (L.ptr) {
      w.pos[s] = pu.beg[s];
      w.end[s] = pu.beg[s] + pu.n[s];
    } else {
      w.pos[s] = 0;
      w.end[s] = pu.n[s];  // arithmetic lists are 0 .. n-1
    }
  }
}

__device__ __forceinline__ bool walk_next(PairWalk& w, const ListParams& L, PairTile& t) {
  int k[2];
  for (int s = 0; s < 2; ++s) {
    if (w.pos[s] >= w.end[s]) {
      k[s] = 0x7FFFFFFF;
    } else if (L.ptr) {
      k[s] = __ldg(L.idx + w.pos[s]);
      if (k[s] < 0 || k[s] >= L.n_blocks) k[s] = 0;  // reported by the softmax side
    } else {
      k[s] = w.pos[s];
    }
  }
  const int m = k[0] < k[1] ? k[0] : k[1];
  if (m == 0x7FFFFFFF) return false;
  t.kb = m;
  for (int s = 0; s < 2; ++s) {
    t.in[s] = (k[s] == m);
    if (t.in[s]) ++w.pos[s];
  }
  return true;
}

template <int HD>
__device__ __forceinline__ void load_tile(const CUtensorMap* m, uint32_t dst, uint32_t b, int row,
                                          int h, int bb) {
#pragma unroll
  for (int c = 0; c < HD / 64; ++c) tma_load_4d(dst + c * (kTile * 128), m, b, c * 64, row, h, bb);
}

template <int HD>
__device__ __forceinline__ void fwd_producer(const FwdParams& p, uint8_t* smem, uint64_t* bars,
                                             volatile int* abort_flag) {
  using L = FwdLayout<HD>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  uint32_t g_cnt = 0, qe_cnt[2] = {0, 0};
  int last_g[L::kSlots];  // last group loaded into each slot, -1 if none
  for (int i = 0; i < L::kSlots; ++i) last_g[i] = -1;
  int last_q[2] = {-1, -1};
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int u = fwd_unit(k);
    if (u >= p.n_units) break;
    const PairUnit pu = decode_pair(u, p);
    if (pu.n[0] + pu.n[1] == 0) continue;
    for (int s = 0; s < 2; ++s) {
      if (pu.n[s] == 0) continue;
      if (!wait_bar(bar(L::kQEmpty + s), (qe_cnt[s] & 1) ^ 1, abort_flag, p.status, 2)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(bar(L::kQFull + s), L::kTileBytes);
      load_tile<HD>(&p.tm_q, smem_u32(smem + L::kQOff + s * L::kTileBytes), bar(L::kQFull + s),
                    int(tile_geo(p.list, pu.q[s], p.N).row0), pu.h, pu.b);
      last_q[s] = int(qe_cnt[s]);
      ++qe_cnt[s];
    }
    if (!ok) break;
    const int hkv = pu.h / p.G;  // key/value head of this query head
    // one ring slot: tile kb_a of map `ma` into its first buffer and, if
    // kb_b >= 0, K tile kb_b into its second
    auto load_group = [&](const CUtensorMap* ma, int kb_a, int kb_b) {
      const int slot = int(g_cnt % L::kSlots);
      if (!wait_bar(bar(L::kKvEmpty + slot), ((g_cnt / L::kSlots) & 1) ^ 1, abort_flag, p.status,
                    3))
        return false;
      mbar_arrive_expect_tx(bar(L::kKvFull + slot), (kb_b >= 0 ? 2 : 1) * L::kTileBytes);
      const uint32_t dst = smem_u32(smem + L::kRingOff + 2 * slot * L::kTileBytes);
      load_tile<HD>(ma, dst, bar(L::kKvFull + slot), int(tile_geo(p.list, kb_a, p.N).row0), hkv,
                    pu.b);
      if (kb_b >= 0)
        load_tile<HD>(&p.tm_k, dst + L::kTileBytes, bar(L::kKvFull + slot),
                      int(tile_geo(p.list, kb_b, p.N).row0), hkv, pu.b);
      last_g[slot] = int(g_cnt);
      ++g_cnt;
      return true;
    };
    PairWalk w;
    walk_init(w, pu, p.list);
    PairTile cur, nxt;
    walk_next(w, p.list, cur);  // the union is non-empty
    ok = load_group(&p.tm_k, cur.kb, -1);  // K of the first tile
    while (ok) {
      const bool more = walk_next(w, p.list, nxt);
      ok = load_group(&p.tm_v, cur.kb, more ? nxt.kb : -1);  // V of cur, K of nxt
      if (!more) break;
      cur = nxt;
    }
  }
  if (!ok) {  // let copies already issued land before the CTA exits
    for (int i = 0; i < L::kSlots; ++i)
      if (last_g[i] >= 0) drain_bar(bar(L::kKvFull + i), (last_g[i] / L::kSlots) & 1);
    for (int s = 0; s < 2; ++s)
      if (last_q[s] >= 0) drain_bar(bar(L::kQFull + s), last_q[s] & 1);
  }
}

template <int HD>
__device__ __forceinline__ void fwd_mma(const FwdParams& p, uint8_t* smem, uint64_t* bars,
                                        uint32_t tmem, volatile int* abort_flag) {
  using L = FwdLayout<HD>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdPV = idesc_bf16_f32(128, HD, false, true);
  uint32_t g_cnt = 0, qf_cnt[2] = {0, 0}, pf_cnt[2] = {0, 0}, oe_cnt[2] = {0, 0};
  const uint32_t ring = smem_u32(smem + L::kRingOff);
  // buffer h of the slot holding group g
  auto buf = [&](uint32_t g, int h) { return ring + (2 * (g % L::kSlots) + h) * L::kTileBytes; };
  auto wait_group = [&](uint32_t g, unsigned where) {
    return wait_bar_warp(bar(L::kKvFull + g % L::kSlots), (g / L::kSlots) & 1, abort_flag, p.status,
                    where);
  };
  bool ok = true;
  // S_s = Q_s K^T for the K tile at shared address kaddr
  auto issue_qk = [&](int s, uint32_t kaddr) {
    const uint32_t qd = sdesc_lo(smem_u32(smem + L::kQOff + s * L::kTileBytes), 16);
    const uint32_t kd = sdesc_lo(kaddr, 16);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      // A = Q, B = K, both K-major: 16-element k-steps are 32 bytes apart
      // inside a 128-byte swizzle row, 64-element chunks 16 KB apart
      const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
      mma_ss(tmem + uint32_t(s * 256), qd + off, kd + off, kIdQK, kk > 0 ? 1u : 0u);
    }
    mma_commit(bar(L::kSFull + s));
  };
  for (int k = 0; ok; ++k) {
    const int u = fwd_unit(k);
    if (u >= p.n_units) break;
    const PairUnit pu = decode_pair(u, p);
    if (pu.n[0] + pu.n[1] == 0) continue;
    int seen[2] = {0, 0};    // P V products issued per slot in this unit
    int issued[2] = {0, 0};  // Q K^T products issued per slot in this unit
    PairWalk w;
    walk_init(w, pu, p.list);
    PairTile cur, nxt;
    walk_next(w, p.list, cur);  // the union is non-empty
    // prologue: Q K^T of the first tile (the unit's first ring group: its K)
    {
      for (int s = 0; s < 2 && ok; ++s)
        if (cur.in[s] && !wait_bar_warp(bar(L::kQFull + s), qf_cnt[s] & 1, abort_flag, p.status, 13))
          ok = false;
      if (ok && !wait_group(g_cnt, 14)) ok = false;
      if (!ok) break;
      tc_fence_after();
      for (int s = 0; s < 2; ++s) {
        if (!cur.in[s]) continue;
        ++qf_cnt[s];
        issue_qk(s, buf(g_cnt, 0));
        if (++issued[s] == pu.n[s]) mma_commit(bar(L::kQEmpty + s));
      }
      mma_commit(bar(L::kKvEmpty + g_cnt % L::kSlots));
      ++g_cnt;
    }
    while (ok) {
      const bool more = walk_next(w, p.list, nxt);
      // this step's group: V of cur (first buffer) and K of nxt (second)
      if (!wait_group(g_cnt, 12)) {
        ok = false;
        break;
      }
      if (more) {
        for (int s = 0; s < 2 && ok; ++s)
          if (nxt.in[s] && issued[s] == 0 &&
              !wait_bar_warp(bar(L::kQFull + s), qf_cnt[s] & 1, abort_flag, p.status, 13))
            ok = false;
        if (!ok) break;
      }
      const uint32_t vaddr = buf(g_cnt, 0), kaddr = buf(g_cnt, 1);
      for (int s = 0; s < 2 && ok; ++s) {
        const uint32_t tS = tmem + uint32_t(s * 256);
        if (cur.in[s]) {  // O_s (+)= P_s V
          if (!wait_bar_warp(bar(L::kPFull + s), pf_cnt[s] & 1, abort_flag, p.status, 10)) {
            ok = false;
            break;
          }
          ++pf_cnt[s];
          if (seen[s] == 0) {
            if (!wait_bar_warp(bar(L::kOEmpty + s), (oe_cnt[s] & 1) ^ 1, abort_flag, p.status, 11)) {
              ok = false;
              break;
            }
            ++oe_cnt[s];
          }
          tc_fence_after();
          // B = V tile, MN-major: 64-column chunks 16 KB apart, 8-row groups
          // 1 KB apart, 16 rows (2 KB) per k-step
          const uint32_t vd = sdesc_lo(vaddr, kTile * 128);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts(tS + 128, tS + kk * 8, vd + kk * (2048 >> 4), kIdPV,
                   (seen[s] > 0 || kk > 0) ? 1u : 0u);
          ++seen[s];
          if (seen[s] == pu.n[s]) mma_commit(bar(L::kOFull + s));
        }
        if (more && nxt.in[s]) {
          if (issued[s] == 0) ++qf_cnt[s];
          tc_fence_after();
          issue_qk(s, kaddr);
          if (++issued[s] == pu.n[s]) mma_commit(bar(L::kQEmpty + s));
        }
      }
      if (!ok) break;
      mma_commit(bar(L::kKvEmpty + g_cnt % L::kSlots));
      ++g_cnt;
      if (!more) break;
      cur = nxt;
    }
  }
  // every MMA issued so far has finished before TMEM is released
  mma_commit(bar(L::kMmaDone));
  drain_bar(bar(L::kMmaDone), 0);
}

template <int HD>
__device__ __forceinline__ void fwd_mma_slot(const FwdParams& p, uint8_t* smem, uint64_t* bars,
                                             uint32_t tmem, int s, volatile int* abort_flag) {
  // MMA issuer of query slot s, used for lists from a block index whose
  // pairs mostly differ (pair_overlap below 1/2): one warp per slot, both
  // walking the same union of key tiles (so both see the same ring groups)
  // and both releasing every group (kKvEmpty then counts two commits).
  // Where the two slots' lists differ, neither slot waits for the other's
  // softmax; where they mostly coincide the single issuer (fwd_mma), whose
  // order staggers the slots, is faster.
  using L = FwdLayout<HD>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdPV = idesc_bf16_f32(128, HD, false, true);
  uint32_t g_cnt = 0, qf_cnt = 0, pf_cnt = 0, oe_cnt = 0;
  const uint32_t ring = smem_u32(smem + L::kRingOff);
  auto buf = [&](uint32_t g, int h) { return ring + (2 * (g % L::kSlots) + h) * L::kTileBytes; };
  // both threads wait for every group they release, used or not: a thread
  // that skipped the wait could release a later use of the slot before the
  // other thread released this one (arrivals are not tagged)
  auto wait_group = [&](uint32_t g, unsigned where) {
    return wait_bar_warp(bar(L::kKvFull + g % L::kSlots), (g / L::kSlots) & 1, abort_flag, p.status,
                    where);
  };
  const uint32_t tS = tmem + uint32_t(s * 256);
  const uint32_t qd = sdesc_lo(smem_u32(smem + L::kQOff + s * L::kTileBytes), 16);
  bool ok = true;
  // S_s = Q_s K^T for the K tile at shared address kaddr
  auto issue_qk = [&](uint32_t kaddr) {
    const uint32_t kd = sdesc_lo(kaddr, 16);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      // A = Q, B = K, both K-major: 16-element k-steps are 32 bytes apart
      // inside a 128-byte swizzle row, 64-element chunks 16 KB apart
      const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
      mma_ss(tS, qd + off, kd + off, kIdQK, kk > 0 ? 1u : 0u);
    }
    mma_commit(bar(L::kSFull + s));
  };
  for (int k = 0; ok; ++k) {
    const int u = fwd_unit(k);
    if (u >= p.n_units) break;
    const PairUnit pu = decode_pair(u, p);
    if (pu.n[0] + pu.n[1] == 0) continue;
    int seen = 0;    // P V products issued in this unit
    int issued = 0;  // Q K^T products issued in this unit
    PairWalk w;
    walk_init(w, pu, p.list);
    PairTile cur, nxt;
    walk_next(w, p.list, cur);  // the union is non-empty
    // prologue: Q K^T of the first tile (the unit's first ring group: its K)
    {
      if (cur.in[s] && !wait_bar_warp(bar(L::kQFull + s), qf_cnt & 1, abort_flag, p.status, 13))
        ok = false;
      if (ok && !wait_group(g_cnt, 14)) ok = false;
      if (!ok) break;
      tc_fence_after();
      if (cur.in[s]) {
        ++qf_cnt;
        issue_qk(buf(g_cnt, 0));
        if (++issued == pu.n[s]) mma_commit(bar(L::kQEmpty + s));
      }
      mma_commit(bar(L::kKvEmpty + g_cnt % L::kSlots));
      ++g_cnt;
    }
    while (ok) {
      const bool more = walk_next(w, p.list, nxt);
      if (!wait_group(g_cnt, 12)) {  // V of cur, K of nxt
        ok = false;
        break;
      }
      if (cur.in[s]) {  // O_s (+)= P_s V
        if (!wait_bar_warp(bar(L::kPFull + s), pf_cnt & 1, abort_flag, p.status, 10)) {
          ok = false;
          break;
        }
        ++pf_cnt;
        if (seen == 0) {
          if (!wait_bar_warp(bar(L::kOEmpty + s), (oe_cnt & 1) ^ 1, abort_flag, p.status, 11)) {
            ok = false;
            break;
          }
          ++oe_cnt;
        }
        tc_fence_after();
        // B = V tile, MN-major: 64-column chunks 16 KB apart, 8-row groups
        // 1 KB apart, 16 rows (2 KB) per k-step
        const uint32_t vd = sdesc_lo(buf(g_cnt, 0), kTile * 128);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(tS + 128, tS + kk * 8, vd + kk * (2048 >> 4), kIdPV,
                 (seen > 0 || kk > 0) ? 1u : 0u);
        ++seen;
        if (seen == pu.n[s]) mma_commit(bar(L::kOFull + s));
      }
      if (more && nxt.in[s]) {
        if (issued == 0 && !wait_bar_warp(bar(L::kQFull + s), qf_cnt & 1, abort_flag, p.status, 13)) {
          ok = false;
          break;
        }
        if (issued == 0) ++qf_cnt;
        tc_fence_after();
        issue_qk(buf(g_cnt, 1));
        if (++issued == pu.n[s]) mma_commit(bar(L::kQEmpty + s));
      }
      mma_commit(bar(L::kKvEmpty + g_cnt % L::kSlots));
      ++g_cnt;
      if (!more) break;
      cur = nxt;
    }
  }
  // every MMA issued so far has finished before TMEM is released
  mma_commit(bar(L::kMmaDone));
  drain_bar(bar(L::kMmaDone), 0);
}

template <int HD>
__device__ __forceinline__ void fwd_softmax(const FwdParams& p, uint64_t* bars, uint32_t tmem,
                                            int slot, volatile int* abort_flag) {
  using L = FwdLayout<HD>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int wq = int(warp_id()) & 3;
  const int row = wq * 32 + int(lane_id());
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t tS = tmem + lane_off + uint32_t(slot * 256);
  const uint32_t tO = tS + 128;
  const float sl2 = p.scale_log2;
  uint32_t sf_cnt = 0, of_cnt = 0;
  for (int k = 0;; ++k) {
    const int u = fwd_unit(k);
    if (u >= p.n_units) break;
    const PairUnit pu = decode_pair(u, p);
    if (pu.q[slot] < 0) continue;
    Unit un;
    un.b = pu.b;
    un.h = pu.h;
    un.ob = pu.q[slot];
    un.begin = pu.beg[slot];
    un.n = pu.n[slot];
    // this row: token i of its sequence (qg.n tokens), token tok of the axis
    const TileGeo qg = tile_geo(p.list, un.ob, p.N);
    const int64_t i = int64_t(qg.lb) * kTile + row;
    const int64_t tok = qg.row0 + row;
    float m_run = -INFINITY, l_run = 0.f;
    for (int t = 0; t < un.n; ++t) {
      const InnerTile it = inner_tile(un, t, p.list, p.status);
      int lo = 0, hi = kTile - 1;
      if (it.dead) {
        hi = -1;
      } else if (it.partial) {
        row_live_range(i, qg.lb, tile_geo(p.list, it.blk, p.N).lb, qg.n, p.mask, lo, hi);
      }
      prefetch_tile_bits(p.list, it.slot, row);
      const bool ok = wait_bar(bar(L::kSFull + slot), sf_cnt & 1, abort_flag, p.status, 20);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;  // tcgen05.ld below needs the whole warp
      ++sf_cnt;
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld_x128(tS, sr);
      if (it.partial || it.dead) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < lo || c > hi) sr[c] = kNegInfBits;
        if (it.slot >= 0) {  // bit-packed mask tile: this row's bits
          uint32_t bw[4];
          load_tile_bits<4>(p.list, it.slot, row, 0, bw);
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (!((bw[c >> 5] >> (c & 31)) & 1u)) sr[c] = kNegInfBits;
        }
      }
      // The tile's row max first (four max3 chains), then one pass of
      // exponentials against the row's reference max.  The reference is
      // raised to the tile's max only when that exceeds it by more than 8
      // (log2 units) -- always on a unit's first live tile -- so P <= 2^8 and
      // O is rescaled rarely.  (An optimistic pass against the old reference
      // with the max formed alongside, redone when a row's max grew, kept two
      // copies of this loop in the kernel and measured slower.)
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float& m = (c & 2) ? mx1 : mx0;
        float& n = (c & 2) ? mx3 : mx2;
        m = max3(m, __uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]));
        n = max3(n, __uint_as_float(sr[2 * c + 2]), __uint_as_float(sr[2 * c + 3]));
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      const float m_new = (mx > m_run + 8.f) ? mx : m_run;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      float sa[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float x0, x1;
        fma2(x0, x1, __uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]), sl2, sl2, -m_use,
             -m_use);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        const int a = 2 * (c & 3);
        add2(sa[a], sa[a + 1], sa[a], sa[a + 1], p0, p1);
        pk[c] = pack_bf16x2(p0, p1);
        if (c == 31) tmem_st_x32(tS, *reinterpret_cast<uint32_t(*)[32]>(pk));
      }
      tmem_st_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      const float alpha = ex2_approx(m_run - m_use);
      const float sum0 = (sa[0] + sa[2]) + (sa[4] + sa[6]);
      const float sum1 = (sa[1] + sa[3]) + (sa[5] + sa[7]);
      l_run = l_run * alpha + (sum0 + sum1);
      if (t > 0 && __any_sync(0xFFFFFFFFu, alpha < 1.f)) {
        // the previous P V has completed: it was issued before this tile's Q K^T
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(tO + c * 32, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st_x32(tO + c * 32, o);
        }
      }
      m_run = m_new;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::kPFull + slot));
    }
    // epilogue: O / l -> bf16, LSE = ln 2 * (m + log2 l)
    if (un.n > 0) {
      const bool ok = wait_bar(bar(L::kOFull + slot), of_cnt & 1, abort_flag, p.status, 21);
      if (!__all_sync(0xFFFFFFFFu, ok)) return;
      ++of_cnt;
      tc_fence_after();
    }
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    __nv_bfloat16* orow =
        p.o + ((int64_t(un.b) * p.N + tok) * p.H + un.h) * int64_t(HD);
    // O into registers with one TMEM load, and its columns released at once:
    // the next unit's first P V may overwrite them while this row is stored
    uint32_t o[HD];
    if (un.n > 0) {
      if constexpr (HD == 128) {
        tmem_ld_x128(tO, o);
      } else {
        tmem_ld_x64(tO, o);
      }
      tc_fence_before();
      mbar_arrive(bar(L::kOEmpty + slot));
    } else {
#pragma unroll
      for (int j = 0; j < HD; ++j) o[j] = 0u;
    }
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float a0, a1;
        mul2(a0, a1, __uint_as_float(o[c * 32 + 2 * j]), __uint_as_float(o[c * 32 + 2 * j + 1]),
             inv_l, inv_l);
        w[j] = pack_bf16x2(a0, a1);
      }
      // pairs of lanes swap 16-byte chunks, so each store writes 32 contiguous
      // bytes (a whole sector) of 16 rows instead of 16 bytes of 32 rows
      uint4 cc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) cc[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      store_rows_transposed<4, 2>(cc, reinterpret_cast<char*>(orow + c * 32),
                                  int64_t(p.H) * HD * 2, i < qg.n);
    }
    if (i < qg.n) {
      p.lse[(int64_t(un.b) * p.H + un.h) * p.N + tok] =
          l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }
  }
}

template <int HD>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = FwdLayout<HD>;
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
    abort_flag[0] = 0;
    abort_flag[1] = p.wait_limit_ms;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(bars + L::kQFull + s), 1);
      mbar_init(smem_u32(bars + L::kQEmpty + s), 1);
      mbar_init(smem_u32(bars + L::kSFull + s), 1);
      mbar_init(smem_u32(bars + L::kPFull + s), 128);
      mbar_init(smem_u32(bars + L::kOFull + s), 1);
      mbar_init(smem_u32(bars + L::kOEmpty + s), 128);
    }
    const uint32_t issuers = p.slot_issuers ? 2 : 1;  // MMA warps (see fwd_mma_slot)
    mbar_init(smem_u32(bars + L::kMmaDone), issuers);
    for (int i = 0; i < L::kSlots; ++i) {
      mbar_init(smem_u32(bars + L::kKvFull + i), 1);
      mbar_init(smem_u32(bars + L::kKvEmpty + i), issuers);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // 384 threads x 168 registers at launch: the producer / MMA warpgroup
  // gives registers to the two softmax warpgroups (128 x 80 + 256 x 208).
  if (warp < 4) {
    regs_shrink<80>();
    if (warp == 0) {
      if (lane == 0) fwd_producer<HD>(p, smem, bars, abort_flag);
    } else if (p.slot_issuers) {  // one MMA-issuing warp per slot (warps 1 and 3)
      if (warp == 1 || warp == 3)
        fwd_mma_slot<HD>(p, smem, bars, tmem, warp == 1 ? 0 : 1, abort_flag);
    } else if (warp == 1) {  // the whole warp: the MMA wrappers elect one lane
      fwd_mma<HD>(p, smem, bars, tmem, abort_flag);
    }
  } else {
    regs_grow<208>();
    fwd_softmax<HD>(p, bars, tmem, (warp - 4) >> 2, abort_flag);
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
static flash_msa_status launch_fwd_hd(const FwdLaunch& a, cudaStream_t stream) {
  using L = FwdLayout<HD>;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  flash_msa_status st;
  if ((st = make_tile_map(&p.tm_q, a.q, a.B, a.N, a.H, HD)) != FLASH_MSA_OK) return st;
  if ((st = make_tile_map(&p.tm_k, a.k, a.B, a.N, a.Hkv, HD)) != FLASH_MSA_OK) return st;
  if ((st = make_tile_map(&p.tm_v, a.v, a.B, a.N, a.Hkv, HD)) != FLASH_MSA_OK) return st;
  p.o = reinterpret_cast<__nv_bfloat16*>(a.o);
  p.G = a.H / a.Hkv;
  p.lse = a.lse;
  p.B = a.B;
  p.H = a.H;
  p.N = int(a.N);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.mask = a.mask;
  p.list = a.list;
  p.n_units = a.B * a.H * ((a.list.n_blocks + 1) / 2);  // pairs of query blocks
  // lists from a block index differ between the two slots of a pair, except
  // for per-sequence tiles, whose pairs are neighbours in one sequence: those
  // (like dense / causal lists) take the single issuer that staggers the slots
  // one MMA-issuing warp per slot where the pairs' lists mostly differ (the
  // fixed interleave of a single issuer would make each slot wait on the
  // other's tiles); one warp interleaving both slots where they mostly
  // coincide, as for arithmetic lists and per-sequence tiles
  p.slot_issuers = (a.list.ptr && !a.list.t_start && a.pair_overlap < 0.5f) ? 1 : 0;
  // one group of all heads: plain rank-major order (groups of a few heads,
  // whose K and V would stay in L2, measured slower: the static deal then
  // leaves CTAs idle at the group boundaries)
  p.order = make_unit_order(a.B, a.H, (a.list.n_blocks + 1) / 2, a.B * a.H);
  p.status = a.status;
  p.wait_limit_ms = int(wait_limit_ms());
  if ((st = enable_smem(reinterpret_cast<const void*>(&fwd_kernel<HD>), L::kSmemBytes,
                        HD == 128 ? 1 : 0, "cudaFuncSetAttribute(fwd)")) != FLASH_MSA_OK)
    return st;
  int grid = p.n_units;
  const int sms = sm_count();
  if (sms > 0 && grid > sms) grid = sms;  // persistent: one CTA per SM
  fwd_kernel<HD><<<grid, kFwdThreads, L::kSmemBytes, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return set_cuda_error("fwd kernel launch");
  return FLASH_MSA_OK;
}

flash_msa_status launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
  if (a.d == 128) return launch_fwd_hd<128>(a, stream);
  return launch_fwd_hd<64>(a, stream);
}

}  // namespace fmsa
