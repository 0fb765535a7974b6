// Device-side pieces shared by the attention kernels: mask evaluation per
// tile and per row, bounded mbarrier waits with an abort path, and decoding
// of work units and their key-tile (or query-tile) lists.
#pragma once
#include <cstdint>

#include "flashmsa.h"
#include "ptx.cuh"

namespace fmsa {

constexpr int kTile = 128;                 // query / key tile edge (tokens)
constexpr uint32_t kNegInfBits = 0xFF800000u;  // fp32 -inf: a dead score
constexpr uint64_t kDrainLimitNs = 50ull * 1000ull * 1000ull;  // draining copies after an abort
constexpr int64_t kUnbounded = int64_t(1) << 40;

// Mask fields in kernel-friendly form (window clamped, absent fields neutral).
struct MaskParams {
  uint32_t flags;
  int32_t dilation, near;
  int32_t stride, phase;
  int64_t window;
  int32_t global_blocks;  // GLOBAL: the first global_blocks blocks of queries and keys
};

// ---------------------------------------------------------------------------
// Mask semantics (see flashmsa.h).  With a 128-token pattern block equal to
// the 128-token tile, the dilation, stride and (block-aligned) global parts
// are constant over a tile, and the causal / window parts depend only on
// delta = i - j.  So over one tile the live entries are exactly those whose
// delta lies in one interval [dlo, dhi] (or none at all).
// ---------------------------------------------------------------------------
struct DeltaRange {
  bool none;  // no entry of the tile can be live
  int64_t lo, hi;
};

__host__ __device__ inline DeltaRange tile_delta_range(int qb, int kb, const MaskParams& m) {
  DeltaRange r{false, -kUnbounded, kUnbounded};
  const uint32_t pat = m.flags & (FLASH_MSA_WINDOW | FLASH_MSA_DILATED | FLASH_MSA_STRIDED |
                                  FLASH_MSA_GLOBAL | FLASH_MSA_STRIDED_REL | FLASH_MSA_DILATED_FAR);
  // a tile of a global query block or global key block: every pair passes
  // the pattern, only the causal part remains
  const bool global_tile =
      (m.flags & FLASH_MSA_GLOBAL) && (qb < m.global_blocks || kb < m.global_blocks);
  bool window_applies = false;
  if (pat && !global_tile) {
    // parts that keep a whole tile (subject to causal): strided key block,
    // relative stride, dilated block distance at any range
    const int dq = qb - kb;
    const int dd = dq < 0 ? -dq : dq;
    int rel = dq % m.stride;
    if (rel < 0) rel += m.stride;
    const bool strided_ok = ((m.flags & FLASH_MSA_STRIDED) && (kb % m.stride == m.phase)) ||
                            ((m.flags & FLASH_MSA_STRIDED_REL) && rel == m.phase) ||
                            ((m.flags & FLASH_MSA_DILATED_FAR) && dd % m.dilation == 0);
    if (!strided_ok) {
      if (!(m.flags & (FLASH_MSA_WINDOW | FLASH_MSA_DILATED))) {
        r.none = true;
        return r;
      }
      if (m.flags & FLASH_MSA_DILATED) {
        if (!(dd < m.near || dd % m.dilation == 0)) {
          r.none = true;
          return r;
        }
      }
      window_applies = (m.flags & FLASH_MSA_WINDOW) != 0;
    }
  }
  if (m.flags & FLASH_MSA_CAUSAL) r.lo = 0;
  if (window_applies) {
    r.lo = r.lo > -m.window ? r.lo : -m.window;
    r.hi = m.window;
  }
  return r;
}

// Tile classification: 0 full, 1 partial, -1 dead.  Rows / columns at or past
// n are dead entries, so a tile that crosses n is never full.
__host__ __device__ inline int classify_tile(int qb, int kb, int64_t n, const MaskParams& m) {
  const DeltaRange r = tile_delta_range(qb, kb, m);
  if (r.none) return -1;
  const int64_t i0 = int64_t(qb) * kTile, j0 = int64_t(kb) * kTile;
  const int64_t i1 = (i0 + kTile < n ? i0 + kTile : n) - 1;
  const int64_t j1 = (j0 + kTile < n ? j0 + kTile : n) - 1;
  if (i1 < i0 || j1 < j0) return -1;
  const int64_t dmin = i0 - j1, dmax = i1 - j0;
  if (dmax < r.lo || dmin > r.hi) return -1;
  const bool clipped = (i1 - i0 + 1 < kTile) || (j1 - j0 + 1 < kTile);
  if (!clipped && dmin >= r.lo && dmax <= r.hi) return 0;
  return 1;
}

// Live tile-local key columns [lo, hi] of query row i in the key tile kb.
__device__ __forceinline__ void row_live_range(int64_t i, int qb, int kb, int64_t n,
                                               const MaskParams& m, int& lo, int& hi) {
  const DeltaRange r = tile_delta_range(qb, kb, m);
  const int64_t j0 = int64_t(kb) * kTile;
  if (r.none || i >= n) {
    lo = 0;
    hi = -1;
    return;
  }
  int64_t clo = i - r.hi - j0;                      // j >= i - hi
  int64_t chi = i - r.lo - j0;                      // j <= i - lo
  const int64_t last = (n - 1 - j0) < (kTile - 1) ? (n - 1 - j0) : (kTile - 1);
  if (clo < 0) clo = 0;
  if (chi > last) chi = last;
  if (chi < -1) chi = -1;
  if (clo > kTile) clo = kTile;
  lo = int(clo);
  hi = int(chi);
}

// Query-side version for the key-stationary backward: live tile-local query
// rows [lo, hi] of key column j in the query tile qb.
__device__ __forceinline__ void col_live_range(int64_t j, int qb, int kb, int64_t n,
                                               const MaskParams& m, int& lo, int& hi) {
  const DeltaRange r = tile_delta_range(qb, kb, m);
  const int64_t i0 = int64_t(qb) * kTile;
  if (r.none || j >= n) {
    lo = 0;
    hi = -1;
    return;
  }
  int64_t rlo = j + r.lo - i0;                      // i >= j + lo
  int64_t rhi = j + r.hi - i0;                      // i <= j + hi
  const int64_t last = (n - 1 - i0) < (kTile - 1) ? (n - 1 - i0) : (kTile - 1);
  if (rlo < 0) rlo = 0;
  if (rhi > last) rhi = last;
  if (rhi < -1) rhi = -1;
  if (rlo > kTile) rlo = kTile;
  lo = int(rlo);
  hi = int(rhi);
}

// ---------------------------------------------------------------------------
// Status word and bounded waits
// ---------------------------------------------------------------------------
// Status encoding: bits 0..7 = flash_msa_status code, bits 8..15 = where
// (kernel-specific wait site), bits 16..31 = block index (low 16 bits).
__device__ __forceinline__ void record_status(unsigned* status, unsigned code, unsigned where) {
  const unsigned word = code | ((where & 0xFFu) << 8) | ((blockIdx.x & 0xFFFFu) << 16);
  atomicCAS(status, 0u, word);
}

// CTA control words in shared memory: abort_flag[0] is the CTA-wide abort
// flag, abort_flag[1] the limit of any single wait in milliseconds (set from
// the launch parameters before the CTA's first barrier).
//
// Wait for the phase with the given parity; gives up (returns false) when the
// CTA-wide abort flag is raised or after the wait limit, raising the flag and
// recording FLASH_MSA_ERR_TIMEOUT.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned* status, unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  const uint64_t limit_ns = uint64_t(unsigned(abort_flag[1])) * 1000000ull;
  while (true) {
#pragma unroll 1
    for (int k = 0; k < 16; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag[0]) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      record_status(status, FLASH_MSA_ERR_TIMEOUT, where);
      return false;
    }
  }
}

// wait_bar for all 32 lanes of a warp (the MMA-issuing warps): every lane
// gets the same answer and the warp is converged afterwards, as the
// warp-elected MMA and commit wrappers require.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, unsigned* status,
                                              unsigned where) {
  return __all_sync(0xFFFFFFFFu, wait_bar(bar, parity, abort_flag, status, where));
}

// Used only on the abort path: wait for copies already in flight, ignoring
// the abort flag, with a short limit.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
// Dynamic work distribution for persistent CTAs (one per SM).  The TMA
// producer thread claims unit indices from the launch's global counter and
// hands them, in claim order, to the CTA's other roles through two
// shared-memory slots, each guarded by a "full" mbarrier (one arrival: the
// producer) and an "empty" mbarrier (one arrival per consumer).  Index -1
// means that no unit is left; it is published exactly once.  Both calls
// return -2 when a wait was abandoned (abort).
//
// The counter is one 64-bit word of a small pool shared by all launches on
// the device.  Before the kernel runs, the host sets both of its 32-bit
// halves to the launch's ticket (a positive number below 2^31, different
// for every launch); a claim adds 1, so the low half minus the ticket is the
// unit index and the high half must still equal the ticket.  A launch that
// finds another ticket there shares the counter with an overlapping launch:
// it records FLASH_MSA_ERR_SCHEDULE and claims nothing more, so aliasing
// counters are reported instead of silently losing work units.
// ---------------------------------------------------------------------------
struct UnitQueue {
  uint32_t full, empty;  // mbarriers of slot 0; slot 1's follow 8 bytes later
  volatile int* slot;    // two shared-memory slots
  uint32_t seq;          // number of pushes / pops done by this thread
};

__device__ __forceinline__ int claim_unit(unsigned long long* counter, unsigned ticket,
                                          int n_units, unsigned* status) {
  const unsigned long long old = atomicAdd(counter, 1ull);
  if (unsigned(old >> 32) != ticket) {
    record_status(status, FLASH_MSA_ERR_SCHEDULE, 0xF4);
    return -1;
  }
  const unsigned u = unsigned(old) - ticket;
  return u < unsigned(n_units) ? int(u) : -1;
}

__device__ __forceinline__ int queue_push(UnitQueue& q, unsigned long long* counter,
                                          unsigned ticket, int n_units,
                                          volatile int* abort_flag, unsigned* status) {
  const uint32_t s = q.seq & 1;
  if (!wait_bar(q.empty + 8 * s, ((q.seq >> 1) & 1) ^ 1, abort_flag, status, 30)) return -2;
  const int u = claim_unit(counter, ticket, n_units, status);
  q.slot[s] = u;
  mbar_arrive(q.full + 8 * s);  // release: the slot write is visible to the waiters
  ++q.seq;
  return u;
}

// kWarp: called by all 32 lanes of a warp, which then arrive once.
template <bool kWarp>
__device__ __forceinline__ int queue_pop(UnitQueue& q, volatile int* abort_flag,
                                         unsigned* status) {
  const uint32_t s = q.seq & 1;
  const bool ok = wait_bar(q.full + 8 * s, (q.seq >> 1) & 1, abort_flag, status, 31);
  if (kWarp ? !__all_sync(0xFFFFFFFFu, ok) : !ok) return -2;
  const int u = q.slot[s];
  if (kWarp) __syncwarp();
  if (!kWarp || (threadIdx.x & 31) == 0) mbar_arrive(q.empty + 8 * s);
  ++q.seq;
  return u;
}

// ---------------------------------------------------------------------------
// Work units and tile lists
// ---------------------------------------------------------------------------
// A list of blocks for one outer block (key tiles of a query block in the
// forward / dQ pass, query tiles of a key block in the dK/dV pass).  With an
// index it is a CSR (or CSC) row; without one it is derived arithmetically
// for dense or causal masks.
struct ListParams {
  const int32_t* ptr;    // row_ptr / col_ptr (null: arithmetic mode)
  const int32_t* idx;    // col_idx / row_idx
  const uint8_t* kind;   // kind / kind_t
  const int32_t* order;  // q_order / k_order
  const int32_t* slot;   // bit-packed masks: bit_slot / bit_slot_t (null otherwise)
  const uint32_t* bits;  // bits / bits_t: 512 words per slot
  int64_t n_bit_tiles;
  int64_t nnz;
  int n_blocks;          // blocks along both axes (square tiling)
  int causal;            // arithmetic mode: causal mask
  int tail;              // N % 128 != 0
  int transposed;        // 0: outer = query block (CSR); 1: outer = key block (CSC)
  // per-sequence tiles (null otherwise): first token of each tile, first
  // token and length of its sequence
  const int32_t* t_start;
  const int32_t* t_seq0;
  const int32_t* t_len;
};

// Where a tile lies: row0 = its first token on the (packed) sequence axis,
// lb = its block index inside its own sequence and n = that sequence's
// length.  Without per-sequence tiles, tile blk of a length-N sequence is the
// 128-token block blk.  Masks are evaluated in the sequence's own coordinates
// (token lb * 128 + r of a sequence of n tokens), outputs go to token row0 + r.
struct TileGeo {
  int64_t row0;
  int lb;
  int64_t n;
};

__device__ __forceinline__ TileGeo tile_geo(const ListParams& L, int blk, int64_t N) {
  if (!L.t_start) return TileGeo{int64_t(blk) * kTile, blk, N};
  const int start = __ldg(L.t_start + blk), s0 = __ldg(L.t_seq0 + blk);
  return TileGeo{start, (start - s0) / kTile, __ldg(L.t_len + blk)};
}

struct Unit {
  int b, h, ob;  // batch, head, outer block
  int begin, n;  // position in idx[] and number of inner tiles
  int n0;        // length of the block list (n = n0 * query heads per unit)
};

// Launch order of the work units: unit u -> (bh = b * H + h, rank), rank =
// position in one head's longest-first block order, in groups of G heads: the
// units of heads [G g, G g + G) come before those of the next group,
// rank-major inside the group (rank 0 of every head of the group, then rank
// 1, ...; the last group may be smaller).  G = BH is plain rank-major order:
// the whole launch runs longest lists first and its last units are short.
// In (b, h)-major order the last heads' longest units started at the very
// end and left most SMs idle (measured: 15% of the forward's span at
// N = 4096); chunks of 4 to 16 ranks per head, which keep more of a head's
// units running together for L2 reuse, recovered less than half of the gain.
// With a small G the CTAs running at any time work on a few heads only, whose
// streamed tiles and accumulators then stay in L2 (the accumulated-dQ
// backward uses that).
//
// Two decoders of that numbering follow.  The forward's divides without
// integer division: a division by a value fixed at launch is a multiply-high
// and a shift (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication"; valid for dividends below 2^31).  The hardware division
// sequence goes through the conversion and reciprocal unit that the softmax
// warps keep busy with exponentials; decoding each unit that way cost the
// forward 3-5%.  The backward's (unit_order_grouped with G, below) keeps the
// hardware division: with the multiply-shift decoder its kernels measured
// 1-2% slower at N = 16384 (1% faster at N = 4096).
struct FastDiv {
  uint32_t mul, shift;
};
// (mul, shift) for d >= 1: shift = ceil(log2 d), mul = floor(2^32 (2^shift - d) / d) + 1
inline FastDiv make_fast_div(uint32_t d) {
  FastDiv f{0u, 0u};
  while ((uint64_t(1) << f.shift) < d) ++f.shift;
  if (d > 1) f.mul = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << f.shift) - d)) / d + 1);
  return f;
}
__device__ __forceinline__ int div_fast(int n, FastDiv f) {
  return int((__umulhi(uint32_t(n), f.mul) + uint32_t(n)) >> f.shift);
}

// The unit numbering of a launch over BH = B H heads of n_blocks ranks each.
struct UnitOrder {
  int group, last, n_full, H;  // heads per group, heads in the last group, whole groups
  FastDiv per_group, by_group, by_last, by_H;
};
inline UnitOrder make_unit_order(int B, int H, int n_blocks, int group) {
  UnitOrder o;
  const int BH = B * H;
  group = group > 0 ? group : 1;
  o.group = group;
  o.n_full = BH / group;
  o.last = BH - o.n_full * group;
  o.H = H;
  o.per_group = make_fast_div(uint32_t(group) * uint32_t(n_blocks));
  o.by_group = make_fast_div(uint32_t(group));
  o.by_last = make_fast_div(uint32_t(o.last > 0 ? o.last : 1));
  o.by_H = make_fast_div(uint32_t(H));
  return o;
}
__device__ __forceinline__ void unit_order_grouped(int u, int n_blocks, const UnitOrder& o,
                                                   int& b, int& h, int& rank) {
  const int per_group = o.group * n_blocks;
  const int gi = div_fast(u, o.per_group);
  int bh;
  if (gi < o.n_full) {
    const int rem = u - gi * per_group;
    rank = div_fast(rem, o.by_group);
    bh = gi * o.group + (rem - rank * o.group);
  } else {
    const int rem = u - o.n_full * per_group;
    rank = div_fast(rem, o.by_last);
    bh = o.n_full * o.group + (rem - rank * o.last);
  }
  b = div_fast(bh, o.by_H);
  h = bh - b * o.H;
}

// Block and list of rank `rank` of one head's order (un.ob, un.begin, un.n,
// un.n0; un.b and un.h are the caller's).
__device__ __forceinline__ void decode_block_at(Unit& un, int rank, const ListParams& L,
                                                unsigned* status) {
  if (L.order) {
    int ob = __ldg(L.order + rank);
    if (ob < 0 || ob >= L.n_blocks) {
      record_status(status, FLASH_MSA_ERR_INDEX, 0xF0);
      ob = rank;
    }
    un.ob = ob;
  } else {
    // arithmetic order, longest list first: causal query blocks descend, key blocks ascend
    un.ob = (L.causal && !L.transposed) ? (L.n_blocks - 1 - rank) : rank;
  }
  if (L.ptr) {
    const int a = __ldg(L.ptr + un.ob), e = __ldg(L.ptr + un.ob + 1);
    if (a < 0 || e < a || int64_t(e) > L.nnz) {
      record_status(status, FLASH_MSA_ERR_INDEX, 0xF1);
      un.begin = 0;
      un.n = 0;
    } else {
      un.begin = a;
      un.n = e - a;
    }
  } else if (L.causal) {
    un.begin = 0;
    un.n = L.transposed ? (L.n_blocks - un.ob) : (un.ob + 1);
  } else {
    un.begin = 0;
    un.n = L.n_blocks;
  }
  un.n0 = un.n;
}

// Unit u of a launch over BH heads in groups of G (the backward's decoder).
__device__ __forceinline__ void unit_order_grouped(int u, int BH, int n_blocks, int G, int& bh,
                                                   int& rank) {
  const int per_group = G * n_blocks;
  const int full = BH / G;
  const int gi = u / per_group;
  if (gi < full) {
    const int rem = u - gi * per_group;
    rank = rem / G;
    bh = gi * G + (rem - rank * G);
  } else {
    const int gl = BH - full * G;
    const int rem = u - full * per_group;
    rank = rem / gl;
    bh = full * G + (rem - rank * gl);
  }
}

// Unit at (bh, rank) of a launch over heads of H (b = bh / H).
__device__ __forceinline__ Unit decode_unit_at(int bh, int rank, int H, const ListParams& L,
                                               unsigned* status) {
  Unit un;
  un.b = bh / H;
  un.h = bh - un.b * H;
  decode_block_at(un, rank, L, status);
  return un;
}

// Inner block t of a unit: block id, whether the element mask must be
// evaluated (partial), and whether the entry was unusable (dead: every entry
// masked; reported as FLASH_MSA_ERR_INDEX, block id replaced by 0).
struct InnerTile {
  int blk;
  bool partial;
  bool dead;
  int slot;  // bit tile of a bit-packed mask, -1 if none
};

__device__ __forceinline__ InnerTile inner_tile(const Unit& un, int t, const ListParams& L,
                                                unsigned* status) {
  InnerTile it;
  it.dead = false;
  it.slot = -1;
  if (L.ptr) {
    it.blk = __ldg(L.idx + un.begin + t);
    it.partial = __ldg(L.kind + un.begin + t) != 0;
    if (it.blk < 0 || it.blk >= L.n_blocks) {
      record_status(status, FLASH_MSA_ERR_INDEX, 0xF2);
      it.blk = 0;
      it.dead = true;
    }
    if (L.slot && it.partial) {
      it.slot = __ldg(L.slot + un.begin + t);
      if (it.slot >= L.n_bit_tiles) {  // corrupt: treat the tile as dead
        record_status(status, FLASH_MSA_ERR_INDEX, 0xF3);
        it.slot = -1;
        it.dead = true;
      }
    }
  } else {
    it.blk = L.transposed ? (L.causal ? un.ob + t : t) : t;
    const int last = L.n_blocks - 1;
    it.partial = (L.causal && it.blk == un.ob) ||
                 (L.tail && (it.blk == last || un.ob == last));
  }
  return it;
}

// Coalesced store of one piece of kC 16-byte chunks per row.  Lane l of the
// warp holds chunks c[0..kC) of its own row's piece, to be written at `dst`;
// the rows of consecutive lanes are `stride` bytes apart.  Written as is,
// every store instruction would touch 32 rows.  Instead the chunks are taken
// in groups of kG (kG divides kC), and for each group the kG lanes of each
// lane group exchange chunks in log2(kG) butterfly steps (a kG x kG
// transpose: afterwards lane i of the lane group holds chunk i of the group
// for every row of the lane group), so that every store instruction writes
// kG * 16 contiguous bytes of each of 32 / kG rows.  row_ok: whether this
// lane's row exists.
template <int kC, int kG>
__device__ __forceinline__ void transpose_chunks(uint4 (&c)[kC]) {
  static_assert(kC % kG == 0 && (kG & (kG - 1)) == 0, "kG: a power of two dividing kC");
  const int i = int(threadIdx.x & 31) & (kG - 1);
#pragma unroll
  for (int q = 0; q < kC; q += kG) {
#pragma unroll
    for (int m = kG / 2; m >= 1; m >>= 1) {
      const bool upper = (i & m) != 0;
#pragma unroll
      for (int j = 0; j < kG; ++j) {
        if (j & m) continue;
        // the lower lane of the pair gives chunk j | m and takes the partner's chunk j
        const uint4 send = upper ? c[q + j] : c[q + (j | m)];
        uint4 recv;
        recv.x = __shfl_xor_sync(0xFFFFFFFFu, send.x, m);
        recv.y = __shfl_xor_sync(0xFFFFFFFFu, send.y, m);
        recv.z = __shfl_xor_sync(0xFFFFFFFFu, send.z, m);
        recv.w = __shfl_xor_sync(0xFFFFFFFFu, send.w, m);
        if (upper) c[q + j] = recv;
        else c[q + (j | m)] = recv;
      }
    }
  }
}

template <int kC, int kG = kC>
__device__ __forceinline__ void store_rows_transposed(uint4 (&c)[kC], char* dst, int64_t stride,
                                                      bool row_ok) {
  transpose_chunks<kC, kG>(c);
  const int lane = int(threadIdx.x & 31);
  const int i = lane & (kG - 1);
  const uint32_t ok = __ballot_sync(0xFFFFFFFFu, row_ok);
  const int base = lane - i;
#pragma unroll
  for (int q = 0; q < kC; q += kG)
#pragma unroll
    for (int k = 0; k < kG; ++k)
      if ((ok >> (base + k)) & 1u)
        *reinterpret_cast<uint4*>(dst + int64_t(k - i) * stride + (q + i) * 16) = c[q + k];
}

// Bits of one row of a bit tile (bit-packed masks): kWords 32-bit words
// starting at word w0 of tile-local row r.  prefetch_tile_bits pulls the row
// into L1 before the tile's barrier wait without holding registers across
// it; load_tile_bits reads it after the wait, only for tiles with bits.
__device__ __forceinline__ const uint32_t* tile_bits_row(const ListParams& L, int slot, int r,
                                                         int w0) {
  return L.bits + int64_t(slot) * 512 + r * 4 + w0;
}
__device__ __forceinline__ void prefetch_tile_bits(const ListParams& L, int slot, int r) {
  if (slot >= 0) asm volatile("prefetch.global.L1 [%0];" ::"l"(tile_bits_row(L, slot, r, 0)));
}
template <int kWords>
__device__ __forceinline__ void load_tile_bits(const ListParams& L, int slot, int r, int w0,
                                               uint32_t (&w)[kWords]) {
  const uint32_t* src = tile_bits_row(L, slot, r, w0);
  if constexpr (kWords == 4) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
    w[0] = v.x; w[1] = v.y;
  }
}

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace fmsa
