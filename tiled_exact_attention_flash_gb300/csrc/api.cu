// C-ABI entry points of libflashmsa (declared in include/flashmsa.h):
// argument validation, the host-side block-index builder and checker, TMA
// descriptor creation, kernel launch and the device status word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <vector>

#include "internal.h"

namespace fmsa {

static thread_local char g_last_error[512] = "";

flash_msa_status set_error(flash_msa_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

flash_msa_status set_cuda_error(const char* what) {
  const cudaError_t e = cudaGetLastError();
  return set_error(FLASH_MSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

flash_msa_status make_tile_map(CUtensorMap* m, const void* base, int B, int64_t N, int H, int d) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return set_error(FLASH_MSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(N), cuuint64_t(H), cuuint64_t(B)};
  const cuuint64_t strides[3] = {cuuint64_t(H) * d * 2, cuuint64_t(d) * 2,
                                 cuuint64_t(N) * H * d * 2};
  const cuuint32_t box[4] = {64, 128, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(FLASH_MSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", int(r));
  return FLASH_MSA_OK;
}

flash_msa_status make_acc_map(CUtensorMap* m, float* base, int B, int H, int64_t NP, int d) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return set_error(FLASH_MSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(NP), cuuint64_t(H), cuuint64_t(B)};
  const cuuint64_t strides[3] = {cuuint64_t(d) * 4, cuuint64_t(NP) * d * 4,
                                 cuuint64_t(H) * NP * d * 4};
  const cuuint32_t box[4] = {32, 128, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(FLASH_MSA_ERR_CUDA, "cuTensorMapEncodeTiled(acc) failed (CUresult %d)", int(r));
  return FLASH_MSA_OK;
}

// ---------------------------------------------------------------------------
// validation helpers
// ---------------------------------------------------------------------------
static constexpr int64_t kMaxN = (int64_t(1) << 31) - 256;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int64_t n_blocks_of(int64_t N) { return (N + kTile - 1) / kTile; }

// Converts the mask into kernel form; `need_index` is set for pattern masks.
static flash_msa_status check_mask(const flash_msa_mask_desc* m, MaskParams& mp,
                                   bool& need_index) {
  memset(&mp, 0, sizeof(mp));
  mp.window = kUnbounded;
  mp.dilation = 1;
  mp.stride = 1;
  need_index = false;
  if (!m) return FLASH_MSA_OK;
  if (m->flags & ~uint32_t(FLASH_MSA_CAUSAL | FLASH_MSA_WINDOW | FLASH_MSA_DILATED |
                           FLASH_MSA_STRIDED | FLASH_MSA_GLOBAL | FLASH_MSA_STRIDED_REL |
                           FLASH_MSA_DILATED_FAR | FLASH_MSA_BITMASK | FLASH_MSA_DOCUMENTS))
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "mask: unknown flag bits 0x%x", m->flags);
  // every flag but CAUSAL needs an index (the bits travel in it)
  const uint32_t pat = m->flags & ~uint32_t(FLASH_MSA_CAUSAL);
  if (m->block != kTile && !(m->block == 0 && pat == 0))
    return set_error(FLASH_MSA_ERR_UNSUPPORTED, "mask: pattern block %d (only 128 is supported)",
                     m->block);
  mp.flags = m->flags;
  if (m->flags & FLASH_MSA_WINDOW) {
    if (m->window < 0) return set_error(FLASH_MSA_ERR_INVALID_ARG, "mask: window < 0");
    mp.window = m->window < kUnbounded ? m->window : kUnbounded;
  }
  if (m->flags & (FLASH_MSA_DILATED | FLASH_MSA_DILATED_FAR)) {
    if (m->dilation < 1 || m->dilation_near < 0)
      return set_error(FLASH_MSA_ERR_INVALID_ARG, "mask: dilation must be >= 1, near >= 0");
    mp.dilation = m->dilation;
    mp.near = m->dilation_near;
  }
  if (m->flags & (FLASH_MSA_STRIDED | FLASH_MSA_STRIDED_REL)) {
    if (m->stride < 1 || m->stride_phase < 0 || m->stride_phase >= m->stride)
      return set_error(FLASH_MSA_ERR_INVALID_ARG, "mask: stride must be >= 1, 0 <= phase < stride");
    mp.stride = m->stride;
    mp.phase = m->stride_phase;
  }
  if (m->flags & FLASH_MSA_GLOBAL) {
    if (m->global_tokens < 1)
      return set_error(FLASH_MSA_ERR_INVALID_ARG, "mask: global_tokens must be >= 1");
    if (m->global_tokens % kTile != 0)
      return set_error(FLASH_MSA_ERR_UNSUPPORTED,
                       "mask: global_tokens %lld is not a multiple of the 128-token block",
                       static_cast<long long>(m->global_tokens));
    const int64_t gb = m->global_tokens / kTile;
    mp.global_blocks = gb < (int64_t(1) << 30) ? int32_t(gb) : int32_t(1) << 30;
  }
  need_index = pat != 0;
  return FLASH_MSA_OK;
}

static flash_msa_status check_dims(int B, int H, int64_t N, int d) {
  if (B < 1 || H < 1) return set_error(FLASH_MSA_ERR_INVALID_ARG, "B and H must be >= 1");
  if (N < 1 || N > kMaxN)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "N must be in [1, 2^31 - 256], got %lld",
                     static_cast<long long>(N));
  if (d != 64 && d != 128)
    return set_error(FLASH_MSA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  const int64_t units = int64_t(B) * H * n_blocks_of(N);
  if (units > int64_t(1) << 30)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "B * H * ceil(N/128) too large");
  return FLASH_MSA_OK;
}

// Lists for the kernels: from a device index, or arithmetic for dense / causal.
static flash_msa_status make_lists(const flash_msa_mask_desc* m, int64_t N, bool need_index,
                                   bool want_csc, ListParams& rows, ListParams& cols) {
  memset(&rows, 0, sizeof(rows));
  memset(&cols, 0, sizeof(cols));
  const int nb = int(n_blocks_of(N));
  rows.n_blocks = cols.n_blocks = nb;
  rows.causal = cols.causal = (m && (m->flags & FLASH_MSA_CAUSAL)) ? 1 : 0;
  rows.tail = cols.tail = (N % kTile) != 0;
  cols.transposed = 1;
  const flash_msa_block_index* ix = m ? m->index : nullptr;
  if (!ix) {
    if (need_index)
      return set_error(FLASH_MSA_ERR_INDEX, "mask has window/dilation/stride flags but no index");
    return FLASH_MSA_OK;
  }
  const int nt = ix->sequence_tiles ? ix->n_q_blocks : nb;  // tiles along each axis
  if (ix->seq_len != N || ix->block != kTile || ix->n_q_blocks != nt || ix->n_k_blocks != nt ||
      ix->nnz < 0 || nt < 1)
    return set_error(FLASH_MSA_ERR_INDEX,
                     "index built for N=%lld block=%d blocks=%dx%d, call has N=%lld",
                     static_cast<long long>(ix->seq_len), ix->block, ix->n_q_blocks,
                     ix->n_k_blocks, static_cast<long long>(N));
  if (ix->sequence_tiles) {
    if (!ix->tile_start || !ix->tile_seq0 || !ix->tile_seq_len)
      return set_error(FLASH_MSA_ERR_INDEX, "index: per-sequence tile arrays missing");
    rows.n_blocks = cols.n_blocks = nt;
    rows.t_start = cols.t_start = ix->tile_start;
    rows.t_seq0 = cols.t_seq0 = ix->tile_seq0;
    rows.t_len = cols.t_len = ix->tile_seq_len;
  }
  if (!ix->row_ptr || !ix->col_idx || !ix->kind || !ix->q_order)
    return set_error(FLASH_MSA_ERR_INDEX, "index: CSR arrays or q_order missing");
  const bool bits = (m->flags & (FLASH_MSA_BITMASK | FLASH_MSA_DOCUMENTS)) && ix->n_bit_tiles > 0;
  if (bits && (!ix->bit_slot || !ix->bits || (want_csc && (!ix->bit_slot_t || !ix->bits_t))))
    return set_error(FLASH_MSA_ERR_INDEX, "index: bit arrays missing");
  rows.ptr = ix->row_ptr;
  rows.idx = ix->col_idx;
  rows.kind = ix->kind;
  rows.order = ix->q_order;
  rows.nnz = ix->nnz;
  if (bits) {
    rows.slot = ix->bit_slot;
    rows.bits = ix->bits;
    rows.n_bit_tiles = ix->n_bit_tiles;
  }
  if (want_csc) {
    if (!ix->col_ptr || !ix->row_idx || !ix->kind_t || !ix->k_order)
      return set_error(FLASH_MSA_ERR_INDEX, "index: CSC arrays or k_order missing");
    cols.ptr = ix->col_ptr;
    cols.idx = ix->row_idx;
    cols.kind = ix->kind_t;
    cols.order = ix->k_order;
    cols.nnz = ix->nnz;
    if (bits) {
      cols.slot = ix->bit_slot_t;
      cols.bits = ix->bits_t;
      cols.n_bit_tiles = ix->n_bit_tiles;
    }
  }
  return FLASH_MSA_OK;
}

static float resolve_scale(float scale, int d) {
  if (!(scale > 0.f) || std::isinf(scale)) return 1.0f / std::sqrt(float(d));
  return scale;
}

}  // namespace fmsa

using namespace fmsa;

extern "C" {

const char* flash_msa_last_error_string(void) { return g_last_error; }

const char* flash_msa_version(void) { return "libflashmsa 0.1 (sm_103a, tcgen05)"; }

// CSC (by counting sort: query blocks come out ascending within each
// column) and the longest-first key-block order, from a filled CSR.
static void finish_lists(flash_msa_block_index* out, int64_t nb,
                         const std::vector<int32_t>& col_count, bool with_bits) {
  out->col_ptr[0] = 0;
  for (int64_t kb = 0; kb < nb; ++kb) out->col_ptr[kb + 1] = out->col_ptr[kb] + col_count[size_t(kb)];
  std::vector<int32_t> fill(out->col_ptr, out->col_ptr + nb);
  for (int64_t qb = 0; qb < nb; ++qb)
    for (int32_t e = out->row_ptr[qb]; e < out->row_ptr[qb + 1]; ++e) {
      const int32_t kb = out->col_idx[e];
      const int32_t dst = fill[size_t(kb)]++;
      out->row_idx[dst] = int32_t(qb);
      out->kind_t[dst] = out->kind[e];
      if (with_bits) out->bit_slot_t[dst] = out->bit_slot[e];
    }
  // k_order: longest first (stable); q_order is filled by the caller
  for (int64_t b = 0; b < nb; ++b) out->k_order[b] = int32_t(b);
  std::stable_sort(out->k_order, out->k_order + nb, [&](int32_t a, int32_t b) {
    return out->col_ptr[a + 1] - out->col_ptr[a] > out->col_ptr[b + 1] - out->col_ptr[b];
  });
}

// Key tiles listed by both query blocks a and b (CSR rows ascend).
static int64_t common_tiles(const flash_msa_block_index* ix, int32_t a, int32_t b) {
  int32_t i = ix->row_ptr[a], j = ix->row_ptr[b];
  const int32_t ie = ix->row_ptr[a + 1], je = ix->row_ptr[b + 1];
  int64_t n = 0;
  while (i < ie && j < je) {
    if (ix->col_idx[i] == ix->col_idx[j]) {
      ++n;
      ++i;
      ++j;
    } else if (ix->col_idx[i] < ix->col_idx[j]) {
      ++i;
    } else {
      ++j;
    }
  }
  return n;
}

// q_order of a packed-axis index: the query blocks in pairs (positions 2r
// and 2r + 1, which the forward runs together, loading their key tiles once)
// chosen to share key tiles.  Blocks are visited longest first (descending
// live-tile count, ties by ascending index); an unpaired block takes, among
// the unpaired blocks 1, 2, 4 or 8 away (tried in the order +1, -1, +2, -2,
// +4, -4, +8, -8), the one with the most key tiles in common with it (the
// first one tried on ties), provided they have any in common.  The blocks
// left over are paired in visiting order.  Pairs are ordered by the live-tile
// count of their first block (descending, ties by its ascending index); a
// last unpaired block, if any, comes at the end.  For causal masks this is
// plain longest-first order; for block dilation it pairs blocks of the same
// parity, for packed documents neighbours of one document.
static void shared_pairs_order(flash_msa_block_index* out, int64_t nb) {
  static const int kOffsets[8] = {1, -1, 2, -2, 4, -4, 8, -8};
  auto len = [&](int32_t b) { return out->row_ptr[b + 1] - out->row_ptr[b]; };
  std::vector<int32_t> visit(static_cast<size_t>(nb));
  for (int64_t b = 0; b < nb; ++b) visit[size_t(b)] = int32_t(b);
  std::stable_sort(visit.begin(), visit.end(),
                   [&](int32_t a, int32_t b) { return len(a) > len(b); });
  std::vector<char> paired(static_cast<size_t>(nb), 0);
  std::vector<std::pair<int32_t, int32_t>> pairs;
  for (const int32_t a : visit) {
    if (paired[size_t(a)]) continue;
    int32_t best = -1;
    int64_t best_common = 0;
    for (const int off : kOffsets) {
      const int64_t c = int64_t(a) + off;
      if (c < 0 || c >= nb || paired[size_t(c)]) continue;
      const int64_t common = common_tiles(out, a, int32_t(c));
      if (common > best_common) {
        best_common = common;
        best = int32_t(c);
      }
    }
    if (best >= 0) {
      paired[size_t(a)] = paired[size_t(best)] = 1;
      pairs.emplace_back(a, best);
    }
  }
  std::vector<int32_t> rest;
  for (const int32_t a : visit)
    if (!paired[size_t(a)]) rest.push_back(a);
  for (size_t i = 0; i + 1 < rest.size(); i += 2) pairs.emplace_back(rest[i], rest[i + 1]);
  std::stable_sort(pairs.begin(), pairs.end(), [&](const std::pair<int32_t, int32_t>& x,
                                                   const std::pair<int32_t, int32_t>& y) {
    const int32_t lx = len(x.first), ly = len(y.first);
    return lx != ly ? lx > ly : x.first < y.first;
  });
  int64_t at = 0;
  for (const auto& pr : pairs) {
    out->q_order[at++] = pr.first;
    out->q_order[at++] = pr.second;
  }
  if (rest.size() % 2) out->q_order[at++] = rest.back();
}

// flash_msa_block_index::pair_overlap from the filled CSR lists (ascending
// within a row) and the final q_order.
static float pair_overlap(const flash_msa_block_index* ix, int64_t nb) {
  int64_t common = 0, either = 0;
  for (int64_t r = 0; r + 1 < nb; r += 2) {
    const int32_t a = ix->q_order[r], b = ix->q_order[r + 1];
    either += (ix->row_ptr[a + 1] - ix->row_ptr[a]) + (ix->row_ptr[b + 1] - ix->row_ptr[b]);
    common += common_tiles(ix, a, b);
  }
  either -= common;
  return either > 0 ? float(double(common) / double(either)) : 0.f;
}

// Live (i, j) pairs of a live tile (qb, kb) of class k (0 full) of one
// sequence of n tokens: all valid entries of a full tile, one interval of
// columns per row of a partial one (the kernels' row_live_range).
static int64_t tile_live_count(int qb, int kb, int k, int64_t n, const MaskParams& mp) {
  const int64_t i0 = int64_t(qb) * kTile, j0 = int64_t(kb) * kTile;
  const int64_t rows = std::min<int64_t>(kTile, n - i0), cols = std::min<int64_t>(kTile, n - j0);
  if (k == 0) return rows * cols;
  const DeltaRange r = tile_delta_range(qb, kb, mp);
  if (r.none) return 0;
  int64_t live = 0;
  for (int64_t row = 0; row < rows; ++row) {
    const int64_t i = i0 + row;
    const int64_t clo = std::max<int64_t>(i - r.hi - j0, 0);
    const int64_t chi = std::min<int64_t>({i - r.lo - j0, n - 1 - j0, int64_t(kTile - 1)});
    if (chi >= clo) live += chi - clo + 1;
  }
  return live;
}

// Per-sequence tiles of packed sequences (flash_msa_block_index,
// sequence_tiles): every sequence is tiled from its own first token and its
// tile pairs are classified with the in-sequence mask parts (causal, window)
// and the sequence's own length; tiles are numbered sequence by sequence.
// Both build phases (counts only when out->row_ptr is null).
static flash_msa_status build_sequence_tiles(const flash_msa_mask_desc* mask,
                                             const MaskParams& mask_params, int64_t N,
                                             flash_msa_block_index* out) {
  MaskParams mp = mask_params;
  mp.flags &= FLASH_MSA_CAUSAL | FLASH_MSA_WINDOW;
  const int64_t* ds = mask->doc_starts;
  const bool window = (mp.flags & FLASH_MSA_WINDOW) != 0;
  const int64_t span = window ? mp.window / kTile + 2 : int64_t(1) << 40;
  // key tiles of query tile m in a sequence of nb tiles that may be live
  auto key_range = [&](int64_t m, int64_t nb, int64_t& k0, int64_t& k1) {
    k0 = std::max<int64_t>(0, m - span);
    k1 = std::min<int64_t>(nb - 1, m + span);
    if (mp.flags & FLASH_MSA_CAUSAL) k1 = std::min(k1, m);
  };
  int64_t nt = 0, nnz = 0, live = 0;
  for (int64_t d = 0; d < mask->n_docs; ++d) {
    const int64_t len = ds[d + 1] - ds[d], nb = (len + kTile - 1) / kTile;
    nt += nb;
    for (int64_t m = 0; m < nb; ++m) {
      int64_t k0, k1;
      key_range(m, nb, k0, k1);
      for (int64_t k = k0; k <= k1; ++k) {
        const int c = classify_tile(int(m), int(k), len, mp);
        if (c < 0) continue;
        ++nnz;
        live += tile_live_count(int(m), int(k), c, len, mp);
      }
    }
  }
  if (nt > INT32_MAX || nnz > INT32_MAX)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: more than 2^31 tiles");
  out->seq_len = N;
  out->block = kTile;
  out->n_q_blocks = out->n_k_blocks = int32_t(nt);
  out->n_bit_tiles = 0;
  out->live_elements = live;
  out->sequence_tiles = 1;
  if (!out->row_ptr) {
    out->nnz = nnz;
    return FLASH_MSA_OK;
  }
  if (out->nnz != nnz)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: nnz %lld, the mask has %lld",
                     static_cast<long long>(out->nnz), static_cast<long long>(nnz));
  if (!out->col_idx || !out->kind || !out->col_ptr || !out->row_idx || !out->kind_t ||
      !out->q_order || !out->k_order || !out->tile_start || !out->tile_seq0 || !out->tile_seq_len)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: some output arrays are null");
  std::vector<int32_t> col_count(size_t(nt), 0);
  int64_t pos = 0, base = 0;
  out->row_ptr[0] = 0;
  for (int64_t d = 0; d < mask->n_docs; ++d) {
    const int64_t len = ds[d + 1] - ds[d], nb = (len + kTile - 1) / kTile;
    for (int64_t m = 0; m < nb; ++m) {
      out->tile_start[base + m] = int32_t(ds[d] + m * kTile);
      out->tile_seq0[base + m] = int32_t(ds[d]);
      out->tile_seq_len[base + m] = int32_t(len);
      int64_t k0, k1;
      key_range(m, nb, k0, k1);
      for (int64_t k = k0; k <= k1; ++k) {
        const int c = classify_tile(int(m), int(k), len, mp);
        if (c < 0) continue;
        out->col_idx[pos] = int32_t(base + k);
        out->kind[pos] = uint8_t(c);
        ++col_count[size_t(base + k)];
        ++pos;
      }
      out->row_ptr[base + m + 1] = int32_t(pos);
    }
    base += nb;
  }
  finish_lists(out, nt, col_count, false);
  // q_order: each sequence's tiles in neighbouring pairs counted from its last
  // tile, so that the forward's pair units (positions 2r, 2r + 1) hold two
  // tiles of one sequence with nearly the same key tiles; pairs by descending
  // live-tile count of their first tile (ties: ascending id), then the single
  // first tiles of sequences with an odd tile count, likewise
  auto count = [&](int32_t t) { return out->row_ptr[t + 1] - out->row_ptr[t]; };
  auto longer = [&](int32_t a, int32_t b) {
    return count(a) != count(b) ? count(a) > count(b) : a < b;
  };
  std::vector<int32_t> firsts, singles;
  base = 0;
  for (int64_t d = 0; d < mask->n_docs; ++d) {
    const int64_t nb = (ds[d + 1] - ds[d] + kTile - 1) / kTile;
    for (int64_t t = base + nb - 1; t > base; t -= 2) firsts.push_back(int32_t(t));
    if (nb % 2) singles.push_back(int32_t(base));
    base += nb;
  }
  std::sort(firsts.begin(), firsts.end(), longer);
  std::sort(singles.begin(), singles.end(), longer);
  int64_t at = 0;
  for (int32_t t : firsts) {
    out->q_order[at++] = t;
    out->q_order[at++] = t - 1;
  }
  for (int32_t t : singles) out->q_order[at++] = t;
  out->pair_overlap = pair_overlap(out, nt);
  return FLASH_MSA_OK;
}

flash_msa_status flash_msa_build_block_index(const flash_msa_mask_desc* mask, int64_t N,
                                             flash_msa_block_index* out) {
  g_last_error[0] = 0;
  if (!mask || !out) return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: null argument");
  if (N < 1 || N > kMaxN) return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: bad N");
  if (mask->block != kTile)
    return set_error(FLASH_MSA_ERR_UNSUPPORTED, "build_block_index: block must be 128");
  MaskParams mp;
  bool need = false;
  flash_msa_status st = check_mask(mask, mp, need);
  if (st != FLASH_MSA_OK) return st;
  out->pair_overlap = 0.f;  // set at the end of the filling call
  const bool with_bitmask = (mask->flags & FLASH_MSA_BITMASK) != 0;
  const bool with_docs = (mask->flags & FLASH_MSA_DOCUMENTS) != 0;
  const bool with_bits = with_bitmask || with_docs;
  if (with_bitmask && !mask->bitmask)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: BITMASK without mask->bitmask");
  // packed documents: the sequence range [doc_lo, doc_hi) of every token
  std::vector<int64_t> doc_lo, doc_hi;
  if (with_docs) {
    const int64_t* ds = mask->doc_starts;
    if (!ds || mask->n_docs < 1 || ds[0] != 0 || ds[mask->n_docs] != N)
      return set_error(FLASH_MSA_ERR_INVALID_ARG,
                       "build_block_index: DOCUMENTS needs offsets from 0 to N=%lld",
                       static_cast<long long>(N));
    doc_lo.resize(size_t(N));
    doc_hi.resize(size_t(N));
    for (int64_t d = 0; d < mask->n_docs; ++d) {
      if (ds[d + 1] <= ds[d])
        return set_error(FLASH_MSA_ERR_INVALID_ARG,
                         "build_block_index: document offsets must rise strictly (at %lld)",
                         static_cast<long long>(d));
      for (int64_t t = ds[d]; t < ds[d + 1]; ++t) {
        doc_lo[size_t(t)] = ds[d];
        doc_hi[size_t(t)] = ds[d + 1];
      }
    }
  }
  // packed sequences with in-sequence (delta-only) parts: one tiling per sequence
  const uint32_t in_sequence = FLASH_MSA_CAUSAL | FLASH_MSA_WINDOW | FLASH_MSA_DOCUMENTS;
  if (with_docs && !with_bitmask && (mask->flags & ~in_sequence) == 0)
    return build_sequence_tiles(mask, mp, N, out);
  out->sequence_tiles = 0;
  const int64_t nb = n_blocks_of(N);
  const int64_t words_per_row = (N + 31) / 32;
  // Tile class with the bits: live entries of row r = interval of the other
  // mask parts AND the row's 128 mask bits.  Returns -1 dead, 0 full,
  // 1 partial; `cut` tells whether the bits removed an entry of the interval
  // (the tile then carries its live entries, written to tb when non-null).
  auto bit_class = [&](int qb, int kb, int c, bool& cut, uint32_t* tb, int64_t* live_out) -> int {
    cut = false;
    if (!with_bits) return c;
    const DeltaRange r = tile_delta_range(qb, kb, mp);
    const int64_t j0 = int64_t(kb) * kTile;
    int64_t live = 0;
    for (int row = 0; row < kTile; ++row) {
      const int64_t i = int64_t(qb) * kTile + row;
      uint32_t iv[4] = {0, 0, 0, 0};
      if (i < N && !r.none) {
        int64_t clo = std::max<int64_t>(i - r.hi - j0, 0);
        int64_t chi = std::min<int64_t>({i - r.lo - j0, N - 1 - j0, int64_t(kTile - 1)});
        for (int64_t col = clo; col <= chi; ++col) iv[col >> 5] |= 1u << (col & 31);
      }
      uint32_t dbits[4] = {~0u, ~0u, ~0u, ~0u};  // keys of row i's own document
      if (with_docs) {
        for (int w = 0; w < 4; ++w) dbits[w] = 0;
        if (i < N) {
          const int64_t a = std::max(doc_lo[size_t(i)] - j0, int64_t(0));
          const int64_t e = std::min(doc_hi[size_t(i)] - j0, int64_t(kTile));
          for (int64_t col = a; col < e; ++col) dbits[col >> 5] |= 1u << (col & 31);
        }
      }
      for (int w = 0; w < 4; ++w) {
        const int64_t word = int64_t(kb) * 4 + w;
        uint32_t mbits = dbits[w];
        if (with_bitmask)
          mbits &= (i < N && word < words_per_row) ? mask->bitmask[i * words_per_row + word] : 0u;
        const uint32_t f = iv[w] & mbits;
        if (f != iv[w]) cut = true;
        live += __builtin_popcount(f);
        if (tb) tb[row * 4 + w] = f;
      }
    }
    if (live_out) *live_out = live;
    if (live == 0) return -1;
    if (c == 0 && !cut) return 0;
    return 1;
  };
  // live (i, j) pairs of a live tile of class k: every valid entry of a full
  // tile, one interval of columns per row of a partial tile (the kernels'
  // row_live_range), the set bits when the mask has bits
  auto tile_live = [&](int qb, int kb, int k, int64_t bits_live) -> int64_t {
    if (with_bits) return bits_live;
    const int64_t i0 = int64_t(qb) * kTile, j0 = int64_t(kb) * kTile;
    const int64_t rows = std::min<int64_t>(kTile, N - i0), cols = std::min<int64_t>(kTile, N - j0);
    if (k == 0) return rows * cols;
    const DeltaRange r = tile_delta_range(qb, kb, mp);
    if (r.none) return 0;
    int64_t live = 0;
    for (int64_t row = 0; row < rows; ++row) {
      const int64_t i = i0 + row;
      const int64_t clo = std::max<int64_t>(i - r.hi - j0, 0);
      const int64_t chi = std::min<int64_t>({i - r.lo - j0, N - 1 - j0, int64_t(kTile - 1)});
      if (chi >= clo) live += chi - clo + 1;
    }
    return live;
  };
  // candidate key blocks per query block: causal and a plain window bound the
  // span; with global tokens the global key blocks come first, and a global
  // query block scans every key block
  const bool window_bound =
      (mp.flags & FLASH_MSA_WINDOW) &&
      !(mp.flags & (FLASH_MSA_STRIDED | FLASH_MSA_STRIDED_REL | FLASH_MSA_DILATED_FAR));
  const int64_t span = window_bound ? mp.window / kTile + 2 : nb;
  const int64_t gb = (mp.flags & FLASH_MSA_GLOBAL) ? std::min<int64_t>(mp.global_blocks, nb) : 0;
  auto for_each_tile = [&](auto&& fn) {
    for (int64_t qb = 0; qb < nb; ++qb) {
      const bool scan_all = !window_bound || qb < gb;
      int64_t k0 = scan_all ? 0 : std::max<int64_t>(0, qb - span);
      int64_t k1 = scan_all ? nb - 1 : std::min<int64_t>(nb - 1, qb + span);
      if (mp.flags & FLASH_MSA_CAUSAL) k1 = std::min(k1, qb);
      const int64_t g_end = std::min(gb, k0);  // global key blocks before the window span
      auto visit = [&](int64_t kb) {
        const int c = classify_tile(int(qb), int(kb), N, mp);
        if (c >= 0) fn(int(qb), int(kb), c);  // the bits are applied by fn
      };
      for (int64_t kb = 0; kb < g_end; ++kb) visit(kb);  // ascending: they precede k0
      for (int64_t kb = k0; kb <= k1; ++kb) visit(kb);
    }
  };
  out->seq_len = N;
  out->block = kTile;
  out->n_q_blocks = out->n_k_blocks = int32_t(nb);
  if (!out->row_ptr) {
    int64_t nnz = 0, n_bits = 0, live = 0;
    for_each_tile([&](int qb, int kb, int c) {
      bool cut;
      int64_t bl = 0;
      const int k = bit_class(qb, kb, c, cut, nullptr, &bl);
      if (k < 0) return;
      ++nnz;
      live += tile_live(qb, kb, k, bl);
      if (k == 1 && cut) ++n_bits;
    });
    out->live_elements = live;
    if (nnz > INT32_MAX)
      return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: more than 2^31 live tiles");
    out->nnz = nnz;
    out->n_bit_tiles = n_bits;
    return FLASH_MSA_OK;
  }
  if (!out->col_idx || !out->kind || !out->col_ptr || !out->row_idx || !out->kind_t ||
      !out->q_order || !out->k_order)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: some output arrays are null");
  if (with_bits && (!out->bit_slot || !out->bit_slot_t ||
                    (out->n_bit_tiles > 0 && (!out->bits || !out->bits_t))))
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "build_block_index: bit arrays are null");
  // CSR
  std::vector<int32_t> col_count(size_t(nb), 0);
  std::vector<uint32_t> tb(size_t(kTile) * 4);
  int64_t pos = 0, slot = 0, live = 0;
  int64_t cur = 0;
  out->row_ptr[0] = 0;
  for_each_tile([&](int qb, int kb, int c) {
    bool cut;
    int64_t bl = 0;
    const int k = bit_class(qb, kb, c, cut, tb.data(), &bl);
    if (k < 0) return;
    live += tile_live(qb, kb, k, bl);
    while (cur < qb) out->row_ptr[++cur] = int32_t(pos);
    if (pos < out->nnz) {
      out->col_idx[pos] = kb;
      out->kind[pos] = uint8_t(k);
      if (with_bits) {
        int32_t s = -1;
        if (k == 1 && cut && slot < out->n_bit_tiles) {
          s = int32_t(slot);
          uint32_t* dst = out->bits + slot * 512;
          uint32_t* dst_t = out->bits_t + slot * 512;
          std::copy(tb.begin(), tb.end(), dst);
          std::fill(dst_t, dst_t + 512, 0u);
          for (int row = 0; row < kTile; ++row)
            for (int col = 0; col < kTile; ++col)
              if ((tb[size_t(row) * 4 + (col >> 5)] >> (col & 31)) & 1u)
                dst_t[col * 4 + (row >> 5)] |= 1u << (row & 31);
        }
        if (k == 1 && cut) ++slot;
        out->bit_slot[pos] = s;
      }
    }
    ++pos;
    ++col_count[size_t(kb)];
  });
  while (cur < nb) out->row_ptr[++cur] = int32_t(pos);
  if (pos != out->nnz || (with_bits && slot != out->n_bit_tiles))
    return set_error(FLASH_MSA_ERR_INVALID_ARG,
                     "build_block_index: nnz %lld / bit tiles %lld do not match the counting pass "
                     "(%lld / %lld)",
                     static_cast<long long>(out->nnz), static_cast<long long>(out->n_bit_tiles),
                     static_cast<long long>(pos), static_cast<long long>(slot));
  if (!with_bits) out->n_bit_tiles = 0;
  out->live_elements = live;
  finish_lists(out, nb, col_count, with_bits);
  shared_pairs_order(out, nb);
  out->pair_overlap = pair_overlap(out, nb);
  return FLASH_MSA_OK;
}

// Per-sequence tiles cover [0, N) sequence by sequence, 128 tokens apart
// inside each sequence.
static bool tile_geometry_ok(const flash_msa_block_index* ix, int64_t N) {
  if (!ix->tile_start || !ix->tile_seq0 || !ix->tile_seq_len) return false;
  int64_t expect = 0;  // first token of the next tile
  for (int64_t t = 0; t < ix->n_q_blocks; ++t) {
    const int64_t st = ix->tile_start[t], s0 = ix->tile_seq0[t], len = ix->tile_seq_len[t];
    if (len < 1 || s0 < 0 || s0 + len > N || st != expect || (st - s0) % kTile != 0 || st < s0 ||
        st >= s0 + len)
      return false;
    expect = st + kTile < s0 + len ? st + kTile : s0 + len;
  }
  return expect == N;
}

flash_msa_status flash_msa_check_block_index(const flash_msa_block_index* ix, int64_t N) {
  g_last_error[0] = 0;
  if (!ix) return set_error(FLASH_MSA_ERR_INVALID_ARG, "check_block_index: null index");
  const int64_t nb = ix->sequence_tiles ? int64_t(ix->n_q_blocks) : n_blocks_of(N);
  if (ix->seq_len != N || ix->block != kTile || ix->n_q_blocks != nb || ix->n_k_blocks != nb ||
      nb < 1)
    return set_error(FLASH_MSA_ERR_INDEX, "index: header does not match N=%lld",
                     static_cast<long long>(N));
  if (ix->sequence_tiles && !tile_geometry_ok(ix, N))
    return set_error(FLASH_MSA_ERR_INDEX, "index: per-sequence tile geometry is inconsistent");
  if (!ix->row_ptr || !ix->col_idx || !ix->kind || !ix->col_ptr || !ix->row_idx || !ix->kind_t ||
      !ix->q_order || !ix->k_order)
    return set_error(FLASH_MSA_ERR_INDEX, "index: missing array");
  auto check_lists = [&](const int32_t* ptr, const int32_t* idx, const uint8_t* kind,
                         const char* what) -> bool {
    if (ptr[0] != 0 || ptr[nb] != ix->nnz) return false;
    for (int64_t b = 0; b < nb; ++b) {
      if (ptr[b + 1] < ptr[b]) return false;
      for (int32_t e = ptr[b]; e < ptr[b + 1]; ++e) {
        if (idx[e] < 0 || idx[e] >= nb || kind[e] > 1) return false;
        if (e > ptr[b] && idx[e] <= idx[e - 1]) return false;
      }
    }
    (void)what;
    return true;
  };
  if (!check_lists(ix->row_ptr, ix->col_idx, ix->kind, "CSR"))
    return set_error(FLASH_MSA_ERR_INDEX, "index: CSR arrays are inconsistent");
  if (ix->sequence_tiles)
    for (int64_t qb = 0; qb < nb; ++qb)
      for (int32_t e = ix->row_ptr[qb]; e < ix->row_ptr[qb + 1]; ++e)
        if (ix->tile_seq0[ix->col_idx[e]] != ix->tile_seq0[qb])
          return set_error(FLASH_MSA_ERR_INDEX, "index: a tile pair spans two sequences");
  if (ix->n_bit_tiles < 0)
    return set_error(FLASH_MSA_ERR_INDEX, "index: negative bit tile count");
  if (ix->n_bit_tiles > 0) {
    if (!ix->bit_slot || !ix->bit_slot_t || !ix->bits || !ix->bits_t)
      return set_error(FLASH_MSA_ERR_INDEX, "index: bit arrays missing");
    for (int64_t e = 0; e < ix->nnz; ++e)
      if (ix->bit_slot[e] < -1 || ix->bit_slot[e] >= ix->n_bit_tiles ||
          (ix->bit_slot[e] >= 0 && ix->kind[e] != 1))
        return set_error(FLASH_MSA_ERR_INDEX, "index: bad bit slot at entry %lld",
                         static_cast<long long>(e));
  }
  if (!check_lists(ix->col_ptr, ix->row_idx, ix->kind_t, "CSC"))
    return set_error(FLASH_MSA_ERR_INDEX, "index: CSC arrays are inconsistent");
  // CSC must be the transpose of CSR
  std::vector<int32_t> fill(ix->col_ptr, ix->col_ptr + nb);
  for (int64_t qb = 0; qb < nb; ++qb)
    for (int32_t e = ix->row_ptr[qb]; e < ix->row_ptr[qb + 1]; ++e) {
      const int32_t kb = ix->col_idx[e];
      const int32_t at = fill[size_t(kb)]++;
      if (at >= ix->col_ptr[kb + 1] || ix->row_idx[at] != qb || ix->kind_t[at] != ix->kind[e])
        return set_error(FLASH_MSA_ERR_INDEX, "index: CSC is not the transpose of CSR");
      if (ix->n_bit_tiles > 0 && ix->bit_slot[e] != ix->bit_slot_t[at])
        return set_error(FLASH_MSA_ERR_INDEX, "index: CSC bit slots differ from CSR");
    }
  for (const int32_t* ord : {ix->q_order, ix->k_order}) {
    std::vector<char> seen(size_t(nb), 0);
    for (int64_t b = 0; b < nb; ++b) {
      if (ord[b] < 0 || ord[b] >= nb || seen[size_t(ord[b])])
        return set_error(FLASH_MSA_ERR_INDEX, "index: order array is not a permutation");
      seen[size_t(ord[b])] = 1;
    }
  }
  return FLASH_MSA_OK;
}

static flash_msa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int Hkv, int64_t N, int d, float scale,
                                 const flash_msa_mask_desc* mask, void* stream) {
  g_last_error[0] = 0;
  flash_msa_status st = check_dims(B, H, N, d);
  if (st != FLASH_MSA_OK) return st;
  if (Hkv < 1 || H % Hkv != 0)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "key/value heads %d must divide query heads %d",
                     Hkv, H);
  if (!q || !k || !v || !o || !lse)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "fwd: null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "fwd: tensors must be 16-byte aligned");
  FwdLaunch a;
  memset(&a, 0, sizeof(a));
  bool need = false;
  if ((st = check_mask(mask, a.mask, need)) != FLASH_MSA_OK) return st;
  ListParams unused;
  if ((st = make_lists(mask, N, need, false, a.list, unused)) != FLASH_MSA_OK) return st;
  a.pair_overlap = (mask && mask->index) ? mask->index->pair_overlap : 0.f;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.d = d;
  a.N = N;
  a.scale = resolve_scale(scale, d);
  a.status = status_word_ptr();
  if (!a.status) return set_cuda_error("status word");
  return launch_fwd(a, static_cast<cudaStream_t>(stream));
}

flash_msa_status flash_msa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int64_t N, int d, float scale,
                               const flash_msa_mask_desc* mask, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, H, N, d, scale, mask, stream);
}

flash_msa_status flash_msa_fwd_gqa(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int Hkv, int64_t N, int d,
                                   float scale, const flash_msa_mask_desc* mask, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Hkv, N, d, scale, mask, stream);
}

// Workspace: two fp32 vectors per (b, h) padded to whole 128-row tiles
// (-LSE * log2(e) and D), then, for the fused backward, the fp32 dQ
// accumulator (B, H, padded N, d).
static size_t vectors_bytes(int B, int H, int64_t N) {
  return 2 * size_t(B) * size_t(H) * size_t(n_blocks_of(N)) * kTile * sizeof(float);
}
static size_t accumulator_bytes(int B, int H, int64_t N, int d) {
  return size_t(B) * size_t(H) * size_t(n_blocks_of(N)) * kTile * size_t(d) * sizeof(float);
}
static size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
static constexpr unsigned kAllStages = FLASH_MSA_BWD_PREPROCESS | FLASH_MSA_BWD_DKDV |
                                       FLASH_MSA_BWD_DQ | FLASH_MSA_BWD_FUSED |
                                       FLASH_MSA_BWD_DQ_CONVERT;
static constexpr unsigned kDefaultStages = FLASH_MSA_BWD_DETERMINISTIC;
static constexpr unsigned kAccumulatorStages = FLASH_MSA_BWD_FUSED | FLASH_MSA_BWD_DQ_CONVERT;

static bool valid_stages(unsigned stages) {
  if (stages == 0 || (stages & ~kAllStages)) return false;
  return !((stages & FLASH_MSA_BWD_FUSED) && (stages & (FLASH_MSA_BWD_DKDV | FLASH_MSA_BWD_DQ)));
}

size_t flash_msa_bwd_stages_workspace_bytes(int B, int H, int64_t N, int d, unsigned stages) {
  if (!valid_stages(stages)) return 0;
  if (B < 1 || H < 1 || N < 1 || N > kMaxN || (d != 64 && d != 128)) return 0;
  size_t bytes = vectors_bytes(B, H, N);
  if (stages & kAccumulatorStages) bytes += accumulator_bytes(B, H, N, d);
  return round256(bytes);
}

size_t flash_msa_bwd_workspace_bytes(int B, int H, int64_t N, int d) {
  return flash_msa_bwd_stages_workspace_bytes(B, H, N, d, kDefaultStages);
}

flash_msa_status flash_msa_bwd(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dO, void* dq, void* dk, void* dv,
                               int B, int H, int64_t N, int d, float scale,
                               const flash_msa_mask_desc* mask, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return flash_msa_bwd_stages(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, mask,
                              workspace, workspace_bytes, kDefaultStages, stream);
}

static flash_msa_status bwd_impl(const void* q, const void* k, const void* v, const void* o,
                                 const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                 int B, int H, int Hkv, int64_t N, int d, float scale,
                                 const flash_msa_mask_desc* mask, void* workspace,
                                 size_t workspace_bytes, unsigned stages, void* stream) {
  g_last_error[0] = 0;
  if (!valid_stages(stages))
    return set_error(FLASH_MSA_ERR_INVALID_ARG,
                     "bwd: stages 0x%x: a non-empty subset of 1|2|4|8|16 without 8 together "
                     "with 2 or 4", stages);
  flash_msa_status st = check_dims(B, H, N, d);
  if (st != FLASH_MSA_OK) return st;
  if (Hkv < 1 || H % Hkv != 0)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "key/value heads %d must divide query heads %d",
                     Hkv, H);
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "bwd: null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "bwd: tensors must be 16-byte aligned");
  BwdLaunch a;
  memset(&a, 0, sizeof(a));
  bool need = false;
  if ((st = check_mask(mask, a.mask, need)) != FLASH_MSA_OK) return st;
  if ((st = make_lists(mask, N, need, true, a.rows, a.cols)) != FLASH_MSA_OK) return st;
  // the vectors hold 128 rows per tile: per-sequence tiles may outnumber
  // ceil(N / 128)
  const int64_t n_rows = int64_t(a.rows.n_blocks) * kTile;
  const bool seq_tiles = a.rows.t_start != nullptr;
  if (seq_tiles && (stages & kAccumulatorStages))
    return set_error(FLASH_MSA_ERR_UNSUPPORTED,
                     "bwd: the accumulated-dQ stages do not take per-sequence tiles");
  const size_t need_ws = flash_msa_bwd_stages_workspace_bytes(B, H, n_rows, d, stages);
  if (need_ws == 0)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "bwd: %lld tile rows are too many",
                     static_cast<long long>(n_rows));
  if (!workspace || workspace_bytes < need_ws || !aligned16(workspace))
    return set_error(FLASH_MSA_ERR_WORKSPACE, "bwd: workspace of %zu bytes required (got %zu)",
                     need_ws, workspace_bytes);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dO;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dsum = static_cast<float*>(workspace);
  // the accumulator follows the two vectors; it is used (and PREPROCESS
  // zeroes it) by the accumulated-dQ stages, and by PREPROCESS run on its own
  // when the workspace holds it (a stage-by-stage accumulated backward)
  const bool acc_call = (stages & kAccumulatorStages) ||
                        (stages == FLASH_MSA_BWD_PREPROCESS && !seq_tiles &&
                         workspace_bytes >= flash_msa_bwd_stages_workspace_bytes(
                                                B, H, N, d, FLASH_MSA_BWD_ACCUMULATED));
  a.dqacc = acc_call
                ? reinterpret_cast<float*>(static_cast<char*>(workspace) + vectors_bytes(B, H, N))
                : nullptr;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.d = d;
  a.N = N;
  a.scale = resolve_scale(scale, d);
  a.status = status_word_ptr();
  a.stages = stages;
  if (!a.status) return set_cuda_error("status word");
  return launch_bwd(a, static_cast<cudaStream_t>(stream));
}

flash_msa_status flash_msa_bwd_stages(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dO, void* dq, void* dk,
                                      void* dv, int B, int H, int64_t N, int d, float scale,
                                      const flash_msa_mask_desc* mask, void* workspace,
                                      size_t workspace_bytes, unsigned stages, void* stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, H, N, d, scale, mask, workspace,
                  workspace_bytes, stages, stream);
}

flash_msa_status flash_msa_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                                   const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                   int B, int H, int Hkv, int64_t N, int d, float scale,
                                   const flash_msa_mask_desc* mask, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, d, scale, mask, workspace,
                  workspace_bytes, kDefaultStages, stream);
}

flash_msa_status flash_msa_bwd_gqa_stages(const void* q, const void* k, const void* v,
                                          const void* o, const float* lse, const void* dO,
                                          void* dq, void* dk, void* dv, int B, int H, int Hkv,
                                          int64_t N, int d, float scale,
                                          const flash_msa_mask_desc* mask, void* workspace,
                                          size_t workspace_bytes, unsigned stages, void* stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, d, scale, mask, workspace,
                  workspace_bytes, stages, stream);
}

flash_msa_status flash_msa_set_wait_limit_ms(unsigned ms) {
  g_last_error[0] = 0;
  if (ms < 1 || ms > 600000)
    return set_error(FLASH_MSA_ERR_INVALID_ARG, "wait limit %u ms outside [1, 600000]", ms);
  set_wait_limit_ms(ms);
  return FLASH_MSA_OK;
}

unsigned flash_msa_get_wait_limit_ms(void) { return wait_limit_ms(); }

flash_msa_status flash_msa_selftest_wait_timeout(void* stream) {
  g_last_error[0] = 0;
  return launch_wait_timeout_probe(static_cast<cudaStream_t>(stream));
}

flash_msa_status flash_msa_get_status(void* stream) {
  g_last_error[0] = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return set_cuda_error("get_status: stream synchronize");
  unsigned* ptr = status_word_ptr();
  if (!ptr) return set_cuda_error("get_status: status word");
  unsigned word = 0;
  if (cudaMemcpy(&word, ptr, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return set_cuda_error("get_status: read");
  if (word == 0) return FLASH_MSA_OK;
  const unsigned zero = 0;
  if (cudaMemcpy(ptr, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return set_cuda_error("get_status: clear");
  const unsigned code = word & 0xFFu;
  return set_error(static_cast<flash_msa_status>(code),
                   "device status %u (site %u, block %u)", code, (word >> 8) & 0xFFu, word >> 16);
}

}  // extern "C"
