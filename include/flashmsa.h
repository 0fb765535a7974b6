/*
 * libflashmsa -- exact tiled ("Flash MSA") scaled-dot-product attention on
 * GB300 (sm_103a), forward and recompute backward, dense / causal /
 * block-sparse masks.
 *
 * Operation (page "Flash MSA Attention Kernel Implementation: A Practical
 * Guide for Production AI", section "Why Standard Attention Broke"; page "How
 * to Use Flash MSA Kernels for Long Context", section "What Flash MSA
 * Actually Does"):
 *
 *     O = softmax(mask(Q K^T * scale)) V,   scale = d^-1/2 unless given,
 *
 * computed tile by tile with an online softmax (running row max and sum, the
 * partial output rescaled per key tile; same page 1, section "The Flash Core:
 * Tiling Over the Memory Hierarchy"), never materialising the N x N matrix.
 * Masked scores are -inf and take no part in the max or the sum (page 1,
 * section "Optimization Tricks That Actually Matter", paragraph "Masking and
 * causal attention").  The forward stores O and the per-row natural-log
 * logsumexp LSE; the backward recomputes the scores from Q, K, V, O, LSE
 * (page 1, section "The Backward Pass: The Real Beast").  Sparse masks are
 * applied inside the tiling loop through a precomputed per-query-block list
 * of live key blocks (page "How Does Flash-MSA Sparse Attention Work",
 * section "How Flash-MSA Sparse Attention Works"), so dead tiles are never
 * loaded.
 *
 * Conventions shared by every entry point:
 *   - q, k, v, o, dO, dq, dk, dv: DEVICE pointers to bf16, contiguous
 *     (B, N, H, d) (token stride H*d elements), 16-byte aligned, owned by the
 *     caller.  lse: DEVICE fp32 (B, H, N).
 *   - d must be 64 or 128 (else FLASH_MSA_ERR_UNSUPPORTED); 1 <= N < 2^31 - 256;
 *     B, H >= 1.
 *   - scale <= 0 or NaN selects the default d^-1/2.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream.  The return value covers argument
 *     validation and launch errors only; a kernel that gives up waiting (see
 *     FLASH_MSA_ERR_TIMEOUT and flash_msa_set_wait_limit_ms()), meets a corrupt
 *     index or loses its work counter records that in a device status word
 *     read by flash_msa_get_status().
 *   - No entry point aborts, throws, or falls back to a CPU implementation.
 *     On error the last message is available from flash_msa_last_error_string().
 */
#ifndef FLASHMSA_H
#define FLASHMSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLASH_MSA_OK = 0,
  FLASH_MSA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, bad mask field */
  FLASH_MSA_ERR_UNSUPPORTED = 2, /* head dimension not 64/128, block != 128, G not whole blocks */
  FLASH_MSA_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
  FLASH_MSA_ERR_TIMEOUT = 4,     /* device: a bounded wait inside a kernel ran out */
  FLASH_MSA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required */
  FLASH_MSA_ERR_INDEX = 6,       /* block index missing, built for another N, or corrupt */
  FLASH_MSA_ERR_SCHEDULE = 7     /* device: a persistent kernel found its work counter taken by
                                    an overlapping launch (more than 256 backward launches in
                                    flight on one device); that call's results are invalid */
} flash_msa_status;

/* Mask flags.  Element predicate for query i, key j of a length-N sequence:
 *   live(i,j) = (i < N) && (j < N) && (!CAUSAL || j <= i) && pattern(i,j)
 *   pattern   = true                          if no pattern flag (all but CAUSAL)
 *             = near || strided || strided_rel || far || global   otherwise
 *   near      = (WINDOW or DILATED set) && (!WINDOW || |i-j| <= window)
 *               && (!DILATED || D < dilation_near || D % dilation == 0),
 *               D = | floor(i/block) - floor(j/block) |
 *   strided   = STRIDED && floor(j/block) % stride == stride_phase
 *   strided_rel = STRIDED_REL && (floor(i/block) - floor(j/block)) mod stride
 *                 == stride_phase   (mod >= 0)
 *   far       = DILATED_FAR && D % dilation == 0
 *   global    = GLOBAL && (i < global_tokens || j < global_tokens)
 * and with BITMASK, live(i,j) is further AND-ed with bit(i,j) of the bit-packed
 * mask given to flash_msa_build_block_index (the mask tiles "in a bit-packed
 * format" of page "Flash MSA Attention Kernel Implementation", section
 * "Optimization Tricks That Actually Matter", "Masking and causal
 * attention"); with DOCUMENTS, with doc(i) == doc(j): variable-length
 * sequences packed back to back on the token axis (offsets doc_starts), each
 * attending only to itself (same page, section "The Production Pipeline:
 * From Kernel to Service", request batching), causal inside each sequence
 * when CAUSAL is set.
 * Window: "Local window -- attend only to +-W tokens"; dilated: "skip every
 * few tokens", read at block level; strided: the fixed pattern of Child et
 * al. (page "How Does Flash-MSA Sparse Attention Work", section "How
 * Flash-MSA Sparse Attention Works", list of masks).  Global: the local
 * window plus a few global tokens in the style of Longformer (same page,
 * section "How Do Sparse Attention Kernels Work in GPU Clusters?"), the
 * first global_tokens tokens attending and attended in both directions.
 * STRIDED_REL and DILATED_FAR are the second readings of the strided and
 * dilated masks: Child et al.'s strides counted from the query block, and
 * a dense window with dilated key blocks kept at every distance. */
enum {
  FLASH_MSA_CAUSAL = 1,
  FLASH_MSA_WINDOW = 2,
  FLASH_MSA_DILATED = 4,
  FLASH_MSA_STRIDED = 8,
  FLASH_MSA_GLOBAL = 16,
  FLASH_MSA_STRIDED_REL = 32,
  FLASH_MSA_DILATED_FAR = 64,
  FLASH_MSA_BITMASK = 128,
  FLASH_MSA_DOCUMENTS = 256
};

/* Per-query-block list of live key blocks ("a precomputed index list", page
 * "How Does Flash-MSA Sparse Attention Work", section "How Flash-MSA Sparse
 * Attention Works").  Tiles are block x block = 128 x 128.  A tile is dead
 * (no live entry; not listed), full (every entry live; kind 0) or partial
 * (kind 1: the kernel evaluates the element predicate).  Rows/columns past N
 * count as dead entries, so tail tiles are never full.
 *   CSR by query block: row_ptr[n_q_blocks+1], col_idx[nnz] (ascending), kind[nnz]
 *   CSC by key block:   col_ptr[n_k_blocks+1], row_idx[nnz] (ascending), kind_t[nnz]
 *   k_order[n_k_blocks]: key blocks by descending live-tile count, ties by
 *   ascending index (longest work is scheduled first).
 *   q_order[n_q_blocks]: query blocks in pairs (the forward runs positions
 *   2r and 2r + 1 together and loads their key tiles once) that share key
 *   tiles: blocks are visited by descending live-tile count (ties: ascending
 *   index); an unpaired block takes, among the unpaired blocks 1, 2, 4 or 8
 *   away (tried as +1, -1, +2, -2, +4, -4, +8, -8), the one with the most key
 *   tiles in common (the first tried on ties), if any is in common; blocks
 *   left over are paired in visiting order; pairs come by descending count
 *   of their first block (ties: ascending index), an odd block out last.
 *   With per-sequence tiles (below) q_order instead holds each sequence's
 *   tiles in neighbouring pairs counted from its last tile, pairs by
 *   descending count of their first tile (ties: ascending id), then the
 *   single first tiles of sequences with an odd tile count.
 * With a BITMASK or DOCUMENTS mask, a partial tile whose live entries are not all given
 * by the other mask parts carries them as bits, in a slot numbered in CSR
 * order: bits[512 slot + 4 r + c / 32] bit c % 32 = live(128 qb + r,
 * 128 kb + c), and bits_t the transpose (4 words per key row over the
 * queries); bit_slot[e] / bit_slot_t[e] give the slot of CSR / CSC entry e or
 * -1.  n_bit_tiles = 0 (and null bit arrays) for every other mask.
 * The struct itself always lives in HOST memory.  Its array pointers are host
 * pointers when filled by flash_msa_build_block_index() and DEVICE pointers
 * when passed to flash_msa_fwd()/flash_msa_bwd() (copy the arrays over and
 * point a second struct at the copies).  The caller owns every array. */
typedef struct flash_msa_block_index {
  int64_t seq_len; /* N the index was built for */
  int32_t n_q_blocks, n_k_blocks, block;
  int64_t nnz;
  int32_t* row_ptr;
  int32_t* col_idx;
  uint8_t* kind;
  int32_t* col_ptr;
  int32_t* row_idx;
  uint8_t* kind_t;
  int32_t* q_order;
  int32_t* k_order;
  int64_t n_bit_tiles;
  int32_t* bit_slot;   /* [nnz] */
  int32_t* bit_slot_t; /* [nnz] */
  uint32_t* bits;      /* [512 n_bit_tiles] */
  uint32_t* bits_t;    /* [512 n_bit_tiles] */
  int64_t live_elements; /* live (i, j) pairs of the mask over N x N; set by both build calls */
  /* Per-sequence tiles (set by both build calls: 1 or 0).  A DOCUMENTS mask
   * without BITMASK whose other flags are only CAUSAL and WINDOW is tiled per
   * sequence: sequence [s0, s1) gets its own tiles starting at s0, s0 + 128,
   * ..., so no tile holds tokens of two sequences and tile pairs of two
   * sequences do not exist.  Tiles are numbered sequence by sequence;
   * n_q_blocks = n_k_blocks = the number of tiles, and the lists above index
   * tiles.  tile_start[t] is the first token of tile t, tile_seq0[t] and
   * tile_seq_len[t] the first token and length of its sequence ([n_q_blocks]
   * int32 each; NULL when sequence_tiles is 0).  Entries of a tile past its
   * sequence's end are dead.  (Other DOCUMENTS masks are tiled on the packed
   * axis, with bit tiles.) */
  int32_t sequence_tiles;
  int32_t* tile_start;
  int32_t* tile_seq0;
  int32_t* tile_seq_len;
  /* Of the key tiles listed by the two query blocks at q_order positions 2r
   * and 2r + 1 (the blocks the forward runs together), the fraction that
   * both of them list: sum over the pairs of |common tiles| / sum of |tiles
   * of either| (0 with fewer than two blocks).  Set by the filling build
   * call (0 after the counting call).  A scheduling hint only: the forward
   * issues the pair's products from one warp, interleaved, when it is at
   * least 1/2, else from one warp per block; 0 (a struct filled by other
   * means) keeps the latter. */
  float pair_overlap;
} flash_msa_block_index;

/* Mask description (host memory).  A NULL mask, or flags == 0, is dense
 * attention.  flags == CAUSAL may pass index = NULL (tiles are derived
 * arithmetically); any other flag requires an index built for the same N
 * and mask, else FLASH_MSA_ERR_INDEX.  block must be 128.
 * window >= 0 (tokens, inclusive); dilation >= 1 (DILATED, DILATED_FAR);
 * dilation_near >= 0; stride >= 1 and 0 <= stride_phase < stride when
 * STRIDED or STRIDED_REL is set;
 * global_tokens >= 1 when GLOBAL is set (FLASH_MSA_ERR_INVALID_ARG
 * otherwise) and a multiple of the 128-token block (else
 * FLASH_MSA_ERR_UNSUPPORTED: every tile then keeps one interval of live
 * keys per row).  bitmask (BITMASK only, HOST memory, read only by
 * flash_msa_build_block_index): N rows of ceil(N/32) little-endian uint32
 * words, bit j % 32 of word j / 32 of row i set iff (i, j) may be live.
 * doc_starts / n_docs (DOCUMENTS only, HOST memory, read only by
 * flash_msa_build_block_index): n_docs + 1 offsets 0 = s_0 < s_1 < ... <
 * s_n_docs = N (cu_seqlens); sequence d holds tokens [s_d, s_{d+1}).  Boundary
 * tiles carry bit tiles, as with BITMASK. */
typedef struct {
  uint32_t flags;
  int32_t block;
  int64_t window;
  int32_t dilation, dilation_near;
  int32_t stride, stride_phase;
  const flash_msa_block_index* index;
  int64_t global_tokens;
  const uint32_t* bitmask;
  const int64_t* doc_starts;
  int64_t n_docs;
} flash_msa_mask_desc;

/* Build the block index for `mask` and sequence length N on the HOST (no GPU
 * work).  Two phases: call with out->row_ptr == NULL to fill only the counts
 * (seq_len, n_q_blocks, n_k_blocks, block, nnz, n_bit_tiles, and
 * live_elements, the mask's live (i, j) pairs, set again by the second call);
 * allocate every
 * array with those sizes (row_ptr/col_ptr n+1 int32, col_idx/row_idx nnz
 * int32, kind/kind_t nnz uint8, q_order/k_order n int32; with BITMASK also
 * bit_slot/bit_slot_t nnz int32 and bits/bits_t 512 n_bit_tiles uint32; with
 * sequence_tiles also tile_start/tile_seq0/tile_seq_len n int32) and call
 * again to fill them.  mask->index is ignored.  Errors: INVALID_ARG
 * (null, N < 1, bad field, BITMASK without mask->bitmask, DOCUMENTS without
 * offsets rising strictly from 0 to N), UNSUPPORTED (block != 128). */
flash_msa_status flash_msa_build_block_index(const flash_msa_mask_desc* mask, int64_t N,
                                             flash_msa_block_index* out);

/* Check a HOST copy of an index for internal consistency against N: sizes,
 * monotone pointers, ascending in-range block ids, kinds in {0,1}, CSC equal
 * to the transpose of CSR, orders being permutations.  Returns OK or
 * ERR_INDEX.  The kernels additionally skip (and report ERR_INDEX for) any
 * out-of-range block id they meet, so a corrupt device index cannot make
 * them read outside the tensors. */
flash_msa_status flash_msa_check_block_index(const flash_msa_block_index* host_index, int64_t N);

/* Forward: o = attention(q, k, v), lse[b,h,i] = log sum_j exp(scale q_i.k_j)
 * over live j (natural log; -inf and o_i = 0 for a row with no live key).
 * One kernel launch on `stream` (one CTA per SM, each working through pairs
 * of query blocks). */
flash_msa_status flash_msa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int64_t N, int d, float scale,
                               const flash_msa_mask_desc* mask, void* stream);

/* Bytes of device workspace flash_msa_bwd() needs: two fp32 vectors per
 * (b, h), each padded to whole 128-row tiles -- -LSE_i * log2(e) and
 * D_i = sum_c dO_ic * O_ic -- rounded up to 256 bytes.  0 for invalid sizes.
 * With a per-sequence tiled index the vectors hold 128 rows per tile: pass
 * N = 128 * index->n_q_blocks. */
size_t flash_msa_bwd_workspace_bytes(int B, int H, int64_t N, int d);

/* Backward: given the forward's o and lse and the upstream gradient dO,
 * write dq, dk, dv (bf16, (B, N, H, d)):
 *   P = exp(scale Q K^T - LSE) on live entries, dV = P^T dO, dP = dO V^T,
 *   D = rowsum(dO o O), dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q
 * (page 1, section "The Backward Pass: The Real Beast"; the scale enters dQ
 * and dK by the chain rule).  `workspace` is a DEVICE buffer of at least
 * flash_msa_bwd_workspace_bytes() bytes owned by the caller (contents are
 * overwritten); else FLASH_MSA_ERR_WORKSPACE.  Three kernel launches on
 * `stream` (D, then a key-stationary dK/dV kernel, then a query-stationary dQ
 * kernel: the "reduced separately" option for dQ, which recomputes S and dP,
 * seven tensor-core products per live tile); no atomics, every output is
 * bitwise reproducible. */
flash_msa_status flash_msa_bwd(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dO, void* dq, void* dk, void* dv,
                               int B, int H, int64_t N, int d, float scale,
                               const flash_msa_mask_desc* mask, void* workspace,
                               size_t workspace_bytes, void* stream);

/* The backward's launches one at a time (same arguments plus a bit set), in
 * two variants.
 * Two-kernel (flash_msa_bwd() is FLASH_MSA_BWD_DETERMINISTIC = PREPROCESS |
 * DKDV | DQ):
 *   PREPROCESS  D and the scaled LSE into the workspace (must run first); run
 *               together with FUSED, or on its own with a workspace large
 *               enough for the accumulated variant, it also zeroes the dQ
 *               accumulator
 *   DKDV        dK and dV (key-stationary, four products per live tile)
 *   DQ          dQ (query-stationary, recomputes S and dP: three products)
 *   DKDV and DQ read the workspace written by PREPROCESS, in either order.
 * Accumulated dQ (FLASH_MSA_BWD_ACCUMULATED = PREPROCESS | FUSED |
 * DQ_CONVERT, run in that order; the "dQ accumulated atomically" option):
 *   FUSED       one key-stationary kernel issuing the five products of every
 *               live tile: dK and dV accumulate on chip, and each tile's dQ
 *               partial product dS K is added into an fp32 accumulator in the
 *               workspace by TMA bulk tensor reductions
 *   DQ_CONVERT  dq = scale * accumulator, rounded to bf16
 *   dK and dV are bitwise equal to the two-kernel variant's; dQ is within
 *   rounding of it, and its low bits may differ between calls (the order of
 *   the fp32 additions varies).  On GB300 this variant is the slower one
 *   (the reductions, 64 KB of fp32 per live tile, cost more than the two
 *   recomputed products); it needs the larger workspace of
 *   flash_msa_bwd_stages_workspace_bytes().
 * FUSED may not be combined with DKDV or DQ (FLASH_MSA_ERR_INVALID_ARG). */
#define FLASH_MSA_BWD_PREPROCESS 1u
#define FLASH_MSA_BWD_DKDV 2u
#define FLASH_MSA_BWD_DQ 4u
#define FLASH_MSA_BWD_FUSED 8u
#define FLASH_MSA_BWD_DQ_CONVERT 16u
#define FLASH_MSA_BWD_DETERMINISTIC 7u
#define FLASH_MSA_BWD_ACCUMULATED 25u
/* Workspace bytes flash_msa_bwd_stages() needs for this set of stages: the
 * two vectors, plus the fp32 dQ accumulator (B, H, padded N, d) when FUSED or
 * DQ_CONVERT is set (0 for invalid sizes or stage bits). */
size_t flash_msa_bwd_stages_workspace_bytes(int B, int H, int64_t N, int d, unsigned stages);
flash_msa_status flash_msa_bwd_stages(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dO, void* dq, void* dk,
                                      void* dv, int B, int H, int64_t N, int d, float scale,
                                      const flash_msa_mask_desc* mask, void* workspace,
                                      size_t workspace_bytes, unsigned stages, void* stream);

/* Grouped-query attention (GQA; MQA when Hkv = 1): H query heads share Hkv
 * key/value heads, query head h using key/value head h / (H / Hkv) (page
 * "Flash MSA Attention Kernel Implementation", FAQ on grouped-query and
 * multi-query attention: the tiling is unchanged, fewer K/V heads are read).
 * q, o, dq and dO are (B, N, H, d); k, v, dk and dv are (B, N, Hkv, d); lse
 * is (B, H, N); the workspace is flash_msa_bwd_workspace_bytes(B, H, N, d).
 * dK and dV sum the contributions of all query heads of the group.  H % Hkv
 * must be 0, else FLASH_MSA_ERR_INVALID_ARG; everything else as in
 * flash_msa_fwd() / flash_msa_bwd(). */
flash_msa_status flash_msa_fwd_gqa(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int B, int H, int Hkv, int64_t N, int d,
                                   float scale, const flash_msa_mask_desc* mask, void* stream);
flash_msa_status flash_msa_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                                   const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                   int B, int H, int Hkv, int64_t N, int d, float scale,
                                   const flash_msa_mask_desc* mask, void* workspace,
                                   size_t workspace_bytes, void* stream);
/* flash_msa_bwd_stages() for grouped-query attention (arguments as in
 * flash_msa_bwd_gqa() plus the stage bits). */
flash_msa_status flash_msa_bwd_gqa_stages(const void* q, const void* k, const void* v,
                                          const void* o, const float* lse, const void* dO,
                                          void* dq, void* dk, void* dv, int B, int H, int Hkv,
                                          int64_t N, int d, float scale,
                                          const flash_msa_mask_desc* mask, void* workspace,
                                          size_t workspace_bytes, unsigned stages, void* stream);

/* Backward for callers that may not allocate device memory at call time (a
 * host framework that owns the whole device memory pool, or a latency-bound
 * loop where cudaMalloc/cudaFree are banned because they can synchronise the
 * device).  No counterpart on the pages: it exists only because such callers
 * cannot hand flash_msa_bwd() a workspace.  Same arguments, kernels and
 * results as flash_msa_bwd() minus the workspace: the scratch is a fixed
 * 16 MiB array inside the library, held on every device that loads the
 * library until the process exits.  Limit: B * H * ceil(N/128) * 128 <= 2^21
 * (flash_msa_bwd_workspace_bytes() <= 16 MiB); larger calls return
 * FLASH_MSA_ERR_WORKSPACE without launching anything.  Allocates nothing and
 * calls no allocating routine.  The first call on a device looks the array's
 * device address up (cudaGetSymbolAddress); make that first call before any
 * stream capture.  CUDA loads a library's device code lazily by default, so
 * the 16 MiB are committed on a device only when the library's device image
 * is first loaded there (at the latest by that first call), and that load
 * can fail with an out-of-memory error if the device has no room left: a
 * caller that reserves the whole device pool for its own allocator should
 * make its first call (or any other call of this library) on each device
 * before reserving the pool.  All calls on a device share the array: calls
 * whose kernels overlap on the GPU (e.g. on unordered streams) race and must
 * be avoided; sequential calls are fine (each rewrites every scratch element
 * it reads). */
flash_msa_status flash_msa_bwd_noalloc(const void* q, const void* k, const void* v,
                                       const void* o, const float* lse, const void* dO, void* dq,
                                       void* dk, void* dv, int B, int H, int64_t N, int d,
                                       float scale, const flash_msa_mask_desc* mask, void* stream);

/* Failure-detection self-test (no counterpart on the pages): launches on
 * `stream` one thread that waits, with the bounded wait every kernel here
 * uses, on an mbarrier that nothing arrives on.  The wait gives up after a
 * fixed 200 ms (independent of flash_msa_set_wait_limit_ms()), records
 * FLASH_MSA_ERR_TIMEOUT in the device status word and returns, so the next
 * flash_msa_get_status() reports TIMEOUT and the context stays usable;
 * nothing faults or hangs.  Returns OK or ERR_CUDA (launch). */
flash_msa_status flash_msa_selftest_wait_timeout(void* stream);

/* Limit, in milliseconds, of any single bounded wait inside the attention
 * kernels (no counterpart on the pages): a CTA whose wait on one of its
 * pipeline barriers exceeds it records FLASH_MSA_ERR_TIMEOUT, stops and
 * leaves its outputs incomplete instead of hanging.  Default 4000 ms, long
 * enough for a GPU time-sliced with other contexts.  Process-wide; applies to
 * launches made after the call.  ms must be in [1, 600000], else
 * FLASH_MSA_ERR_INVALID_ARG.  flash_msa_get_wait_limit_ms() returns the
 * current value. */
flash_msa_status flash_msa_set_wait_limit_ms(unsigned ms);
unsigned flash_msa_get_wait_limit_ms(void);

/* Synchronise `stream`, then read and clear the device status word shared by
 * every kernel of this library on the current device.  Returns OK, or the
 * first device-side error recorded since the last call (TIMEOUT, INDEX,
 * SCHEDULE), or
 * ERR_CUDA if the synchronisation itself failed. */
flash_msa_status flash_msa_get_status(void* stream);

/* Message for the last error returned on this host thread ("" if none). */
const char* flash_msa_last_error_string(void);

/* Library version string. */
const char* flash_msa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLASHMSA_H */
