"""Element-level attention mask predicate (oracle; test infrastructure only).

Definitions, one per mask kind named on the pages:

* causal -- key j is visible to query i iff j <= i.  Masked scores are -inf,
  never multiplied by zero ("Flash MSA Attention Kernel Implementation",
  section "Optimization Tricks That Actually Matter", paragraph "Masking and
  causal attention"; FAQ "How do I debug a flash attention kernel that
  produces NaN?").
* local window -- |i - j| <= W, inclusive ("How Does Flash-MSA Sparse
  Attention Work", section "How Flash-MSA Sparse Attention Works", mask kind
  "Local window").
* dilated -- read at block level: with Delta = |i // blk - j // blk|, keep the
  pair iff Delta < near or Delta % dilation == 0 (same section, mask kind
  "Dilated").
* strided -- fixed pattern in the style of Child et al.: every key in key
  block kb with kb % stride == phase (same section, mask kind "Fixed
  pattern").
* relative strided -- the strided pattern of Child et al. read relative to
  the query: with Delta = i // blk - j // blk, keep the pair iff
  Delta mod stride == phase (the alternative to the absolute reading above).
* far dilation -- the alternative reading of dilation: the window stays
  dense and dilated blocks (|Delta| mod dilation == 0) are kept at every
  distance, beyond the window too.
* global tokens -- the hybrid of a local window with a few global tokens in
  the style of Longformer (same page, section "How Do Sparse Attention
  Kernels Work in GPU Clusters?", the paragraph after the benchmark table;
  the FAQ "How does Flash-MSA affect model accuracy compared to dense
  attention?" gives 512 global tokens with an 8K window at 128K).  Read
  symmetrically: the first G tokens are global, so a global query attends
  every key and every query attends the global keys.

* bit-packed mask -- an arbitrary element mask given as bits, the mask tiles
  "in a bit-packed format" of "Flash MSA Attention Kernel Implementation",
  section "Optimization Tricks That Actually Matter", paragraph "Masking and
  causal attention": row i is ceil(N/32) little-endian 32-bit words, bit
  j % 32 of word j // 32 set iff the pair may be live.  It is AND-ed with
  everything else.
* documents (variable-length batches) -- sequences of different lengths
  packed back to back on one token axis, with offsets doc_starts (0 = s_0 <
  s_1 < ... < s_D = N); a token attends only to tokens of its own sequence,
  the batch being handled by masking (same page, section "The Production
  Pipeline: From Kernel to Service", request batching; "How to Use Flash
  MSA Kernels for Long Context", FAQ on flash-batch inference).  AND-ed with
  everything else, so causal means causal inside each sequence.

Combination: live = in_range AND causal_part AND pattern [AND bit], where pattern is
true when no window/dilation/stride/global part is set, and otherwise
(window AND dilation part) OR (strided part) OR (far dilation part) OR
(global part).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np


@dataclass(frozen=True)
class MaskSpec:
    causal: bool = False
    window: Optional[int] = None     # W, inclusive: |i - j| <= W
    dilation: Optional[int] = None   # block dilation factor
    dilation_near: int = 0           # block distances below this are always kept
    stride: Optional[int] = None     # key block kb live iff kb % stride == stride_phase
    stride_phase: int = 0
    block: int = 128                 # pattern block, in tokens
    global_tokens: Optional[int] = None  # G: queries and keys 0..G-1 are global
    stride_relative: bool = False    # stride part relative to the query block
    dilation_far: bool = False       # dilation as its own part, at every distance
    bitmask: Optional[bytes] = None  # packed rows, N x ceil(N/32) little-endian uint32
    doc_starts: Optional[tuple] = None  # packed sequences: offsets 0 = s_0 < ... < s_D = N

    @property
    def has_pattern(self) -> bool:
        return (self.window is not None or self.dilation is not None or self.stride is not None
                or self.global_tokens is not None)

    @property
    def window_bounded(self) -> bool:
        """Only the window reaches far keys' blocks (no strided / far-dilated part)."""
        return self.window is not None and self.stride is None and not self.dilation_far


DENSE = MaskSpec()
CAUSAL = MaskSpec(causal=True)


def live_matrix(rows, cols, n: int, spec: MaskSpec) -> np.ndarray:
    """Boolean matrix live[a, b] = live(rows[a], cols[b]) for a length-n sequence."""
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.asarray(cols, dtype=np.int64)[None, :]
    ok = (i >= 0) & (i < n) & (j >= 0) & (j < n)
    if spec.causal:
        ok = ok & (j <= i)
    if spec.has_pattern:
        part = np.zeros(ok.shape, dtype=bool)
        near_dilated = spec.dilation is not None and not spec.dilation_far
        if spec.window is not None or near_dilated:
            near_part = np.ones(ok.shape, dtype=bool)
            if spec.window is not None:
                near_part &= np.abs(i - j) <= spec.window
            if near_dilated:
                delta = np.abs(i // spec.block - j // spec.block)
                near_part &= (delta < spec.dilation_near) | (delta % spec.dilation == 0)
            part |= near_part
        if spec.dilation is not None and spec.dilation_far:
            part |= np.abs(i // spec.block - j // spec.block) % spec.dilation == 0
        if spec.stride is not None:
            if spec.stride_relative:
                part |= np.mod(i // spec.block - j // spec.block, spec.stride) == spec.stride_phase
            else:
                part |= (j // spec.block) % spec.stride == spec.stride_phase
        if spec.global_tokens is not None:
            part |= (i < spec.global_tokens) | (j < spec.global_tokens)
        ok = ok & part
    if spec.bitmask is not None:
        ok = ok & bit_matrix(spec.bitmask, n, i, j)
    if spec.doc_starts is not None:
        starts = np.asarray(spec.doc_starts, dtype=np.int64)
        if starts[0] != 0 or starts[-1] != n or (np.diff(starts) <= 0).any():
            raise ValueError("doc_starts must rise strictly from 0 to n")
        ok = ok & (document_of(starts, i) == document_of(starts, j))
    return ok


def document_of(starts: np.ndarray, t) -> np.ndarray:
    """Index of the sequence holding token t (clipped into [0, D))."""
    return np.clip(np.searchsorted(starts, t, side="right") - 1, 0, len(starts) - 2)


def bit_matrix(bitmask: bytes, n: int, i, j) -> np.ndarray:
    """bit(i, j) of a packed row-major mask (indices outside [0, n) read as 0)."""
    w = (n + 31) // 32
    words = np.frombuffer(bitmask, dtype="<u4")
    if words.size != n * w:
        raise ValueError(f"bitmask has {words.size} words, expected {n} x {w}")
    words = words.reshape(n, w)
    inside = (i >= 0) & (i < n) & (j >= 0) & (j < n)
    ii = np.clip(i, 0, n - 1)
    jj = np.clip(j, 0, n - 1)
    bit = (words[ii, jj // 32] >> (jj % 32).astype(np.uint32)) & np.uint32(1)
    return inside & (bit != 0)


def candidate_cols(r0: int, r1: int, n: int, spec: MaskSpec) -> tuple[int, int]:
    """Half-open key range [c0, c1) outside of which rows r0..r1-1 have no live key.

    Pure bound from the definitions above (causal: j <= i; window without a
    strided part: |i - j| <= W, and with global tokens the global keys
    j < G stay candidates while global rows i < G see every key); it only
    skips keys that the predicate kills.
    """
    c0, c1 = 0, n
    if spec.causal:
        c1 = min(c1, r1)
    if spec.window_bounded:
        g = spec.global_tokens
        if g is None:
            c0 = max(c0, r0 - spec.window)
        if g is None or r0 >= g:
            c1 = min(c1, r1 + spec.window)
    return c0, max(c0, c1)


def candidate_col_array(r0: int, r1: int, n: int, spec: MaskSpec) -> np.ndarray:
    """Key indices outside of which rows r0..r1-1 have no live key.

    The span of ``candidate_cols``, narrowed for a window with global tokens
    to the global keys [0, G) plus the window span of the rows (rows r0 >= G;
    same definitions as above, so only dead keys are left out).
    """
    c0, c1 = candidate_cols(r0, r1, n, spec)
    g = spec.global_tokens
    if g is None or not spec.window_bounded or r0 < g:
        return np.arange(c0, c1)
    lo = max(g, r0 - spec.window)
    return np.concatenate([np.arange(0, min(g, c1)), np.arange(lo, max(lo, c1))])
