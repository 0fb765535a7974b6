"""Brute-force tile classification and the per-block index lists (oracle).

"How Does Flash-MSA Sparse Attention Work" (section "How Flash-MSA Sparse
Attention Works") applies the mask inside the tiling loop through a per-block
mask or "a precomputed index list", so that dead key/value tiles are never
loaded.  Here every tile (qb, kb) of `tile` x `tile` entries is classified by
evaluating the element predicate on ALL of its entries (rows and columns past
the end of the sequence count as dead entries):

    dead    -- no live entry;  full -- every entry live;  partial -- otherwise

and the lists are built from that classification:

    CSR  by query block: row_ptr, col_idx (ascending kb), kind (0 full, 1 partial)
    CSC  by key block:   col_ptr, row_idx (ascending qb), kind_t
    k_order:             key blocks sorted by descending live-tile count,
                         ties by ascending index (longest work first)
    q_order:             query blocks in pairs that share key tiles, pairs
                         longest first (see _shared_pairs_order)

With a bit-packed mask (or packed documents), a partial tile whose live set
differs from the live set of the same mask without the bits (and without
the documents) carries its live entries as bits:
slots are numbered in CSR order; bits[slot] holds 128 rows (query) of four
32-bit words (key bit c in word c // 32, bit c % 32) and bits_t[slot] the
transpose (128 key rows of four words over the queries); bit_slot /
bit_slot_t give each CSR / CSC entry its slot or -1.

Packed sequences (variable-length batches) whose other mask parts depend
only on i - j (causal, local window) and that carry no bit-packed mask are
tiled per sequence instead: sequence [s0, s1) gets its own tiles starting at
s0, s0 + 128, ..., so no tile holds tokens of two sequences (the way P1's
request batching keeps each request's attention to itself), and only tile
pairs of one sequence exist.  Tiles are numbered sequence by sequence; for
tile t, tile_start[t] is its first token, tile_seq0[t] and tile_seq_len[t]
its sequence's first token and length.  q_order then keeps neighbouring
tiles of one sequence together in pairs (see _pair_order).  Entries of a tile past its
sequence's end count as dead, and each tile pair is classified by evaluating
the predicate on all of its entries, as above.

For masks with a local window and no strided part, key blocks farther than
the window from the query block are skipped without evaluation: by the window
definition none of their entries is live (with global tokens, the key
blocks holding global keys and every block of a global query block are
still evaluated).  Tests check this shortcut against the full evaluation.
"""
from __future__ import annotations

import numpy as np

import dataclasses

from .mask import MaskSpec, live_matrix

DEAD, FULL, PARTIAL = -1, 0, 1


def classify(n: int, spec: MaskSpec, tile: int = 128, prune: bool = True) -> np.ndarray:
    """kinds[qb, kb] in {DEAD, FULL, PARTIAL}."""
    nb = (n + tile - 1) // tile
    kinds = np.full((nb, nb), DEAD, dtype=np.int8)
    span = None
    if prune and spec.window_bounded:
        span = spec.window // tile + 2
    g = spec.global_tokens
    for qb in range(nb):
        rows = np.arange(qb * tile, qb * tile + tile)
        if span is None or (g is not None and qb * tile < g):
            kbs = range(nb)
        else:
            kbs = range(max(0, qb - span), min(nb, qb + span + 1))
            if g is not None:
                kbs = sorted(set(kbs) | set(range(min(nb, (g + tile - 1) // tile))))
        for kb in kbs:
            cols = np.arange(kb * tile, kb * tile + tile)
            live = live_matrix(rows, cols, n, spec)
            cnt = int(live.sum())
            if cnt == 0:
                continue
            kinds[qb, kb] = FULL if cnt == tile * tile else PARTIAL
    return kinds


def _pack_rows(live: np.ndarray) -> np.ndarray:
    """(rows, 128) booleans -> (rows, 4) uint32 words, column c in word c // 32, bit c % 32."""
    weights = (np.uint32(1) << np.arange(32, dtype=np.uint32))
    return (live.reshape(live.shape[0], 4, 32).astype(np.uint32) * weights).sum(axis=2).astype(np.uint32)


def sequence_tiled(spec: MaskSpec) -> bool:
    """Whether a mask is tiled per sequence (see the module docstring)."""
    return (spec.doc_starts is not None and spec.bitmask is None and spec.dilation is None
            and spec.stride is None and spec.global_tokens is None)


def sequence_tiles(spec: MaskSpec, tile: int = 128):
    """(tile_start, tile_seq0, tile_seq_len) of the per-sequence tiling."""
    start, seq0, seq_len = [], [], []
    for s0, s1 in zip(spec.doc_starts[:-1], spec.doc_starts[1:]):
        for m in range((s1 - s0 + tile - 1) // tile):
            start.append(s0 + m * tile)
            seq0.append(s0)
            seq_len.append(s1 - s0)
    return (np.array(start, dtype=np.int32), np.array(seq0, dtype=np.int32),
            np.array(seq_len, dtype=np.int32))


def _pair_order(spec: MaskSpec, row_len, tile: int) -> np.ndarray:
    """q_order of per-sequence tiles: every sequence's tiles in neighbouring
    pairs counted from its last tile ((t, t - 1), (t - 2, t - 3), ...; a
    sequence with an odd tile count leaves its first tile single).  Pairs come
    first, by descending live-tile count of their first tile, ties by
    ascending tile id, each pair's tiles in that order; then the single
    tiles, by descending count, ties by ascending id.  Positions 2r and
    2r + 1 thus hold two neighbouring tiles of one sequence (or two singles)."""
    starts = spec.doc_starts
    pairs, singles, base = [], [], 0
    for s0, s1 in zip(starts[:-1], starts[1:]):
        nt = (s1 - s0 + tile - 1) // tile
        last = base + nt - 1
        for t in range(last, base, -2):
            pairs.append((t, t - 1))
        if nt % 2:
            singles.append(base)
        base += nt
    pairs.sort(key=lambda pr: (-row_len[pr[0]], pr[0]))
    singles.sort(key=lambda t: (-row_len[t], t))
    return np.array([t for pr in pairs for t in pr] + singles, dtype=np.int32)


# Candidate partners of a query block, in the order they are tried.
PAIR_OFFSETS = (1, -1, 2, -2, 4, -4, 8, -8)


def _shared_pairs_order(row_ptr, col_idx) -> np.ndarray:
    """q_order of a packed-axis index: the query blocks in pairs (positions
    2r and 2r + 1, which the forward runs together, loading their key tiles
    once) chosen to share key tiles.  Blocks are visited longest first
    (descending live-tile count, ties by ascending index); an unpaired block
    takes, among the unpaired blocks PAIR_OFFSETS away, the one whose list
    has the most key tiles in common with its own (the first one tried on
    ties), provided they have any in common.  The blocks left over are paired
    in visiting order.  The pairs are then ordered by the live-tile count of
    their first block (descending, ties by its ascending index); a last
    unpaired block, if any, comes at the end."""
    nb = len(row_ptr) - 1
    lens = np.diff(row_ptr)
    lists = [set(col_idx[row_ptr[b]:row_ptr[b + 1]].tolist()) for b in range(nb)]
    visit = sorted(range(nb), key=lambda b: (-lens[b], b))
    paired = [False] * nb
    pairs = []
    for a in visit:
        if paired[a]:
            continue
        best, best_common = -1, 0
        for off in PAIR_OFFSETS:
            c = a + off
            if 0 <= c < nb and not paired[c]:
                common = len(lists[a] & lists[c])
                if common > best_common:
                    best, best_common = c, common
        if best >= 0:
            paired[a] = paired[best] = True
            pairs.append((a, best))
    rest = [a for a in visit if not paired[a]]
    pairs += [(rest[i], rest[i + 1]) for i in range(0, len(rest) - 1, 2)]
    pairs.sort(key=lambda pr: (-lens[pr[0]], pr[0]))
    order = [b for pr in pairs for b in pr]
    if len(rest) % 2:
        order.append(rest[-1])
    return np.array(order, dtype=np.int32)


def classify_sequence_tiles(n: int, spec: MaskSpec, tile: int = 128) -> np.ndarray:
    """kinds[qt, kt] over the per-sequence tiles; pairs of two sequences are dead."""
    start, seq0, seq_len = sequence_tiles(spec, tile)
    nt = len(start)
    kinds = np.full((nt, nt), DEAD, dtype=np.int8)
    for qt in range(nt):
        end = int(seq0[qt]) + int(seq_len[qt])
        rows = np.arange(start[qt], start[qt] + tile)
        for kt in np.nonzero(seq0 == seq0[qt])[0]:
            cols = np.arange(start[kt], start[kt] + tile)
            live = live_matrix(rows, cols, n, spec) & (rows < end)[:, None] & (cols < end)[None, :]
            cnt = int(live.sum())
            if cnt:
                kinds[qt, kt] = FULL if cnt == tile * tile else PARTIAL
    return kinds


def build(n: int, spec: MaskSpec, tile: int = 128, prune: bool = True) -> dict:
    seq = sequence_tiled(spec)
    kinds = classify_sequence_tiles(n, spec, tile) if seq else classify(n, spec, tile, prune)
    nb = kinds.shape[0]
    row_ptr = np.zeros(nb + 1, dtype=np.int32)
    col_idx, kind = [], []
    for qb in range(nb):
        kbs = np.nonzero(kinds[qb] != DEAD)[0]
        col_idx.extend(kbs.tolist())
        kind.extend(kinds[qb, kbs].tolist())
        row_ptr[qb + 1] = row_ptr[qb] + len(kbs)
    col_ptr = np.zeros(nb + 1, dtype=np.int32)
    row_idx, kind_t = [], []
    for kb in range(nb):
        qbs = np.nonzero(kinds[:, kb] != DEAD)[0]
        row_idx.extend(qbs.tolist())
        kind_t.extend(kinds[qbs, kb].tolist())
        col_ptr[kb + 1] = col_ptr[kb] + len(qbs)
    # bit tiles (bit-packed masks only)
    bit_slot = np.full(len(col_idx), -1, dtype=np.int32)
    bits, bits_t = [], []
    if (spec.bitmask is not None or spec.doc_starts is not None) and not seq:
        plain = dataclasses.replace(spec, bitmask=None, doc_starts=None)
        for qb in range(nb):
            rows = np.arange(qb * tile, qb * tile + tile)
            for e in range(row_ptr[qb], row_ptr[qb + 1]):
                if kind[e] != PARTIAL:
                    continue
                cols = np.arange(col_idx[e] * tile, col_idx[e] * tile + tile)
                live = live_matrix(rows, cols, n, spec)
                if np.array_equal(live, live_matrix(rows, cols, n, plain)):
                    continue
                bit_slot[e] = len(bits)
                bits.append(_pack_rows(live))
                bits_t.append(_pack_rows(live.T))
    slot_of = {(qb, int(col_idx[e])): int(bit_slot[e])
               for qb in range(nb) for e in range(row_ptr[qb], row_ptr[qb + 1])}
    bit_slot_t = np.array([slot_of[(int(qb), kb)] for kb in range(nb)
                           for qb in row_idx[col_ptr[kb]:col_ptr[kb + 1]]], dtype=np.int32)
    row_len = np.diff(row_ptr)
    col_len = np.diff(col_ptr)
    if seq:
        q_order = _pair_order(spec, row_len, tile)
    else:
        q_order = _shared_pairs_order(row_ptr, np.array(col_idx, dtype=np.int32))
    k_order = np.array(sorted(range(nb), key=lambda b: (-col_len[b], b)), dtype=np.int32)
    empty = np.zeros(0, dtype=np.int32)
    tile_start, tile_seq0, tile_seq_len = sequence_tiles(spec, tile) if seq else (empty,) * 3
    return {
        "tile_start": tile_start,
        "tile_seq0": tile_seq0,
        "tile_seq_len": tile_seq_len,
        "n_blocks": nb,
        "nnz": int(row_ptr[-1]),
        "row_ptr": row_ptr,
        "col_idx": np.array(col_idx, dtype=np.int32),
        "kind": np.array(kind, dtype=np.uint8),
        "col_ptr": col_ptr,
        "row_idx": np.array(row_idx, dtype=np.int32),
        "kind_t": np.array(kind_t, dtype=np.uint8),
        "q_order": q_order,
        "k_order": k_order,
        "n_bit_tiles": len(bits),
        "bit_slot": bit_slot,
        "bit_slot_t": bit_slot_t,
        "bits": (np.concatenate(bits).reshape(-1) if bits else np.zeros(0, np.uint32)),
        "bits_t": (np.concatenate(bits_t).reshape(-1) if bits_t else np.zeros(0, np.uint32)),
    }
