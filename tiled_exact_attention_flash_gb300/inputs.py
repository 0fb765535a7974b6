"""Seeded synthetic inputs and workload descriptions (no attention arithmetic here).

Shared by the tests, ``bench.py`` and ``__graft_entry__``: every tensor is
``numpy.random.default_rng(seed).standard_normal(shape, dtype=float32)`` in
(B, N, H, d) layout, rounded once to bf16 (round-to-nearest-even via
``torch.Tensor.to(torch.bfloat16)``).  The CUDA path consumes the bf16 tensor;
the oracle consumes the same values promoted exactly to float64.

Workloads: the five attention configurations the pages' discussion motivates
(7B-style layer, d = 128, long context; causal, local window + strided, and
local window with block dilation), plus a sixth for the local window with
global tokens hybrid (8K window, 512 global tokens, 128K tokens), two more
with the second readings of the strided and dilated masks, one of packed
documents under a bit-packed mask and one variable-length batch.  Seeds: Q, K, V, dO of workload c use
1000*c + 1 .. 1000*c + 4.
"""
from __future__ import annotations

import functools
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    cid: int
    name: str
    B: int
    H: int
    N: int
    d: int
    # mask description: plain fields, converted by each side into its own type
    mask: dict = field(default_factory=dict)
    # packed documents: (mean length, seed) of the seeded document lengths,
    # added by mask_fields() as a bit-packed mask ("bitmask") or as sequence
    # offsets ("starts": a variable-length batch)
    docs: Optional[tuple] = None
    docs_as: str = "bitmask"

    @property
    def shape(self):
        return (self.B, self.N, self.H, self.d)

    def mask_fields(self) -> dict:
        """The mask fields with the packed-documents bitmask when there is one."""
        f = dict(self.mask)
        if self.docs is not None:
            if self.docs_as == "starts":
                lens = document_lengths(self.N, self.docs[1], self.docs[0])
                f["doc_starts"] = tuple(int(x) for x in np.cumsum([0] + lens))
            else:
                f["bitmask"] = _documents_bitmask(self.N, *self.docs)
        return f


WORKLOADS = {
    1: Workload(1, "dense B1 H1 N256 d64", 1, 1, 256, 64, {}),
    2: Workload(2, "causal B4 H16 N4096 d128", 4, 16, 4096, 128, {"causal": True}),
    3: Workload(3, "causal B1 H32 N16384 d128", 1, 32, 16384, 128, {"causal": True}),
    4: Workload(4, "causal window1024 + strided8 B1 H32 N32768 d128", 1, 32, 32768, 128,
                {"causal": True, "window": 1024, "stride": 8, "stride_phase": 0}),
    5: Workload(5, "causal window4096 dilation2 B1 H8 N131072 d128", 1, 8, 131072, 128,
                {"causal": True, "window": 4096, "dilation": 2, "dilation_near": 2}),
    # local window plus global tokens: 8K window and 512 global tokens at 128K
    6: Workload(6, "causal window8192 + global512 B1 H8 N131072 d128", 1, 8, 131072, 128,
                {"causal": True, "window": 8192, "global_tokens": 512}),
    # the second readings of the strided and dilated masks on the shapes of 4 and 5
    7: Workload(7, "causal window1024 + relative strided8 B1 H32 N32768 d128", 1, 32, 32768, 128,
                {"causal": True, "window": 1024, "stride": 8, "stride_phase": 0,
                 "stride_relative": True}),
    8: Workload(8, "causal window4096 + far dilation2 B1 H8 N131072 d128", 1, 8, 131072, 128,
                {"causal": True, "window": 4096, "dilation": 2, "dilation_far": True}),
    # packed documents under a bit-packed mask, causal inside each document
    9: Workload(9, "causal packed documents (mean 2048 tokens) B1 H16 N32768 d128", 1, 16, 32768,
                128, {"causal": True}, docs=(2048, 9009)),
    # a variable-length batch: seeded sequence lengths (mean 2048) packed into
    # 65536 tokens, causal inside each sequence
    10: Workload(10, "causal varlen batch (mean 2048 tokens) T65536 H16 d128", 1, 16, 65536, 128,
                 {"causal": True}, docs=(2048, 10010), docs_as="starts"),
}


def normal_bf16(shape, seed: int) -> torch.Tensor:
    """float32 N(0, 1) from a seeded generator, rounded to bf16 (CPU tensor)."""
    x = np.random.default_rng(seed).standard_normal(shape, dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def workload_inputs(w: Workload, names=("q", "k", "v", "do")) -> dict:
    seeds = {"q": 1, "k": 2, "v": 3, "do": 4}
    return {n: normal_bf16(w.shape, 1000 * w.cid + seeds[n]) for n in names}


def small_inputs(B, N, H, d, seed: int, names=("q", "k", "v", "do")) -> dict:
    """Inputs for extra test cases (ragged N, tiny shapes): seeds seed*10 + 1..4."""
    seeds = {"q": 1, "k": 2, "v": 3, "do": 4}
    return {n: normal_bf16((B, N, H, d), 10 * seed + seeds[n]) for n in names}


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact promotion of a (bf16) tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# bit-packed masks: row i is ceil(N/32) little-endian uint32 words, bit j % 32
# of word j // 32 set iff the pair (i, j) may be live
# ---------------------------------------------------------------------------
def pack_bitmask(live: np.ndarray) -> bytes:
    """(N, N) booleans -> packed rows."""
    n = live.shape[0]
    w = (n + 31) // 32
    padded = np.zeros((n, w * 32), dtype=bool)
    padded[:, :n] = live
    words = np.packbits(padded.reshape(n, w, 4, 8)[..., ::-1], axis=-1).reshape(n, w, 4)
    return words.astype(np.uint8).tobytes()


def document_lengths(n: int, seed: int, mean: int) -> list:
    """Seeded lengths of the documents packed into one sequence of n tokens
    (exponentially distributed around `mean`, at least 1 token each)."""
    rng = np.random.default_rng(seed)
    lens, total = [], 0
    while total < n:
        ln = max(1, int(rng.exponential(mean)))
        ln = min(ln, n - total)
        lens.append(ln)
        total += ln
    return lens


def document_bitmask(n: int, lengths) -> bytes:
    """Packed mask of a sequence of packed documents: (i, j) may be live iff
    both tokens belong to the same document (built row block by row block,
    without an (N, N) boolean matrix)."""
    w = (n + 31) // 32
    words = np.zeros((n, w), dtype=np.uint32)
    start = 0
    for ln in lengths:
        end = start + ln
        row = np.zeros(w * 32, dtype=bool)
        row[start:end] = True
        packed = (row.reshape(w, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(axis=1)
        words[start:end] = packed.astype(np.uint32)
        start = end
    return words.astype("<u4").tobytes()


@functools.lru_cache(maxsize=2)
def _documents_bitmask(n: int, mean: int, seed: int) -> bytes:
    return document_bitmask(n, document_lengths(n, seed, mean))
