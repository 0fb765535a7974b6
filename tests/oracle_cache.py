"""Memoised oracle block indices (the brute-force build takes seconds at full N)."""
import functools

from oracle import block_index
from oracle.mask import MaskSpec


@functools.lru_cache(maxsize=None)
def oracle_index(n: int, fields: tuple):
    return block_index.build(n, MaskSpec(**dict(fields)))
