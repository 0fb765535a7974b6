"""(B, N, H, d) wrappers over the per-head oracle, with an optional process pool.

Heads are independent (each (b, h) pair is its own attention problem), so the
wrappers just loop -- or fan out over worker processes started with the
``spawn`` method -- and gather.  BLAS threads per worker are left to the
caller's environment.
"""
from __future__ import annotations

import multiprocessing as mp

import numpy as np

from . import attention
from .mask import MaskSpec


def _fwd_one(args):
    q, k, v, scale, spec, rows = args
    return attention.forward_rows(q, k, v, scale, spec, rows)


def _bwd_one(args):
    q, k, v, do, scale, spec = args
    return attention.backward_head(q, k, v, do, scale, spec)


def forward(q, k, v, scale, spec: MaskSpec, heads=None, rows=None, workers: int = 1):
    """q, k, v: float64 (B, N, H, d).  Returns {(b, h): (O_rows, LSE_rows)}."""
    B, N, H, _ = q.shape
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)
    jobs = [(q[b, :, h], k[b, :, h], v[b, :, h], scale, spec, rows) for b, h in heads]
    if workers > 1 and len(jobs) > 1:
        with mp.get_context("spawn").Pool(min(workers, len(jobs))) as pool:
            res = pool.map(_fwd_one, jobs)
    else:
        res = [_fwd_one(j) for j in jobs]
    return dict(zip(heads, res))


def backward(q, k, v, do, scale, spec: MaskSpec, heads=None, workers: int = 1):
    """Full per-head gradients {(b, h): (dQ, dK, dV)}."""
    B, N, H, _ = q.shape
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)
    jobs = [(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], scale, spec) for b, h in heads]
    if workers > 1 and len(jobs) > 1:
        with mp.get_context("spawn").Pool(min(workers, len(jobs))) as pool:
            res = pool.map(_bwd_one, jobs)
    else:
        res = [_bwd_one(j) for j in jobs]
    return dict(zip(heads, res))


def full_forward(q, k, v, scale, spec: MaskSpec):
    """Dense (B, N, H, d) output and (B, H, N) LSE for small problems."""
    B, N, H, d = q.shape
    o = np.zeros(q.shape[:3] + (v.shape[3],))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, :, h], lse[b, h] = attention.forward_head(q[b, :, h], k[b, :, h], v[b, :, h], scale, spec)
    return o, lse


def full_backward(q, k, v, do, scale, spec: MaskSpec):
    B, N, H, d = q.shape
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            dq[b, :, h], dk[b, :, h], dv[b, :, h] = attention.backward_head(
                q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], scale, spec)
    return dq, dk, dv
