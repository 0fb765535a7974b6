"""Two independent restatements used only to pin the vectorised oracle.

* ``forward_loops`` / ``backward_loops``: scalar pure-Python loops straight
  from the definitions (tiny N only), with their own scalar mask predicate.
* ``forward_tiled``: the tiled forward with an online softmax -- per query
  block keep the running row max m and running sum l, rescale the partial
  output by exp(m_old - m_new) for every key block, divide by l at the end
  ("Flash MSA Attention Kernel Implementation", section "The Flash Core:
  Tiling Over the Memory Hierarchy").  Masked scores are -inf; a row whose
  running max is still -inf contributes nothing.
"""
from __future__ import annotations

import math

import numpy as np

from .mask import MaskSpec


def live_scalar(i: int, j: int, n: int, spec: MaskSpec) -> bool:
    if not (0 <= i < n and 0 <= j < n):
        return False
    if spec.causal and j > i:
        return False
    if spec.doc_starts is not None:
        doc_i = max(d for d, st in enumerate(spec.doc_starts[:-1]) if st <= i)
        doc_j = max(d for d, st in enumerate(spec.doc_starts[:-1]) if st <= j)
        if doc_i != doc_j:
            return False
    if spec.bitmask is not None:
        w = (n + 31) // 32
        at = 4 * (i * w + j // 32)
        word = int.from_bytes(spec.bitmask[at:at + 4], "little")
        if not (word >> (j % 32)) & 1:
            return False
    if not spec.has_pattern:
        return True
    qb, kb = i // spec.block, j // spec.block
    near_ok = False
    near_dilated = spec.dilation is not None and not spec.dilation_far
    if spec.window is not None or near_dilated:
        near_ok = True
        if spec.window is not None and abs(i - j) > spec.window:
            near_ok = False
        if near_dilated:
            delta = abs(qb - kb)
            if not (delta < spec.dilation_near or delta % spec.dilation == 0):
                near_ok = False
    far_ok = spec.dilation is not None and spec.dilation_far and abs(qb - kb) % spec.dilation == 0
    stride_ok = False
    if spec.stride is not None:
        if spec.stride_relative:
            stride_ok = (qb - kb) % spec.stride == spec.stride_phase   # Python % is non-negative
        else:
            stride_ok = kb % spec.stride == spec.stride_phase
    global_ok = spec.global_tokens is not None and (i < spec.global_tokens or j < spec.global_tokens)
    return near_ok or far_ok or stride_ok or global_ok


def _dot(a, b):
    t = 0.0
    for x, y in zip(a, b):
        t += float(x) * float(y)
    return t


def _probs_loops(q, k, scale, spec):
    n = len(q)
    p = [[0.0] * n for _ in range(n)]
    lse = [-math.inf] * n
    for i in range(n):
        s = [scale * _dot(q[i], k[j]) if live_scalar(i, j, n, spec) else -math.inf for j in range(n)]
        m = max(s) if n else -math.inf
        if m == -math.inf:
            continue
        z = sum(math.exp(x - m) for x in s if x != -math.inf)
        lse[i] = m + math.log(z)
        for j in range(n):
            if s[j] != -math.inf:
                p[i][j] = math.exp(s[j] - lse[i])
    return p, lse


def forward_loops(q, k, v, scale, spec: MaskSpec):
    n, d = len(q), len(v[0])
    p, lse = _probs_loops(q, k, scale, spec)
    o = [[sum(p[i][j] * float(v[j][c]) for j in range(n)) for c in range(d)] for i in range(n)]
    return np.array(o), np.array(lse)


def backward_loops(q, k, v, do, scale, spec: MaskSpec):
    n, d = len(q), len(q[0])
    p, _ = _probs_loops(q, k, scale, spec)
    dp = [[_dot(do[i], v[j]) for j in range(n)] for i in range(n)]
    dsum = [sum(p[i][j] * dp[i][j] for j in range(n)) for i in range(n)]
    ds = [[p[i][j] * (dp[i][j] - dsum[i]) for j in range(n)] for i in range(n)]
    dq = [[scale * sum(ds[i][j] * float(k[j][c]) for j in range(n)) for c in range(d)] for i in range(n)]
    dk = [[scale * sum(ds[i][j] * float(q[i][c]) for i in range(n)) for c in range(d)] for j in range(n)]
    dv = [[sum(p[i][j] * float(do[i][c]) for i in range(n)) for c in range(len(do[0]))] for j in range(n)]
    return np.array(dq), np.array(dk), np.array(dv)


def forward_tiled(q, k, v, scale, spec: MaskSpec, block: int = 128):
    """Online-softmax forward over query and key blocks of `block` rows."""
    n, dv = q.shape[0], v.shape[1]
    out = np.zeros((n, dv))
    lse = np.full(n, -np.inf)
    for q0 in range(0, n, block):
        rows = np.arange(q0, min(q0 + block, n))
        m = np.full(len(rows), -np.inf)
        l = np.zeros(len(rows))
        o = np.zeros((len(rows), dv))
        for k0 in range(0, n, block):
            cols = np.arange(k0, min(k0 + block, n))
            s = scale * (q[rows] @ k[cols].T)
            live = np.array([[live_scalar(int(i), int(j), n, spec) for j in cols] for i in rows])
            s = np.where(live, s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            # rows that have seen no live key keep m = -inf; shift by 0 there
            shift = np.where(np.isfinite(m_new), m_new, 0.0)
            alpha = np.exp(m - shift)                 # exp(-inf) = 0 on the first live block
            e = np.exp(s - shift[:, None])
            l = alpha * l + e.sum(axis=1)
            o = alpha[:, None] * o + e @ v[cols]
            m = m_new
        seen = l > 0
        out[rows] = np.where(seen[:, None], o / np.where(seen, l, 1.0)[:, None], 0.0)
        lse[rows] = np.where(seen, m + np.log(np.where(seen, l, 1.0)), -np.inf)
    return out, lse
