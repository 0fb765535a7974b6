"""Dense float64 attention and its analytic gradients (oracle; test infrastructure only).

Definition followed ("Flash MSA Attention Kernel Implementation", section
"Why Standard Attention Broke": O = softmax(Q K^T / sqrt(d)) V; "How to Use
Flash MSA Kernels for Long Context", section "What Flash MSA Actually Does":
the fused kernel computes the same exact function), with the mask applied as
-inf before the softmax.  For one head with inputs q, k, v of shape (N, d):

    S_ij   = scale * q_i . k_j        if live(i, j), else -inf
    LSE_i  = m_i + log(sum_j exp(S_ij - m_i)),  m_i = max_j S_ij
    P_ij   = exp(S_ij - LSE_i)
    O_i    = sum_j P_ij v_j

A row with no live key has O_i = 0, LSE_i = -inf and contributes nothing to
any gradient (reading of an edge case the pages leave open).

Gradients ("Flash MSA Attention Kernel Implementation", section "The Backward
Pass: The Real Beast": dP = dO V^T, dS = P o (dP - rowsum(P o dP)),
dQ = dS K, dK = dS^T Q, dV = P^T dO; the softmax scale enters dQ and dK by the
chain rule, which the page's sketch leaves out):

    dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P o (dP - D)
    dQ = scale * dS K,  dK = scale * dS^T Q

``forward_head`` / ``backward_head`` materialise S over the whole (N, N)
matrix.  ``forward_rows`` / ``row_stats`` / ``backward_sampled`` evaluate the
same definitions for chosen rows or key columns, materialising S one chunk of
rows at a time over the rows' candidate key span (keys outside that span are
dead by definition); tests check them against the full versions.
"""
from __future__ import annotations

import numpy as np

from .mask import MaskSpec, candidate_col_array, live_matrix


def default_scale(d: int) -> float:
    return 1.0 / np.sqrt(d)


def _masked_scores(q_rows, k_cols, scale, live):
    s = scale * (q_rows @ k_cols.T)
    return np.where(live, s, -np.inf)


def _softmax_rows(s):
    """Row softmax of a masked score matrix; returns (P, LSE); empty rows -> P = 0, LSE = -inf."""
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 for dead entries
    l = e.sum(axis=1)
    l_safe = np.where(empty, 1.0, l)
    p = e / l_safe[:, None]
    lse = np.where(empty, -np.inf, m_safe + np.log(l_safe))
    return p, lse


def forward_head(q, k, v, scale, spec: MaskSpec):
    """O (N, d) and LSE (N,) for one head, full (N, N) materialisation."""
    n = q.shape[0]
    idx = np.arange(n)
    s = _masked_scores(q, k, scale, live_matrix(idx, idx, n, spec))
    p, lse = _softmax_rows(s)
    return p @ v, lse


def probabilities(q, k, scale, spec: MaskSpec):
    """The full P matrix (N, N) for one head."""
    n = q.shape[0]
    idx = np.arange(n)
    s = _masked_scores(q, k, scale, live_matrix(idx, idx, n, spec))
    return _softmax_rows(s)[0]


def backward_head(q, k, v, do, scale, spec: MaskSpec):
    """dQ, dK, dV (each (N, d)) for one head, full (N, N) materialisation."""
    p = probabilities(q, k, scale, spec)
    dv = p.T @ do
    dp = do @ v.T
    dsum = (p * dp).sum(axis=1)
    ds = p * (dp - dsum[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Row-chunked evaluation of the same definitions (large N)
# ---------------------------------------------------------------------------
def _chunks(rows, chunk):
    rows = np.asarray(rows, dtype=np.int64)
    for a in range(0, len(rows), chunk):
        yield rows[a:a + chunk]


def _row_block(q, k, scale, spec, rows):
    """Masked scores for `rows` over their candidate key span; returns (cols, S).

    Key columns that are dead for every row of the chunk are dropped before
    the product (they would only contribute exp(-inf) = 0)."""
    n = q.shape[0]
    cols = candidate_col_array(int(rows.min()), int(rows.max()) + 1, n, spec)
    live = live_matrix(rows, cols, n, spec)
    keep = live.any(axis=0)
    if keep.size and keep.mean() < 0.75:
        cols, live = cols[keep], live[:, keep]
    s = _masked_scores(q[rows], k[cols], scale, live)
    return cols, s


def forward_rows(q, k, v, scale, spec: MaskSpec, rows=None, chunk=256):
    """O[rows], LSE[rows] for one head (rows default: all)."""
    n, d = q.shape
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.zeros((len(rows), v.shape[1]))
    lse = np.full(len(rows), -np.inf)
    pos = 0
    for r in _chunks(rows, chunk):
        cols, s = _row_block(q, k, scale, spec, r)
        p, l = _softmax_rows(s)
        o[pos:pos + len(r)] = p @ v[cols]
        lse[pos:pos + len(r)] = l
        pos += len(r)
    return o, lse


def row_stats(q, k, v, do, scale, spec: MaskSpec, chunk=256, rows=None):
    """LSE_i and D_i = sum_j P_ij dP_ij for every row of one head, or only for
    `rows` (the others are left at LSE = -inf, D = 0).  A causal mask makes
    column j of P depend only on rows i >= j, so the statistics of rows
    i >= min(cols) suffice for the key columns cols of ``backward_sampled``."""
    n = q.shape[0]
    lse = np.full(n, -np.inf)
    dsum = np.zeros(n)
    for r in _chunks(np.arange(n) if rows is None else rows, chunk):
        cols, s = _row_block(q, k, scale, spec, r)
        p, l = _softmax_rows(s)
        dp = do[r] @ v[cols].T
        lse[r] = l
        dsum[r] = (p * dp).sum(axis=1)
    return lse, dsum


def backward_sampled(q, k, v, do, scale, spec: MaskSpec, q_rows, k_cols, chunk=256, stats=None):
    """dQ[q_rows] and dK[k_cols], dV[k_cols] for one head.

    dQ_i needs only row i of P and dP.  dK_j, dV_j need column j of P, i.e.
    LSE_i and D_i of every row, which ``row_stats`` provides (pass them in
    through ``stats`` to reuse them).
    """
    n = q.shape[0]
    lse, dsum = row_stats(q, k, v, do, scale, spec, chunk) if stats is None else stats
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_cols = np.asarray(k_cols, dtype=np.int64)
    dq = np.zeros((len(q_rows), q.shape[1]))
    pos = 0
    for r in _chunks(q_rows, chunk):
        cols, s = _row_block(q, k, scale, spec, r)
        p, _ = _softmax_rows(s)
        dp = do[r] @ v[cols].T
        ds = p * (dp - dsum[r][:, None])
        dq[pos:pos + len(r)] = scale * (ds @ k[cols])
        pos += len(r)
    # columns: P_ij = exp(S_ij - LSE_i) for every row i
    all_rows = np.arange(n)
    live = live_matrix(all_rows, k_cols, n, spec)
    s = np.where(live, scale * (q @ k[k_cols].T), -np.inf)
    lse_safe = np.where(np.isfinite(lse), lse, 0.0)
    p = np.where(live, np.exp(s - lse_safe[:, None]), 0.0)
    dp = do @ v[k_cols].T
    ds = p * (dp - dsum[:, None])
    dv = p.T @ do
    dk = scale * (ds.T @ q)
    return dq, dk, dv
