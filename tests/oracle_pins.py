"""Pin checks for the oracle: each returns the largest violation it finds.

They are plain functions of an oracle-like callable so that the negative
controls in ``test_oracle_pins.py`` can run the same checks against copies of
the oracle with a mistake planted in them.
"""
import numpy as np

from oracle.mask import MaskSpec, live_matrix


def uniform_q_zero(fwd, n, d, spec, rng):
    """Q = 0: O_i = mean of v_j over live j, LSE_i = ln(#live_i)."""
    q = np.zeros((n, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    o, lse = fwd(q, k, v, 1.0 / np.sqrt(d), spec)
    live = live_matrix(np.arange(n), np.arange(n), n, spec)
    cnt = live.sum(axis=1)
    err = 0.0
    for i in range(n):
        if cnt[i] == 0:
            err = max(err, np.abs(o[i]).max(), 0.0 if lse[i] == -np.inf else np.inf)
            continue
        err = max(err, np.abs(o[i] - v[live[i]].mean(axis=0)).max(), abs(lse[i] - np.log(cnt[i])))
    return err


def causal_row0(fwd, n, d, rng):
    """Causal: O_0 = v_0 and LSE_0 = scale * q_0 . k_0."""
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    scale = 1.0 / np.sqrt(d)
    o, lse = fwd(q, k, v, scale, MaskSpec(causal=True))
    return max(np.abs(o[0] - v[0]).max(), abs(lse[0] - scale * q[0] @ k[0]))


def one_hot_dominant(fwd, n, d, rng):
    """q_i = c * k_t(i) with a score gap >= 40: O_i = v_t(i) within e^-40 (dense mask)."""
    k = np.linalg.qr(rng.standard_normal((max(n, d), max(n, d))))[0][:n, :d] * 1.0
    # orthonormal-ish keys: q_i . k_t = c, q_i . k_j ~ 0 for j != t when n <= d
    v = rng.standard_normal((n, d))
    target = rng.permutation(n)
    c = 80.0
    q = c * k[target] * np.sqrt(d)   # scale 1/sqrt(d) -> score c * |k_t|^2
    o, _ = fwd(q, k, v, 1.0 / np.sqrt(d), MaskSpec())
    s = q @ k.T / np.sqrt(d)
    gap = np.sort(s, axis=1)[:, -1] - np.sort(s, axis=1)[:, -2]
    assert gap.min() >= 40, gap.min()
    return np.abs(o - v[target]).max()


def constant_v(fwd, bwd, n, d, spec, rng):
    """V = c: O = c, dQ = dK = 0, dV_j = sum_i P_ij dO_i."""
    q, k, do = (rng.standard_normal((n, d)) for _ in range(3))
    v = np.full((n, d), 0.75)
    scale = 1.0 / np.sqrt(d)
    o, lse = fwd(q, k, v, scale, spec)
    dq, dk, dv = bwd(q, k, v, do, scale, spec)
    live = live_matrix(np.arange(n), np.arange(n), n, spec)
    has = live.any(axis=1)
    err = np.abs(o[has] - 0.75).max()
    err = max(err, np.abs(dq).max(), np.abs(dk).max())
    # P from the definition, not from the callable under test
    s = np.where(live, scale * q @ k.T, -np.inf)
    m = np.where(has, s.max(axis=1), 0.0)
    e = np.where(live, np.exp(s - m[:, None]), 0.0)
    p = e / np.where(has, e.sum(axis=1), 1.0)[:, None]
    return max(err, np.abs(dv - p.T @ do).max())


def gradient_invariants(fwd, bwd, n, d, spec, rng):
    """sum_j dK_j = 0; sum_j dV_j = sum over rows with a live key of dO_i."""
    q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
    dq, dk, dv = bwd(q, k, v, do, 1.0 / np.sqrt(d), spec)
    has = live_matrix(np.arange(n), np.arange(n), n, spec).any(axis=1)
    return max(np.abs(dk.sum(axis=0)).max(), np.abs(dv.sum(axis=0) - do[has].sum(axis=0)).max())


def permutation_invariance(fwd, n, d, rng):
    """Dense mask: permuting (K, V) rows jointly leaves O and LSE unchanged."""
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    perm = rng.permutation(n)
    o1, l1 = fwd(q, k, v, 1.0 / np.sqrt(d), MaskSpec())
    o2, l2 = fwd(q, k[perm], v[perm], 1.0 / np.sqrt(d), MaskSpec())
    return max(np.abs(o1 - o2).max(), np.abs(l1 - l2).max())


def finite_differences(fwd, bwd, n, d, spec, rng, h=1e-5):
    """Relative error of the analytic gradient of L = sum(O * dO) vs central differences."""
    q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
    scale = 1.0 / np.sqrt(d)

    def loss(qq, kk, vv):
        o, _ = fwd(qq, kk, vv, scale, spec)
        return float((o * do).sum())

    grads = bwd(q, k, v, do, scale, spec)
    worst = 0.0
    for which, g in enumerate(grads):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            num[idx] = (lp - lm) / (2 * h)
        denom = max(np.abs(num).max(), 1e-12)
        worst = max(worst, np.abs(num - g).max() / denom)
    return worst
