"""The oracle pinned to facts that do not come from the oracle itself (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import attention, block_index, loops
from oracle.mask import MaskSpec, candidate_col_array, candidate_cols, live_matrix
from tests import oracle_pins as pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# small-N mask family: block 4 so dilation / stride patterns appear at N <= 64
SMALL_SPECS = {
    "dense": MaskSpec(),
    "causal": MaskSpec(causal=True),
    "window": MaskSpec(window=5),
    "causal_window": MaskSpec(causal=True, window=6),
    "causal_window_strided": MaskSpec(causal=True, window=3, stride=3, stride_phase=1, block=4),
    "causal_window_dilated": MaskSpec(causal=True, window=14, dilation=2, dilation_near=2, block=4),
    "dilated_only": MaskSpec(dilation=3, dilation_near=1, block=4),
    "strided_only": MaskSpec(causal=True, stride=2, stride_phase=0, block=4),
    "causal_window_global": MaskSpec(causal=True, window=4, global_tokens=8, block=4),
    "window_global": MaskSpec(window=3, global_tokens=4, block=4),
    "causal_window_relstride": MaskSpec(causal=True, window=3, stride=3, stride_phase=0,
                                        stride_relative=True, block=4),
    "relstride_noncausal": MaskSpec(stride=2, stride_phase=1, stride_relative=True, block=4),
    "causal_window_fardil": MaskSpec(causal=True, window=5, dilation=3, dilation_far=True, block=4),
}

fwd_full = attention.forward_head
bwd_full = attention.backward_head


def rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- mask predicate
def test_mask_hand_examples():
    n = 20
    # causal: diagonal included
    live = live_matrix([5], [4, 5, 6], n, MaskSpec(causal=True))
    assert live.tolist() == [[True, True, False]]
    # window inclusive at W, dead at W + 1, both sides when not causal
    live = live_matrix([10], [6, 7, 13, 14], n, MaskSpec(window=3))
    assert live.tolist() == [[False, True, True, False]]
    # block dilation: block 4, near 2, dilation 2 -> block distance 0,1,2,4 live; 3 dead
    live = live_matrix([19], [19, 15, 11, 7, 3], n, MaskSpec(dilation=2, dilation_near=2, block=4))
    assert live.tolist() == [[True, True, True, False, True]]
    # strided: key blocks with kb % 3 == 1 (block 4): keys 4..7 and 16..19
    live = live_matrix([19], [0, 4, 7, 8, 16], n, MaskSpec(stride=3, stride_phase=1, block=4))
    assert live.tolist() == [[False, True, True, False, True]]
    # union: window OR strided, intersected with causal
    spec = MaskSpec(causal=True, window=2, stride=3, stride_phase=1, block=4)
    live = live_matrix([19], [17, 16, 5, 12, 20], 21, spec)
    assert live.tolist() == [[True, True, True, False, False]]
    # out of range entries are dead
    assert not live_matrix([3], [7], 5, MaskSpec()).any()
    # global tokens (G = 4): global keys visible from every query, a global
    # query sees every key; window 2 elsewhere; causal on top when set
    spec = MaskSpec(window=2, global_tokens=4)
    live = live_matrix([15], [0, 3, 4, 12, 13, 17, 18], 20, spec)
    assert live.tolist() == [[True, True, False, False, True, True, False]]
    live = live_matrix([2], [0, 9, 19], 20, spec)
    assert live.tolist() == [[True, True, True]]
    live = live_matrix([2, 15], [0, 9, 19], 20, MaskSpec(causal=True, window=2, global_tokens=4))
    assert live.tolist() == [[True, False, False], [True, False, False]]
    # relative strided (block 4, stride 3, phase 0): query block 4 keeps key
    # blocks 4, 1 (distance 0, 3) and, not causal, 7 (distance -3)
    spec = MaskSpec(stride=3, stride_phase=0, stride_relative=True, block=4)
    live = live_matrix([17], [17, 4, 7, 8, 12, 28, 24], 32, spec)
    assert live.tolist() == [[True, True, True, False, False, True, False]]
    # phase 1 keeps distances 1, 4, -2, -5 (mod 3 = 1)
    spec = MaskSpec(stride=3, stride_phase=1, stride_relative=True, block=4)
    live = live_matrix([17], [12, 0, 24, 17], 32, spec)
    assert live.tolist() == [[True, True, True, False]]
    # far dilation (block 4, dilation 3): dense window 2 plus key blocks at
    # block distance 0, 3, 6, ... anywhere
    spec = MaskSpec(causal=True, window=2, dilation=3, dilation_far=True, block=4)
    live = live_matrix([29], [27, 26, 25, 17, 16, 12, 5, 4], 32, spec)
    assert live.tolist() == [[True, False, False, True, True, False, True, True]]


@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
def test_vector_predicate_matches_scalar(name):
    spec = SMALL_SPECS[name]
    n = 37
    idx = np.arange(-2, n + 3)
    m = live_matrix(idx, idx, n, spec)
    ref = np.array([[loops.live_scalar(int(i), int(j), n, spec) for j in idx] for i in idx])
    assert (m == ref).all()


@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
def test_candidate_span_only_drops_dead_keys(name):
    spec = SMALL_SPECS[name]
    n = 60
    for r0 in range(0, n, 7):
        r1 = min(n, r0 + 7)
        c0, c1 = candidate_cols(r0, r1, n, spec)
        live = live_matrix(np.arange(r0, r1), np.arange(n), n, spec)
        outside = np.ones(n, dtype=bool)
        outside[c0:c1] = False
        assert not live[:, outside].any()
        kept = candidate_col_array(r0, r1, n, spec)
        assert len(np.unique(kept)) == len(kept)
        outside = np.ones(n, dtype=bool)
        outside[kept] = False
        assert not live[:, outside].any()


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
def test_uniform_attention_when_q_is_zero(name):
    assert pins.uniform_q_zero(fwd_full, 29, 6, SMALL_SPECS[name], rng(1)) < 1e-12


def test_causal_row_zero():
    assert pins.causal_row0(fwd_full, 17, 8, rng(2)) < 1e-12


def test_one_hot_dominant_row():
    assert pins.one_hot_dominant(fwd_full, 8, 16, rng(3)) < 1e-15


@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
def test_constant_v(name):
    assert pins.constant_v(fwd_full, bwd_full, 23, 5, SMALL_SPECS[name], rng(4)) < 1e-12


@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
def test_probability_rows_sum_to_one(name):
    spec = SMALL_SPECS[name]
    r = rng(5)
    q, k = r.standard_normal((31, 4)), r.standard_normal((31, 4))
    p = attention.probabilities(q, k, 0.5, spec)
    has = live_matrix(np.arange(31), np.arange(31), 31, spec).any(axis=1)
    assert np.abs(p[has].sum(axis=1) - 1).max() < 1e-13
    assert (p[~has] == 0).all()
    assert (p >= 0).all()


@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
def test_gradient_sum_invariants(name):
    assert pins.gradient_invariants(fwd_full, bwd_full, 26, 5, SMALL_SPECS[name], rng(6)) < 1e-11


def test_permutation_invariance_dense():
    assert pins.permutation_invariance(fwd_full, 40, 8, rng(7)) < 1e-12


@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
def test_finite_differences(name):
    # N <= 8 rows with block 4 would hide the patterns; use N = 8, d = 3
    assert pins.finite_differences(fwd_full, bwd_full, 8, 3, SMALL_SPECS[name], rng(8)) < 1e-6


# ---------------------------------------------------------------- restatements
@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
def test_scalar_loops_agree(name):
    spec = SMALL_SPECS[name]
    r = rng(9)
    n, d = 16, 3
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    o, lse = fwd_full(q, k, v, 0.6, spec)
    o2, lse2 = loops.forward_loops(q.tolist(), k.tolist(), v.tolist(), 0.6, spec)
    assert np.abs(o - o2).max() < 1e-12
    fin = np.isfinite(lse)
    assert (np.isfinite(lse2) == fin).all() and np.abs(lse[fin] - lse2[fin]).max(initial=0) < 1e-12
    g = bwd_full(q, k, v, do, 0.6, spec)
    g2 = loops.backward_loops(q.tolist(), k.tolist(), v.tolist(), do.tolist(), 0.6, spec)
    for a, b in zip(g, g2):
        assert np.abs(a - b).max() < 1e-12


@pytest.mark.parametrize("name", sorted(SMALL_SPECS))
@pytest.mark.parametrize("n,blk", [(50, 8), (61, 16), (130, 128)])
def test_tiled_online_softmax_agrees(name, n, blk):
    spec = SMALL_SPECS[name]
    r = rng(10)
    q, k, v = (r.standard_normal((n, 8)) for _ in range(3))
    o, lse = fwd_full(q, k, v, 0.35, spec)
    o2, lse2 = loops.forward_tiled(q, k, v, 0.35, spec, block=blk)
    assert np.abs(o - o2).max() < 1e-12
    fin = np.isfinite(lse)
    assert (np.isfinite(lse2) == fin).all()
    assert np.abs(lse[fin] - lse2[fin]).max(initial=0) < 1e-12


@pytest.mark.parametrize("spec", [
    MaskSpec(causal=True),
    MaskSpec(causal=True, window=100, stride=4, stride_phase=0, block=32),
    MaskSpec(causal=True, window=150, dilation=2, dilation_near=2, block=32),
    MaskSpec(window=90),
    MaskSpec(causal=True, window=70, global_tokens=64, block=32),
    MaskSpec(window=50, global_tokens=96, block=32),
])
def test_chunked_evaluation_matches_full(spec):
    r = rng(11)
    n, d = 333, 8
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    o, lse = fwd_full(q, k, v, 0.3, spec)
    o2, lse2 = attention.forward_rows(q, k, v, 0.3, spec, chunk=50)
    assert np.abs(o - o2).max() < 1e-12 and np.abs(lse - lse2).max() < 1e-12
    dq, dk, dv = bwd_full(q, k, v, do, 0.3, spec)
    rows = np.array([0, 1, 77, 200, 332])
    cols = np.array([0, 5, 128, 331, 332])
    dq2, dk2, dv2 = attention.backward_sampled(q, k, v, do, 0.3, spec, rows, cols, chunk=64)
    assert np.abs(dq[rows] - dq2).max() < 1e-12
    assert np.abs(dk[cols] - dk2).max() < 1e-12
    assert np.abs(dv[cols] - dv2).max() < 1e-12


@pytest.mark.parametrize("spec", [
    MaskSpec(causal=True),
    MaskSpec(causal=True, window=60, dilation=2, dilation_far=True, block=32),
])
def test_row_stats_of_tail_rows_give_tail_columns(spec):
    # under a causal mask, column j of P involves only rows i >= j: the
    # statistics of the rows from min(cols) on reproduce the full-materialisation
    # gradients of those key columns, and match the full statistics there
    r = rng(13)
    n, d = 333, 8
    q, k, v, do = (r.standard_normal((n, d)) for _ in range(4))
    dq, dk, dv = bwd_full(q, k, v, do, 0.3, spec)
    cols = np.array([250, 251, 300, 331, 332])
    tail = np.arange(cols.min(), n)
    stats = attention.row_stats(q, k, v, do, 0.3, spec, chunk=40, rows=tail)
    full = attention.row_stats(q, k, v, do, 0.3, spec, chunk=40)
    assert np.abs(stats[0][tail] - full[0][tail]).max() < 1e-12
    assert np.abs(stats[1][tail] - full[1][tail]).max() < 1e-12
    assert (stats[0][:cols.min()] == -np.inf).all() and (stats[1][:cols.min()] == 0).all()
    _, dk2, dv2 = attention.backward_sampled(q, k, v, do, 0.3, spec, [], cols, stats=stats)
    assert np.abs(dk[cols] - dk2).max() < 1e-12
    assert np.abs(dv[cols] - dv2).max() < 1e-12


def test_empty_rows_are_zero_not_nan():
    # strided-only causal mask at block 4 with phase 1: rows 0..3 have no live key
    spec = MaskSpec(causal=True, stride=2, stride_phase=1, block=4)
    r = rng(12)
    q, k, v, do = (r.standard_normal((12, 3)) for _ in range(4))
    o, lse = fwd_full(q, k, v, 0.5, spec)
    assert (o[:4] == 0).all() and (lse[:4] == -np.inf).all() and np.isfinite(o).all()
    g = bwd_full(q, k, v, do, 0.5, spec)
    assert all(np.isfinite(x).all() for x in g)


# ---------------------------------------------------------------- block index
def _counts(idx):
    kind = idx["kind"]
    return idx["nnz"], int((kind == 0).sum()), int((kind == 1).sum())


def test_golden_tile_counts():
    gold = json.load(open(os.path.join(GOLDEN, "tile_counts.json")))
    cases = {
        "causal_n4096": (4096, MaskSpec(causal=True)),
        "causal_n16384": (16384, MaskSpec(causal=True)),
        "window1024_strided8_n32768": (32768, MaskSpec(causal=True, window=1024, stride=8)),
        "window4096_dilation2_n131072": (131072, MaskSpec(causal=True, window=4096, dilation=2, dilation_near=2)),
        "window8192_global512_n32768": (32768, MaskSpec(causal=True, window=8192, global_tokens=512)),
        "window1024_relstride8_n32768": (32768, MaskSpec(causal=True, window=1024, stride=8, stride_relative=True)),
        "window4096_fardilation2_n16384": (16384, MaskSpec(causal=True, window=4096, dilation=2, dilation_far=True)),
    }
    for key, (n, spec) in cases.items():
        idx = block_index.build(n, spec)
        g = gold[key]
        assert _counts(idx) == (g["nnz"], g["full"], g["partial"]), key


def test_closed_form_counts_formulas():
    # the same numbers, recomputed from the closed forms in the fixture
    assert sum(range(1, 33)) == 528 and sum(range(1, 129)) == 8256
    win = sum(qb + 1 for qb in range(8)) + 248 * 9
    strided = sum((qb - 9) // 8 + 1 for qb in range(9, 256))
    assert (win, strided, win + strided) == (2268, 3937, 6205)
    dil = 992 * 18 + sum(1 + min(qb, 1) + qb // 2 for qb in range(32))
    assert dil == 18159
    # causal window of w = 64 blocks plus gb = 4 global blocks: a query block
    # sees [0, qb] while its window reaches the global blocks, else 65 + 4
    def glob(nb, w=64, gb=4):
        return sum(qb + 1 if qb - w <= gb - 1 else w + 1 + gb for qb in range(nb))
    assert (glob(1024), glob(256)) == (68310, 15318)
    # causal window of w blocks plus key blocks at block distances divisible
    # by p beyond it (relative strides of p = 8, far dilation p = 2)
    def beyond(nb, w, p):
        return sum(min(qb, w) + 1 + sum(1 for dd in range(w + 1, qb + 1) if dd % p == 0)
                   for qb in range(nb))
    assert (beyond(256, 8, 8), beyond(1024, 32, 2), beyond(128, 32, 2)) == (5988, 278784, 5952)
    # partial: the diagonal plus the window edge kb = qb - 64 when it is not global
    assert (1024 + sum(1 for qb in range(1024) if qb - 64 >= 4),
            256 + sum(1 for qb in range(256) if qb - 64 >= 4)) == (1980, 444)


@pytest.mark.parametrize("n,spec", [
    (1000, MaskSpec(causal=True, window=200)),
    (1500, MaskSpec(window=300, dilation=2, dilation_near=1)),
    (2100, MaskSpec(causal=True, window=129, dilation=3, dilation_near=2)),
    (2000, MaskSpec(causal=True, window=300, global_tokens=256)),
    (1700, MaskSpec(window=200, global_tokens=384)),
])
def test_window_shortcut_matches_full_scan(n, spec):
    a = block_index.classify(n, spec, prune=True)
    b = block_index.classify(n, spec, prune=False)
    assert (a == b).all()


@pytest.mark.parametrize("n", [1, 127, 128, 129, 300, 1000])
def test_tail_tiles_are_partial_and_structure_consistent(n):
    spec = MaskSpec(causal=True, window=200, stride=3, stride_phase=2)
    idx = block_index.build(n, spec)
    nb = idx["n_blocks"]
    assert nb == (n + 127) // 128
    kinds = block_index.classify(n, spec)
    if n % 128:
        assert not (kinds[-1] == block_index.FULL).any()
        assert not (kinds[:, -1] == block_index.FULL).any()
    # CSR and CSC describe the same set of tiles with the same kinds
    csr = {(qb, int(kb)): int(t) for qb in range(nb)
           for kb, t in zip(idx["col_idx"][idx["row_ptr"][qb]:idx["row_ptr"][qb + 1]],
                            idx["kind"][idx["row_ptr"][qb]:idx["row_ptr"][qb + 1]])}
    csc = {(int(qb), kb): int(t) for kb in range(nb)
           for qb, t in zip(idx["row_idx"][idx["col_ptr"][kb]:idx["col_ptr"][kb + 1]],
                            idx["kind_t"][idx["col_ptr"][kb]:idx["col_ptr"][kb + 1]])}
    assert csr == csc
    lens = np.diff(idx["row_ptr"])
    assert sorted(idx["q_order"].tolist()) == list(range(nb))
    # pairs (positions 2r, 2r + 1) come by descending count of their first block
    firsts = idx["q_order"][0:nb - nb % 2:2]
    assert all(lens[a] >= lens[b] for a, b in zip(firsts, firsts[1:]))


def test_smoke_golden_shape():
    g = json.load(open(os.path.join(GOLDEN, "smoke_shape.json")))
    B, N, H, d = g["input_shape"]
    r = rng(13)
    q, k, v = (r.standard_normal((N, d)) for _ in range(3))
    o, _ = fwd_full(q, k, v, d ** -0.5, MaskSpec(causal=g["causal"]))
    assert [B, o.shape[0], H, o.shape[1]] == g["output_shape"]


# ---------------------------------------------------------------- negative controls
def _mutant_zero_mask(q, k, v, scale, spec):
    """Masking by multiplying scores by zero instead of -inf (a page's sketch does this)."""
    n = q.shape[0]
    live = live_matrix(np.arange(n), np.arange(n), n, spec)
    s = scale * (q @ k.T) * live
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return (e / e.sum(axis=1, keepdims=True)) @ v, m[:, 0] + np.log(e.sum(axis=1))


def _mutant_lse_sum(q, k, v, scale, spec, block=4):
    """Online recurrence that adds log-sums and divides without the running-max rescale."""
    n = q.shape[0]
    o = np.zeros_like(v)
    lse_out = np.zeros(n)
    for r0 in range(0, n, block):
        rows = np.arange(r0, min(n, r0 + block))
        acc = np.zeros((len(rows), v.shape[1]))
        lse = np.zeros(len(rows))
        for c0 in range(0, n, block):
            cols = np.arange(c0, min(n, c0 + block))
            s = np.where(live_matrix(rows, cols, n, spec), scale * q[rows] @ k[cols].T, -np.inf)
            mx = np.where(np.isfinite(s.max(axis=1)), s.max(axis=1), 0)
            p = np.exp(s - mx[:, None])
            lse = lse + np.log(p.sum(axis=1) + 1e-10)
            acc = acc + (p @ v[cols]) / np.exp(lse)[:, None]
        o[rows] = acc
        lse_out[rows] = lse
    return o, lse_out


def _mutant_no_scale(q, k, v, scale, spec):
    return fwd_full(q, k, v, 1.0, spec)


def _mutant_strict_causal(q, k, v, scale, spec):
    n = q.shape[0]
    s = np.where(np.tril(np.ones((n, n), bool), -1) | ~np.array(spec.causal), scale * q @ k.T, -np.inf)
    m = s.max(axis=1)
    m = np.where(np.isfinite(m), m, 0)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    return (e / np.where(l > 0, l, 1)[:, None]) @ v, m + np.log(np.where(l > 0, l, 1))


def _mutant_bwd_sign(q, k, v, do, scale, spec):
    p = attention.probabilities(q, k, scale, spec)
    dp = do @ v.T
    ds = p * (dp + (p * dp).sum(axis=1)[:, None])
    return scale * ds @ k, scale * ds.T @ q, p.T @ do


def _mutant_bwd_transposed(q, k, v, do, scale, spec):
    p = attention.probabilities(q, k, scale, spec)
    dp = do @ v.T
    ds = p * (dp - (p * dp).sum(axis=1)[:, None])
    return scale * ds @ k, scale * ds.T @ q, p @ do


def _mutant_bwd_no_scale(q, k, v, do, scale, spec):
    dq, dk, dv = bwd_full(q, k, v, do, scale, spec)
    return dq / scale, dk / scale, dv


@pytest.mark.parametrize("mutant", [_mutant_zero_mask, _mutant_lse_sum, _mutant_no_scale,
                                    _mutant_strict_causal])
def test_forward_mistakes_fail_a_pin(mutant):
    r = rng(20)
    errs = [
        max(pins.uniform_q_zero(mutant, 29, 6, s, r) for s in SMALL_SPECS.values()),
        pins.causal_row0(mutant, 17, 8, r),
        pins.permutation_invariance(mutant, 40, 8, r),
    ]
    # the mutant must also disagree with the scalar loops on random inputs
    q, k, v = (r.standard_normal((12, 3)) for _ in range(3))
    o_m, _ = mutant(q, k, v, 0.6, MaskSpec(causal=True))
    o_l, _ = loops.forward_loops(q.tolist(), k.tolist(), v.tolist(), 0.6, MaskSpec(causal=True))
    errs.append(np.abs(o_m - o_l).max())
    assert max(errs) > 1e-3, errs


@pytest.mark.parametrize("mutant", [_mutant_bwd_sign, _mutant_bwd_transposed, _mutant_bwd_no_scale])
def test_backward_mistakes_fail_a_pin(mutant):
    r = rng(21)
    spec = MaskSpec(causal=True, window=6)
    errs = [
        pins.gradient_invariants(fwd_full, mutant, 26, 5, spec, r),
        pins.finite_differences(fwd_full, mutant, 6, 2, spec, r),
    ]
    assert max(errs) > 1e-3, errs


# ---------------------------------------------------------------- bit-packed masks
def _random_bits(n, seed, p=0.5):
    return np.random.default_rng(seed).random((n, n)) < p


def test_bitmask_hand_example():
    from tiled_exact_attention_flash_gb300.inputs import pack_bitmask
    live = np.zeros((8, 8), dtype=bool)
    live[5, [0, 2, 5, 7]] = True
    live[1, 1] = True
    b = pack_bitmask(live)
    spec = MaskSpec(bitmask=b)
    assert live_matrix([5], range(8), 8, spec).tolist() == [[True, False, True, False, False, True, False, True]]
    # AND-ed with causal and with the pattern parts
    spec = MaskSpec(causal=True, bitmask=b)
    assert live_matrix([5], range(8), 8, spec).tolist() == [[True, False, True, False, False, True, False, False]]
    spec = MaskSpec(window=2, bitmask=b)
    assert live_matrix([5], range(8), 8, spec).tolist() == [[False] * 5 + [True, False, True]]
    # the packed layout itself: row 5 is one word with bits 0, 2, 5, 7
    assert int.from_bytes(b[4 * 5:4 * 6], "little") == 1 | 4 | 32 | 128


BIT_CASES = [(37, {}), (37, {"causal": True}), (41, {"causal": True, "window": 6}),
             (29, {"window": 4, "stride": 2, "stride_phase": 1, "block": 4})]


@pytest.mark.parametrize("case", range(len(BIT_CASES)))
def test_bitmask_scalar_and_closed_forms(case):
    from tiled_exact_attention_flash_gb300.inputs import pack_bitmask
    n, fields = BIT_CASES[case]
    bits = _random_bits(n, 100 + case)
    spec = MaskSpec(bitmask=pack_bitmask(bits), **fields)
    idx = np.arange(-2, n + 3)
    m = live_matrix(idx, idx, n, spec)
    ref = np.array([[loops.live_scalar(int(i), int(j), n, spec) for j in idx] for i in idx])
    assert (m == ref).all()
    # the bits act as an AND on top of the mask without them
    plain = live_matrix(np.arange(n), np.arange(n), n, MaskSpec(**fields))
    assert (live_matrix(np.arange(n), np.arange(n), n, spec) == (plain & bits)).all()
    # Q = 0: O_i is the mean of v_j over j with bit and mask set, counted from the
    # boolean matrix the bits were packed from
    r = rng(case)
    q = np.zeros((n, 5))
    k, v = r.standard_normal((n, 5)), r.standard_normal((n, 5))
    o, lse = fwd_full(q, k, v, 0.4, spec)
    for i in range(n):
        sel = plain[i] & bits[i]
        if sel.any():
            assert np.abs(o[i] - v[sel].mean(axis=0)).max() < 1e-12
            assert abs(lse[i] - np.log(sel.sum())) < 1e-12
        else:
            assert lse[i] == -np.inf and not o[i].any()


def test_bitmask_finite_differences():
    from tiled_exact_attention_flash_gb300.inputs import pack_bitmask
    bits = _random_bits(8, 5, 0.6)
    spec = MaskSpec(causal=True, bitmask=pack_bitmask(bits))
    assert pins.finite_differences(fwd_full, bwd_full, 8, 3, spec, rng(9)) < 1e-6


@pytest.mark.parametrize("n,fields", [(300, {}), (300, {"causal": True, "window": 100}),
                                      (519, {"causal": True})])
def test_bitmask_index_tiles_hold_the_live_entries(n, fields):
    # every partial tile that the bits cut carries exactly its live entries,
    # unpacked here with numpy's unpackbits (independent of the packing code)
    from tiled_exact_attention_flash_gb300.inputs import document_bitmask, document_lengths
    spec = MaskSpec(bitmask=document_bitmask(n, document_lengths(n, n, 60)), **fields)
    idx = block_index.build(n, spec)
    full = live_matrix(np.arange(n), np.arange(n), n, spec)
    plain = live_matrix(np.arange(n), np.arange(n), n, MaskSpec(**fields))
    nb = idx["n_blocks"]

    def unpack(words):
        return np.unpackbits(words.astype("<u4").view(np.uint8).reshape(128, 16), axis=1,
                             bitorder="little").astype(bool)

    def tile(mat, qb, kb):
        t = np.zeros((128, 128), dtype=bool)
        sub = mat[qb * 128:(qb + 1) * 128, kb * 128:(kb + 1) * 128]
        t[:sub.shape[0], :sub.shape[1]] = sub
        return t
    slots = 0
    for qb in range(nb):
        for e in range(idx["row_ptr"][qb], idx["row_ptr"][qb + 1]):
            kb, slot = int(idx["col_idx"][e]), int(idx["bit_slot"][e])
            cut = not np.array_equal(tile(full, qb, kb), tile(plain, qb, kb))
            assert (slot >= 0) == (cut and idx["kind"][e] == 1)
            if slot >= 0:
                slots += 1
                assert np.array_equal(unpack(idx["bits"][slot * 512:(slot + 1) * 512]), tile(full, qb, kb))
                assert np.array_equal(unpack(idx["bits_t"][slot * 512:(slot + 1) * 512]), tile(full, qb, kb).T)
    assert slots == idx["n_bit_tiles"]
    # the CSC entries point at the same slots
    for kb in range(nb):
        for e in range(idx["col_ptr"][kb], idx["col_ptr"][kb + 1]):
            qb = int(idx["row_idx"][e])
            row = np.nonzero(idx["col_idx"][idx["row_ptr"][qb]:idx["row_ptr"][qb + 1]] == kb)[0][0]
            assert idx["bit_slot_t"][e] == idx["bit_slot"][idx["row_ptr"][qb] + row]


# ---------------------------------------------------------------- packed documents (varlen)
def test_documents_hand_example():
    starts = (0, 3, 7, 10)
    spec = MaskSpec(causal=True, doc_starts=starts)
    # token 8 (third sequence, positions 7..9) sees 7 and 8 only
    assert live_matrix([8], range(10), 10, spec).tolist() == [[False] * 7 + [True, True, False]]
    # without causal: the whole first sequence for token 1
    spec = MaskSpec(doc_starts=starts)
    assert live_matrix([1], range(10), 10, spec).tolist() == [[True, True, True] + [False] * 7]
    with pytest.raises(ValueError):
        live_matrix([1], [1], 10, MaskSpec(doc_starts=(0, 5, 5, 10)))


@pytest.mark.parametrize("fields", [{}, {"causal": True}, {"causal": True, "window": 5},
                                    {"window": 3, "stride": 2, "stride_phase": 0, "block": 4}])
def test_documents_equal_their_bitmask_and_scalar(fields):
    from tiled_exact_attention_flash_gb300.inputs import document_bitmask
    lens = [5, 1, 9, 13, 4, 8]
    n = sum(lens)
    starts = tuple(int(x) for x in np.cumsum([0] + lens))
    a = MaskSpec(doc_starts=starts, **fields)
    b = MaskSpec(bitmask=document_bitmask(n, lens), **fields)
    idx = np.arange(-2, n + 3)
    la = live_matrix(idx, idx, n, a)
    assert (la == live_matrix(idx, idx, n, b)).all()
    ref = np.array([[loops.live_scalar(int(i), int(j), n, a) for j in idx] for i in idx])
    assert (la == ref).all()


def test_packed_documents_equal_separate_sequences():
    # attention over packed sequences equals attention over each sequence
    # alone (outputs, LSE and all three gradients)
    lens = [17, 3, 30, 1, 12]
    n = sum(lens)
    starts = np.cumsum([0] + lens)
    r = rng(21)
    q, k, v, do = (r.standard_normal((n, 8)) for _ in range(4))
    spec = MaskSpec(causal=True, doc_starts=tuple(int(x) for x in starts))
    o, lse = fwd_full(q, k, v, 0.3, spec)
    dq, dk, dv = bwd_full(q, k, v, do, 0.3, spec)
    for a, e in zip(starts[:-1], starts[1:]):
        sl = slice(a, e)
        o1, l1 = fwd_full(q[sl], k[sl], v[sl], 0.3, MaskSpec(causal=True))
        g = bwd_full(q[sl], k[sl], v[sl], do[sl], 0.3, MaskSpec(causal=True))
        assert np.abs(o[sl] - o1).max() < 1e-12 and np.abs(lse[sl] - l1).max() < 1e-12
        for got, ref in zip((dq, dk, dv), g):
            assert np.abs(got[sl] - ref).max() < 1e-12


def test_documents_index_equals_bitmask_index():
    from tiled_exact_attention_flash_gb300.inputs import document_bitmask, document_lengths
    n = 700
    lens = document_lengths(n, 4, 90)
    starts = tuple(int(x) for x in np.cumsum([0] + lens))
    # a block-level part (strides) keeps the packed tiling for the documents
    # given as offsets, so both builds tile the packed axis
    a = block_index.build(n, MaskSpec(causal=True, stride=3, doc_starts=starts))
    b = block_index.build(n, MaskSpec(causal=True, stride=3, bitmask=document_bitmask(n, lens)))
    assert a["n_bit_tiles"] > 0
    for key in a:
        assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), key


def test_sequence_tiles_hand_example():
    # sequences [0,1) [1,201) [201,208) [208,337) [337,401): tiles start at
    # each sequence's first token, 128 tokens apart, causal pairs only inside
    # a sequence (1 + 3 + 1 + 3 + 1 = 9), every one cut by the diagonal or a
    # sequence end
    spec = MaskSpec(causal=True, doc_starts=(0, 1, 201, 208, 337, 401))
    r = block_index.build(401, spec)
    assert r["tile_start"].tolist() == [0, 1, 129, 201, 208, 336, 337]
    assert r["tile_seq0"].tolist() == [0, 1, 1, 201, 208, 208, 337]
    assert r["tile_seq_len"].tolist() == [1, 200, 200, 7, 129, 129, 64]
    assert r["nnz"] == 9 and (r["kind"] == block_index.PARTIAL).all()
    assert r["row_ptr"].tolist() == [0, 1, 2, 4, 5, 6, 8, 9]
    assert r["col_idx"].tolist() == [0, 1, 1, 2, 3, 4, 4, 5, 6]
    assert r["n_bit_tiles"] == 0
    # pairs of neighbouring tiles from each sequence's end: (2, 1) and (5, 4),
    # longest first (counts 2 and 2, tie by id), then the single tiles 0, 3, 6
    assert r["q_order"].tolist() == [2, 1, 5, 4, 0, 3, 6]


@pytest.mark.parametrize("causal,window", [(True, None), (False, None), (True, 150), (False, 70)])
def test_sequence_tiles_are_the_sequences_own_tiles(causal, window):
    # the per-sequence index is the block-diagonal concatenation of every
    # sequence's index built on its own (the plain single-sequence builder)
    lens = [1, 300, 128, 129, 7, 511]
    starts = tuple(int(x) for x in np.cumsum([0] + lens))
    spec = MaskSpec(causal=causal, window=window, doc_starts=starts)
    got = block_index.build(starts[-1], spec)
    base, nnz = 0, 0
    for s0, ln in zip(starts[:-1], lens):
        own = block_index.build(ln, MaskSpec(causal=causal, window=window))
        nb = own["n_blocks"]
        rows = slice(base, base + nb)
        assert (got["tile_start"][rows] == s0 + 128 * np.arange(nb)).all()
        assert (got["tile_seq_len"][rows] == ln).all() and (got["tile_seq0"][rows] == s0).all()
        for qb in range(nb):
            a, e = got["row_ptr"][base + qb], got["row_ptr"][base + qb + 1]
            oa, oe = own["row_ptr"][qb], own["row_ptr"][qb + 1]
            assert (got["col_idx"][a:e] == base + own["col_idx"][oa:oe]).all()
            assert (got["kind"][a:e] == own["kind"][oa:oe]).all()
        base += nb
        nnz += own["nnz"]
    assert got["n_blocks"] == base and got["nnz"] == nnz


def test_documents_with_block_patterns_keep_packed_tiles():
    # block-level parts (dilation, strides, global tokens) and bit-packed
    # masks are defined on the packed axis's 128-token blocks: those masks
    # keep the packed tiling with bit tiles
    starts = (0, 100, 300)
    for spec in (MaskSpec(causal=True, stride=2, doc_starts=starts),
                 MaskSpec(causal=True, window=50, global_tokens=128, doc_starts=starts)):
        r = block_index.build(300, spec)
        assert not block_index.sequence_tiled(spec) and r["tile_start"].size == 0
        assert r["n_blocks"] == 3


def test_shared_pairs_hand_example():
    # six 128-token blocks; blocks of the same parity attend to each other's
    # keys only: 0, 2, 4 list key blocks {0, 2, 4}, and 1, 3, 5 list {1, 3, 5}.
    # Visited in id order (equal counts): 0 pairs with 2 (3 common tiles; 1
    # shares none), 1 with 3, then 4 and 5 share nothing with any unpaired
    # block within reach and are paired as leftovers.  Longest-first order
    # alone would have paired 0 with 1 and 2 with 3, which share nothing.
    from tiled_exact_attention_flash_gb300.inputs import pack_bitmask
    par = np.arange(768) // 128 % 2
    spec = MaskSpec(bitmask=pack_bitmask(par[:, None] == par[None, :]))
    r = block_index.build(768, spec)
    assert np.diff(r["row_ptr"]).tolist() == [3] * 6
    assert r["q_order"].tolist() == [0, 2, 1, 3, 4, 5]


@pytest.mark.parametrize("n", [129, 1000, 1024, 2100])
def test_shared_pairs_of_causal_masks_are_longest_first(n):
    # causal block qb lists qb + 1 tiles: its best partner is qb - 1, so the
    # pairs are (nb-1, nb-2), (nb-3, nb-4), ... -- plain longest-first order
    r = block_index.build(n, MaskSpec(causal=True, window=n))
    lens = np.diff(r["row_ptr"])
    assert r["q_order"].tolist() == sorted(range(len(lens)), key=lambda b: (-lens[b], b))
