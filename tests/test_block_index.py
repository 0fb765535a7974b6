"""The C++ block-index builder is bit-exact with the oracle's brute-force build."""
import numpy as np
import pytest

from tests.oracle_cache import oracle_index
from tiled_exact_attention_flash_gb300 import api
from tiled_exact_attention_flash_gb300.inputs import WORKLOADS

ARRAYS = ("row_ptr", "col_idx", "kind", "col_ptr", "row_idx", "kind_t", "q_order", "k_order")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tests.libbuild import ensure_built
    ensure_built()


def compare(n, fields):
    ref = oracle_index(n, tuple(sorted(fields.items())))
    got = api.build_block_index(api.Mask(**fields), n)
    assert got.nnz == ref["nnz"]
    assert got.header.n_q_blocks == ref["n_blocks"] == got.header.n_k_blocks
    names = ARRAYS
    if fields.get("bitmask") is not None:
        assert got.header.n_bit_tiles == ref["n_bit_tiles"]
        names = ARRAYS + ("bit_slot", "bit_slot_t", "bits", "bits_t")
    assert got.sequence_tiles == (ref["tile_start"].size > 0)
    if got.sequence_tiles:
        names = names + ("tile_start", "tile_seq0", "tile_seq_len")
    for name in names:
        a, b = got.host[name], ref[name]
        assert a.dtype == b.dtype, name
        assert np.array_equal(a, b), name
    assert api.check_block_index(got) == api.OK
    return got


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5, 6, 7, 9, 10])
def test_workload_indices_bit_exact(cid):
    w = WORKLOADS[cid]
    compare(w.N, w.mask_fields())


def test_far_dilation_index_bit_exact_at_32k():
    # workload 8's mask (dense window 4096, even block distances at any
    # range): the brute-force build scans every tile, so it is compared at
    # N = 32768 (20352 live tiles per head); the full-size counts are pinned
    # by hand in tests/golden/tile_counts.json
    w = WORKLOADS[8]
    got = compare(32768, w.mask_fields())
    assert got.nnz == 20352


MASKS = [
    {},
    {"causal": True},
    {"window": 300},
    {"causal": True, "window": 1},
    {"causal": True, "window": 129, "stride": 3, "stride_phase": 1},
    {"causal": True, "window": 700, "dilation": 2, "dilation_near": 2},
    {"window": 513, "dilation": 3, "dilation_near": 1},
    {"dilation": 2, "dilation_near": 0},
    {"causal": True, "stride": 4, "stride_phase": 3},
    {"stride": 2, "stride_phase": 0, "window": 64},
    {"causal": True, "window": 200, "global_tokens": 128},
    {"window": 130, "global_tokens": 256},
    {"causal": True, "global_tokens": 384},
    {"causal": True, "window": 300, "dilation": 2, "dilation_near": 1, "global_tokens": 128},
    {"causal": True, "window": 200, "stride": 3, "stride_phase": 0, "stride_relative": True},
    {"stride": 2, "stride_phase": 1, "stride_relative": True},
    {"causal": True, "window": 300, "dilation": 3, "dilation_far": True},
    {"window": 129, "dilation": 2, "dilation_far": True},
]


@pytest.mark.parametrize("n", [1, 5, 127, 128, 129, 255, 256, 1000, 2047])
@pytest.mark.parametrize("mi", range(len(MASKS)))
def test_small_indices_bit_exact(n, mi):
    compare(n, MASKS[mi])


def test_random_indices_bit_exact():
    rng = np.random.default_rng(7)
    for _ in range(25):
        n = int(rng.integers(1, 2049))
        f = {"causal": bool(rng.integers(0, 2))}
        if rng.integers(0, 2):
            f["window"] = int(rng.integers(0, 1500))
        if rng.integers(0, 2):
            f["dilation"] = int(rng.integers(1, 5))
            f["dilation_near"] = int(rng.integers(0, 4))
        if rng.integers(0, 2):
            s = int(rng.integers(1, 9))
            f["stride"] = s
            f["stride_phase"] = int(rng.integers(0, s))
        if rng.integers(0, 3) == 0:
            f["global_tokens"] = 128 * int(rng.integers(1, 5))
        if "stride" in f and rng.integers(0, 2):
            f["stride_relative"] = True
        if "dilation" in f and rng.integers(0, 2):
            f["dilation_far"] = True
        compare(n, f)


def test_pattern_indices_match_hand_counts():
    # global tokens, relative strides and far dilation at benchmark sizes,
    # against the counts derived by hand in tests/golden/tile_counts.json
    import json, os
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tile_counts.json")))
    cases = (("window8192_global512_n131072", 131072, dict(causal=True, window=8192, global_tokens=512)),
             ("window8192_global512_n32768", 32768, dict(causal=True, window=8192, global_tokens=512)),
             ("window1024_relstride8_n32768", 32768,
              dict(causal=True, window=1024, stride=8, stride_relative=True)),
             ("window4096_fardilation2_n131072", 131072,
              dict(causal=True, window=4096, dilation=2, dilation_far=True)),
             ("window4096_fardilation2_n16384", 16384,
              dict(causal=True, window=4096, dilation=2, dilation_far=True)))
    for key, n, fields in cases:
        idx = api.build_block_index(api.Mask(**fields), n)
        kind = idx.host["kind"]
        g = gold[key]
        assert (idx.nnz, int((kind == 0).sum()), int((kind == 1).sum())) == \
            (g["nnz"], g["full"], g["partial"]), key
        assert api.check_block_index(idx) == api.OK


@pytest.mark.parametrize("lens", [(1, 300, 128, 129, 7, 511), (5000,), (127, 1, 1, 2, 256)])
@pytest.mark.parametrize("fields", [{"causal": True}, {}, {"causal": True, "window": 150},
                                    {"window": 70}])
def test_sequence_tile_indices_bit_exact(lens, fields):
    # packed sequences with a causal / window mask are tiled per sequence,
    # bit-exact with the oracle's per-sequence build
    starts = tuple(int(x) for x in np.cumsum((0,) + lens))
    got = compare(starts[-1], dict(fields, doc_starts=starts))
    assert got.sequence_tiles and got.n_tiles == sum((n + 127) // 128 for n in lens)


def test_checker_rejects_corruption():
    idx = api.build_block_index(api.Mask(causal=True, window=500, stride=2), 2000)
    assert api.check_block_index(idx) == api.OK
    for name, pos, val in [("col_idx", 3, 99), ("kind", 0, 7), ("row_idx", 1, -1),
                           ("q_order", 0, 1), ("row_ptr", 2, 0)]:
        saved = idx.host[name][pos]
        idx.host[name][pos] = val
        assert api.check_block_index(idx) == api.ERR_INDEX, name
        idx.host[name][pos] = saved
    assert api.check_block_index(idx) == api.OK


@pytest.mark.parametrize("n,fields,seed", [
    (300, {}, 1), (519, {"causal": True}, 2), (1000, {"causal": True, "window": 200}, 3),
    (700, {"window": 130, "stride": 2, "stride_phase": 1}, 4),
    (640, {"causal": True, "global_tokens": 128, "window": 100}, 5)])
def test_bitmask_indices_bit_exact(n, fields, seed):
    from tiled_exact_attention_flash_gb300.inputs import (document_bitmask, document_lengths,
                                                          pack_bitmask)
    # packed documents, then a random element mask
    compare(n, dict(fields, bitmask=document_bitmask(n, document_lengths(n, seed, 90))))
    live = np.random.default_rng(seed).random((n, n)) < 0.7
    live[:, :64] = True  # some tiles stay untouched by the bits
    compare(n, dict(fields, bitmask=pack_bitmask(live)))


def test_bitmask_requires_the_bits():
    m = api.Mask(causal=True)
    desc = m.desc()
    desc.flags |= api.BITMASK
    hdr = api.BlockIndexStruct()
    import ctypes
    assert api.lib().flash_msa_build_block_index(ctypes.byref(desc), 300, ctypes.byref(hdr)) == \
        api.ERR_INVALID_ARG


@pytest.mark.parametrize("n,fields,seed", [
    (300, {}, 11), (519, {"causal": True}, 12), (1000, {"causal": True, "window": 200}, 13),
    (777, {"causal": True, "global_tokens": 128, "window": 64}, 14)])
def test_document_indices_bit_exact(n, fields, seed):
    from tiled_exact_attention_flash_gb300.inputs import document_lengths
    lens = document_lengths(n, seed, 120)
    starts = tuple(int(x) for x in np.cumsum([0] + lens))
    compare(n, dict(fields, doc_starts=starts))


def test_documents_require_valid_offsets():
    import ctypes
    for starts in ((0, 50, 50, 300), (0, 100, 299), (1, 300)):
        desc = api.Mask(causal=True, doc_starts=starts).desc()
        hdr = api.BlockIndexStruct()
        assert api.lib().flash_msa_build_block_index(ctypes.byref(desc), 300, ctypes.byref(hdr)) == \
            api.ERR_INVALID_ARG, starts


def _oracle_live_count(n, fields):
    from oracle.mask import MaskSpec, live_matrix
    idx = np.arange(n)
    return int(live_matrix(idx, idx, n, MaskSpec(**fields)).sum())


@pytest.mark.parametrize("n", [1, 129, 517, 1000])
@pytest.mark.parametrize("mi", range(len(MASKS)))
def test_live_element_counts_match_the_mask(n, mi):
    """live_elements (both build calls) equals the number of live (i, j)
    pairs of the mask's definition."""
    import ctypes
    fields = MASKS[mi]
    got = api.build_block_index(api.Mask(**fields), n)
    want = _oracle_live_count(n, fields)
    assert got.live_elements == want
    hdr = api.BlockIndexStruct()  # the counting call alone
    assert api.lib().flash_msa_build_block_index(ctypes.byref(api.Mask(**fields).desc()), n,
                                                 ctypes.byref(hdr)) == api.OK
    assert hdr.live_elements == want


@pytest.mark.parametrize("n,fields,seed", [
    (519, {"causal": True}, 2), (700, {"window": 130, "stride": 2, "stride_phase": 1}, 4)])
def test_live_element_counts_with_bits(n, fields, seed):
    from tiled_exact_attention_flash_gb300.inputs import document_lengths, pack_bitmask
    live = np.random.default_rng(seed).random((n, n)) < 0.7
    for extra in ({"bitmask": pack_bitmask(live)},
                  {"doc_starts": tuple(int(x) for x in np.cumsum([0] + document_lengths(n, seed, 90)))}):
        f = dict(fields, **extra)
        assert api.build_block_index(api.Mask(**f), n).live_elements == _oracle_live_count(n, f)


def _pair_overlap(host):
    """Sum over q_order pairs of the common key tiles / sum of the tiles of
    either block, from the lists as sets."""
    rp, ci, qo = host["row_ptr"], host["col_idx"], host["q_order"]
    common = either = 0
    for r in range(0, len(qo) - 1, 2):
        a = set(ci[rp[qo[r]]:rp[qo[r] + 1]].tolist())
        b = set(ci[rp[qo[r + 1]]:rp[qo[r + 1] + 1]].tolist())
        common += len(a & b)
        either += len(a | b)
    return common / either if either else 0.0


def _random_block_mask(nb, density, seed):
    """Block-sparse bit-packed mask: each 128 x 128 tile live or dead at random."""
    from tiled_exact_attention_flash_gb300.inputs import pack_bitmask
    blocks = np.random.default_rng(seed).random((nb, nb)) < density
    return pack_bitmask(np.kron(blocks, np.ones((128, 128), dtype=bool)))


@pytest.mark.parametrize("cid,low", [(2, 0.9), (4, 0.75), (5, 0.75), (6, 0.9), (7, 0.5), (8, 0.9),
                                     (9, 0.85), (10, 0.9), (None, None)])
def test_pair_overlap(cid, low):
    """pair_overlap (the forward's choice between one interleaving MMA warp and
    one per query slot) is the overlap of the paired blocks' key-tile lists;
    with q_order pairing blocks that share key tiles it is high for every
    workload mask, and low for tiles live at random; the counting call leaves
    it 0."""
    import ctypes
    if cid is None:
        n = 40 * 128
        m = api.Mask(bitmask=_random_block_mask(40, 0.08, 3))
    else:
        w = WORKLOADS[cid]
        n = w.N
        m = api.Mask(**w.mask_fields())
    got = api.build_block_index(m, n)
    assert got.header.pair_overlap == pytest.approx(_pair_overlap(got.host), rel=1e-6)
    if low is None:
        assert got.header.pair_overlap < 0.5
    else:
        assert got.header.pair_overlap >= low
    hdr = api.BlockIndexStruct()
    assert api.lib().flash_msa_build_block_index(ctypes.byref(m.desc()), n,
                                                 ctypes.byref(hdr)) == api.OK
    assert hdr.pair_overlap == 0.0


@pytest.mark.parametrize("density,seed", [(0.08, 3), (0.3, 4), (0.7, 5)])
def test_random_block_masks_bit_exact(density, seed):
    """Block-sparse random masks: the shared-pairs q_order (and the rest of
    the index) of the C++ builder equals the oracle's."""
    n = 40 * 128 - 57
    compare(n, {"bitmask": _random_block_mask_n(n, density, seed)})


def _random_block_mask_n(n, density, seed):
    """As _random_block_mask, cut to n tokens (a ragged tail)."""
    from tiled_exact_attention_flash_gb300.inputs import pack_bitmask
    nb = (n + 127) // 128
    blocks = np.random.default_rng(seed).random((nb, nb)) < density
    return pack_bitmask(np.kron(blocks, np.ones((128, 128), dtype=bool))[:n, :n])
