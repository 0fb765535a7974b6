"""GPU parity: the CUDA path (through the C-ABI) against the float64 oracle.

Small cases compare every element; the full-size workloads compare sampled
heads, query rows and key columns that the oracle computes one by one.
Tolerances: |O - O_ref| <= 1e-2, |LSE - LSE_ref| <= 2e-3 on finite rows (-inf
rows must match exactly), |g - g_ref| <= 3e-2 * max|g_ref| per gradient."""
import numpy as np
import pytest
import torch

from tests import gpu_cases as gc
from tiled_exact_attention_flash_gb300 import api
from tiled_exact_attention_flash_gb300.inputs import WORKLOADS, small_inputs, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.libbuild import ensure_built
    ensure_built()


SMALL_MASKS = {
    "dense": {},
    "causal": {"causal": True},
    "window_strided": {"causal": True, "window": 150, "stride": 2, "stride_phase": 1},
    "window_dilated": {"causal": True, "window": 400, "dilation": 2, "dilation_near": 1},
    "window_noncausal": {"window": 100},
    "strided_only": {"causal": True, "stride": 3, "stride_phase": 2},
    "window_global": {"causal": True, "window": 130, "global_tokens": 128},
    "global_noncausal": {"window": 100, "global_tokens": 256},
    "relstride": {"causal": True, "window": 150, "stride": 2, "stride_phase": 0,
                  "stride_relative": True},
    "relstride_noncausal": {"stride": 3, "stride_phase": 1, "stride_relative": True},
    "fardil": {"causal": True, "window": 200, "dilation": 2, "dilation_far": True},
}


def test_workload1_full():
    w = WORKLOADS[1]
    inp = workload_inputs(w)
    res = gc.run_gpu(inp, w.mask_fields())
    gc.full_compare(inp, w.mask_fields(), res)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [1, 127, 129, 200, 384, 517])
@pytest.mark.parametrize("mname", sorted(SMALL_MASKS))
def test_small_cases(d, n, mname):
    fields = SMALL_MASKS[mname]
    inp = small_inputs(2, n, 3, d, seed=n * 7 + d)
    res = gc.run_gpu(inp, fields)
    gc.full_compare(inp, fields, res)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [129, 517])
@pytest.mark.parametrize("mname", sorted(SMALL_MASKS))
def test_small_cases_accumulated_backward(d, n, mname):
    # the fused backward with dQ added into an fp32 accumulator, against the oracle
    fields = SMALL_MASKS[mname]
    inp = small_inputs(2, n, 3, d, seed=n * 5 + d)
    res = gc.run_gpu(inp, fields, accumulated=True)
    gc.full_compare(inp, fields, res)


@pytest.mark.parametrize("cid", [3, 4, 9])
def test_full_size_workloads_accumulated_backward(cid):
    w = WORKLOADS[cid]
    inp = workload_inputs(w)
    res = gc.run_gpu(inp, w.mask_fields(), accumulated=True)
    rng = np.random.default_rng(cid + 100)
    gc.sampled_compare(inp, w.mask_fields(), res, [(0, w.H // 2)], gc.sample_positions(w.N, rng),
                       gc.sample_positions(w.N, rng))


@pytest.mark.parametrize("cid", [2, 3, 4, 5, 6, 7, 9, 10])
def test_full_size_workloads(cid):
    w = WORKLOADS[cid]
    inp = workload_inputs(w)
    res = gc.run_gpu(inp, w.mask_fields())
    rng = np.random.default_rng(cid)
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    rows = gc.sample_positions(w.N, rng)
    cols = gc.sample_positions(w.N, rng)
    gc.sampled_compare(inp, w.mask_fields(), res, heads, rows, cols)
    # outputs are finite everywhere (spot check of the whole tensors)
    for name in ("o", "dq", "dk", "dv"):
        assert np.isfinite(res[name]).all(), name


def test_full_size_far_dilation_workload():
    # 278784 live tiles per head: the oracle checks sampled forward rows and
    # dQ rows at full size, and dK / dV element by element on key columns
    # sampled from the last 4096 tokens of one head (a causal mask: their
    # columns of P involve only the rows from there on, whose statistics the
    # oracle computes in full); at N = 16384 the same mask is compared on
    # sampled rows and columns spread over the whole sequence
    w = WORKLOADS[8]
    inp = workload_inputs(w)
    res = gc.run_gpu(inp, w.mask_fields())
    rng = np.random.default_rng(8)
    rows = gc.sample_positions(w.N, rng)
    gc.sampled_compare(inp, w.mask_fields(), res, [(w.B - 1, w.H - 1)], rows, [], backward=False)
    cols = np.unique(np.concatenate([w.N - 1 - np.arange(24),
                                     rng.integers(w.N - 4096, w.N, size=24)]))
    gc.sampled_compare(inp, w.mask_fields(), res, [(0, 0)], rows[::4], cols, tail_stats=True)
    for name in ("o", "dq", "dk", "dv"):
        assert np.isfinite(res[name]).all(), name
    small = small_inputs(1, 16384, 2, 128, seed=88)
    res = gc.run_gpu(small, w.mask_fields())
    rng = np.random.default_rng(88)
    gc.sampled_compare(small, w.mask_fields(), res, [(0, 0), (0, 1)], gc.sample_positions(16384, rng),
                       gc.sample_positions(16384, rng))


def test_closed_form_uniform_on_gpu():
    # Q = 0: every live score is 0, so O_i is the mean of V over the live keys
    B, N, H, d = 1, 300, 2, 128
    inp = small_inputs(B, N, H, d, seed=99)
    inp["q"] = torch.zeros_like(inp["q"])
    fields = {"causal": True, "window": 130}
    res = gc.run_gpu(inp, fields, backward=False)
    v = inp["v"].double().numpy()
    for h in range(H):
        for i in range(N):
            lo = max(0, i - 130)
            ref = v[0, lo:i + 1, h].mean(axis=0)
            assert np.abs(res["o"][0, i, h] - ref).max() <= gc.O_TOL
            assert abs(res["lse"][0, h, i] - np.log(i + 1 - lo)) <= gc.LSE_TOL


def test_closed_form_uniform_global_tokens_on_gpu():
    # Q = 0 with a causal window of 130 and 256 global tokens: O_i is the mean
    # of V over keys j <= i with j < 256 or i - j <= 130, or over all j <= i
    # when i itself is global
    B, N, H, d = 1, 700, 2, 128
    inp = small_inputs(B, N, H, d, seed=98)
    inp["q"] = torch.zeros_like(inp["q"])
    fields = {"causal": True, "window": 130, "global_tokens": 256}
    res = gc.run_gpu(inp, fields, backward=False)
    v = inp["v"].double().numpy()
    for h in range(H):
        for i in range(N):
            keys = [j for j in range(i + 1) if i < 256 or j < 256 or i - j <= 130]
            ref = v[0, keys, h].mean(axis=0)
            assert np.abs(res["o"][0, i, h] - ref).max() <= gc.O_TOL
            assert abs(res["lse"][0, h, i] - np.log(len(keys))) <= gc.LSE_TOL


def test_smoke_shape_from_the_pages():
    # (1, 128, 8, 128) causal -> output (1, 128, 8, 128)
    inp = small_inputs(1, 128, 8, 128, seed=5)
    res = gc.run_gpu(inp, {"causal": True}, backward=False)
    assert res["o"].shape == (1, 128, 8, 128)


def test_repeat_calls_are_deterministic():
    # every output of the default path is bitwise reproducible; the
    # accumulated variant gives bitwise the same dK, dV (the same products in
    # the same order) and a dQ within the gradient tolerance (its fp32
    # additions run in a varying order)
    inp = small_inputs(2, 1000, 4, 128, seed=11)
    a = gc.run_gpu(inp, {"causal": True})
    b = gc.run_gpu(inp, {"causal": True})
    c = gc.run_gpu(inp, {"causal": True}, accumulated=True)
    for name in ("o", "lse", "dq", "dk", "dv"):
        assert np.array_equal(a[name], b[name]), name
    for name in ("o", "lse", "dk", "dv"):
        assert np.array_equal(a[name], c[name]), name
    gc.check_grad(c["dq"], a["dq"].astype(np.float64), "dQ")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n", [129, 300, 517])
@pytest.mark.parametrize("kind", ["random_causal", "documents_causal", "documents_window"])
def test_bitmask_small_cases(d, n, kind):
    from tiled_exact_attention_flash_gb300.inputs import (document_bitmask, document_lengths,
                                                          pack_bitmask)
    if kind == "random_causal":
        live = np.random.default_rng(n + d).random((n, n)) < 0.7
        fields = {"causal": True, "bitmask": pack_bitmask(live)}
    elif kind == "documents_causal":
        fields = {"causal": True, "bitmask": document_bitmask(n, document_lengths(n, n, 70))}
    else:
        fields = {"window": 90, "bitmask": document_bitmask(n, document_lengths(n, n + 1, 100))}
    inp = small_inputs(2, n, 3, d, seed=n * 11 + d)
    res = gc.run_gpu(inp, fields)
    gc.full_compare(inp, fields, res)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lens", [(1, 200, 7, 129, 64), (300,), (128, 128, 5, 1, 250, 33)])
def test_varlen_equals_separate_sequences(d, causal, lens):
    # a variable-length batch through fwd_varlen / bwd_varlen against the
    # oracle run on every sequence alone
    from oracle import attention
    from oracle.mask import MaskSpec
    T, H = sum(lens), 3
    inp = small_inputs(1, T, H, d, seed=sum(lens) + d)
    cu = np.cumsum([0] + list(lens))
    q, k, v, do = (inp[n][0].cuda() for n in ("q", "k", "v", "do"))
    o, lse = api.fwd_varlen(q, k, v, cu, causal=causal)
    dq, dk, dv = api.bwd_varlen(q, k, v, o, lse, do, cu, causal=causal)
    assert api.get_status() == api.OK
    got = {n: t.float().cpu().numpy() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    f64 = {n: inp[n][0].double().numpy() for n in ("q", "k", "v", "do")}
    for h in range(H):
        for a, e in zip(cu[:-1], cu[1:]):
            sl = slice(int(a), int(e))
            args = [f64[n][sl, h] for n in ("q", "k", "v")]
            o_ref, l_ref = attention.forward_head(*args, d ** -0.5, MaskSpec(causal=causal))
            g_ref = attention.backward_head(*args, f64["do"][sl, h], d ** -0.5, MaskSpec(causal=causal))
            gc.check_o(got["o"][sl, h], o_ref)
            gc.check_lse(got["lse"][h, sl], l_ref)
            for name, ref in zip(("dq", "dk", "dv"), g_ref):
                gc.check_grad(got[name][sl, h], ref, name)


@pytest.mark.parametrize("mname", ["causal", "window_global"])
def test_many_units_per_cta(mname):
    """More work units than SMs, so the persistent kernels (one CTA per SM)
    take several units each, dealt in rank-major order: B=2, H=96, N=300 gives
    384 forward pair units and 576 units per backward kernel.  Sampled heads
    spread over the unit order are compared element by element; every head
    must have been computed."""
    fields = SMALL_MASKS[mname]
    inp = small_inputs(2, 300, 96, 128, seed=4242)
    res = gc.run_gpu(inp, fields)
    heads = [(b, h) for b in range(2) for h in range(96) if (b * 96 + h) % 11 == 0] + [(1, 95)]
    gc.full_compare(inp, fields, res, heads=heads)
    for name in ("o", "dq", "dk", "dv"):
        per_head = np.abs(res[name]).max(axis=(1, 3))  # (B, N, H, d) -> (B, H)
        assert (per_head > 0).all(), name


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("scale", [0.05, 0.3])
@pytest.mark.parametrize("mname", ["dense", "causal", "window_dilated"])
def test_custom_scale(d, scale, mname):
    """A softmax scale other than d^-1/2 reaches every step that uses it: the
    forward's exponent and LSE, and the backward's dQ = scale dS K and
    dK = scale dS^T Q (a backward that kept the default would be off by the
    ratio of the two scales)."""
    fields = SMALL_MASKS[mname]
    inp = small_inputs(1, 300, 2, d, seed=900 + d)
    res = gc.run_gpu(inp, fields, scale=scale)
    gc.full_compare(inp, fields, res, scale=scale)


@pytest.mark.parametrize("order", ["dkdv_first", "dq_first"])
@pytest.mark.parametrize("mname", ["causal", "window_strided"])
def test_bwd_stages_match_full_backward(order, mname):
    """flash_msa_bwd_stages, two-kernel variant: the preprocessing stage,
    then dK/dV and dQ in either order on one workspace, gives bit-for-bit
    the gradients of flash_msa_bwd; a stage leaves the other stage's outputs
    untouched."""
    fields = SMALL_MASKS[mname]
    inp = small_inputs(2, 517, 3, 128, seed=31)
    mask = api.Mask(**fields)
    N = inp["q"].shape[1]
    index = api.build_block_index(mask, N).to("cuda") if mask.needs_index else None
    q, k, v, do = (inp[n].to("cuda") for n in ("q", "k", "v", "do"))
    o, lse = api.fwd(q, k, v, mask=mask, index=index)
    dq, dk, dv = api.bwd(q, k, v, o, lse, do, mask=mask, index=index)
    B, _, H, d = q.shape
    ws = torch.empty(api.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    sentinel = torch.tensor(7.0, dtype=torch.bfloat16)
    sq, sk, sv = (torch.full_like(t, 7.0) for t in (dq, dk, dv))
    api.bwd(q, k, v, o, lse, do, mask=mask, index=index, dq=sq, dk=sk, dv=sv, workspace=ws,
            stages=api.BWD_PREPROCESS)
    first, second = ((api.BWD_DKDV, api.BWD_DQ) if order == "dkdv_first"
                     else (api.BWD_DQ, api.BWD_DKDV))
    api.bwd(q, k, v, o, lse, do, mask=mask, index=index, dq=sq, dk=sk, dv=sv, workspace=ws,
            stages=first)
    torch.cuda.synchronize()
    untouched = (sq,) if first == api.BWD_DKDV else (sk, sv)
    for t in untouched:
        assert bool((t.cpu() == sentinel).all())
    api.bwd(q, k, v, o, lse, do, mask=mask, index=index, dq=sq, dk=sk, dv=sv, workspace=ws,
            stages=second)
    assert api.get_status() == api.OK
    for a, b in ((sq, dq), (sk, dk), (sv, dv)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("mname", ["causal", "window_strided", "window_global"])
def test_fused_bwd_stages_match_full_backward(mname):
    """flash_msa_bwd_stages, accumulated variant: PREPROCESS, FUSED and
    DQ_CONVERT launched one at a time give the gradients of flash_msa_bwd
    (dK, dV bit for bit, dQ within the gradient tolerance); FUSED writes no
    dq and DQ_CONVERT no dk / dv; PREPROCESS zeroes an accumulator that holds
    garbage (the workspace is filled with NaN first)."""
    fields = SMALL_MASKS[mname]
    inp = small_inputs(2, 517, 3, 128, seed=37)
    mask = api.Mask(**fields)
    N = inp["q"].shape[1]
    index = api.build_block_index(mask, N).to("cuda") if mask.needs_index else None
    q, k, v, do = (inp[n].to("cuda") for n in ("q", "k", "v", "do"))
    o, lse = api.fwd(q, k, v, mask=mask, index=index)
    dq, dk, dv = api.bwd(q, k, v, o, lse, do, mask=mask, index=index)
    B, _, H, d = q.shape
    nbytes = api.bwd_stages_workspace_bytes(B, H, N, d, api.BWD_ACCUMULATED)
    ws = torch.full((nbytes // 4,), float("nan"), device="cuda")
    sentinel = torch.tensor(7.0, dtype=torch.bfloat16)
    sq, sk, sv = (torch.full_like(t, 7.0) for t in (dq, dk, dv))
    for stage, untouched in ((api.BWD_PREPROCESS, (sq, sk, sv)), (api.BWD_FUSED, (sq,)),
                             (api.BWD_DQ_CONVERT, ())):
        api.bwd(q, k, v, o, lse, do, mask=mask, index=index, dq=sq, dk=sk, dv=sv, workspace=ws,
                stages=stage)
        torch.cuda.synchronize()
        for t in untouched:
            assert bool((t.cpu() == sentinel).all())
    assert api.get_status() == api.OK
    assert torch.equal(sk, dk) and torch.equal(sv, dv)
    gc.check_grad(sq.float().cpu().numpy(), dq.float().cpu().numpy().astype(np.float64), "dQ")


def test_side_streams_match_default_stream():
    """The calls run on the caller's current stream: forward and backward
    issued on two side streams at once (each with its own work counters)
    give bit-for-bit the results of the default stream."""
    fields = {"causal": True, "window": 300, "dilation": 2, "dilation_near": 1}
    inp = small_inputs(2, 517, 3, 128, seed=77)
    mask = api.Mask(**fields)
    N = inp["q"].shape[1]
    index = api.build_block_index(mask, N).to("cuda")
    dev = {n: inp[n].to("cuda") for n in ("q", "k", "v", "do")}
    o, lse = api.fwd(dev["q"], dev["k"], dev["v"], mask=mask, index=index)
    ref = (o, lse) + api.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], mask=mask, index=index)
    torch.cuda.synchronize()
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            so, slse = api.fwd(dev["q"], dev["k"], dev["v"], mask=mask, index=index)
            outs.append((so, slse) + api.bwd(dev["q"], dev["k"], dev["v"], so, slse, dev["do"],
                                              mask=mask, index=index))
    torch.cuda.synchronize()
    assert api.get_status() == api.OK
    for got in outs:
        for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), got, ref):
            assert torch.equal(a, b), name


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens", [(1, 300, 128, 129, 7, 211), (517,), (90, 1, 2, 300, 130)])
@pytest.mark.parametrize("extra", [{"causal": True}, {}, {"causal": True, "window": 150},
                                   {"window": 70}, {"causal": True, "stride": 2}])
def test_packed_sequences(d, lens, extra):
    """Sequences packed on one axis (the DOCUMENTS mask): with causal / window
    parts the index tiles every sequence from its own first token (no tile
    spans two sequences); with a block-level part (strides) it keeps the
    packed 128-token tiles with bit tiles.  Both against the oracle, element
    by element."""
    starts = tuple(int(x) for x in np.cumsum((0,) + lens))
    fields = dict(extra, doc_starts=starts)
    inp = small_inputs(2, starts[-1], 3, d, seed=sum(lens) + 3 * d + len(extra))
    mask = api.Mask(**fields)
    assert api.build_block_index(mask, starts[-1]).sequence_tiles == ("stride" not in extra)
    res = gc.run_gpu(inp, fields)
    gc.full_compare(inp, fields, res)


@pytest.mark.parametrize("mname", ["window_strided", "window_dilated", "window_global", "relstride"])
def test_forward_issuer_modes_agree(mname):
    """The forward issues a query-block pair's products from one interleaving
    MMA warp or from one warp per block, chosen by the index's pair_overlap.
    Each block's products run in the same order either way, so forcing
    either mode (through the hint) gives bitwise the same O and LSE, and
    both match the oracle."""
    n = 1500
    inp = small_inputs(2, n, 3, 128, seed=23)
    fields = SMALL_MASKS[mname]
    mask = api.Mask(**fields)
    index = api.build_block_index(mask, n).to("cuda")
    q, k, v = (inp[t].to("cuda") for t in ("q", "k", "v"))
    outs = []
    for overlap in (0.0, 1.0):
        index.device_struct.pair_overlap = overlap
        o, lse = api.fwd(q, k, v, mask=mask, index=index)
        torch.cuda.synchronize()
        assert api.get_status() == api.OK
        outs.append((o.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    res = {"o": outs[0][0].float().cpu().numpy(), "lse": outs[0][1].cpu().numpy()}
    gc.full_compare(inp, fields, res, backward=False)


def test_backward_head_groups_with_a_remainder():
    """The backward numbers its units within groups of heads whose streamed
    tiles fit 64 MB of L2: at N = 32768, d = 128 a head streams 16 MB, so six
    heads form groups of 4 and 2.  Every head -- the last group's included --
    matches the oracle on sampled rows and columns."""
    B, N, H, d = 1, 32768, 6, 128
    inp = small_inputs(B, N, H, d, seed=29)
    fields = {"causal": True}
    res = gc.run_gpu(inp, fields)
    rng = np.random.default_rng(29)
    rows = gc.sample_positions(N, rng, k=48)
    cols = gc.sample_positions(N, rng, k=48)
    gc.sampled_compare(inp, fields, res, [(0, 0), (0, 4), (0, 5)], rows, cols)


@pytest.mark.parametrize("cid", [3, 4, 9, 10])
def test_full_size_constant_values_every_row(cid):
    """Every output row of every head at full size.  With all value rows of a
    head equal (V[b, j, h] = c[b, h] for every key j) each softmax row sums to
    one, so O[b, i, h] = c[b, h] for every query row with a live key (every
    row here: each attends to itself).  The kernel rounds P to bf16 before
    P V (bf16 keeps 8 significant bits: unit roundoff u = 2^-8 per entry, so
    the weights sum to within u of the fp32 row sum that divides them) and
    rounds O to bf16 (within u |O|): |O - c| <= (2u + u^2) |c| up to fp32
    accumulation.  O and LSE start as NaN, so a row that no work unit wrote
    fails the check."""
    w = WORKLOADS[cid]
    inp = workload_inputs(w)
    B, N, H, d = inp["q"].shape
    rng = np.random.default_rng(1000 + cid)
    c = torch.from_numpy(rng.standard_normal((B, 1, H, d)).astype(np.float32)).to(torch.bfloat16)
    fields = w.mask_fields()
    mask = api.Mask(**fields) if fields else None
    index = api.build_block_index(mask, N).to("cuda") if (mask and mask.needs_index) else None
    q, k = inp["q"].to("cuda"), inp["k"].to("cuda")
    v = c.expand(B, N, H, d).contiguous().to("cuda")
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    api.fwd(q, k, v, mask=mask, index=index, out=o, lse=lse)
    assert api.get_status() == api.OK
    got = o.float().cpu().numpy()
    cc = c.float().numpy()
    assert np.isfinite(got).all(), "an output row was not written"
    assert np.isfinite(lse.cpu().numpy()).all(), "an LSE entry was not written"
    err = np.abs(got - cc)
    u = 2.0 ** -8
    bound = (2 * u + u * u) * np.abs(cc) + 1e-6
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())} entries off; worst {err.max():.3e} at "
                           f"{np.unravel_index(np.argmax(err - bound), err.shape)}")


@pytest.mark.parametrize("cid", [3, 4, 9, 10])
def test_full_size_zero_output_gradient_every_row(cid):
    """Every gradient row of every head at full size.  With dO = 0, D = 0 and
    dP = 0, so dS = P (dP - D) = 0 and dQ, dK, dV are exactly zero.  The
    gradients start as NaN, so a row that no backward work unit wrote fails
    the check (their values are covered by the sampled oracle comparisons)."""
    w = WORKLOADS[cid]
    inp = workload_inputs(w)
    B, N, H, d = inp["q"].shape
    fields = w.mask_fields()
    mask = api.Mask(**fields) if fields else None
    index = api.build_block_index(mask, N).to("cuda") if (mask and mask.needs_index) else None
    q, k, v = (inp[n].to("cuda") for n in ("q", "k", "v"))
    o, lse = api.fwd(q, k, v, mask=mask, index=index)
    do = torch.zeros_like(q)
    grads = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    api.bwd(q, k, v, o, lse, do, mask=mask, index=index, dq=grads[0], dk=grads[1], dv=grads[2])
    assert api.get_status() == api.OK
    for name, g in zip(("dq", "dk", "dv"), grads):
        assert bool((g == 0).all()), f"{name}: {int((g != 0).sum())} entries not exactly zero"
