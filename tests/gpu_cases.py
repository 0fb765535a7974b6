"""Helpers for the GPU parity tests: run the CUDA path through the C-ABI
binding and compare with the oracle on the same seeded inputs."""
import numpy as np
import torch

from oracle import attention
from oracle.mask import MaskSpec
from tiled_exact_attention_flash_gb300 import api
from tiled_exact_attention_flash_gb300.inputs import as_f64

# tolerances (bf16 inputs, fp32 accumulation)
O_TOL = 1e-2
LSE_TOL = 2e-3
GRAD_REL_TOL = 3e-2
# Where a reference gradient vanishes identically (e.g. N = 1 causal: dS = 0)
# the relative bound above is 0; bf16 rounding of O in D = rowsum(dO o O)
# still leaves ~1e-7 there.  Absolute floor, far below bf16 resolution of any
# non-trivial gradient in these tests.
GRAD_ABS_FLOOR = 1e-4


def run_gpu(inp: dict, fields: dict, device="cuda", backward=True, scale=None,
            accumulated=False):
    """scale: softmax scale passed to the library (None: its default d^-1/2);
    accumulated: the fused backward with dQ added into an fp32 accumulator
    instead of the default two-kernel backward."""
    mask = api.Mask(**fields) if fields else None
    N = inp["q"].shape[1]
    index = None
    if mask is not None and mask.needs_index:
        index = api.build_block_index(mask, N).to(device)
    q, k, v, do = (inp[n].to(device) for n in ("q", "k", "v", "do"))
    o, lse = api.fwd(q, k, v, mask=mask, index=index, scale=scale)
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv = api.bwd(q, k, v, o, lse, do, mask=mask, index=index, scale=scale,
                             accumulated=accumulated)
        out.update(dq=dq, dk=dk, dv=dv)
    st = api.get_status()
    assert st == api.OK, f"device status {st}"
    return {k2: t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
            for k2, t in out.items()}


def head(t: torch.Tensor, b: int, h: int) -> np.ndarray:
    return as_f64(t[b, :, h])


def check_lse(got, ref):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "LSE -inf pattern differs"
    assert (got[~fin] == -np.inf).all()
    if fin.any():
        err = np.abs(got[fin] - ref[fin]).max()
        assert err <= LSE_TOL, f"LSE max err {err}"


# O is returned in bf16: the kernel accumulates in fp32 and rounds its
# result once, to nearest even.  The stated 1e-2 bound applies to that fp32
# result, so the check is exactly "O is the bf16 rounding of some value within
# 1e-2 of O_ref": rounding is monotone, so that holds iff
# bf16(O_ref - 1e-2) <= O <= bf16(O_ref + 1e-2).  (A plain |O - O_ref| bound
# would have to allow for the rounding on top: a kernel error e moves the
# rounded output by up to |bf16(O_ref) - O_ref| + 2 e.)
def bf16_round(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def check_o(got, ref):
    lo, hi = bf16_round(ref - O_TOL), bf16_round(ref + O_TOL)
    bad = (got < lo) | (got > hi)
    if bad.any():
        k = np.argmax(bad)
        raise AssertionError(
            f"O outside the bf16 rounding of O_ref +- {O_TOL}: got {got.flat[k]}, ref "
            f"{ref.flat[k]:.5f}, allowed [{lo.flat[k]}, {hi.flat[k]}]; max |err| "
            f"{np.abs(got - ref).max():.5f}")


def check_grad(got, ref, name):
    scale = np.abs(ref).max() if ref.size else 0.0
    err = np.abs(got - ref).max() if ref.size else 0.0
    tol = max(GRAD_REL_TOL * scale, GRAD_ABS_FLOOR)
    assert err <= tol, f"{name} max err {err} vs max(3e-2 x {scale}, {GRAD_ABS_FLOOR})"


def full_compare(inp, fields, res, heads=None, backward=True, scale=None):
    """Element-by-element comparison for every (or the given) head."""
    B, N, H, d = inp["q"].shape
    spec = MaskSpec(**fields)
    scale = d ** -0.5 if scale is None else scale
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in heads:
        q, k, v, do = (head(inp[n], b, h) for n in ("q", "k", "v", "do"))
        o_ref, lse_ref = attention.forward_head(q, k, v, scale, spec)
        check_o(res["o"][b, :, h], o_ref)
        check_lse(res["lse"][b, h], lse_ref)
        if backward:
            dq, dk, dv = attention.backward_head(q, k, v, do, scale, spec)
            check_grad(res["dq"][b, :, h], dq, "dQ")
            check_grad(res["dk"][b, :, h], dk, "dK")
            check_grad(res["dv"][b, :, h], dv, "dV")


def sampled_compare(inp, fields, res, heads, rows, cols, backward=True, tail_stats=False):
    """Full-size comparison on sampled heads / query rows / key columns.
    tail_stats (causal masks only): the row statistics are computed for the
    sampled rows and the rows >= min(cols) only (column j of P involves rows
    i >= j alone)."""
    B, N, H, d = inp["q"].shape
    spec = MaskSpec(**fields)
    scale = d ** -0.5
    for b, h in heads:
        q, k, v, do = (head(inp[n], b, h) for n in ("q", "k", "v", "do"))
        o_ref, lse_ref = attention.forward_rows(q, k, v, scale, spec, rows)
        check_o(res["o"][b, rows, h], o_ref)
        check_lse(res["lse"][b, h, rows], lse_ref)
        if backward:
            need = None
            if tail_stats and len(cols):
                need = np.union1d(np.asarray(rows, dtype=np.int64), np.arange(int(np.min(cols)), N))
            stats = attention.row_stats(q, k, v, do, scale, spec, rows=need)
            dq, dk, dv = attention.backward_sampled(q, k, v, do, scale, spec, rows, cols,
                                                    stats=stats)
            check_grad(res["dq"][b, rows, h], dq, "dQ")
            check_grad(res["dk"][b, cols, h], dk, "dK")
            check_grad(res["dv"][b, cols, h], dv, "dV")


def sample_positions(N, rng, k=96):
    pos = set(range(min(N, 40))) | set(range(max(0, N - 40), N))
    pos |= set(rng.integers(0, N, size=k).tolist())
    return np.array(sorted(pos))


# ---------------------------------------------------------------------------
# grouped-query attention: query head h reads key/value head h // G
# ---------------------------------------------------------------------------
def gqa_reference(q, k, v, do, scale, spec, backward=True):
    """Per-head oracle for (N, H, d) query tensors and (N, Hkv, d) key/value
    tensors (float64); dK / dV of a shared head sum the group's contributions."""
    N, H, d = q.shape
    Hkv = k.shape[1]
    G = H // Hkv
    o = np.zeros(q.shape)
    lse = np.zeros((H, N))
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for h in range(H):
        j = h // G
        o[:, h], lse[h] = attention.forward_head(q[:, h], k[:, j], v[:, j], scale, spec)
        if backward:
            gq, gk, gv = attention.backward_head(q[:, h], k[:, j], v[:, j], do[:, h], scale, spec)
            dq[:, h] = gq
            dk[:, j] += gk
            dv[:, j] += gv
    return o, lse, dq, dk, dv


def run_gpu_gqa(inp, fields, device="cuda", accumulated=False):
    mask = api.Mask(**fields) if fields else None
    N = inp["q"].shape[1]
    index = api.build_block_index(mask, N).to(device) if (mask and mask.needs_index) else None
    q, k, v, do = (inp[n].to(device) for n in ("q", "k", "v", "do"))
    o, lse = api.fwd(q, k, v, mask=mask, index=index)
    dq, dk, dv = api.bwd(q, k, v, o, lse, do, mask=mask, index=index, accumulated=accumulated)
    assert api.get_status() == api.OK
    f = lambda t: t.float().cpu().numpy()
    return {"o": f(o), "lse": lse.cpu().numpy(), "dq": f(dq), "dk": f(dk), "dv": f(dv)}


def gqa_full_compare(inp, fields, res):
    B = inp["q"].shape[0]
    d = inp["q"].shape[3]
    spec = MaskSpec(**fields)
    for b in range(B):
        q, k, v, do = (as_f64(inp[n][b]) for n in ("q", "k", "v", "do"))
        o, lse, dq, dk, dv = gqa_reference(q, k, v, do, d ** -0.5, spec)
        for h in range(q.shape[1]):
            check_o(res["o"][b, :, h], o[:, h])
            check_lse(res["lse"][b, h], lse[h])
        check_grad(res["dq"][b], dq, "dQ")
        check_grad(res["dk"][b], dk, "dK")
        check_grad(res["dv"][b], dv, "dV")
