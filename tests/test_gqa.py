"""Grouped-query / multi-query attention (K/V heads shared by groups of query
heads; "Flash MSA Attention Kernel Implementation", FAQ on GQA and MQA).

CPU: the grouped reference (per-head oracle, gradients of a shared head
summed over its group) is pinned by central finite differences of the total
loss with respect to the shared K and V.  GPU: parity of flash_msa_fwd_gqa /
flash_msa_bwd_gqa with that reference."""
import numpy as np
import pytest
import torch

from oracle import attention
from oracle.mask import MaskSpec
from tests import gpu_cases as gc
from tiled_exact_attention_flash_gb300.inputs import normal_bf16


def _loss(q, k, v, do, scale, spec):
    o, *_ = gc.gqa_reference(q, k, v, do, scale, spec, backward=False)
    return float((o * do).sum())


@pytest.mark.parametrize("spec", [MaskSpec(), MaskSpec(causal=True, window=3),
                                  MaskSpec(causal=True, stride=2, stride_phase=0, block=2)])
def test_grouped_reference_gradients_by_finite_differences(spec):
    rng = np.random.default_rng(31)
    N, H, Hkv, d = 6, 4, 2, 3
    q, do = rng.standard_normal((N, H, d)), rng.standard_normal((N, H, d))
    k, v = rng.standard_normal((N, Hkv, d)), rng.standard_normal((N, Hkv, d))
    scale = 0.7
    _, _, dq, dk, dv = gc.gqa_reference(q, k, v, do, scale, spec)
    eps = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, do=do, scale=scale, spec=spec)
            lm = _loss(**{**args, name: xm}, do=do, scale=scale, spec=spec)
            num[idx] = (lp - lm) / (2 * eps)
        assert np.abs(num - g).max() <= 1e-6 * max(1.0, np.abs(num).max()), name


def test_group_of_one_is_multi_head():
    rng = np.random.default_rng(32)
    N, H, d = 9, 3, 4
    q, k, v, do = (rng.standard_normal((N, H, d)) for _ in range(4))
    o, lse, dq, dk, dv = gc.gqa_reference(q, k, v, do, 0.5, MaskSpec(causal=True))
    for h in range(H):
        o1, l1 = attention.forward_head(q[:, h], k[:, h], v[:, h], 0.5, MaskSpec(causal=True))
        assert np.array_equal(o[:, h], o1) and np.array_equal(lse[h], l1)


def _inputs(B, N, H, Hkv, d, seed):
    return {"q": normal_bf16((B, N, H, d), 10 * seed + 1), "k": normal_bf16((B, N, Hkv, d), 10 * seed + 2),
            "v": normal_bf16((B, N, Hkv, d), 10 * seed + 3), "do": normal_bf16((B, N, H, d), 10 * seed + 4)}


@pytest.mark.gpu
@pytest.mark.parametrize("H,Hkv", [(4, 2), (8, 2), (4, 1)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("fields", [{"causal": True}, {"causal": True, "window": 150, "stride": 2, "stride_phase": 1}, {}])
def test_gqa_parity(H, Hkv, d, fields):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.libbuild import ensure_built
    ensure_built()
    inp = _inputs(2, 389, H, Hkv, d, seed=H * 10 + Hkv + d)
    res = gc.run_gpu_gqa(inp, fields)
    gc.gqa_full_compare(inp, fields, res)


@pytest.mark.gpu
@pytest.mark.parametrize("H,Hkv", [(4, 2), (4, 1)])
@pytest.mark.parametrize("fields", [{"causal": True}, {"causal": True, "window": 150, "stride": 2, "stride_phase": 1}])
def test_gqa_parity_accumulated_backward(H, Hkv, fields):
    # the fused backward walks each key/value head's group of query heads and
    # adds every query head's dQ partial products into its own accumulator rows
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.libbuild import ensure_built
    ensure_built()
    inp = _inputs(2, 389, H, Hkv, 128, seed=H * 7 + Hkv)
    res = gc.run_gpu_gqa(inp, fields, accumulated=True)
    gc.gqa_full_compare(inp, fields, res)
