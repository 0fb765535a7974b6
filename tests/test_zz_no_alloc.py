"""flash_msa_bwd_noalloc: the backward for callers that may not allocate
device memory per call -- a framework that owns the whole device memory pool
and hands out no extra buffers, or a loop where cudaMalloc / cudaFree are
banned because they can synchronise the device.  Its scratch is a fixed
16 MiB array inside the library instead of a caller-provided workspace.

Checked through the C-ABI on two calls in a row: bit for bit against
flash_msa_bwd with a caller-provided workspace (the same kernels), and
within the gradient tolerance of the parity tests as well.  The first call is the larger problem and the second a ragged
one (N not a multiple of 128), so the second call finds the first call's
finite values in the scratch rows its padding uses.  This file is collected
last on purpose."""
import numpy as np
import pytest
import torch

from tests import gpu_cases as gc
from tiled_exact_attention_flash_gb300 import api
from tiled_exact_attention_flash_gb300.inputs import small_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tests.libbuild import ensure_built
    ensure_built()


def _run(B, N, H, d, fields, seed):
    dev = torch.device("cuda")
    inp = small_inputs(B, N, H, d, seed=seed)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    mask = api.Mask(**fields) if fields else None
    index = api.build_block_index(mask, N).to(dev) if (mask and mask.needs_index) else None
    o, lse = api.fwd(q, k, v, mask=mask, index=index)
    ref = api.bwd(q, k, v, o, lse, do, mask=mask, index=index)
    got = api.bwd_noalloc(q, k, v, o, lse, do, mask=mask, index=index)
    assert api.get_status() == api.OK
    for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(a, b), name
        gc.check_grad(a.float().cpu().numpy(), b.float().cpu().numpy().astype(np.float64), name)
    return got


def test_noalloc_matches_workspace_entry_on_two_calls():
    # a large problem first, then a ragged one whose padding rows of the
    # shared scratch still hold the first call's values
    _run(1, 4096, 8, 128, {"causal": True}, 42)
    _run(2, 1000, 4, 128, {"causal": True, "window": 300, "stride": 3, "stride_phase": 1}, 41)


def test_noalloc_rejects_sizes_beyond_the_scratch():
    L = api.lib()
    fake = 0x10000  # never dereferenced: the size check comes first
    # B * H * ceil(N/128) * 128 = 4 * 16 * 32768 = 2^21 fits; one more block does not
    args = [fake] * 9
    code = L.flash_msa_bwd_noalloc(*args, 4, 16, 32768 + 1, 128, 0.0, None, None)
    assert code == api.ERR_WORKSPACE
    assert b"16777216" in L.flash_msa_last_error_string()
