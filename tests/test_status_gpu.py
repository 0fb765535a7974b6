"""Failure detection without a GPU fault: a bounded wait that must run out.

flash_msa_selftest_wait_timeout launches one thread that waits, through the
library's own bounded wait, on an mbarrier nothing arrives on.  The wait
gives up after its limit and records FLASH_MSA_ERR_TIMEOUT in the device
status word; the host reads it through flash_msa_get_status, and the next
attention call runs normally on the same context."""
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


def test_bounded_wait_reports_timeout_and_context_survives():
    assert api.get_status() == api.OK
    assert api.selftest_wait_timeout() == api.OK
    assert api.get_status() == api.ERR_TIMEOUT
    assert b"site 238" in api.lib().flash_msa_last_error_string()
    assert api.get_status() == api.OK  # read and cleared
    # the same context still computes correct attention
    inp = small_inputs(1, 300, 2, 128, seed=77)
    res = gc.run_gpu(inp, {"causal": True})
    gc.full_compare(inp, {"causal": True}, res)
