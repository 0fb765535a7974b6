"""The C-ABI library loads, exports what include/flashmsa.h declares, and
validates arguments on the host (no GPU needed: every call here fails
validation before any CUDA call)."""
import ctypes
import os
import re

import pytest

from tiled_exact_attention_flash_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from tests.libbuild import ensure_built
    ensure_built()
    return api.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "flashmsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flash_msa_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(L, name), name
    assert sorted(api.SYMBOLS) == names


def test_version(L):
    assert "sm_103a" in api.version()


FAKE = 0x10000  # aligned, never dereferenced: validation fails first


def fwd_raw(L, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=256, d=128, scale=0.0,
            mask=None):
    return L.flash_msa_fwd(q, k, v, o, lse, B, H, N, d, scale,
                           ctypes.byref(mask) if mask is not None else None, None)


def test_fwd_argument_errors(L):
    assert fwd_raw(L, d=96) == api.ERR_UNSUPPORTED
    assert fwd_raw(L, N=0) == api.ERR_INVALID_ARG
    assert fwd_raw(L, N=1 << 31) == api.ERR_INVALID_ARG
    assert fwd_raw(L, B=0) == api.ERR_INVALID_ARG
    assert fwd_raw(L, q=0) == api.ERR_INVALID_ARG
    assert fwd_raw(L, k=FAKE + 2) == api.ERR_INVALID_ARG
    assert fwd_raw(L, lse=FAKE + 1) == api.ERR_INVALID_ARG
    assert b"aligned" in L.flash_msa_last_error_string()
    bad_flags = api.MaskDescStruct(512, 128, 0, 1, 0, 1, 0, None)
    assert fwd_raw(L, mask=bad_flags) == api.ERR_INVALID_ARG
    bad_block = api.Mask(causal=True, window=10, block=64).desc()
    assert fwd_raw(L, mask=bad_block) == api.ERR_UNSUPPORTED
    no_index = api.Mask(causal=True, window=100).desc()
    assert fwd_raw(L, mask=no_index) == api.ERR_INDEX
    bad_stride = api.Mask(stride=4, stride_phase=4).desc()
    assert fwd_raw(L, mask=bad_stride) == api.ERR_INVALID_ARG
    neg_window = api.MaskDescStruct(api.WINDOW, 128, -1, 1, 0, 1, 0, None)
    assert fwd_raw(L, mask=neg_window) == api.ERR_INVALID_ARG
    no_global = api.MaskDescStruct(api.WINDOW | api.GLOBAL, 128, 10, 1, 0, 1, 0, None, 0)
    assert fwd_raw(L, mask=no_global) == api.ERR_INVALID_ARG
    ragged_global = api.Mask(causal=True, window=100, global_tokens=100).desc()
    assert fwd_raw(L, mask=ragged_global) == api.ERR_UNSUPPORTED
    assert b"multiple of the 128-token block" in L.flash_msa_last_error_string()
    bad_rel = api.Mask(causal=True, stride=4, stride_phase=5, stride_relative=True).desc()
    assert fwd_raw(L, mask=bad_rel) == api.ERR_INVALID_ARG
    bad_far = api.MaskDescStruct(api.WINDOW | api.DILATED_FAR, 128, 100, 0, 0, 1, 0, None, 0)
    assert fwd_raw(L, mask=bad_far) == api.ERR_INVALID_ARG


def test_index_for_another_n_is_rejected(L):
    m = api.Mask(causal=True, window=300)
    idx = api.build_block_index(m, 1000)
    hs = idx.host_struct()
    desc = m.desc(ctypes.addressof(hs))
    assert fwd_raw(L, N=2000, mask=desc) == api.ERR_INDEX


def test_bwd_workspace_errors(L):
    need = L.flash_msa_bwd_workspace_bytes(2, 3, 300, 128)
    assert need == 2 * 2 * 3 * 384 * 4  # two fp32 vectors per (b, h), padded rows
    assert L.flash_msa_bwd_workspace_bytes(0, 3, 300, 128) == 0
    ws = L.flash_msa_bwd_stages_workspace_bytes
    assert ws(2, 3, 300, 128, api.BWD_DETERMINISTIC) == need
    big = ws(2, 3, 300, 128, api.BWD_ACCUMULATED)
    assert big == need + 2 * 3 * 384 * 128 * 4  # plus the fp32 dQ accumulator
    assert ws(2, 3, 300, 128, api.BWD_DQ_CONVERT) == big
    assert ws(2, 3, 300, 128, api.BWD_FUSED | api.BWD_DKDV) == 0
    assert ws(2, 3, 300, 128, 32) == 0
    stage_args = [FAKE] * 9 + [2, 3, 300, 128, 0.0, None, FAKE, big]
    assert L.flash_msa_bwd_stages(*stage_args, api.BWD_FUSED | api.BWD_DQ, None) == api.ERR_INVALID_ARG
    assert L.flash_msa_bwd_stages(*stage_args[:-1], need, api.BWD_FUSED, None) == api.ERR_WORKSPACE
    args = [FAKE] * 9 + [2, 3, 300, 128, 0.0, None]
    assert L.flash_msa_bwd(*args, None, need, None) == api.ERR_WORKSPACE
    assert L.flash_msa_bwd(*args, FAKE, need - 4, None) == api.ERR_WORKSPACE
    args2 = [FAKE] * 9 + [2, 3, 300, 64, 0.0, None]
    assert L.flash_msa_bwd(*([0] + args2[1:]), FAKE, need, None) == api.ERR_INVALID_ARG


def test_build_index_argument_errors(L):
    hdr = api.BlockIndexStruct()
    d = api.Mask(causal=True).desc()
    assert L.flash_msa_build_block_index(None, 100, ctypes.byref(hdr)) == api.ERR_INVALID_ARG
    assert L.flash_msa_build_block_index(ctypes.byref(d), 0, ctypes.byref(hdr)) == api.ERR_INVALID_ARG
    d64 = api.Mask(causal=True, block=64).desc()
    assert L.flash_msa_build_block_index(ctypes.byref(d64), 100, ctypes.byref(hdr)) == api.ERR_UNSUPPORTED


def test_gqa_head_count_errors(L):
    args = [FAKE] * 5
    assert L.flash_msa_fwd_gqa(*args, 1, 6, 4, 256, 128, 0.0, None, None) == api.ERR_INVALID_ARG
    assert L.flash_msa_fwd_gqa(*args, 1, 6, 0, 256, 128, 0.0, None, None) == api.ERR_INVALID_ARG
    need = L.flash_msa_bwd_workspace_bytes(1, 6, 256, 128)
    assert L.flash_msa_bwd_gqa(*([FAKE] * 9), 1, 6, 4, 256, 128, 0.0, None, FAKE, need,
                               None) == api.ERR_INVALID_ARG


def test_wait_limit_setting(L):
    old = api.get_wait_limit_ms()
    assert old == 4000
    try:
        assert L.flash_msa_set_wait_limit_ms(0) == api.ERR_INVALID_ARG
        assert L.flash_msa_set_wait_limit_ms(600001) == api.ERR_INVALID_ARG
        assert api.get_wait_limit_ms() == old
        api.set_wait_limit_ms(12000)
        assert api.get_wait_limit_ms() == 12000
    finally:
        api.set_wait_limit_ms(old)
