"""ctypes binding over libflashmsa (argument marshalling only).

Every step of the computation runs in the CUDA library; this module checks
tensor dtypes / devices / shapes, allocates outputs with PyTorch (which is
used here only for device memory and streams), passes raw pointers and the
current CUDA stream, and turns non-zero status codes into exceptions.  There
is no fallback: if ``libflashmsa.so`` is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflashmsa.so")

(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_INDEX,
 ERR_SCHEDULE) = range(8)
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT",
                5: "WORKSPACE", 6: "INDEX", 7: "SCHEDULE"}
CAUSAL, WINDOW, DILATED, STRIDED, GLOBAL, STRIDED_REL, DILATED_FAR, BITMASK, DOCUMENTS = \
    1, 2, 4, 8, 16, 32, 64, 128, 256

# exported symbols, in the order include/flashmsa.h declares them
SYMBOLS = (
    "flash_msa_build_block_index",
    "flash_msa_check_block_index",
    "flash_msa_fwd",
    "flash_msa_bwd_workspace_bytes",
    "flash_msa_bwd",
    "flash_msa_bwd_stages",
    "flash_msa_bwd_stages_workspace_bytes",
    "flash_msa_fwd_gqa",
    "flash_msa_bwd_gqa",
    "flash_msa_bwd_gqa_stages",
    "flash_msa_bwd_noalloc",
    "flash_msa_selftest_wait_timeout",
    "flash_msa_set_wait_limit_ms",
    "flash_msa_get_wait_limit_ms",
    "flash_msa_get_status",
    "flash_msa_last_error_string",
    "flash_msa_version",
)


class BlockIndexStruct(ctypes.Structure):
    _fields_ = [
        ("seq_len", ctypes.c_int64),
        ("n_q_blocks", ctypes.c_int32),
        ("n_k_blocks", ctypes.c_int32),
        ("block", ctypes.c_int32),
        ("nnz", ctypes.c_int64),
        ("row_ptr", ctypes.c_void_p),
        ("col_idx", ctypes.c_void_p),
        ("kind", ctypes.c_void_p),
        ("col_ptr", ctypes.c_void_p),
        ("row_idx", ctypes.c_void_p),
        ("kind_t", ctypes.c_void_p),
        ("q_order", ctypes.c_void_p),
        ("k_order", ctypes.c_void_p),
        ("n_bit_tiles", ctypes.c_int64),
        ("bit_slot", ctypes.c_void_p),
        ("bit_slot_t", ctypes.c_void_p),
        ("bits", ctypes.c_void_p),
        ("bits_t", ctypes.c_void_p),
        ("live_elements", ctypes.c_int64),
        ("sequence_tiles", ctypes.c_int32),
        ("tile_start", ctypes.c_void_p),
        ("tile_seq0", ctypes.c_void_p),
        ("tile_seq_len", ctypes.c_void_p),
        ("pair_overlap", ctypes.c_float),
    ]


class MaskDescStruct(ctypes.Structure):
    _fields_ = [
        ("flags", ctypes.c_uint32),
        ("block", ctypes.c_int32),
        ("window", ctypes.c_int64),
        ("dilation", ctypes.c_int32),
        ("dilation_near", ctypes.c_int32),
        ("stride", ctypes.c_int32),
        ("stride_phase", ctypes.c_int32),
        ("index", ctypes.c_void_p),
        ("global_tokens", ctypes.c_int64),
        ("bitmask", ctypes.c_void_p),
        ("doc_starts", ctypes.c_void_p),
        ("n_docs", ctypes.c_int64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libflashmsa.so (once); raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    L.flash_msa_build_block_index.argtypes = [ctypes.POINTER(MaskDescStruct), i64,
                                              ctypes.POINTER(BlockIndexStruct)]
    L.flash_msa_check_block_index.argtypes = [ctypes.POINTER(BlockIndexStruct), i64]
    L.flash_msa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, i32, f32,
                                ctypes.POINTER(MaskDescStruct), vp]
    L.flash_msa_bwd_workspace_bytes.argtypes = [i32, i32, i64, i32]
    L.flash_msa_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.flash_msa_bwd_stages_workspace_bytes.argtypes = [i32, i32, i64, i32, ctypes.c_uint]
    L.flash_msa_bwd_stages_workspace_bytes.restype = ctypes.c_size_t
    L.flash_msa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, i32, f32,
                                ctypes.POINTER(MaskDescStruct), vp, ctypes.c_size_t, vp]
    L.flash_msa_bwd_stages.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, i32,
                                       f32, ctypes.POINTER(MaskDescStruct), vp, ctypes.c_size_t,
                                       ctypes.c_uint, vp]
    L.flash_msa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, f32,
                                    ctypes.POINTER(MaskDescStruct), vp]
    L.flash_msa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i32,
                                    f32, ctypes.POINTER(MaskDescStruct), vp, ctypes.c_size_t, vp]
    L.flash_msa_bwd_gqa_stages.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i64,
                                           i32, f32, ctypes.POINTER(MaskDescStruct), vp,
                                           ctypes.c_size_t, ctypes.c_uint, vp]
    L.flash_msa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, i32,
                                        f32, ctypes.POINTER(MaskDescStruct), vp]
    L.flash_msa_get_status.argtypes = [vp]
    L.flash_msa_selftest_wait_timeout.argtypes = [vp]
    L.flash_msa_set_wait_limit_ms.argtypes = [ctypes.c_uint]
    L.flash_msa_get_wait_limit_ms.restype = ctypes.c_uint
    L.flash_msa_last_error_string.restype = ctypes.c_char_p
    L.flash_msa_version.restype = ctypes.c_char_p
    for name in ("flash_msa_build_block_index", "flash_msa_check_block_index", "flash_msa_fwd",
                 "flash_msa_bwd", "flash_msa_bwd_stages", "flash_msa_bwd_noalloc",
                 "flash_msa_fwd_gqa", "flash_msa_bwd_gqa", "flash_msa_bwd_gqa_stages", "flash_msa_get_status",
                 "flash_msa_selftest_wait_timeout", "flash_msa_set_wait_limit_ms"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


class FlashMSAError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().flash_msa_last_error_string().decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({msg})")
        self.code = code


def _check(code: int, where: str):
    if code != OK:
        raise FlashMSAError(code, where)


# ---------------------------------------------------------------------------
# masks and block indices
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Mask:
    """Attention mask description (semantics in include/flashmsa.h)."""
    causal: bool = False
    window: Optional[int] = None
    dilation: Optional[int] = None
    dilation_near: int = 0
    stride: Optional[int] = None
    stride_phase: int = 0
    block: int = 128
    global_tokens: Optional[int] = None
    stride_relative: bool = False  # the stride counted from the query block
    dilation_far: bool = False     # dilated key blocks at every distance, window dense
    # bit-packed element mask (flag BITMASK): N rows of ceil(N/32) little-endian
    # uint32 words, read by build_block_index only (see inputs.pack_bitmask)
    bitmask: Optional[bytes] = field(default=None, repr=False)
    # packed sequences (flag DOCUMENTS): offsets 0 = s_0 < s_1 < ... < s_D = N
    doc_starts: Optional[tuple] = field(default=None, repr=False)

    @classmethod
    def from_fields(cls, fields: dict) -> "Mask":
        return cls(**fields)

    @property
    def flags(self) -> int:
        f = CAUSAL if self.causal else 0
        f |= WINDOW if self.window is not None else 0
        if self.dilation is not None:
            f |= DILATED_FAR if self.dilation_far else DILATED
        if self.stride is not None:
            f |= STRIDED_REL if self.stride_relative else STRIDED
        f |= GLOBAL if self.global_tokens is not None else 0
        f |= BITMASK if self.bitmask is not None else 0
        f |= DOCUMENTS if self.doc_starts is not None else 0
        return f

    @property
    def needs_index(self) -> bool:
        return bool(self.flags & ~CAUSAL)

    def desc(self, index_ptr=None) -> MaskDescStruct:
        bits = ctypes.cast(ctypes.c_char_p(self.bitmask), ctypes.c_void_p) if self.bitmask else None
        starts = None
        if self.doc_starts is not None:
            starts = np.ascontiguousarray(self.doc_starts, dtype=np.int64)
        d = MaskDescStruct(self.flags, self.block, self.window or 0, self.dilation or 1,
                           self.dilation_near, self.stride or 1, self.stride_phase,
                           index_ptr, self.global_tokens or 0, bits,
                           starts.ctypes.data if starts is not None else None,
                           len(starts) - 1 if starts is not None else 0)
        d._keep = starts  # the offsets must outlive the struct
        return d


_INDEX_ARRAYS = (("row_ptr", np.int32, "nq1"), ("col_idx", np.int32, "nnz"),
                 ("kind", np.uint8, "nnz"), ("col_ptr", np.int32, "nk1"),
                 ("row_idx", np.int32, "nnz"), ("kind_t", np.uint8, "nnz"),
                 ("q_order", np.int32, "nq"), ("k_order", np.int32, "nk"),
                 ("bit_slot", np.int32, "nnz"), ("bit_slot_t", np.int32, "nnz"),
                 ("bits", np.uint32, "nbits"), ("bits_t", np.uint32, "nbits"),
                 ("tile_start", np.int32, "ntiles"), ("tile_seq0", np.int32, "ntiles"),
                 ("tile_seq_len", np.int32, "ntiles"))


class BlockIndex:
    """Host arrays of a block index and (after ``to``) their device copies."""

    def __init__(self, mask: Mask, n: int, host: dict, header: BlockIndexStruct):
        self.mask, self.n, self.host, self.header = mask, n, host, header
        self.device: dict = {}
        self.device_struct: Optional[BlockIndexStruct] = None

    @property
    def nnz(self) -> int:
        return int(self.header.nnz)

    @property
    def live_elements(self) -> int:
        """Live (i, j) pairs of the mask over the N x N score matrix."""
        return int(self.header.live_elements)

    @property
    def sequence_tiles(self) -> bool:
        """Tiled per sequence (packed sequences with a causal / window mask)."""
        return bool(self.header.sequence_tiles)

    @property
    def n_tiles(self) -> int:
        return int(self.header.n_q_blocks)

    def _copy_header(self, s: BlockIndexStruct):
        s.n_bit_tiles = self.header.n_bit_tiles
        s.live_elements = self.header.live_elements
        s.sequence_tiles = self.header.sequence_tiles
        s.pair_overlap = self.header.pair_overlap

    def host_struct(self) -> BlockIndexStruct:
        s = BlockIndexStruct(self.header.seq_len, self.header.n_q_blocks, self.header.n_k_blocks,
                             self.header.block, self.header.nnz)
        self._copy_header(s)
        for name, _, kind in _INDEX_ARRAYS:
            if kind == "ntiles" and not self.sequence_tiles:
                continue  # null: packed tiling
            setattr(s, name, self.host[name].ctypes.data)
        return s

    def to(self, device) -> "BlockIndex":
        # at least one element per array, so every device pointer is non-null
        self.device = {name: torch.from_numpy(arr.copy() if arr.size else np.zeros(1, arr.dtype)).to(device)
                       for name, arr in self.host.items()}
        s = BlockIndexStruct(self.header.seq_len, self.header.n_q_blocks, self.header.n_k_blocks,
                             self.header.block, self.header.nnz)
        self._copy_header(s)
        for name, _, kind in _INDEX_ARRAYS:
            if kind == "ntiles" and not self.sequence_tiles:
                continue
            setattr(s, name, self.device[name].data_ptr())
        self.device_struct = s
        return self


def build_block_index(mask: Mask, n: int) -> BlockIndex:
    """Host-side build (two-phase C call); returns host numpy arrays."""
    L = lib()
    desc = mask.desc()
    hdr = BlockIndexStruct()
    _check(L.flash_msa_build_block_index(ctypes.byref(desc), n, ctypes.byref(hdr)),
           "build_block_index(count)")
    sizes = {"nq1": hdr.n_q_blocks + 1, "nk1": hdr.n_k_blocks + 1, "nnz": hdr.nnz,
             "nq": hdr.n_q_blocks, "nk": hdr.n_k_blocks, "nbits": 512 * hdr.n_bit_tiles,
             "ntiles": hdr.n_q_blocks if hdr.sequence_tiles else 0}
    host = {name: np.zeros(max(1, sizes[kind]), dtype=dt) for name, dt, kind in _INDEX_ARRAYS}
    out = BlockIndexStruct(hdr.seq_len, hdr.n_q_blocks, hdr.n_k_blocks, hdr.block, hdr.nnz)
    out.n_bit_tiles = hdr.n_bit_tiles
    for name, _, kind in _INDEX_ARRAYS:
        if kind == "ntiles" and not hdr.sequence_tiles:
            continue
        setattr(out, name, host[name].ctypes.data)
    _check(L.flash_msa_build_block_index(ctypes.byref(desc), n, ctypes.byref(out)),
           "build_block_index(fill)")
    host = {name: host[name][:sizes[kind]] for name, _, kind in _INDEX_ARRAYS}
    return BlockIndex(mask, n, host, out)


def check_block_index(index: BlockIndex) -> int:
    s = index.host_struct()
    return lib().flash_msa_check_block_index(ctypes.byref(s), index.n)


_VARLEN_INDEX: dict = {}


def varlen_mask(cu_seqlens, causal: bool = True, device="cuda"):
    """Mask and (cached) device index of a variable-length batch: sequences
    packed back to back on one token axis with offsets cu_seqlens."""
    starts = tuple(int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens))
    key = (starts, bool(causal), str(device))
    if key not in _VARLEN_INDEX:
        mask = Mask(causal=bool(causal), doc_starts=starts)
        _VARLEN_INDEX.clear()  # keep one layout: indices can be large
        _VARLEN_INDEX[key] = (mask, build_block_index(mask, starts[-1]).to(device))
    return _VARLEN_INDEX[key]


def fwd_varlen(q, k, v, cu_seqlens, causal: bool = True, scale: Optional[float] = None,
               out=None, lse=None, stream=None):
    """Forward of a variable-length batch: q, k, v of shape (T, H, d) hold the
    sequences back to back (offsets cu_seqlens, T = cu_seqlens[-1]); returns
    O (T, H, d) and LSE (H, T).  Runs flash_msa_fwd on the packed axis with the
    DOCUMENTS mask."""
    mask, index = varlen_mask(cu_seqlens, causal, q.device)
    o, l = fwd(q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), mask=mask, index=index,
               scale=scale, out=None if out is None else out.unsqueeze(0),
               lse=None if lse is None else lse.unsqueeze(0), stream=stream)
    return o[0], l[0]


def bwd_varlen(q, k, v, o, lse, do, cu_seqlens, causal: bool = True,
               scale: Optional[float] = None, stream=None):
    """dQ, dK, dV of a variable-length batch (shapes as in fwd_varlen)."""
    mask, index = varlen_mask(cu_seqlens, causal, q.device)
    dq, dk, dv = bwd(q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), o.unsqueeze(0),
                     lse.unsqueeze(0), do.unsqueeze(0), mask=mask, index=index, scale=scale,
                     stream=stream)
    return dq[0], dk[0], dv[0]


# ---------------------------------------------------------------------------
# attention calls
# ---------------------------------------------------------------------------
def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_qkv(name, t, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (B, N, H, d)")
    if t.dim() != 4:
        raise ValueError(f"{name} must have shape (B, N, H, d)")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _mask_desc(mask: Optional[Mask], index: Optional[BlockIndex], n: int):
    if mask is None:
        return None, None
    if index is not None:
        if index.device_struct is None:
            raise ValueError("block index has no device copy: call index.to(device)")
        if index.n != n:
            raise ValueError(f"block index built for N={index.n}, tensors have N={n}")
        holder = index.device_struct
        return mask.desc(ctypes.addressof(holder)), holder
    return mask.desc(), None


def _kv_shape(q, k):
    """(B, N, Hkv, d) of k; Hkv may be smaller than q's head count (GQA / MQA)."""
    _check_qkv("k", k)
    B, N, H, d = q.shape
    if k.shape[0] != B or k.shape[1] != N or k.shape[3] != d or H % k.shape[2] != 0:
        raise ValueError(f"k has shape {tuple(k.shape)}: expected (B, N, Hkv, d) with Hkv | {H}")
    return tuple(k.shape)


def fwd(q, k, v, mask: Optional[Mask] = None, index: Optional[BlockIndex] = None,
        scale: Optional[float] = None, out=None, lse=None, stream=None):
    """O (bf16, like q) and LSE (fp32, (B, H, N)).  k and v may have fewer
    heads than q (grouped-query attention): flash_msa_fwd_gqa."""
    _check_qkv("q", q)
    B, N, H, d = q.shape
    kv_shape = _kv_shape(q, k)
    _check_qkv("v", v, kv_shape)
    Hkv = kv_shape[2]
    o = torch.empty_like(q) if out is None else out
    _check_qkv("out", o, q.shape)
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if l.dtype != torch.float32 or not l.is_contiguous() or tuple(l.shape) != (B, H, N):
        raise ValueError("lse must be contiguous float32 (B, H, N)")
    desc, _keep = _mask_desc(mask, index, N)
    dptr = ctypes.byref(desc) if desc is not None else None
    if Hkv == H:
        code = lib().flash_msa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   l.data_ptr(), B, H, N, d, float(scale or 0.0), dptr,
                                   _stream_ptr(stream))
    else:
        code = lib().flash_msa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       l.data_ptr(), B, H, Hkv, N, d, float(scale or 0.0), dptr,
                                       _stream_ptr(stream))
    _check(code, "flash_msa_fwd")
    return o, l


def bwd_workspace_bytes(B, H, N, d, index: Optional["BlockIndex"] = None) -> int:
    """Workspace of flash_msa_bwd; with a per-sequence tiled index the vectors
    hold 128 rows per tile."""
    if index is not None and index.sequence_tiles:
        N = 128 * index.n_tiles
    return int(lib().flash_msa_bwd_workspace_bytes(B, H, N, d))


BWD_PREPROCESS, BWD_DKDV, BWD_DQ, BWD_FUSED, BWD_DQ_CONVERT = 1, 2, 4, 8, 16
BWD_DETERMINISTIC = BWD_PREPROCESS | BWD_DKDV | BWD_DQ      # flash_msa_bwd: two kernels
BWD_ACCUMULATED = BWD_PREPROCESS | BWD_FUSED | BWD_DQ_CONVERT  # dQ accumulated in fp32


def bwd_stages_workspace_bytes(B, H, N, d, stages, index: Optional["BlockIndex"] = None) -> int:
    """Workspace of flash_msa_bwd_stages for this set of stages."""
    if index is not None and index.sequence_tiles:
        N = 128 * index.n_tiles
    return int(lib().flash_msa_bwd_stages_workspace_bytes(B, H, N, d, stages))


def bwd(q, k, v, o, lse, do, mask: Optional[Mask] = None, index: Optional[BlockIndex] = None,
        scale: Optional[float] = None, dq=None, dk=None, dv=None, workspace=None, stream=None,
        stages: Optional[int] = None, accumulated: bool = False):
    """dQ, dK, dV (bf16, like q).  ``stages`` (bits BWD_*) runs a subset of the
    launches through flash_msa_bwd_stages; ``accumulated`` runs the fused
    kernel with dQ added into an fp32 accumulator (stages BWD_ACCUMULATED);
    default: flash_msa_bwd (two kernels, bitwise deterministic)."""
    _check_qkv("q", q)
    B, N, H, d = q.shape
    kv_shape = _kv_shape(q, k)
    Hkv = kv_shape[2]
    _check_qkv("v", v, kv_shape)
    for name, t in (("o", o), ("do", do)):
        _check_qkv(name, t, q.shape)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be contiguous float32 (B, H, N)")
    if accumulated:
        if stages is not None:
            raise ValueError("pass either stages or accumulated")
        stages = BWD_ACCUMULATED
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = (bwd_workspace_bytes(B, H, N, d, index) if stages is None
                else bwd_stages_workspace_bytes(B, H, N, d, stages, index))
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    desc, _keep = _mask_desc(mask, index, N)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
            float(scale or 0.0), ctypes.byref(desc) if desc is not None else None,
            workspace.data_ptr(), workspace.numel() * workspace.element_size())
    if Hkv != H and stages is None:
        code = lib().flash_msa_bwd_gqa(*args[:11], Hkv, *args[11:], _stream_ptr(stream))  # after H
    elif Hkv != H:
        code = lib().flash_msa_bwd_gqa_stages(*args[:11], Hkv, *args[11:], stages,
                                              _stream_ptr(stream))
    elif stages is None:
        code = lib().flash_msa_bwd(*args, _stream_ptr(stream))
    else:
        code = lib().flash_msa_bwd_stages(*args, stages, _stream_ptr(stream))
    _check(code, "flash_msa_bwd")
    return dq, dk, dv


def bwd_noalloc(q, k, v, o, lse, do, mask: Optional[Mask] = None,
                index: Optional[BlockIndex] = None, scale: Optional[float] = None,
                dq=None, dk=None, dv=None, stream=None):
    """dQ, dK, dV through flash_msa_bwd_noalloc: the library's fixed 16 MiB
    device scratch replaces the workspace (for callers that may not allocate
    device memory per call; the outputs here still come from torch unless
    passed in).  Calls overlapping on the GPU share that scratch and race."""
    _check_qkv("q", q)
    B, N, H, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        _check_qkv(name, t, q.shape)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be contiguous float32 (B, H, N)")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    desc, _keep = _mask_desc(mask, index, N)
    code = lib().flash_msa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                       dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                       float(scale or 0.0),
                                       ctypes.byref(desc) if desc is not None else None,
                                       _stream_ptr(stream))
    _check(code, "flash_msa_bwd_noalloc")
    return dq, dk, dv


def get_status(stream=None) -> int:
    """Synchronise the stream and read + clear the device status word."""
    return lib().flash_msa_get_status(_stream_ptr(stream))


def selftest_wait_timeout(stream=None) -> int:
    """Launch the bounded-wait probe (a wait that must run out); the next
    get_status() then reports ERR_TIMEOUT."""
    return lib().flash_msa_selftest_wait_timeout(_stream_ptr(stream))


def set_wait_limit_ms(ms: int):
    """Limit of any single bounded wait inside the kernels (process-wide)."""
    _check(lib().flash_msa_set_wait_limit_ms(int(ms)), "flash_msa_set_wait_limit_ms")


def get_wait_limit_ms() -> int:
    return int(lib().flash_msa_get_wait_limit_ms())


def check_status(stream=None):
    _check(get_status(stream), "device status")


def version() -> str:
    return lib().flash_msa_version().decode()
