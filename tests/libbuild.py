"""Build the CUDA library once per test session if it is missing or stale."""
import os

from tiled_exact_attention_flash_gb300 import build as _build

_done = False


def _stale() -> bool:
    if not os.path.exists(_build.LIB):
        return True
    t = os.path.getmtime(_build.LIB)
    srcs = [os.path.join(_build.CSRC, f) for f in os.listdir(_build.CSRC)]
    srcs.append(os.path.join(_build.ROOT, "include", "flashmsa.h"))
    return any(os.path.getmtime(s) > t for s in srcs)


def ensure_built():
    global _done
    if not _done:
        if _stale():
            _build.build()
        _done = True
