"""libflashmsa: exact tiled ("Flash MSA") attention for GB300 (sm_103a).

The compute path is the C-ABI shared library ``libflashmsa.so`` built from
``csrc/`` (hand-written CUDA with tcgen05 / TMA inline PTX); ``api`` is a thin
ctypes binding over it.  Importing this package does not load the library;
the first call into ``api`` does, and fails loudly if it is missing.
"""
__all__ = ["api", "inputs"]
