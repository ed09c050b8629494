"""decode_attention_kv_gb300 -- decode-phase KV-cache attention on GB300.

``kvd`` is the ctypes binding of libkvd.so (C ABI in include/kvd.h): KV
append, masked and paged split-KV decode attention, paged gather and the
log-sum-exp combine, all as hand-written sm_103a kernels.  ``build()``
compiles the library in-tree.
"""
from . import kvd  # noqa: F401
from ._build import build  # noqa: F401

__all__ = ["kvd", "build"]
