"""Position-independent KV stitching for GB300 (sm_103a).

The product is libpic (C ABI in include/pic.h, CUDA kernels in csrc/);
``pic`` is its thin ctypes binding with the same function names.
"""

from . import pic  # noqa: F401
from .pic import PicError  # noqa: F401

__all__ = ["pic", "PicError"]
