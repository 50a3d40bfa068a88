"""OSCAR INT2 KV-cache serving path for GB300 (sm_103a).

The compute lives in liboscar.so (CUDA, C ABI in include/oscar.h); this
package is its ctypes binding plus host-side helpers:

  abi        the C-ABI calls (load_rotations, quant_append, decode_attn, ...)
  cache      caller-owned device buffers, page allocation, prefix forks
  calibrate  offline computation of R_K, R_V and the clip values
  build      compiles liboscar.so in-tree for sm_103a
"""

from . import abi  # noqa: F401
from .abi import Context, OscarConfig, OscarError, SeqState, make_config  # noqa: F401

__all__ = ["abi", "Context", "OscarConfig", "OscarError", "SeqState", "make_config"]
