"""GB300-native exact ring / context-parallel attention (libcp + binding).

The compute path is libcp.so (CUDA kernels for sm_103a behind the C ABI of
include/cp.h); this package only loads it and marshals arguments.
"""
from . import api, inputs  # noqa: F401
from ._lib import (CP_BF16, CP_EBOUNDS, CP_EHEADS, CP_EINVAL, CP_ESMEM, CP_ETIMEOUT,  # noqa: F401
                   CP_EUNSUPPORTED, CP_F32,
                   CP_LAYOUT_CONTIGUOUS, CP_LAYOUT_STRIPED, CP_LAYOUT_ZIGZAG, CP_OK,
                   CpError)

__all__ = ["api", "inputs", "CpError"]
