"""VBQ mixed-bit decode for B300 (sm_103a): packed per-group {1,2,4,8}-bit weights
with fused dequantize-and-multiply kernels behind a C ABI (include/vbq.h).

Importing this package loads libvbq.so and fails if it is missing: there is no
CPU or PyTorch fallback. Build it with ``python mixed_precision_weight_bit_b300/build.py``
(by path: importing the package needs a library that is already built).
"""

from .vbq import *  # noqa: F401,F403
from .vbq import LIB_PATH, HEADER_PATH, Matrix, Model, VbqError, load_library  # noqa: F401

load_library()
