"""B300 (sm_103a) sparse MoE layer forward pass: router + top-k, bucketing, slot-table lookup,
int8 block-32 SwiGLU experts, combine. The kernels live in libmoe_b300.so (include/moe.h);
_lib is its ctypes binding and layer chains the calls for one layer."""
from . import _lib  # noqa: F401
from ._lib import *  # noqa: F401,F403
