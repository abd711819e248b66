"""Single-GPU MoE layer (route, dispatch, grouped SwiGLU experts, combine;
forward and backward) for GB300 (sm_103a), exposed as a C-ABI library
(include/moe_abi.h) with this thin ctypes binding."""
from .binding import *  # noqa: F401,F403
from . import binding  # noqa: F401
