"""GB300-native routed mixture-of-experts expert layer (libmoe): CUDA kernels behind a C ABI,
with a thin ctypes binding (`binding`)."""
from . import binding  # noqa: F401
from .binding import (GraphedForward, GraphedStack, Layer, MoeError, dispatch, e4m3_encode, forward,  # noqa: F401
                      forward_stack, get_status, route, workspace, workspace_bytes)
