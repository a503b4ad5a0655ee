"""GB300-native routed mixture-of-experts expert layer (libmoe): CUDA kernels behind a C ABI,
with a thin ctypes binding (`binding`)."""
from . import binding  # noqa: F401
from .binding import (GraphedForward, Layer, MoeError, dispatch, e4m3_encode, forward, forward_stack,  # noqa: F401
                      get_status, route, workspace, workspace_bytes)
