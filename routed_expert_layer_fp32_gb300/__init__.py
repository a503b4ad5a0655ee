"""GB300-native routed mixture-of-experts expert layer (libmoe): CUDA kernels behind a C ABI,
with a thin ctypes binding (`binding`)."""
from . import binding  # noqa: F401
from .binding import (Layer, MoeError, dispatch, e4m3_encode, forward, forward_stack, get_status,  # noqa: F401
                      route, workspace, workspace_bytes)
