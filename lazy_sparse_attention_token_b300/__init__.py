"""FlashLoop lazy loop step on one B300: C-ABI library (libflashloop.so) and its binding."""
from .flashloop import *  # noqa: F401,F403
from .flashloop import Cache, Dims, FlashLoopError, lib, make_dims, workspace_for  # noqa: F401
