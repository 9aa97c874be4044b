"""CPU oracle for the W4A8 quantized linear (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product path (the CUDA library and its Python binding) never
does, and shares no code with it.
"""
from .oracle import *  # noqa: F401,F403
from . import oracle as _impl  # noqa: F401
