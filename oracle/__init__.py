"""CPU oracle of the ResidualKV cache codec (float64, NumPy).

TEST INFRASTRUCTURE ONLY.  This package is the correctness authority for the
CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the C-ABI library and its Python binding) never imports,
links or executes anything here, and nothing here comes from the CUDA path.

Parity status of each function is recorded in its docstring; every function
is pinned by a ``-m "not gpu"`` test against something other than itself
(closed forms, printed values of the page, brute force, library routines).
"""
from . import formats, codec, storage  # noqa: F401
from .codec import *  # noqa: F401,F403
