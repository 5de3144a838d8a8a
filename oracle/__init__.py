"""Float64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The CUDA library and its Python binding
never import it.  See ``g4_oracle.py`` for what each function computes.
"""
from . import g4_oracle  # noqa: F401
