"""fp64 CPU oracle for exact attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference legs may import this package.  The CUDA library neither imports nor
links anything here; the two share no code.  See ``oracle/attention.py`` for
what each function computes, the passages it follows and how it is pinned.
"""
from .attention import *  # noqa: F401,F403
from .attention import __all__  # noqa: F401
