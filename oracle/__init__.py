"""fp64 CPU oracle for exact attention: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The attention library never does.
"""
from . import attention  # noqa: F401
