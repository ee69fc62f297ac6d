"""CPU oracle (test infrastructure only).

Imported by the test suite, by ``__graft_entry__.smoke()`` and by the CPU
baseline leg of ``bench.py``; never by the library itself.
"""
from . import tern_oracle  # noqa: F401
