"""fp64 CPU oracle for MLA decode with weight absorption.

TEST INFRASTRUCTURE ONLY: used by the tests, by ``__graft_entry__.smoke()`` and by
the CPU-baseline leg of ``bench.py``.  The product path never imports it.
"""
from .mla_oracle import *  # noqa: F401,F403
from .mla_oracle import __all__  # noqa: F401
