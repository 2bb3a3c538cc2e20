"""fp64 CPU oracle of the DyRA linear layer -- test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library never imports it.
"""
from .dyra_oracle import *  # noqa: F401,F403
from .dyra_oracle import __all__  # noqa: F401
