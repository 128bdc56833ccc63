"""Oracle package: plain CPU reference of the DiT step.  Test infrastructure only --
imported by the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``, never by the library."""
from . import dit_oracle  # noqa: F401
