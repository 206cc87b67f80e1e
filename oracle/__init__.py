"""CPU oracle for the OSCAR INT2 KV-cache path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) imports, calls or links this package; only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.  It shares no code, tables or constants with
the CUDA path.
"""
from .oscar_oracle import *  # noqa: F401,F403
