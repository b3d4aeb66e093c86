"""CPU oracle of the CFG sampler step (test infrastructure only).

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs.  Shares no code with the CUDA library.
"""
from . import cfg_oracle  # noqa: F401
