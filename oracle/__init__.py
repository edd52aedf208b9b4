"""CPU oracle of the Flint-shaped MoE decode step (test infrastructure).

Only the tests, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline /
reference arm may import this package.  The CUDA library never does, and this
package imports nothing from it.

Parity status of each function is listed in `oracle/model.py`'s header.
"""
from .model import Oracle, ContiguousKV, PagedKV  # noqa: F401
from . import numerics  # noqa: F401
