"""Persistent MoE decode megakernel for GB300 (sm_103a).

The product is the C-ABI library libmk.so (include/mk.h), built in-tree by
`_build.build()`; `_lib` is its ctypes binding under the same names and
`engine` a thin driver (Engine, Batcher) over it.
"""
from . import _build  # noqa: F401


def build(force: bool = False, verbose: bool = False) -> str:
    return _build.build(force=force, verbose=verbose)
