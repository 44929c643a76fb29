"""Paged grouped-query attention with per-head attention sinks for GB300 (sm_103a).

The compute lives in libsinkattn.so (hand-written CUDA kernels behind a C ABI,
declared in include/sinkattn.h).  `sinkattn` is its thin ctypes binding; the
library is loaded on first use and a missing or unbuildable library raises.
`inputs` holds the seeded synthetic workload generators.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "sinkattn"]


def __getattr__(name):
    if name == "sinkattn":
        import importlib
        return importlib.import_module(__name__ + ".sinkattn")
    raise AttributeError(name)
