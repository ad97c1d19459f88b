"""GB300-native Ulysses 4D sequence/head relayout (fast-ulysses' all_to_all_4d, one GPU, W virtual
ranks held as separate HBM buffers).

The compute lives in ``libulysses.so`` (hand-written sm_103a kernels behind a C ABI declared in
``include/ulysses.h``); ``binding`` marshals tensors and pointers into it. Importing this package
does not load the library; the first call into ``binding`` does, and raises if it is missing.
"""
from . import workloads  # noqa: F401  (pure-Python input generators)

__all__ = ["workloads", "binding"]


def __getattr__(name):
    if name == "binding":
        from . import binding
        return binding
    raise AttributeError(name)
