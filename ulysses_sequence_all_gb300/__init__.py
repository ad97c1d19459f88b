"""GB300-native Ulysses 4D sequence/head relayout (fast-ulysses' all_to_all_4d, one GPU, W virtual
ranks held as separate HBM buffers).

The compute lives in ``libulysses.so`` (hand-written sm_103a kernels behind a C ABI declared in
``include/ulysses.h``); ``binding`` marshals tensors and pointers into it. Importing this package
does not load the library; the first call into ``binding`` does, and raises if it is missing.
"""
from . import binding, workloads  # noqa: F401

__all__ = ["binding", "workloads"]
