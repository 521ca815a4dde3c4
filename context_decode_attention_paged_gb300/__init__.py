"""GB300-native Decode Context Parallelism (DCP) decode attention.

The compute path is the C-ABI library ``libdcp.so`` (hand-written CUDA for
sm_103a, declared in ``include/dcp.h``).  ``binding`` is a thin ctypes layer
that passes tensor pointers and the current CUDA stream to it; ``workloads``
draws seeded synthetic inputs.  Import ``binding`` explicitly: it raises if the
library has not been built.
"""

__all__ = ["binding", "workloads", "build"]
