"""B300-native Fast Multipole Method (Morton octree, Cartesian multipoles).

The compute path is the CUDA library ``lib/libbfm_fmm.so`` (C ABI in
``include/fmm.h``), reached through :mod:`body_forces_morton_b300.native`.
Importing this package does not load the library; ``native.lib()`` does, and
raises if it has not been built (``python body_forces_morton_b300/build.py``).
"""
from . import workloads  # noqa: F401  (seeded inputs; no method arithmetic)

__all__ = ["workloads", "native"]


def __getattr__(name):
    if name == "native":
        import importlib
        return importlib.import_module(__name__ + ".native")
    raise AttributeError(name)
