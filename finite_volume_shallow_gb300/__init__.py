"""GB300-native first-order Roe-type (IR-Roe) finite-volume solver for the 2D
shallow-water equations with a passive pollutant.

``swe``     the Python binding of the C ABI in include/swe.h (libswe).
``inputs``  seeded synthetic workloads (bathymetry and initial states).
``build``   compiles libswe in-tree with nvcc for sm_103a.

The library is loaded lazily on the first call into ``swe``.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "swe", "build"]


def __getattr__(name):
    if name in ("swe", "build"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
