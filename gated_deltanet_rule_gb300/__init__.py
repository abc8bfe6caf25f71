"""Gated delta rule forward on GB300 (sm_103a).

The computation lives in the CUDA library ``libgdr.so`` behind a C ABI (``include/gdr.h``).
This package is its thin Python binding (``gated_deltanet_rule_gb300.gdr``: argument
marshalling only) plus a seeded synthetic input generator (``inputs``).

Importing the package does not load the library; the first call into ``gdr`` does, and
raises if the library has not been built (there is no CPU fallback).
"""

__all__ = ["gdr", "inputs"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
